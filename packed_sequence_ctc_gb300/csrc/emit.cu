// Emission gather of the forward: for every frame of every utterance, the
// log probabilities of the utterance's target labels and of the blank,
// lp[t, l_1..l_U] and lp[t, blank], converted once into extended-range
// probabilities (ctc_common.cuh, XP) and written as one contiguous row of the
// workspace's emission matrix.  Entry em[row][w] pairs label l_{w+1} (w < U)
// with the frame's blank; em[row][U] pairs a zero emission with the blank,
// for the recursion lanes that hold no label.
//
// Page "feat(asr): native CTC loss kernel over sequence-packed log
// probabilities", ctc_loss.py ``_alpha_kernel`` and ``_beta_grad_kernel``:
// both recursions read exactly these columns, lp[t, l'_s], each frame.
//
// Why a kernel of its own: the label columns are scattered through rows of
// D elements, so each read costs a whole DRAM sector.  Gathered inside the
// serial recursions (one chain per SM, both the alpha and the beta chain of
// an utterance reading the same columns), they run into the number of reads
// an SM can keep in flight.  Here every SM gathers with many independent
// loads per thread, each column once, and the recursions then read short
// contiguous rows, mostly from L2.
#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

// Frame rows per CTA (independent loads in flight per thread) and threads
// per CTA.  Measured on the 8193-class workload: 4 rows beat 2 and 8 (16 is
// much slower: more rows open at once per CTA), 192 threads beat 128 and 256.
constexpr int kEmitRows = 4;
constexpr int kEmitThreads = 192;

__device__ __forceinline__ int utterance_of_row(const int32_t* cu, int B, int64_t row) {
    int lo = 0, hi = B - 1, ans = -1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)cu[mid] <= row) {
            ans = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    return ans;
}

// One log probability.  The loads are scattered, so each asks L2 to fetch
// only the 64-byte segment around it from DRAM (the default fetch is larger
// and mostly wasted here).
template <int DT>
__device__ __forceinline__ float load_lp(const void* lp, int64_t idx) {
    if constexpr (DT == 0) {
        const float* p = reinterpret_cast<const float*>(lp) + idx;
        float v;
        asm volatile("ld.global.nc.L2::64B.f32 %0, [%1];" : "=f"(v) : "l"(p));
        return v;
    } else {
        const unsigned short* p = reinterpret_cast<const unsigned short*>(lp) + idx;
        unsigned short h;
        asm volatile("ld.global.nc.L2::64B.u16 %0, [%1];" : "=h"(h) : "l"(p));
        return bits_to_float<DT>((uint32_t)h);
    }
}

// Label records the backward needs, one CTA per utterance: for each target
// position whether it is the first occurrence of its class (then it owns the
// class's posterior sum and gets the next rank), the next position with the
// same class, and whether the id equals the blank (then its posterior joins
// the blank column).  Every position compares its class with all others,
// which pass through shared memory one tile at a time.
__device__ void run_label_block(const ChainArgs& a, int b) {
    __shared__ int s_tile[kEmitThreads];
    __shared__ int s_warp[kEmitThreads / 32];
    __shared__ int s_bad;
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    const UttInfo info = utt[b];
    const int U = info.U;
    const int32_t* tg = a.targets + info.toff;
    LabelRec* lbl = ws_at<LabelRec>(a.ws, a.L.off_lbl) + info.moff;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    int running = 0;  // distinct classes ranked so far
    for (int j0 = 0; j0 < U; j0 += kEmitThreads) {
        const int j = j0 + tid;
        const int c = j < U ? tg[j] : -1;
        const bool is_blank = c == a.blank;
        bool first = j < U && !is_blank;
        int nx = -1;
        if (j < U && (c < 0 || c >= a.D)) s_bad = 1;
        for (int k0 = 0; k0 < U; k0 += kEmitThreads) {
            __syncthreads();
            s_tile[tid] = k0 + tid < U ? tg[k0 + tid] : -1;
            __syncthreads();
            const int n = min(kEmitThreads, U - k0);
            if (j < U && !is_blank) {
                for (int kk = 0; kk < n; ++kk) {
                    if (s_tile[kk] == c) {
                        const int k = k0 + kk;
                        if (k < j) first = false;
                        if (k > j && nx < 0) nx = k;
                    }
                }
            }
        }
        // ranks of the first occurrences, in target order
        const unsigned m = __ballot_sync(0xffffffffu, first);
        if (lane == 0) s_warp[warp] = __popc(m);
        __syncthreads();
        int before = running;
        for (int w = 0; w < warp; ++w) before += s_warp[w];
        int total = 0;
        for (int w = 0; w < kEmitThreads / 32; ++w) total += s_warp[w];
        const int r = before + __popc(m & ((1u << lane) - 1u));
        if (j < U) lbl[j] = LabelRec{first ? r : (is_blank ? -2 : -1), nx, c, 0};
        running += total;
        __syncthreads();
    }
    __syncthreads();
    if (tid == 0) {
        utt[b].n_owners = running + 1;
        utt[b].labels_ok = s_bad ? 0 : 1;
        if (s_bad) set_status(ctrl, CTC_PACKED_DEV_LABEL_OUT_OF_RANGE);
    }
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kEmitThreads) emit_kernel(ChainArgs a) {
    __shared__ int s_b[kEmitRows], s_u[kEmitRows], s_toff[kEmitRows];
    __shared__ XP s_blank[kEmitRows];
    __shared__ int s_maxw;
    const UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    UttInfo* uttw = ws_at<UttInfo>(a.ws, a.L.off_utt);
    XP2* em = ws_at<XP2>(a.ws, em_base(a.L));
    const int64_t r0 = (int64_t)blockIdx.x * kEmitRows;
    const int tid = threadIdx.x;
    pdl_wait();  // utterance metadata from the prep kernel
    // the blocks after the gather's are the label analysis of the backward,
    // one per utterance with frames (before the chains, so that the gradient
    // stream of the forward-backward call can use it while they run)
    const int64_t n_gather = (a.L.T_total + kEmitRows - 1) / kEmitRows;
    if ((int64_t)blockIdx.x >= n_gather) {
        const Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
        const int k = (int)((int64_t)blockIdx.x - n_gather);
        if (k < ctrl->n_lab) run_label_block(a, ws_at<int32_t>(a.ws, a.L.off_queue)[2 * a.L.B + 1 + k]);
        return;
    }
    if (tid == 0) s_maxw = 0;
    __syncthreads();
    if (tid < kEmitRows) {
        const int64_t row = r0 + tid;
        int b = -1, U = -1, toff = 0;
        if (row < a.L.T_total) {
            b = utterance_of_row(a.cu, a.L.B, row);
            if (b >= 0) {
                const UttInfo u = utt[b];
                const int64_t t = row - u.start;
                if (u.valid && t >= 0 && t < u.T) {
                    U = u.U;
                    toff = u.toff;
                } else {
                    b = -1;
                }
            }
        }
        s_b[tid] = b;
        s_u[tid] = U;
        s_toff[tid] = toff;
        if (b >= 0) {
            float x = load_lp<DT>(a.lp, row * (int64_t)a.D + a.blank);
            if (a.lse != nullptr) x -= a.lse[row];  // logits: log_softmax of the row
            s_blank[tid] = xp_from_log(x);
            if (x != x) atomicOr(&uttw[b].has_nan, 1);
            atomicMax(&s_maxw, U + 1);
        }
    }
    __syncthreads();
    const int maxw = s_maxw;
    float lse_r[kEmitRows];
#pragma unroll
    for (int rr = 0; rr < kEmitRows; ++rr)
        lse_r[rr] = (a.lse != nullptr && s_b[rr] >= 0) ? a.lse[r0 + rr] : 0.0f;
    for (int w = tid; w < maxw; w += kEmitThreads) {
        int cls[kEmitRows];
#pragma unroll
        for (int rr = 0; rr < kEmitRows; ++rr) {
            cls[rr] = -1;  // no entry
            if (s_b[rr] >= 0 && w < s_u[rr]) cls[rr] = a.targets[s_toff[rr] + w];
            if (s_b[rr] >= 0 && w == s_u[rr]) cls[rr] = -2;  // (zero, blank): read by lanes without a label
        }
        float x[kEmitRows];
#pragma unroll
        for (int rr = 0; rr < kEmitRows; ++rr) {
            // an id outside [0, D) is not read (the chain reports it); its emission is 0
            const bool live = cls[rr] >= 0 && cls[rr] < a.D;
            x[rr] = live ? load_lp<DT>(a.lp, (r0 + rr) * (int64_t)a.D + cls[rr]) - lse_r[rr] : -INFINITY;
        }
#pragma unroll
        for (int rr = 0; rr < kEmitRows; ++rr) {
            if (cls[rr] != -1) {
                XP2 v;
                v.l = cls[rr] == -2 ? XP{0.0f, kEZeroEm} : xp_from_log(x[rr]);
                v.b = s_blank[rr];
                em[(r0 + rr) * (int64_t)a.L.epitch + w] = v;
                if (x[rr] != x[rr]) atomicOr(&uttw[s_b[rr]].has_nan, 1);
            }
        }
    }
}

template __global__ void emit_kernel<0>(ChainArgs);
template __global__ void emit_kernel<1>(ChainArgs);
template __global__ void emit_kernel<2>(ChainArgs);

cudaError_t launch_emit(const ChainArgs& a, int dtype, cudaStream_t s) {
    if (a.L.T_total == 0 || a.L.B == 0) return cudaSuccess;
    // gather blocks, then one label block per utterance
    const int64_t grid = (a.L.T_total + kEmitRows - 1) / kEmitRows + a.L.B;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    if (dtype == 0) return launch_pdl(emit_kernel<0>, dim3((unsigned)grid), dim3(kEmitThreads), 0, s, a);
    if (dtype == 1) return launch_pdl(emit_kernel<1>, dim3((unsigned)grid), dim3(kEmitThreads), 0, s, a);
    return launch_pdl(emit_kernel<2>, dim3((unsigned)grid), dim3(kEmitThreads), 0, s, a);
}

}  // namespace ctcp
