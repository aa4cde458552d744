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
    const int64_t grid = (a.L.T_total + kEmitRows - 1) / kEmitRows;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    if (dtype == 0) return launch_pdl(emit_kernel<0>, dim3((unsigned)grid), dim3(kEmitThreads), 0, s, a);
    if (dtype == 1) return launch_pdl(emit_kernel<1>, dim3((unsigned)grid), dim3(kEmitThreads), 0, s, a);
    return launch_pdl(emit_kernel<2>, dim3((unsigned)grid), dim3(kEmitThreads), 0, s, a);
}

}  // namespace ctcp
