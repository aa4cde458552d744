// Class sums of every row when the forward kept only checkpoint rows.
//
// Page "feat(asr): native CTC loss kernel over sequence-packed log
// probabilities", ctc_loss.py ``_PackedCTCLoss``: the forward keeps alpha
// for the backward.  Storing every frame's states costs the serial chains an
// encode and a store each frame, and the backward a reload of every row.
// With a checkpoint interval K the chains keep only the rows whose absolute
// index is a multiple of K, and this kernel recomputes the rest.
//
// One CTA takes K consecutive rows at a time.  For each utterance part in
// them (frames t0 .. t1 - 1 of utterance b) it
//   1. runs the beta recursion down from the checkpoint at frame t1 (or from
//      the terminal states when t1 is the utterance's end), keeping each
//      frame's beta in shared memory;
//   2. runs the alpha recursion up from the checkpoint at frame t0 (or from
//      the start states when t0 = 0); at each frame, before the emission, it
//      forms the posteriors alpha_t(s) beta_t(s) / p_t(l'_s), normalises them
//      by their sum over the row (every frame carries the whole path
//      probability), sums them per distinct class in a fixed order and writes
//      the row's class sums and header in the format the gradient kernels
//      read.
// The recursions are those of the chain kernel, on extended-range values
// (a float mantissa and an int exponent per state), one state pair per
// thread and pass.  Rows outside every utterance get "not covered" headers.
#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

constexpr int kSegThreads = 256;
constexpr int kSegWarps = kSegThreads / 32;
constexpr int kSegMaxPairsPerThread = 4;  // state pairs a thread holds: max_U + 1 <= 1024

__device__ __forceinline__ XP dec_state(int w, int off) {
    if (w == kFixZero) return XP{0.0f, kEZero};
    return XP{__int_as_float(((w & 0x7ffff) << 4) | 0x3f800000), (w >> kFixFrac) + off};
}

__device__ __forceinline__ float pow2i(int k) { return pow2_nonpos(k); }

}  // namespace

__global__ void __launch_bounds__(kSegThreads) segpost_kernel(GradArgs a) {
    extern __shared__ __align__(16) unsigned char seg_smem[];
    const int K = a.ckpt;
    const int Up = a.L.max_U + 1;  // pairs of the widest target
    XP2* bst = reinterpret_cast<XP2*>(seg_smem);                       // [K][Up] beta (label, blank) per frame
    XP2* emx = bst + (size_t)K * Up;                                   // [K][Up] the part's emission rows
    XP* xs = reinterpret_cast<XP*>(emx + (size_t)K * Up);              // [2][Up + 1] neighbour exchange
    float* lab_m = reinterpret_cast<float*>(xs + 2 * (Up + 1));        // [Up] label posterior terms
    int* lab_e = reinterpret_cast<int*>(lab_m + Up);
    int* red = lab_e + Up;                                             // [3][kSegWarps]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    const int* alpha = ws_at<int>(a.ws, a.L.off_alpha);
    const int* beta = ws_at<int>(a.ws, a.L.off_beta);
    const LabelRec* lbl = ws_at<LabelRec>(a.ws, a.L.off_lbl);
    const XP2* em = ws_at<XP2>(a.ws, em_base(a.L));
    RowHead* head = ws_at<RowHead>(a.ws, a.L.off_head);
    int2* ent = ws_at<int2>(a.ws, a.L.off_ent);
    pdl_wait();  // the forward's checkpoint rows and metadata
    pdl_trigger();
    const bool ready = ctrl->grad_ready != 0 && (int)ctrl->ckpt == K;
    if (blockIdx.x == 0 && tid == 0 && a.L.T_total > 0 && !ready) set_status(ctrl, CTC_PACKED_DEV_NO_GRAD_STATE);
    const bool bad_cu = (ctrl->status & CTC_PACKED_DEV_BAD_CU_SEQLENS) != 0;
    const int B = a.L.B;
    const int64_t T_total = a.L.T_total;
    const int64_t n_blocks = (T_total + K - 1) / K;
    const float inv_count = a.reduction == CTC_PACKED_MEAN_VOLUME ? (float)ctrl->tl_total : (float)B;
    const XP zero{0.0f, kEZero};

    auto uncovered = [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0 + tid; r < r1; r += kSegThreads) head[r] = RowHead{0, 0.0f, 0, 0};
    };

    for (int64_t blk = blockIdx.x; blk < n_blocks; blk += gridDim.x) {
        const int64_t r_lo = blk * K, r_hi = min(r_lo + K, T_total);
        if (!ready || bad_cu || B == 0) {
            uncovered(r_lo, r_hi);
            continue;
        }
        // the utterance whose span holds r_lo (cu_seqlens is non-decreasing here)
        int b = -1;
        {
            int lo = 0, hi = B - 1;
            while (lo <= hi) {
                const int mid = (lo + hi) >> 1;
                if ((int64_t)a.cu[mid] <= r_lo) {
                    b = mid;
                    lo = mid + 1;
                } else {
                    hi = mid - 1;
                }
            }
        }
        int64_t r = r_lo;
        while (r < r_hi) {
            while (b + 1 < B && (int64_t)a.cu[b + 1] <= r) ++b;
            if (b < 0) {  // rows before the first span
                const int64_t e = min(r_hi, (int64_t)a.cu[0]);
                uncovered(r, e);
                r = e;
                continue;
            }
            const UttInfo u = utt[b];
            const int64_t span_end = b + 1 < B ? (int64_t)a.cu[b + 1] : T_total;
            const int64_t fr_end = (int64_t)u.start + (u.valid ? u.T : 0);
            if (!u.valid || !u.labels_ok || r >= fr_end) {  // not a frame of a well-formed utterance
                const int64_t e = min(r_hi, max(span_end, r + 1));
                uncovered(r, e);
                r = e;
                continue;
            }
            // utterance b, frames t0 .. t1 - 1
            const int T = u.T, U = u.U;
            const int t0 = (int)(r - u.start), t1 = (int)(min(r_hi, fr_end) - u.start);
            float sc;
            if (a.reduction == CTC_PACKED_NONE) {
                sc = a.grad_loss[b];
            } else if (a.reduction == CTC_PACKED_SUM) {
                sc = a.grad_loss[0];
            } else if (a.reduction == CTC_PACKED_MEAN) {
                sc = __fdiv_rn(a.grad_loss[0], (float)B * (float)max(U, 1));
            } else {
                sc = __fdiv_rn(a.grad_loss[0], inv_count);
            }
            const LabelRec* lb = lbl + u.moff;
            const int32_t* tg = a.targets + u.toff;
            // my pairs j = tid + i * kSegThreads, with their skip flags
            bool mine[kSegMaxPairsPerThread], skip[kSegMaxPairsPerThread];
#pragma unroll
            for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                const int j = tid + i * kSegThreads;
                mine[i] = j <= U;
                skip[i] = j >= 1 && j < U && tg[j] != tg[j - 1];
            }
            // the part's emission rows, all at once (every recursion step needs one)
            {
                const int n = (t1 - t0) * (U + 1);
                const XP2* src = em + (int64_t)(u.start + t0) * a.L.epitch;
                for (int idx = tid; idx < n; idx += kSegThreads) {
                    const int kk = idx / (U + 1), w = idx - kk * (U + 1);
                    emx[kk * Up + w] = src[(int64_t)kk * a.L.epitch + w];
                }
                __syncthreads();
            }
            // 1. beta, from frame t1 (a checkpoint) or the utterance's last frame down to t0
            XP vb[kSegMaxPairsPerThread], vl[kSegMaxPairsPerThread];  // beta pair j = (label 2j-1, blank 2j)
            int k;
            if (t1 == T) {
                const XP2* er = emx + (T - 1 - t0) * Up;
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    vb[i] = vl[i] = zero;
                    if (j == U) {
                        const XP2 e = er[U == 0 ? U : U - 1];
                        vb[i] = xp_norm(e.b.m, e.b.e);
                        if (U >= 1) vl[i] = xp_norm(e.l.m, e.l.e);
                    }
                }
                k = T - 1;
            } else {
                const int* br = beta + (int64_t)(u.start + t1) * a.L.spitch;
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    vb[i] = vl[i] = zero;
                    if (mine[i]) {
                        const int g = (int)(((uint32_t)j * a.gp_mul) >> 21);
                        const int off = br[g];
                        const int2 w = *reinterpret_cast<const int2*>(br + a.L.owo + 2 * j);
                        vl[i] = j >= 1 ? dec_state(w.x, off) : zero;
                        vb[i] = dec_state(w.y, off);
                    }
                }
                k = t1;  // one step down gives frame t1 - 1
            }
            int buf = 0;
            for (;;) {
                if (k < t1) {  // store beta at frame k
#pragma unroll
                    for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                        const int j = tid + i * kSegThreads;
                        if (mine[i]) bst[(k - t0) * Up + j] = XP2{vl[i], vb[i]};
                    }
                }
                if (k == t0) break;
                // step to frame k - 1: new_j from old_j and the label of pair j + 1
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    if (mine[i]) xs[buf * (Up + 1) + j] = vl[i];
                }
                __syncthreads();
                const XP2* er = emx + (k - 1 - t0) * Up;
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    if (!mine[i]) continue;
                    const XP o = j < U ? xs[buf * (Up + 1) + j + 1] : zero;
                    const XP2 e = er[j == 0 ? U : j - 1];
                    float Sl, Sb;
                    int El, Eb;
                    xp_sum3(vl[i], vb[i], skip[i] ? o : zero, Sl, El);
                    xp_sum2(vb[i], o, Sb, Eb);
                    vl[i] = j >= 1 ? xp_norm(Sl * e.l.m, El + e.l.e) : zero;
                    vb[i] = xp_norm(Sb * e.b.m, Eb + e.b.e);
                }
                buf ^= 1;
                --k;
            }
            // 2. alpha, from frame t0 (the start or a checkpoint) up to t1 - 1;
            // A = alpha before the frame's emission
            XP ab[kSegMaxPairsPerThread], al[kSegMaxPairsPerThread];  // alpha pair j = (blank 2j, label 2j+1)
            if (t0 == 0) {
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    ab[i] = j == 0 ? XP{1.0f, 0} : zero;
                    al[i] = (j == 0 && U >= 1) ? XP{1.0f, 0} : zero;
                }
            } else {
                const int* ar = alpha + (int64_t)(u.start + t0) * a.L.spitch;
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    ab[i] = al[i] = zero;
                    if (mine[i]) {
                        const int g = (int)(((uint32_t)j * a.gp_mul) >> 21);
                        const int off = ar[g];
                        const int2 w = *reinterpret_cast<const int2*>(ar + a.L.owo + 2 * j);
                        ab[i] = dec_state(w.x, off);
                        al[i] = j < U ? dec_state(w.y, off) : zero;
                    }
                }
            }
            __syncthreads();  // beta rows of the part are in shared memory
            for (k = t0; k < t1; ++k) {
                const int64_t row = u.start + k;
                // posterior terms: blank 2j = A(2j) B(2j), label 2j+1 = A(2j+1) B(2j+1)
                const XP2* bk = bst + (k - t0) * Up;
                int emax = kEZero;
                float pbm[kSegMaxPairsPerThread];
                int pbe[kSegMaxPairsPerThread];
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    pbm[i] = 0.0f;
                    pbe[i] = kEZero;
                    if (!mine[i]) continue;
                    const XP bb = bk[j].b;
                    if (ab[i].m != 0.0f && bb.m != 0.0f) {
                        pbm[i] = ab[i].m * bb.m;
                        pbe[i] = ab[i].e + bb.e;
                        emax = max(emax, pbe[i]);
                    }
                    if (j < U) {
                        const XP bl = bk[j + 1].l;
                        float m = 0.0f;
                        int e = kEZero;
                        if (al[i].m != 0.0f && bl.m != 0.0f) {
                            m = al[i].m * bl.m;
                            e = al[i].e + bl.e;
                            emax = max(emax, e);
                        }
                        lab_m[j] = m;
                        lab_e[j] = e;
                    }
                }
                emax = __reduce_max_sync(0xffffffffu, emax);
                if (lane == 0) red[warp] = emax;
                __syncthreads();
                int M = red[0];
                for (int w = 1; w < kSegWarps; ++w) M = max(M, red[w]);
                float zs = 0.0f, bs = 0.0f;
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    if (!mine[i]) continue;
                    const float pb = pbm[i] * pow2i(pbe[i] - M);
                    zs += pb;
                    bs += pb;
                    if (j < U) {
                        const float pl = lab_m[j] * pow2i(lab_e[j] - M);
                        zs += pl;
                        if (lb[j].rank == -2) bs += pl;  // a target id equal to the blank
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    zs += __shfl_xor_sync(0xffffffffu, zs, o);
                    bs += __shfl_xor_sync(0xffffffffu, bs, o);
                }
                if (lane == 0) {
                    red[kSegWarps + warp] = __float_as_int(zs);
                    red[2 * kSegWarps + warp] = __float_as_int(bs);
                }
                __syncthreads();
                float Z = __int_as_float(red[kSegWarps]), Bsum = __int_as_float(red[2 * kSegWarps]);
                for (int w = 1; w < kSegWarps; ++w) {
                    Z += __int_as_float(red[kSegWarps + w]);
                    Bsum += __int_as_float(red[2 * kSegWarps + w]);
                }
                float s = sc;
                if (Z == 0.0f && a.zero_infinity) s = 0.0f;  // no path: zeroed with its loss
                const bool live = s != 0.0f;
                if (live) {
                    const float ns = -s * __frcp_rn(Z);
                    const bool nan_row = u.has_nan != 0;
                    for (int j = tid; j < U; j += kSegThreads) {
                        const LabelRec lr = lb[j];
                        if (lr.rank < 0) continue;
                        float sum = lab_m[j] * pow2i(lab_e[j] - M);
                        for (int jj = lr.next; jj >= 0; jj = lb[jj].next) sum = fmaf(lab_m[jj], pow2i(lab_e[jj] - M), sum);
                        ent[row * a.L.ecap + lr.rank] =
                            make_int2(lr.cls, __float_as_int(nan_row ? __int_as_float(0x7fc00000) : ns * sum));
                    }
                    if (tid == 0)
                        ent[row * a.L.ecap + u.n_owners - 1] =
                            make_int2(a.blank, __float_as_int(nan_row ? __int_as_float(0x7fc00000) : ns * Bsum));
                }
                if (tid == 0) head[row] = RowHead{live ? u.n_owners : 0, s, 1, 0};
                if (k + 1 == t1) break;
                // alpha at frame k (after its emission), then A at frame k + 1
                const XP2* er = emx + (k - t0) * Up;
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    if (!mine[i]) continue;
                    const XP2 e = er[j];  // (label j or zero, blank)
                    ab[i] = xp_norm(ab[i].m * e.b.m, ab[i].e + e.b.e);
                    al[i] = xp_norm(al[i].m * e.l.m, al[i].e + e.l.e);
                    xs[buf * (Up + 1) + j] = al[i];
                }
                __syncthreads();  // also: every thread is done with this row's label terms
#pragma unroll
                for (int i = 0; i < kSegMaxPairsPerThread; ++i) {
                    const int j = tid + i * kSegThreads;
                    if (!mine[i]) continue;
                    const XP o = j >= 1 ? xs[buf * (Up + 1) + j - 1] : zero;
                    float Sl, Sb;
                    int El, Eb;
                    xp_sum3(al[i], ab[i], skip[i] ? o : zero, Sl, El);
                    xp_sum2(ab[i], o, Sb, Eb);
                    al[i] = j < U ? xp_norm(Sl, El) : zero;
                    ab[i] = xp_norm(Sb, Eb);
                }
                buf ^= 1;
            }
            __syncthreads();  // the part's beta rows and label terms are free again
            r = (int64_t)u.start + t1;
        }
    }
}

cudaError_t launch_segpost(const GradArgs& a, cudaStream_t s) {
    if (a.L.T_total == 0) return cudaSuccess;
    const int Up = a.L.max_U + 1;
    const size_t smem = 32 * (size_t)a.ckpt * Up + 8 * 2 * (size_t)(Up + 1) + 8 * (size_t)Up + 4 * 3 * kSegWarps;
    cudaError_t e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(segpost_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, segpost_kernel, kSegThreads, smem)) !=
        cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const long long blocks = (a.L.T_total + a.ckpt - 1) / a.ckpt;
    long long grid = (long long)sms * per_sm;
    if (blocks < grid) grid = blocks;
    return launch_pdl(segpost_kernel, dim3((unsigned)grid), dim3(kSegThreads), smem, s, a);
}

// Largest supported checkpoint interval for these sizes (0: none): the beta
// rows and emission rows of K frames must fit a CTA's shared memory (two
// CTAs an SM) beside the rest, and
// each thread holds at most kSegMaxPairsPerThread pairs.
int segpost_max_ckpt(const Layout& L) {
    const int Up = L.max_U + 1;
    if (Up > kSegThreads * kSegMaxPairsPerThread) return 0;
    int k = 64;
    while (k > 1 && 32 * (size_t)k * Up + 24 * (size_t)(Up + 1) > 110 * 1024) k >>= 1;
    return k > 1 ? k : 0;
}

}  // namespace ctcp
