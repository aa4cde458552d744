// Row log-sum-exp of logits input (CTC_PACKED_FLAG_LOGITS): one dense read
// of the (T_total, D) logits, lse[t] = log(sum_c exp(z[t, c])), so that the
// emission gather and the gradient stream can use log_softmax(z)[t, c] =
// z[t, c] - lse[t] without a normalised copy of the rows ever being written.
//
// Page "feat(asr): native CTC loss kernel over sequence-packed log
// probabilities", ctc_loss.py, ``packed_ctc_loss``: the path's input is the
// log_softmax of a model's logits, and the gradient it returns is
// scale * exp(lp) - P; with lp = z - lse that is scale * softmax(z) - P, the
// gradient with respect to the logits.
//
// One warp per row, rows strided over a persistent grid.  A row is read as
// the 16-byte chunks that cover its bytes, 2 per lane in flight; the ragged
// chunks at the two ends of the buffer are read element by element.  Each lane keeps a running maximum m
// and a sum s of exp(z - m) (rescaled when m grows), the warp combines the
// lanes' pairs, and lane 0 writes m + log(s).  A row of -inf gives -inf; a
// NaN or +inf logit gives NaN, as log_softmax does.
#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

constexpr int kLseWarps = 8;    // warps per CTA
// 16-byte chunks in flight per lane.  Measured on the 8193-class workload:
// 2 beat 1, 4 and 8, and an L2 prefetch of the whole row cost 2 to 6 us.
constexpr int kLseUnroll = 2;

__device__ __forceinline__ uint4 ld_row_chunk(uintptr_t p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Folds the valid values of one chunk into the running (m, s); a NaN or a
// +inf value marks the row bad (its log_softmax is NaN).
template <int N>
__device__ __forceinline__ void fold(const float (&x)[N], const bool (&ok)[N], float& m, float& s, bool& bad) {
    float cm = -INFINITY;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if (ok[i]) {
            bad |= !(x[i] < INFINITY) && !(x[i] == -INFINITY);  // NaN or +inf
            cm = fmaxf(cm, x[i]);
        }
    }
    if (bad || cm == -INFINITY) return;
    if (cm > m) {
        s = m == -INFINITY ? 0.0f : s * fast_ex2((m - cm) * kLog2e);
        m = cm;
    }
    const float mb = -m * kLog2e;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (ok[i]) s += fast_ex2(fmaf(x[i], kLog2e, mb));  // exp(x - m); exactly 0 for x = -inf
}

// The same for a chunk whose values all belong to the row (every chunk but
// the row's two ends): no per-value checks.  A NaN, or +inf against a finite
// maximum, turns s into NaN, which marks the row bad at the end.
template <int N>
__device__ __forceinline__ void fold_inner(const float (&x)[N], float& m, float& s) {
    float cm = x[0];
#pragma unroll
    for (int i = 1; i < N; ++i) cm = fmaxf(cm, x[i]);
    if (cm > m) {
        s *= fast_ex2((m - cm) * kLog2e);  // 0 * 0 while m is still -inf
        m = cm;
    }
    if (m == -INFINITY) return;  // nothing but -inf so far
    const float2 l2e = make_float2(kLog2e, kLog2e), mb = make_float2(-m * kLog2e, -m * kLog2e);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const float2 t = __ffma2_rn(make_float2(x[i], x[i + 1]), l2e, mb);
        acc = __fadd2_rn(acc, make_float2(fast_ex2(t.x), fast_ex2(t.y)));
    }
    s += acc.x + acc.y;
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kLseWarps * 32) lse_kernel(ChainArgs a) {
    constexpr int E = Elem<DT>::bytes;
    constexpr int V = 16 / E;
    const int lane = threadIdx.x & 31;
    const int64_t T = a.L.T_total;
    const int D = a.D;
    const uintptr_t z0 = reinterpret_cast<uintptr_t>(a.lp);
    const uintptr_t z_end = z0 + (uintptr_t)T * D * E;
    float* lse = ws_at<float>(a.ws, a.L.off_lse);
    const int64_t warps = (int64_t)gridDim.x * kLseWarps;
    pdl_wait();  // the workspace may still be read by the stream's earlier work
    for (int64_t row = (int64_t)blockIdx.x * kLseWarps + (threadIdx.x >> 5); row < T; row += warps) {
        const uintptr_t r0 = z0 + (uintptr_t)(row * D * E), r1 = r0 + (uintptr_t)D * E;
        const uintptr_t qb = r0 & ~uintptr_t(15);
        const int nq = (int)((((r1 + 15) & ~uintptr_t(15)) - qb) / 16);
        float m = -INFINITY, s = 0.0f;
        bool bad = false;
        for (int q0 = 0; q0 < nq; q0 += 32 * kLseUnroll) {
            uint4 in[kLseUnroll];
            bool whole[kLseUnroll];
#pragma unroll
            for (int k = 0; k < kLseUnroll; ++k) {
                const uintptr_t c = qb + (uintptr_t)(q0 + k * 32 + lane) * 16;
                whole[k] = q0 + k * 32 + lane < nq && c >= z0 && c + 16 <= z_end;
                if (whole[k]) in[k] = ld_row_chunk(c);
            }
#pragma unroll
            for (int k = 0; k < kLseUnroll; ++k) {
                const int q = q0 + k * 32 + lane;
                if (q >= nq) continue;
                const uintptr_t c = qb + (uintptr_t)q * 16;
                float x[V];
                bool ok[V];
                if (whole[k]) {
                    const uint32_t w[4] = {in[k].x, in[k].y, in[k].z, in[k].w};
#pragma unroll
                    for (int i = 0; i < V; ++i) {
                        uint32_t bits;
                        if constexpr (E == 4) {
                            bits = w[i];
                        } else {
                            bits = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu);
                        }
                        x[i] = bits_to_float<DT>(bits);
                    }
                    if (c >= r0 && c + 16 <= r1) {
                        fold_inner(x, m, s);
                        continue;
                    }
#pragma unroll
                    for (int i = 0; i < V; ++i) {
                        const uintptr_t ad = c + (uintptr_t)i * E;
                        ok[i] = ad >= r0 && ad < r1;
                    }
                } else {
                    // a chunk at an end of the buffer: only the row's own elements are read
#pragma unroll
                    for (int i = 0; i < V; ++i) {
                        const uintptr_t ad = c + (uintptr_t)i * E;
                        ok[i] = ad >= r0 && ad < r1;
                        x[i] = 0.0f;
                        if (ok[i]) {
                            if constexpr (E == 4) {
                                x[i] = __uint_as_float(*reinterpret_cast<const uint32_t*>(ad));
                            } else {
                                x[i] = bits_to_float<DT>(*reinterpret_cast<const unsigned short*>(ad));
                            }
                        }
                    }
                }
                fold(x, ok, m, s, bad);
            }
        }
        // combine the lanes' (m, s): M = max m, S = sum s * exp(m - M)
        const bool row_bad = __any_sync(0xffffffffu, bad || s != s || m == INFINITY);
        float M = m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float part = m == -INFINITY ? 0.0f : s * fast_ex2((m - M) * kLog2e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0)
            lse[row] = row_bad ? __int_as_float(0x7fc00000) : (M == -INFINITY ? -INFINITY : M + logf(part));
    }
}

template __global__ void lse_kernel<0>(ChainArgs);
template __global__ void lse_kernel<1>(ChainArgs);
template __global__ void lse_kernel<2>(ChainArgs);

cudaError_t launch_lse(const ChainArgs& a, int dtype, cudaStream_t s) {
    if (a.L.T_total == 0) return cudaSuccess;
    cudaError_t e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    void (*k)(ChainArgs) = dtype == 0 ? lse_kernel<0> : dtype == 1 ? lse_kernel<1> : lse_kernel<2>;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kLseWarps * 32, 0)) != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)sms * per_sm;
    const long long want = (a.L.T_total + kLseWarps - 1) / kLseWarps;
    if (want < grid) grid = want;
    return launch_pdl(k, dim3((unsigned)grid), dim3(kLseWarps * 32), 0, s, a);
}

}  // namespace ctcp
