// Gradient of the packed CTC loss, written row by row in the token-flat layout.
//
// Page "feat(asr): native CTC loss kernel over sequence-packed log
// probabilities", ctc_loss.py ``_beta_grad_kernel``:
//
//   posterior_t(s) = exp(alpha_t(s) + beta_t(s) - lp[t, l'_s] + nll) * scale,
//   grad[t, c]     = exp(lp[t, c]) * scale - sum over s with l'_s = c of posterior_t(s),
//   scale          = upstream gradient of the utterance, 0 when zero_infinity
//                    meets an infinite loss (then the posteriors are skipped);
//   a frame outside every utterance gets a zero gradient.
//
// One kernel, one warp per group of consecutive rows (one row when D is
// large), no CTA-wide barrier:
//   1. posteriors: for each row of the group the warp reads the stored alpha
//      and beta rows and sums the posteriors of each distinct class of the
//      row's utterance.  Blank states are summed lane-strided and then by a
//      fixed butterfly; each distinct label class is summed by its first
//      occurrence walking the chain of its later occurrences.  No atomics and
//      a fixed order, so the gradient is bitwise reproducible.  The sums wait
//      in the warp's slice of shared memory as (row, class, scale * sum).
//   2. the group's rows are one contiguous span, streamed in batches of
//      16-byte chunks (vector loads and stores, several in flight per lane):
//      grad = scale * exp(lp) - P, or 0 outside every utterance.  Before a
//      batch the warp drops the batch's few class sums into a small shared
//      tile P and marks their chunks, so a chunk reads P only when marked and
//      every gradient element is written exactly once, in one rounding.
//
// The stored rows hold alpha_t(s) / p_t(s) (before the emission) and
// beta_t(s) as exact mantissa-exponent words, each relative to an integer
// offset of its (frame, warp).  A posterior is the product of two mantissas
// and the per-utterance constant 2^frac(nll log2 e), scaled by 2 to the
// integer sum of the exponents, the offsets and floor(nll log2 e).
#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

constexpr int kMaxWarpsPerBlock = 8;
constexpr int kUnroll = 4;                   // 16-byte chunks in flight per lane
constexpr int kBatchChunks = 32 * kUnroll;   // chunks a warp streams per batch

__device__ __forceinline__ int find_utterance(const int32_t* cu, int B, int64_t row) {
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

// Posterior of one state from its stored alpha / beta words (see enc_state):
// (ma * mb * c) * 2^(ka + kb + base), where base = A + B + floor(nll log2 e)
// and c = 2^frac(nll log2 e).  Results below 2^-126 flush to 0.
__device__ __forceinline__ float posterior(int va, int vb, int base, float c) {
    if (va == kFixZero || vb == kFixZero) return 0.0f;
    const float ma = __int_as_float(((va & 0x7ffff) << 4) | 0x3f800000);
    const float mb = __int_as_float(((vb & 0x7ffff) << 4) | 0x3f800000);
    const int n = min(max((va >> kFixFrac) + (vb >> kFixFrac) + base, -200), 64);
    return __int_as_float(max(__float_as_int(ma * mb * c) + (n << 23), 0));
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int DT>
__device__ __forceinline__ uint32_t load_elem(uintptr_t addr) {
    if constexpr (Elem<DT>::bytes == 4) {
        return *reinterpret_cast<const uint32_t*>(addr);
    } else {
        return *reinterpret_cast<const unsigned short*>(addr);
    }
}
template <int DT>
__device__ __forceinline__ void store_elem(uintptr_t addr, uint32_t bits) {
    if constexpr (Elem<DT>::bytes == 4) {
        *reinterpret_cast<uint32_t*>(addr) = bits;
    } else {
        *reinterpret_cast<unsigned short*>(addr) = (unsigned short)bits;
    }
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kMaxWarpsPerBlock * 32, 3) grad_kernel(GradArgs a) {
    constexpr int E = Elem<DT>::bytes;
    constexpr int V = 16 / E;  // elements per 16-byte chunk
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int K = a.rows_per_tile;   // rows per group
    const int cap = a.entry_cap;     // corrections a group can hold
    const int ulen = a.L.max_U + 1;  // label posteriors a row can hold
    // this warp's slice: row scales, corrections (packed row/class, value), label posteriors
    unsigned char* ws = smem_raw + (size_t)warp * a.warp_smem;
    float* row_scale = reinterpret_cast<float*>(ws);  // K entries, NaN-free: 0 when not covered
    int* row_cov = reinterpret_cast<int*>(ws + align_up(4 * (size_t)K, 16));
    int* e_key = reinterpret_cast<int*>(ws + 2 * align_up(4 * (size_t)K, 16));
    float* e_val = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(e_key) + align_up(4 * (size_t)cap, 16));
    float* gam = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(e_val) + align_up(4 * (size_t)cap, 16));
    float* ptile = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(gam) + align_up(4 * (size_t)ulen, 16));
    uint32_t* pmark = reinterpret_cast<uint32_t*>(ptile + kBatchChunks * V);  // kBatchChunks / 32 words

    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    const double* nll = ws_at<double>(a.ws, a.L.off_nll);
    const int32_t* __restrict__ aoff = ws_at<int32_t>(a.ws, a.L.off_aoff);
    const int32_t* __restrict__ boff = ws_at<int32_t>(a.ws, a.L.off_boff);
    const int* __restrict__ alpha = ws_at<int>(a.ws, a.L.off_alpha);
    const int* __restrict__ beta = ws_at<int>(a.ws, a.L.off_beta);
    const int32_t* __restrict__ nxt = ws_at<int32_t>(a.ws, a.L.off_nxt);
    const int32_t* __restrict__ rank = ws_at<int32_t>(a.ws, a.L.off_rank);
    const int GP = a.L.gpairs;  // pairs per offset group of a stored row
    const bool ready = ctrl->grad_ready != 0;
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.L.T_total > 0 && !ready)
        set_status(ctrl, CTC_PACKED_DEV_NO_GRAD_STATE);
    const int D = a.D;
    const int B = a.L.B;
    const uintptr_t lp0 = reinterpret_cast<uintptr_t>(a.lp);
    const uintptr_t gr0 = reinterpret_cast<uintptr_t>(a.grad);
    const int64_t n_groups = a.n_tiles;
    const int wpb = blockDim.x >> 5;
    const int64_t warps = (int64_t)gridDim.x * wpb;

    for (int i = lane; i < kBatchChunks * V; i += 32) ptile[i] = 0.0f;
    if (lane < kBatchChunks / 32) pmark[lane] = 0u;
    __syncwarp();

    for (int64_t grp = (int64_t)blockIdx.x * wpb + warp; grp < n_groups; grp += warps) {
        const int64_t r0 = grp * K;
        const int nrows = (int)min((int64_t)K, a.L.T_total - r0);

        // the next group's stored rows start their way into L2
        {
            const int64_t nr0 = (grp + warps) * K;
            const int64_t nrows_next = nr0 < a.L.T_total ? min((int64_t)K, a.L.T_total - nr0) : 0;
            const int64_t bytes = nrows_next * (int64_t)a.L.pitch * 4;
            for (int64_t off = (int64_t)lane * 128; off < bytes; off += 32 * 128) {
                asm volatile("prefetch.global.L2 [%0];" ::"l"(alpha + nr0 * a.L.pitch + off / 4));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(beta + nr0 * a.L.pitch + off / 4));
            }
        }
        // 1. posteriors of every row of the group
        int count = 0;  // corrections so far (warp-uniform)
        int b = find_utterance(a.cu, B, r0);
        for (int rr = 0; rr < nrows; ++rr) {
            const int64_t row = r0 + rr;
            while (b + 1 < B && (int64_t)a.cu[b + 1] <= row) ++b;  // rows ascend: walk forward
            int covered = 0;
            float scale = 0.0f;
            UttInfo u{};
            if (b >= 0) {
                u = utt[b];
                const int64_t t = row - u.start;
                covered = ready && u.valid && u.labels_ok && t >= 0 && t < u.T;
                if (covered) {
                    if (a.reduction == CTC_PACKED_NONE) {
                        scale = a.grad_loss[b];
                    } else if (a.reduction == CTC_PACKED_SUM) {
                        scale = a.grad_loss[0];
                    } else {
                        scale = (float)((double)a.grad_loss[0] / ((double)B * (double)max(u.U, 1)));
                    }
                    const double v = nll[b];
                    if (a.zero_infinity && isinf(v) && v > 0) scale = 0.0f;
                }
            }
            if (lane == 0) {
                row_scale[rr] = covered ? scale : 0.0f;
                row_cov[rr] = covered;
            }
            if (!covered || scale == 0.0f) continue;

            // an infinite nll (no alignment, zero_infinity off) leaves these rows unspecified: NaN scale factor
            const double nl2 = nll[b] * kLog2eD;
            const bool nfin = isfinite(nl2);
            const double kfl = nfin ? floor(nl2) : 0.0;
            const int kint = (int)fmin(fmax(kfl, -1.0e9), 1.0e9);
            const float cfrac = nfin ? (float)exp2(nl2 - kfl) : __int_as_float(0x7fc00000);
            const int32_t* ao = aoff + row * a.L.nwo;
            const int32_t* bo = boff + row * a.L.nwo;
            const int* ar = alpha + row * a.L.pitch;
            const int* br = beta + row * a.L.pitch;
            const int32_t* rk = rank + u.moff;
            const int32_t* nx = nxt + u.moff;
            const int32_t* tg = a.targets + u.toff;
            // alpha pair j holds states (2j, 2j+1) at positions 2j, 2j+1 (offset group j / GP of its chain);
            // beta pair j holds states (2j-1, 2j) at positions 2j, 2j+1, so state s sits at s+1
            auto base_of = [&](int ja, int jb) -> int { return ao[ja / GP] + bo[jb / GP] + kint; };
            float blank_sum = 0.0f;
            for (int j = lane; j <= u.U; j += 32) {
                const int2 av = *reinterpret_cast<const int2*>(ar + 2 * j);
                const int2 bv = *reinterpret_cast<const int2*>(br + 2 * j);
                blank_sum += posterior(av.x, bv.y, base_of(j, j), cfrac);
                if (j < u.U) {
                    const float gl = posterior(av.y, br[2 * j + 2], base_of(j, j + 1), cfrac);
                    gam[j] = gl;
                    if (rk[j] == -2) blank_sum += gl;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) blank_sum += __shfl_xor_sync(0xffffffffu, blank_sum, o);
            __syncwarp();
            // each distinct class, summed by its first occurrence in target order
            for (int j = lane; j < u.U; j += 32) {
                const int kind = rk[j];
                if (kind >= 0) {
                    float s = gam[j];
                    for (int jj = nx[j]; jj >= 0; jj = nx[jj]) s += gam[jj];
                    e_key[count + kind] = rr * D + tg[j];
                    e_val[count + kind] = scale * s;
                }
            }
            if (lane == 0) {
                e_key[count + u.n_owners - 1] = rr * D + a.blank;
                e_val[count + u.n_owners - 1] = scale * blank_sum;
            }
            count += u.n_owners;
            __syncwarp();
        }
        __syncwarp();

        // 2. the dense span of the group, 16 bytes at a time
        const uintptr_t a0 = lp0 + (uintptr_t)(r0 * D * E);
        const uintptr_t g0 = gr0 + (uintptr_t)(r0 * D * E);
        const uintptr_t g1 = g0 + (uintptr_t)nrows * D * E;
        const uintptr_t qb = g0 & ~uintptr_t(15);
        const int pshift = (int)((g0 - qb) / E);  // element f of the group lies in chunk (f + pshift) / V
        const int nq = (int)((((g1 + 15) & ~uintptr_t(15)) - qb) / 16);
        const float invD = 1.0f / (float)D;
        // element index (within the group) of the first element of chunk q, and its row
        auto chunk_row = [&](int f) {
            int r = 0;
            if (K > 1) {
                r = __float2int_rz((float)f * invD);
                if (r * D > f) --r;
                if ((r + 1) * D <= f) ++r;
            }
            return r;
        };
        if (nrows == 1 && a.congruent) {
            // one row, lp and grad congruent modulo 16: chunks [qf0, qf1) are whole and aligned
            const int qf0 = pshift > 0 ? 1 : 0;
            const int qf1 = (int)((g1 - qb) / 16);
            const uintptr_t lpq = qb + (a0 - g0);  // lp address of chunk 0
            const bool cov = row_cov[0] != 0;
            const float s = row_scale[0];
            for (int q0 = 0; q0 < nq; q0 += kBatchChunks) {
                uint4 in[kUnroll];
#pragma unroll
                for (int k = 0; k < kUnroll; ++k) {
                    const int q = q0 + k * 32 + lane;
                    if (cov && q >= qf0 && q < qf1) in[k] = ld_stream(reinterpret_cast<const void*>(lpq + (uintptr_t)q * 16));
                }
                const int f_begin = q0 * V - pshift, f_end = f_begin + kBatchChunks * V;
                for (int e = lane; e < count; e += 32) {
                    const int f = e_key[e];
                    if (f >= f_begin && f < f_end) {
                        const int idx = f - f_begin;
                        ptile[idx] = e_val[e];
                        atomicOr(&pmark[idx / (32 * V)], 1u << ((idx / V) & 31));
                    }
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < kUnroll; ++k) {
                    const int q = q0 + k * 32 + lane;
                    if (q >= nq) continue;
                    const int ql = k * 32 + lane;
                    const bool marked = (pmark[k] >> lane) & 1u;
                    const uintptr_t c0 = qb + (uintptr_t)q * 16;
                    if (q >= qf0 && q < qf1) {
                        float pv[V];
#pragma unroll
                        for (int i = 0; i < V; ++i) pv[i] = 0.0f;
                        if (marked) {
#pragma unroll
                            for (int i = 0; i < V; i += 4) {
                                const float4 v = reinterpret_cast<const float4*>(ptile + ql * V)[i / 4];
                                pv[i] = v.x;
                                pv[i + 1] = v.y;
                                pv[i + 2] = v.z;
                                pv[i + 3] = v.w;
                                reinterpret_cast<float4*>(ptile + ql * V)[i / 4] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
                        uint4 o = make_uint4(0u, 0u, 0u, 0u);
                        if (cov) {
                            const uint32_t w[4] = {in[k].x, in[k].y, in[k].z, in[k].w};
                            float out[V];
#pragma unroll
                            for (int i = 0; i < V; ++i) {
                                float x;
                                if constexpr (E == 4) {
                                    x = __uint_as_float(w[i]);
                                } else if constexpr (DT == 1) {  // bfloat16: the high half is already a float
                                    x = __uint_as_float((i & 1) ? (w[i >> 1] & 0xffff0000u) : (w[i >> 1] << 16));
                                } else {
                                    x = bits_to_float<DT>((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu));
                                }
                                out[i] = fmaf(s, fast_ex2(x * kLog2e), -pv[i]);
                            }
                            if constexpr (E == 4) {
                                o = make_uint4(__float_as_uint(out[0]), __float_as_uint(out[1]), __float_as_uint(out[2]),
                                               __float_as_uint(out[3]));
                            } else {
                                o = make_uint4(pack2<DT>(out[0], out[1]), pack2<DT>(out[2], out[3]),
                                               pack2<DT>(out[4], out[5]), pack2<DT>(out[6], out[7]));
                            }
                        }
                        *reinterpret_cast<uint4*>(c0) = o;
                    } else {
                        // the ragged first / last chunk of the row
                        const uintptr_t lo = c0 > g0 ? c0 : g0;
                        const uintptr_t hi = c0 + 16 < g1 ? c0 + 16 : g1;
                        for (uintptr_t ad = lo; ad < hi; ad += E) {
                            const size_t f = (ad - g0) / E;
                            const float x = bits_to_float<DT>(load_elem<DT>(a0 + f * E));
                            const float pk = marked ? ptile[ql * V + (int)(f + pshift) - q * V] : 0.0f;
                            const float gv = cov ? fmaf(s, fast_ex2(x * kLog2e), -pk) : 0.0f;
                            store_elem<DT>(ad, pack1<DT>(gv));
                        }
                        if (marked) {
                            for (int i = 0; i < V; ++i) ptile[ql * V + i] = 0.0f;
                        }
                    }
                }
                __syncwarp();
                if (lane < kBatchChunks / 32) pmark[lane] = 0u;
                __syncwarp();
            }
            continue;
        }
        for (int q0 = 0; q0 < nq; q0 += kBatchChunks) {
            uint4 in[kUnroll];
            bool fast[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int q = q0 + k * 32 + lane;
                const uintptr_t c0 = qb + (uintptr_t)q * 16;
                fast[k] = q < nq && c0 >= g0 && c0 + 16 <= g1 && a.congruent;
                if (fast[k]) in[k] = ld_stream(reinterpret_cast<const void*>(a0 + (c0 - g0)));
            }
            // this batch's class sums into the tile: element f sits at ptile[f + pshift - q0 * V]
            const int f_begin = q0 * V - pshift, f_end = (q0 + kBatchChunks) * V - pshift;
            for (int e = lane; e < count; e += 32) {
                const int f = e_key[e];
                if (f >= f_begin && f < f_end) {
                    const int idx = f - f_begin;
                    ptile[idx] = e_val[e];
                    atomicOr(&pmark[idx / V / 32], 1u << ((idx / V) & 31));
                }
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int q = q0 + k * 32 + lane;
                if (q >= nq) continue;
                const uintptr_t c0 = qb + (uintptr_t)q * 16;
                const uintptr_t lo = c0 > g0 ? c0 : g0;
                const uintptr_t hi = c0 + 16 < g1 ? c0 + 16 : g1;
                const int f_lo = (int)((lo - g0) / E);
                int r = chunk_row(f_lo);
                int c = f_lo - r * D;
                // the chunk's class sums (zero unless marked), cleared once read
                const int ql = q - q0;
                const bool marked = (pmark[ql >> 5] >> (ql & 31)) & 1u;
                if (fast[k] && c + V <= D) {
                    float pv[V];
#pragma unroll
                    for (int i = 0; i < V; ++i) pv[i] = 0.0f;
                    if (marked) {
#pragma unroll
                        for (int i = 0; i < V; i += 4) {
                            const float4 v = reinterpret_cast<const float4*>(ptile + ql * V)[i / 4];
                            pv[i] = v.x;
                            pv[i + 1] = v.y;
                            pv[i + 2] = v.z;
                            pv[i + 3] = v.w;
                            reinterpret_cast<float4*>(ptile + ql * V)[i / 4] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                    // a whole chunk inside one row
                    uint4 o = make_uint4(0u, 0u, 0u, 0u);
                    if (row_cov[r]) {
                        const float s = row_scale[r];
                        const uint32_t w[4] = {in[k].x, in[k].y, in[k].z, in[k].w};
                        float out[V];
#pragma unroll
                        for (int i = 0; i < V; ++i) {
                            uint32_t bits;
                            if constexpr (E == 4) {
                                bits = w[i];
                            } else {
                                bits = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu);
                            }
                            out[i] = fmaf(s, fast_ex2(bits_to_float<DT>(bits) * kLog2e), -pv[i]);
                        }
                        if constexpr (E == 4) {
                            o = make_uint4(__float_as_uint(out[0]), __float_as_uint(out[1]), __float_as_uint(out[2]),
                                           __float_as_uint(out[3]));
                        } else {
                            o = make_uint4(pack2<DT>(out[0], out[1]), pack2<DT>(out[2], out[3]),
                                           pack2<DT>(out[4], out[5]), pack2<DT>(out[6], out[7]));
                        }
                    }
                    *reinterpret_cast<uint4*>(c0) = o;
                } else {
                    // ragged end of the span, a chunk across two rows, or misaligned buffers
                    const int f_hi = (int)((hi - g0) / E);
                    for (int f = f_lo; f < f_hi; ++f) {
                        while (c >= D) {
                            c -= D;
                            ++r;
                        }
                        const float x = bits_to_float<DT>(load_elem<DT>(a0 + (size_t)f * E));
                        const float pk = marked ? ptile[ql * V + f + pshift - q * V] : 0.0f;
                        const float gv = row_cov[r] ? fmaf(row_scale[r], fast_ex2(x * kLog2e), -pk) : 0.0f;
                        store_elem<DT>(g0 + (size_t)f * E, pack1<DT>(gv));
                        ++c;
                    }
                    if (marked) {
                        for (int i = 0; i < V; ++i) ptile[ql * V + i] = 0.0f;
                    }
                }
            }
            __syncwarp();
            if (lane < kBatchChunks / 32) pmark[lane] = 0u;
            __syncwarp();
        }
        __syncwarp();
    }
}

template __global__ void grad_kernel<0>(GradArgs);
template __global__ void grad_kernel<1>(GradArgs);
template __global__ void grad_kernel<2>(GradArgs);

template <int DT>
static cudaError_t launch_grad_t(const GradArgs& a, cudaStream_t s) {
    // as many warps per block (up to 8) as 200 KB of shared memory hold
    int wpb = (int)(200 * 1024 / (a.warp_smem > 0 ? a.warp_smem : 1));
    wpb = wpb < 1 ? 1 : (wpb > kMaxWarpsPerBlock ? kMaxWarpsPerBlock : wpb);
    const size_t smem = (size_t)wpb * a.warp_smem;
    cudaError_t e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(grad_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, grad_kernel<DT>, wpb * 32, smem)) != cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)sms * per_sm;
    const long long want = (a.n_tiles + wpb - 1) / wpb;
    if (want < grid) grid = want;
    if (grid < 1) return cudaSuccess;
    grad_kernel<DT><<<(unsigned)grid, wpb * 32, smem, s>>>(a);
    return cudaGetLastError();
}

// Rows per warp group and the shared memory each warp needs.
void grad_geometry(const Layout& L, int D, int& rows, int& entry_cap, size_t& warp_smem) {
    const int ecap = L.ecap;
    int k = 2048 / D;
    const int k2 = 512 / (ecap > 0 ? ecap : 1);
    if (k2 < k) k = k2;
    if (k < 1) k = 1;
    rows = k;
    entry_cap = k * ecap;
    warp_smem = 2 * align_up(4 * (size_t)k, 16) + 2 * align_up(4 * (size_t)entry_cap, 16) +
                align_up(4 * (size_t)(L.max_U + 1), 16) + 4 * (size_t)kBatchChunks * 8 + 4 * (kBatchChunks / 32);
    warp_smem = align_up(warp_smem, 16);
}

cudaError_t launch_grad(const GradArgs& a, int dtype, cudaStream_t s) {
    if (dtype == 0) return launch_grad_t<0>(a, s);
    if (dtype == 1) return launch_grad_t<1>(a, s);
    if (dtype == 2) return launch_grad_t<2>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace ctcp
