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
// Two kernels.
//
// post_kernel (latency-bound, small): one warp per row sums the posteriors
// of each distinct class of the row's utterance from the stored alpha / beta
// rows.  Blank states are summed lane-strided and then by a fixed butterfly;
// each distinct label class is summed by its first occurrence walking the
// chain of later occurrences (no atomics, fixed order: bitwise reproducible).
// The sums land in a compact row post[r][o], o = the class's owner rank
// (the blank last), unscaled.
//
// dense_kernel (bandwidth-bound, the dominant kernel): the (T_total, D)
// output is cut into tiles of whole rows (about kTileElems elements).
// Persistent CTAs stream the tiles:
//   * one thread keeps kBuffers tiles of log probabilities in flight with
//     bulk (TMA) copies of each tile's 16-byte-aligned interior into shared
//     memory (ragged head/tail bytes come with plain loads);
//   * one warp per row scatters the row's few class sums into a shared
//     dense row P (and marks the 16-byte chunks they fall in);
//   * every 16-byte chunk of the gradient is computed as
//     scale * (exp(lp) - P) and leaves with one vector store (ragged chunks
//     at the tile ends element by element); marked chunks are cleared.
//
// The stored rows are fixed-point log2 values of alpha_t(s) / p_t(s) (before
// the emission) and of beta_t(s), each relative to an integer offset of its
// (frame, warp); the posterior's exponent alpha~ + beta~ + offsets + nll is
// summed exactly in 64-bit integers and meets one ex2 at the end.
#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

constexpr int kBuffers = 2;  // tiles of log probabilities in flight per CTA

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

struct RowInfo {
    int b;        // utterance, -1 for none
    int covered;  // the row is a frame of a well-formed utterance
    float scale;  // upstream gradient of the row's utterance (0 if zeroed)
};

__device__ __forceinline__ RowInfo row_info(const GradArgs& a, int64_t row) {
    const UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    const double* nll = ws_at<double>(a.ws, a.L.off_nll);
    const Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    RowInfo ri{-1, 0, 0.0f};
    const int B = a.L.B;
    const int b = find_utterance(a.cu, B, row);
    if (b < 0) return ri;
    ri.b = b;
    const UttInfo u = utt[b];
    const int64_t t = row - u.start;
    ri.covered = ctrl->grad_ready && u.valid && u.labels_ok && t >= 0 && t < u.T;
    if (!ri.covered) return ri;
    float scale;
    if (a.reduction == CTC_PACKED_NONE) {
        scale = a.grad_loss[b];
    } else if (a.reduction == CTC_PACKED_SUM) {
        scale = a.grad_loss[0];
    } else {
        scale = (float)((double)a.grad_loss[0] / ((double)B * (double)max(u.U, 1)));
    }
    const double v = nll[b];
    if (a.zero_infinity && isinf(v) && v > 0) scale = 0.0f;
    ri.scale = scale;
    return ri;
}

}  // namespace

// ------------------------------------------------------------ posteriors

// Posterior of one state from its stored alpha / beta fixed-point values and
// the integer part `base` = ((A + B) << frac) + round(nll * log2 e << frac).
__device__ __forceinline__ float posterior(int va, int vb, long long base) {
    if (va == kFixZero || vb == kFixZero) return 0.0f;
    long long t = (long long)va + (long long)vb + base;
    t = t < -(200ll << kFixFrac) ? -(200ll << kFixFrac) : (t > (200ll << kFixFrac) ? (200ll << kFixFrac) : t);
    return fast_ex2((float)(int)t * (1.0f / (float)(1 << kFixFrac)));
}

__global__ void __launch_bounds__(256) post_kernel(GradArgs a) {
    const UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    const double* nll = ws_at<double>(a.ws, a.L.off_nll);
    const int32_t* aoff = ws_at<int32_t>(a.ws, a.L.off_aoff);
    const int32_t* boff = ws_at<int32_t>(a.ws, a.L.off_boff);
    const int* alpha = ws_at<int>(a.ws, a.L.off_alpha);
    const int* beta = ws_at<int>(a.ws, a.L.off_beta);
    const int32_t* nxt = ws_at<int32_t>(a.ws, a.L.off_nxt);
    const int32_t* rank = ws_at<int32_t>(a.ws, a.L.off_rank);
    float* post = ws_at<float>(a.ws, a.L.off_post);
    const int lane = threadIdx.x & 31;
    const int P = pairs_for_max_u(a.L.max_U);
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.L.T_total > 0) {
        Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
        if (!ctrl->grad_ready) set_status(ctrl, CTC_PACKED_DEV_NO_GRAD_STATE);
    }
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < a.L.T_total;
         row += warps) {
        const RowInfo ri = row_info(a, row);
        if (!ri.covered || ri.scale == 0.0f) continue;
        const UttInfo u = utt[ri.b];
        const long long kfix = __double2ll_rn(nll[ri.b] * kLog2eD * (double)(1 << kFixFrac));
        const int32_t* ao = aoff + row * a.L.nwo;
        const int32_t* bo = boff + row * a.L.nwo;
        const int* ar = alpha + row * a.L.pitch;
        const int* br = beta + row * a.L.pitch;
        const int32_t* rk = rank + u.moff;
        const int32_t* nx = nxt + u.moff;
        float* pr = post + row * a.L.post_pitch;
        // alpha pair j holds states (2j, 2j+1) at positions 2j, 2j+1 (warp (j/P)/32 of its chain);
        // beta pair j holds states (2j-1, 2j) at positions 2j, 2j+1, so state s sits at s+1
        auto base_of = [&](int ja, int jb) -> long long {
            return ((long long)ao[(ja / P) >> 5] + (long long)bo[(jb / P) >> 5]) * (1ll << kFixFrac) + kfix;
        };
        auto label_post = [&](int j) {  // state 2j+1
            return posterior(ar[2 * j + 1], br[2 * j + 2], base_of(j, j + 1));
        };
        float blank_sum = 0.0f;
        for (int j = lane; j <= u.U; j += 32) {
            const int2 av = *reinterpret_cast<const int2*>(ar + 2 * j);
            const int2 bv = *reinterpret_cast<const int2*>(br + 2 * j);
            blank_sum += posterior(av.x, bv.y, base_of(j, j));
            if (j < u.U) {
                const int kind = rk[j];
                if (kind == -2) {
                    blank_sum += label_post(j);
                } else if (kind >= 0) {
                    float s = label_post(j);
                    for (int jj = nx[j]; jj >= 0; jj = nx[jj]) s += label_post(jj);
                    pr[kind] = s;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) blank_sum += __shfl_xor_sync(0xffffffffu, blank_sum, o);
        if (lane == 0) pr[u.n_owners - 1] = blank_sum;
    }
}

// ------------------------------------------------------------ dense rows

template <int DT>
__global__ void __launch_bounds__(kGradThreads) dense_kernel(GradArgs a) {
    constexpr int E = Elem<DT>::bytes;
    constexpr int V = 16 / E;  // elements per 16-byte chunk
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int K = a.rows_per_tile;
    const int D = a.D;
    const int tile_elems = K * D;
    const int max_chunks = tile_elems / V + 2;
    const int bitmap_words = (max_chunks + 31) / 32;
    // shared memory: barriers, flag, row info, chunk bitmap, P, log-probability tiles
    unsigned char* p = smem_raw;
    uint64_t* bar = reinterpret_cast<uint64_t*>(p);
    p += 8 * kBuffers;
    int* flag = reinterpret_cast<int*>(p);
    p += 8;
    p = reinterpret_cast<unsigned char*>(align_up(reinterpret_cast<uintptr_t>(p), 16));
    int* row_cov = reinterpret_cast<int*>(p);
    p += align_up(sizeof(int) * K, 16);
    float* row_scale = reinterpret_cast<float*>(p);
    p += align_up(sizeof(float) * K, 16);
    uint32_t* bitmap = reinterpret_cast<uint32_t*>(p);
    p += align_up(sizeof(uint32_t) * bitmap_words, 16);
    float* P = reinterpret_cast<float*>(p);
    p += align_up(sizeof(float) * (size_t)max_chunks * V, 16);
    const size_t buf_bytes = align_up((size_t)tile_elems * E + 32, 16);
    unsigned char* lpbuf = p;

    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    const float* post = ws_at<float>(a.ws, a.L.off_post);
    const int32_t* owner = ws_at<int32_t>(a.ws, a.L.off_owner);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NT = blockDim.x, NW = NT >> 5;
    const uintptr_t lp0 = reinterpret_cast<uintptr_t>(a.lp);
    const uintptr_t gr0 = reinterpret_cast<uintptr_t>(a.grad);

    for (int i = tid; i < max_chunks * V / 4; i += NT) reinterpret_cast<float4*>(P)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = tid; i < bitmap_words; i += NT) bitmap[i] = 0u;
    if (tid == 0) {
        for (int k = 0; k < kBuffers; ++k) mbar_init(&bar[k], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // geometry of tile `tile` of this CTA: byte range of its log probabilities
    auto tile_rows = [&](int64_t tile, int64_t& r0, int& nrows) {
        r0 = tile * K;
        nrows = (int)min((int64_t)K, a.L.T_total - r0);
    };
    // start the copy of tile `tile` into buffer `buf` (thread 0); returns whether a bulk copy was issued
    auto issue_tile = [&](int64_t tile, int buf) {
        int64_t r0;
        int nrows;
        tile_rows(tile, r0, nrows);
        const uintptr_t a0 = lp0 + (uintptr_t)(r0 * D * E);
        const uintptr_t a1 = a0 + (uintptr_t)nrows * D * E;
        const uintptr_t A16 = (a0 + 15) & ~uintptr_t(15);
        const uintptr_t B16 = a1 & ~uintptr_t(15);
        if (A16 + 16 <= B16) {
            mbar_expect_tx(&bar[buf], (uint32_t)(B16 - A16));
            bulk_g2s(lpbuf + buf * buf_bytes + (A16 - (a0 & ~uintptr_t(15))), reinterpret_cast<const void*>(A16),
                     (uint32_t)(B16 - A16), &bar[buf]);
        }
    };
    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    if (tid == 0) {
        for (int k = 0; k < kBuffers; ++k) {
            const int64_t tile = first + k * stride;
            if (tile < a.n_tiles) issue_tile(tile, k);
        }
    }
    uint32_t phases = 0;  // bit k: parity of buffer k's next completion

    int it = 0;
    for (int64_t tile = first; tile < a.n_tiles; tile += stride, ++it) {
        const int buf = it % kBuffers;
        int64_t r0;
        int nrows;
        tile_rows(tile, r0, nrows);
        const int nelem = nrows * D;
        const uintptr_t a0 = lp0 + (uintptr_t)(r0 * D * E);
        const uintptr_t a1 = a0 + (uintptr_t)nelem * E;
        const uintptr_t abase = a0 & ~uintptr_t(15);
        const uintptr_t A16 = (a0 + 15) & ~uintptr_t(15);
        const uintptr_t B16 = a1 & ~uintptr_t(15);
        const bool bulk = A16 + 16 <= B16;
        unsigned char* lb = lpbuf + buf * buf_bytes;
        const size_t shift = a0 - abase;
        const uintptr_t g0 = gr0 + (uintptr_t)(r0 * D * E);
        const uintptr_t g1 = g0 + (uintptr_t)nelem * E;
        const uintptr_t qb = g0 & ~uintptr_t(15);
        const int pshift = (int)((g0 - qb) / E);  // element f of the tile sits at P[f + pshift]

        // 1. ragged head/tail of the log probabilities, plain loads
        {
            const int head = bulk ? (int)((A16 - a0) / E) : nelem;
            const int tail = bulk ? (int)((B16 - a0) / E) : nelem;
            for (int f = tid; f < head; f += NT) {
                if constexpr (E == 4) {
                    *reinterpret_cast<uint32_t*>(lb + shift + (size_t)f * 4) = *reinterpret_cast<const uint32_t*>(a0 + (size_t)f * 4);
                } else {
                    *reinterpret_cast<unsigned short*>(lb + shift + (size_t)f * 2) = *reinterpret_cast<const unsigned short*>(a0 + (size_t)f * 2);
                }
            }
            for (int f = tail + tid; f < nelem; f += NT) {
                if constexpr (E == 4) {
                    *reinterpret_cast<uint32_t*>(lb + shift + (size_t)f * 4) = *reinterpret_cast<const uint32_t*>(a0 + (size_t)f * 4);
                } else {
                    *reinterpret_cast<unsigned short*>(lb + shift + (size_t)f * 2) = *reinterpret_cast<const unsigned short*>(a0 + (size_t)f * 2);
                }
            }
        }
        // 2. rows: scale, and the class sums scattered into P
        for (int r = warp; r < nrows; r += NW) {
            const int64_t row = r0 + r;
            const RowInfo ri = row_info(a, row);
            if (lane == 0) {
                row_cov[r] = ri.covered;
                row_scale[r] = ri.scale;
            }
            if (!ri.covered || ri.scale == 0.0f) continue;
            const UttInfo u = utt[ri.b];
            const float* pr = post + row * a.L.post_pitch;
            const int32_t* oc = owner + u.moff;
            for (int o = lane; o < u.n_owners; o += 32) {
                const int idx = r * D + oc[o] + pshift;
                P[idx] = pr[o];
                atomicOr(&bitmap[(idx / V) >> 5], 1u << ((idx / V) & 31));
            }
        }
        __syncthreads();
        if (bulk) {
            // one thread waits (bounded) for the copy; the barrier then
            // publishes both the data and the verdict to the whole CTA
            if (tid == 0) {
                long long spins = 0;
                int ok = 1;
                while (!mbar_try_wait(&bar[buf], (phases >> buf) & 1u)) {
                    if (++spins > kSpinLimit) {
                        ok = 0;
                        break;
                    }
                }
                *flag = ok;
                if (!ok) set_status(ctrl, CTC_PACKED_DEV_WAIT_TIMEOUT);
            }
            phases ^= 1u << buf;
            __syncthreads();
            if (!*flag) return;  // the copy never landed: leave rather than read a partial tile
        }
        // 3. the gradient tile, 16 bytes at a time
        const int nq = (int)((((g1 + 15) & ~uintptr_t(15)) - qb) / 16);
        {
            const float invD = 1.0f / (float)D;
            for (int q = tid; q < nq; q += NT) {
                const uintptr_t c0 = qb + (uintptr_t)q * 16;
                const uintptr_t lo = c0 > g0 ? c0 : g0;
                const uintptr_t hi = c0 + 16 < g1 ? c0 + 16 : g1;
                const int f_lo = (int)((lo - g0) / E);
                const int f_hi = (int)((hi - g0) / E);
                int r = __float2int_rz((float)f_lo * invD);
                if (r * D > f_lo) --r;
                if ((r + 1) * D <= f_lo) ++r;
                int c = f_lo - r * D;
                const bool marked = (bitmap[q >> 5] >> (q & 31)) & 1u;
                float pv[V];
                if (marked) {
#pragma unroll
                    for (int k = 0; k < V; k += 4) {
                        const float4 v = reinterpret_cast<const float4*>(P + q * V)[k / 4];
                        pv[k] = v.x;
                        pv[k + 1] = v.y;
                        pv[k + 2] = v.z;
                        pv[k + 3] = v.w;
                        reinterpret_cast<float4*>(P + q * V)[k / 4] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < V; ++k) pv[k] = 0.0f;
                }
                if (lo == c0 && hi == c0 + 16) {
                    uint32_t w[4];
                    if (a.congruent) {
                        const uint4 v = *reinterpret_cast<const uint4*>(lb + shift + (size_t)f_lo * E);
                        w[0] = v.x;
                        w[1] = v.y;
                        w[2] = v.z;
                        w[3] = v.w;
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if constexpr (E == 4) {
                                w[k] = *reinterpret_cast<const uint32_t*>(lb + shift + (size_t)(f_lo + k) * 4);
                            } else {
                                const uint32_t l0 = *reinterpret_cast<const unsigned short*>(lb + shift + (size_t)(f_lo + 2 * k) * 2);
                                const uint32_t l1 = *reinterpret_cast<const unsigned short*>(lb + shift + (size_t)(f_lo + 2 * k + 1) * 2);
                                w[k] = l0 | (l1 << 16);
                            }
                        }
                    }
                    float out[V];
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        while (c >= D) {
                            c -= D;
                            ++r;
                        }
                        uint32_t bits;
                        if constexpr (E == 4) {
                            bits = w[k];
                        } else {
                            bits = (k & 1) ? (w[k >> 1] >> 16) : (w[k >> 1] & 0xffffu);
                        }
                        const float x = bits_to_float<DT>(bits);
                        out[k] = row_cov[r] ? row_scale[r] * (fast_ex2(x * kLog2e) - pv[k]) : 0.0f;
                        ++c;
                    }
                    uint4 o;
                    if constexpr (E == 4) {
                        o = make_uint4(__float_as_uint(out[0]), __float_as_uint(out[1]), __float_as_uint(out[2]),
                                       __float_as_uint(out[3]));
                    } else {
                        o = make_uint4(pack2<DT>(out[0], out[1]), pack2<DT>(out[2], out[3]), pack2<DT>(out[4], out[5]),
                                       pack2<DT>(out[6], out[7]));
                    }
                    *reinterpret_cast<uint4*>(c0) = o;
                } else {
                    for (int f = f_lo; f < f_hi; ++f) {
                        while (c >= D) {
                            c -= D;
                            ++r;
                        }
                        uint32_t bits;
                        if constexpr (E == 4) {
                            bits = *reinterpret_cast<const uint32_t*>(lb + shift + (size_t)f * 4);
                        } else {
                            bits = *reinterpret_cast<const unsigned short*>(lb + shift + (size_t)f * 2);
                        }
                        const float x = bits_to_float<DT>(bits);
                        const float pk = pv[f + pshift - q * V];
                        const float gv = row_cov[r] ? row_scale[r] * (fast_ex2(x * kLog2e) - pk) : 0.0f;
                        const uint32_t ob = pack1<DT>(gv);
                        if constexpr (E == 4) {
                            *reinterpret_cast<uint32_t*>(g0 + (size_t)f * 4) = ob;
                        } else {
                            *reinterpret_cast<unsigned short*>(g0 + (size_t)f * 2) = (unsigned short)ob;
                        }
                        ++c;
                    }
                }
            }
        }
        __syncthreads();  // buffer `buf` and P are free again
        for (int k = tid; k < (nq + 31) / 32; k += NT) bitmap[k] = 0u;
        if (tid == 0) {
            const int64_t next = tile + (int64_t)kBuffers * stride;
            if (next < a.n_tiles) issue_tile(next, buf);
        }
        __syncthreads();
    }
}

template __global__ void dense_kernel<0>(GradArgs);
template __global__ void dense_kernel<1>(GradArgs);
template __global__ void dense_kernel<2>(GradArgs);

static size_t dense_smem_bytes(int rows_per_tile, int D, int E) {
    const size_t K = (size_t)rows_per_tile;
    const int V = 16 / E;
    const size_t max_chunks = K * D / V + 2;
    const size_t bitmap_words = (max_chunks + 31) / 32;
    return 16 + 8 * kBuffers + 8 + 2 * align_up(4 * K, 16) + align_up(4 * bitmap_words, 16) +
           align_up(4 * max_chunks * V, 16) + kBuffers * align_up(K * D * E + 32, 16);
}

template <int DT>
static cudaError_t launch_dense_t(const GradArgs& a, cudaStream_t s) {
    const size_t smem = dense_smem_bytes(a.rows_per_tile, a.D, Elem<DT>::bytes);
    cudaError_t e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(dense_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dense_kernel<DT>, kGradThreads, smem)) !=
        cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)sms * per_sm;
    if (a.n_tiles < grid) grid = a.n_tiles;
    if (grid < 1) return cudaSuccess;
    dense_kernel<DT><<<(unsigned)grid, kGradThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_grad(const GradArgs& a, int dtype, cudaStream_t s) {
    cudaError_t e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (a.L.B > 0 && a.L.T_total > 0) {
        long long want = (a.L.T_total + 7) / 8;  // blocks of 8 warps, one row per warp
        long long grid = (long long)sms * 8;
        if (want < grid) grid = want;
        post_kernel<<<(unsigned)grid, 256, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (dtype == 0) return launch_dense_t<0>(a, s);
    if (dtype == 1) return launch_dense_t<1>(a, s);
    if (dtype == 2) return launch_dense_t<2>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace ctcp
