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
// How it maps to the GPU.  The (T_total, D) output is cut into tiles of
// whole rows (about kTileElems elements).  Persistent CTAs walk the tiles:
//   1. one thread starts a bulk (TMA) copy of the tile's 16-byte-aligned
//      interior of log probabilities into shared memory; the few ragged
//      head/tail bytes come in with plain loads;
//   2. while it flies, each row finds its utterance (binary search over
//      cu_seqlens), its frame and its scale;
//   3. one warp per row forms the posteriors from the stored alpha / beta
//      rows: blank states are summed in registers (lane-strided, then a
//      fixed butterfly), each distinct label class is summed by its first
//      occurrence walking the chain of later occurrences, and the sums land
//      in a shared-memory row P[r][c] -- no global atomics, and a fixed order
//      so the result is bitwise reproducible;
//   4. every 16-byte chunk of the gradient tile is computed as
//      scale * (exp(lp) - P) and stored with one vector store (ragged chunks
//      at the tile ends element by element); P is then cleared.
//
// The stored rows are alpha~ = alpha - lp - A_t (pre-emission) and
// beta~ = beta - B_t in base-2 log units, so the exponent of the posterior is
// alpha~ + beta~ + (A_t + B_t + nll * log2 e), the last term formed in
// float64 once per row.
#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

struct TileSmem {
    uint64_t* bar;
    int* flag;
    int* row_b;
    int* row_cov;
    float* row_scale;
    float* P;              // rows_per_tile * D floats, zero between tiles
    unsigned char* lpbuf;  // 16-byte aligned image of the tile's log probabilities
};

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

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kGradThreads) grad_kernel(GradArgs a) {
    constexpr int E = Elem<DT>::bytes;
    constexpr int V = 16 / E;  // elements per 16-byte chunk
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int K = a.rows_per_tile;
    const int D = a.D;
    TileSmem sm;
    {
        unsigned char* p = smem_raw;
        sm.bar = reinterpret_cast<uint64_t*>(p);
        sm.flag = reinterpret_cast<int*>(p + 8);
        p += 16;
        sm.row_b = reinterpret_cast<int*>(p);
        p += align_up(sizeof(int) * K, 16);
        sm.row_cov = reinterpret_cast<int*>(p);
        p += align_up(sizeof(int) * K, 16);
        sm.row_scale = reinterpret_cast<float*>(p);
        p += align_up(sizeof(float) * K, 16);
        sm.P = reinterpret_cast<float*>(p);
        p += align_up(sizeof(float) * (size_t)K * D, 16);
        sm.lpbuf = p;
    }
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    const double* nll = ws_at<double>(a.ws, a.L.off_nll);
    const int32_t* aoff = ws_at<int32_t>(a.ws, a.L.off_aoff);
    const int32_t* boff = ws_at<int32_t>(a.ws, a.L.off_boff);
    const float* alpha = ws_at<float>(a.ws, a.L.off_alpha);
    const float* beta = ws_at<float>(a.ws, a.L.off_beta);
    const int32_t* nxt = ws_at<int32_t>(a.ws, a.L.off_nxt);
    const int32_t* rank = ws_at<int32_t>(a.ws, a.L.off_rank);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NT = blockDim.x, NW = NT >> 5;
    const int B = a.L.B;
    const bool ready = __ldcg(&ctrl->grad_ready) != 0;
    const unsigned char* lp = static_cast<const unsigned char*>(a.lp);
    unsigned char* grad = static_cast<unsigned char*>(a.grad);

    for (int i = tid; i < (int)(((size_t)K * D + 3) / 4); i += NT)
        reinterpret_cast<float4*>(sm.P)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid == 0) {
        mbar_init(sm.bar, 1);
        fence_mbar_init();
        if (!ready) set_status(ctrl, CTC_PACKED_DEV_NO_GRAD_STATE);
    }
    __syncthreads();
    uint32_t phase = 0;

    for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
        const int64_t r0 = tile * K;
        const int nrows = (int)min((int64_t)K, a.L.T_total - r0);
        const int nelem = nrows * D;
        // 1. log probabilities of the tile into shared memory
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(lp) + (uintptr_t)(r0 * D * E);
        const uintptr_t a1 = a0 + (uintptr_t)nelem * E;
        const uintptr_t abase = a0 & ~uintptr_t(15);
        const uintptr_t A16 = (a0 + 15) & ~uintptr_t(15);
        const uintptr_t B16 = a1 & ~uintptr_t(15);
        const bool bulk = A16 + 16 <= B16;
        if (tid == 0 && bulk) {
            mbar_expect_tx(sm.bar, (uint32_t)(B16 - A16));
            bulk_g2s(sm.lpbuf + (A16 - abase), reinterpret_cast<const void*>(A16), (uint32_t)(B16 - A16), sm.bar);
        }
        {
            const int head = bulk ? (int)((A16 - a0) / E) : nelem;
            const int tail = bulk ? (int)((B16 - a0) / E) : nelem;
            const size_t shift = a0 - abase;
            for (int f = tid; f < head; f += NT) {
                if constexpr (E == 4) {
                    *reinterpret_cast<uint32_t*>(sm.lpbuf + shift + (size_t)f * 4) =
                        *reinterpret_cast<const uint32_t*>(a0 + (size_t)f * 4);
                } else {
                    *reinterpret_cast<unsigned short*>(sm.lpbuf + shift + (size_t)f * 2) =
                        *reinterpret_cast<const unsigned short*>(a0 + (size_t)f * 2);
                }
            }
            for (int f = tail + tid; f < nelem; f += NT) {
                if constexpr (E == 4) {
                    *reinterpret_cast<uint32_t*>(sm.lpbuf + shift + (size_t)f * 4) =
                        *reinterpret_cast<const uint32_t*>(a0 + (size_t)f * 4);
                } else {
                    *reinterpret_cast<unsigned short*>(sm.lpbuf + shift + (size_t)f * 2) =
                        *reinterpret_cast<const unsigned short*>(a0 + (size_t)f * 2);
                }
            }
        }
        // 2. which utterance, frame and scale each row has
        for (int r = tid; r < nrows; r += NT) {
            const int64_t row = r0 + r;
            const int b = find_utterance(a.cu, B, row);
            int cov = 0;
            float scale = 0.0f;
            if (b >= 0) {
                const UttInfo u = utt[b];
                const int64_t t = row - u.start;
                cov = ready && u.valid && u.labels_ok && t >= 0 && t < u.T;
                if (cov) {
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
            sm.row_b[r] = b;
            sm.row_cov[r] = cov;
            sm.row_scale[r] = scale;
        }
        __syncthreads();
        // 3. posteriors, one warp per row, into the shared row P
        for (int r = warp; r < nrows; r += NW) {
            if (!sm.row_cov[r] || sm.row_scale[r] == 0.0f) continue;
            const int64_t row = r0 + r;
            const int b = sm.row_b[r];
            const UttInfo u = utt[b];
            const double kd = (double)aoff[row] + (double)boff[row] + nll[b] * kLog2eD;
            const float kf = (float)kd;
            const float* ar = alpha + row * a.L.pitch;
            const float* br = beta + row * a.L.pitch;
            const int32_t* rk = rank + u.moff;
            const int32_t* nx = nxt + u.moff;
            const int32_t* tg = a.targets + u.toff;
            float* Prow = sm.P + (size_t)r * D;
            float blank_sum = 0.0f;
            for (int j = lane; j <= u.U; j += 32) {
                blank_sum += fast_ex2(ar[2 * j] + br[2 * j + 1] + kf);
                if (j < u.U) {
                    const int kind = rk[j];
                    if (kind == -2) {
                        blank_sum += fast_ex2(ar[2 * j + 1] + br[2 * j + 2] + kf);
                    } else if (kind >= 0) {
                        float s = 0.0f;
                        for (int jj = j; jj >= 0; jj = nx[jj]) s += fast_ex2(ar[2 * jj + 1] + br[2 * jj + 2] + kf);
                        Prow[tg[j]] = s;
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) blank_sum += __shfl_xor_sync(0xffffffffu, blank_sum, o);
            if (lane == 0) Prow[a.blank] = blank_sum;
        }
        if (bulk) {
            // one thread waits (bounded) for the copy; the barrier then
            // publishes both the data and the verdict to the whole CTA
            if (tid == 0) {
                long long spins = 0;
                int ok = 1;
                while (!mbar_try_wait(sm.bar, phase)) {
                    if (++spins > kSpinLimit) {
                        ok = 0;
                        break;
                    }
                }
                *sm.flag = ok;
                if (!ok) set_status(ctrl, CTC_PACKED_DEV_WAIT_TIMEOUT);
            }
            phase ^= 1u;
        }
        __syncthreads();
        if (bulk && !*sm.flag) return;  // the copy never landed: leave rather than read a partial tile
        // 4. the gradient tile, 16 bytes at a time
        {
            const uintptr_t g0 = reinterpret_cast<uintptr_t>(grad) + (uintptr_t)(r0 * D * E);
            const uintptr_t g1 = g0 + (uintptr_t)nelem * E;
            const uintptr_t qb = g0 & ~uintptr_t(15);
            const int nq = (int)(((g1 + 15) & ~uintptr_t(15)) - qb) / 16;
            const size_t shift = a0 - abase;
            const float invD = 1.0f / (float)D;
            for (int qi = tid; qi < nq; qi += NT) {
                const uintptr_t c0 = qb + (uintptr_t)qi * 16;
                const uintptr_t lo = c0 > g0 ? c0 : g0;
                const uintptr_t hi = c0 + 16 < g1 ? c0 + 16 : g1;
                const int f_lo = (int)((lo - g0) / E);
                const int f_hi = (int)((hi - g0) / E);
                int r = __float2int_rz((float)f_lo * invD);
                if (r * D > f_lo) --r;
                if ((r + 1) * D <= f_lo) ++r;
                int c = f_lo - r * D;
                if (lo == c0 && hi == c0 + 16) {
                    uint32_t w[4];
                    if (a.congruent) {
                        const uint4 v = *reinterpret_cast<const uint4*>(sm.lpbuf + shift + (size_t)f_lo * E);
                        w[0] = v.x;
                        w[1] = v.y;
                        w[2] = v.z;
                        w[3] = v.w;
                    } else {
#pragma unroll
                        for (int i = 0; i < V; ++i) {
                            uint32_t bits;
                            if constexpr (E == 4) {
                                bits = *reinterpret_cast<const uint32_t*>(sm.lpbuf + shift + (size_t)(f_lo + i) * 4);
                            } else {
                                bits = *reinterpret_cast<const unsigned short*>(sm.lpbuf + shift + (size_t)(f_lo + i) * 2);
                            }
                            if constexpr (E == 4) {
                                w[i] = bits;
                            } else {
                                if (i & 1)
                                    w[i >> 1] |= bits << 16;
                                else
                                    w[i >> 1] = bits;
                            }
                        }
                    }
                    float out[V];
#pragma unroll
                    for (int i = 0; i < V; ++i) {
                        while (c >= D) {
                            c -= D;
                            ++r;
                        }
                        uint32_t bits;
                        if constexpr (E == 4) {
                            bits = w[i];
                        } else {
                            bits = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu);
                        }
                        const float x = bits_to_float<DT>(bits);
                        const float pr = sm.P[f_lo + i];
                        out[i] = sm.row_cov[r] ? sm.row_scale[r] * (fast_ex2(x * kLog2e) - pr) : 0.0f;
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
                            bits = *reinterpret_cast<const uint32_t*>(sm.lpbuf + shift + (size_t)f * 4);
                        } else {
                            bits = *reinterpret_cast<const unsigned short*>(sm.lpbuf + shift + (size_t)f * 2);
                        }
                        const float x = bits_to_float<DT>(bits);
                        const float g = sm.row_cov[r] ? sm.row_scale[r] * (fast_ex2(x * kLog2e) - sm.P[f]) : 0.0f;
                        const uint32_t ob = pack1<DT>(g);
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
        __syncthreads();
        // 5. clear P for the next tile
        for (int i = tid; i < (nelem + 3) / 4; i += NT)
            reinterpret_cast<float4*>(sm.P)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncthreads();
    }
}

template __global__ void grad_kernel<0>(GradArgs);
template __global__ void grad_kernel<1>(GradArgs);
template __global__ void grad_kernel<2>(GradArgs);

static size_t grad_smem_bytes(int rows_per_tile, int D, int elem_bytes) {
    const size_t K = (size_t)rows_per_tile;
    return 16 + 3 * align_up(4 * K, 16) + align_up(4 * K * (size_t)D, 16) + align_up(K * D * elem_bytes + 32, 16);
}

template <int DT>
static cudaError_t launch_grad_t(const GradArgs& a, cudaStream_t s) {
    const size_t smem = grad_smem_bytes(a.rows_per_tile, a.D, Elem<DT>::bytes);
    cudaError_t e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(grad_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, grad_kernel<DT>, kGradThreads, smem)) !=
        cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)sms * per_sm;
    if (a.n_tiles < grid) grid = a.n_tiles;
    if (grid < 1) return cudaSuccess;
    grad_kernel<DT><<<(unsigned)grid, kGradThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_grad(const GradArgs& a, int dtype, cudaStream_t s) {
    if (dtype == 0) return launch_grad_t<0>(a, s);
    if (dtype == 1) return launch_grad_t<1>(a, s);
    if (dtype == 2) return launch_grad_t<2>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace ctcp
