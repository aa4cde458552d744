// Forward and backward CTC recursions over packed log probabilities.
//
// Page "feat(asr): native CTC loss kernel over sequence-packed log
// probabilities", ctc_loss.py ``_alpha_kernel`` and ``_beta_grad_kernel``:
//
//   alpha_0(s) = lp[0, l'_s] for s in {0, 1};
//   alpha_t(s) = lse(alpha_{t-1}(s), alpha_{t-1}(s-1), [skip(s)] alpha_{t-1}(s-2)) + lp[t, l'_s],
//     skip(s): s odd, s >= 2 and l'_s != l'_{s-2};
//   nll = -lse(alpha_{T-1}(S-1), alpha_{T-1}(S-2));
//   beta_{T-1}(s) = lp[T-1, l'_s] for s in {S-2, S-1};
//   beta_t(s) = lse(beta_{t+1}(s), beta_{t+1}(s+1), [skip'(s)] beta_{t+1}(s+2)) + lp[t, l'_s],
//     skip'(s): s odd, s + 2 < S and l'_s != l'_{s+2}.
//
// How it maps to the GPU.  Each utterance is two independent work items, its
// alpha chain and its beta chain, so both serial recursions of an utterance
// run at the same time on different SMs (the page runs beta inside its
// backward program, after the forward).  A chain item is run by a group of
// threads: the whole CTA when the target is long, one warp when 2U+1 states
// fit in a warp.  Thread j of a group holds P consecutive *state pairs*:
//   alpha pair j = (blank 2j, label 2j+1),   beta pair j = (label 2j-1, blank 2j),
// so a frame step needs the state just below (alpha) or above (beta) the
// thread's pairs only: one warp shuffle, plus a shared-memory halo across
// warps and one CTA barrier per frame.
//
// Label columns: every frame a chain reads lp[t, blank] and lp[t, l_j] for its
// labels.  Each thread gathers its own labels' words with 4-byte cp.async
// kRing-1 frames ahead into a shared-memory ring (the word that holds a
// 2-byte element is fetched whole and the right half picked on use), so no
// global-memory latency sits on the recursion.
//
// Accuracy: the recursion runs in base-2 log space in float32, and each frame
// subtracts an integer offset delta_t from every state, so the states near
// the maximum stay near 0 where float32 is dense (the page's absolute float32
// alphas reach |1e4| and lose ~1e-3).  delta_t is chosen two frames late from
// the exact maximum of frame t-2 (delta_t = round(max_{t-2}) - delta_{t-1},
// a dead-beat correction), so the reduction never sits on the critical path.
// The running offsets are exact int32 sums, stored per frame (aoff / boff)
// and added back in float64 where the log-likelihood is assembled.
//
// What is stored for the backward: alpha rows hold the *pre-emission* value
// alpha_t(s) - lp[t, l'_s] - A_t (so the backward needs no lp gather), beta
// rows hold beta_t(s) - B_t, both in (T_total, pitch) float32 rows.
#include <cstdio>

#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

struct Group {
    int tid;         // thread index within the group
    int n;           // threads in the group
    int warp;        // warp index within the CTA (CTA mode)
    int nw;          // warps in the CTA (CTA mode)
    uint32_t* ring;  // kRing slots of (n * P + 1) words
    float* halo;     // [2][nw]   (CTA mode)
    float* maxima;   // [4][nw]   (CTA mode)
    float* fin;      // 2 floats private to the group
};

template <bool CTA>
__device__ __forceinline__ void group_sync() {
    if constexpr (CTA) {
        __syncthreads();
    } else {
        __syncwarp();
    }
}

// Issue the gather of element `elem` of the log probabilities into `dst`.
template <int DT>
__device__ __forceinline__ void gather_word(uint32_t* dst, const unsigned char* lp, int64_t lp_bytes, int64_t elem) {
    const unsigned char* p = lp + elem * Elem<DT>::bytes;
    if constexpr (DT == 0) {
        cp_async4(smem_addr(dst), p);
    } else {
        const uintptr_t addr = reinterpret_cast<uintptr_t>(p);
        const uintptr_t word = addr & ~uintptr_t(3);
        const uintptr_t lo = reinterpret_cast<uintptr_t>(lp);
        if (word >= lo && word + 4 <= lo + (uintptr_t)lp_bytes) {
            cp_async4(smem_addr(dst), reinterpret_cast<const void*>(word));
        } else {
            // the aligned word would leave the buffer: read the element alone
            reinterpret_cast<unsigned short*>(dst)[(addr >> 1) & 1] = *reinterpret_cast<const unsigned short*>(p);
        }
    }
}

// The gathered value of element `elem` in base-2 log units, -inf clamped to kNeg.
template <int DT>
__device__ __forceinline__ float gathered_log2(uint32_t w, const unsigned char* lp, int64_t elem) {
    int half = 0;
    if constexpr (DT != 0) half = (int)((reinterpret_cast<uintptr_t>(lp + elem * 2) >> 1) & 1);
    return max_nan(word_to_float<DT>(w, half) * kLog2e, kNeg);
}

// Maximum of one value per thread over the group, for the offset controller.
template <bool CTA>
__device__ __forceinline__ void publish_max(const Group& g, int slot, float m) {
    const float wm = warp_max(m);
    if constexpr (CTA) {
        if ((g.tid & 31) == 0) g.maxima[slot * g.nw + g.warp] = wm;
    }
}

template <int P, int DT, bool CTA>
__device__ void run_chain_item(const ChainArgs& a, int item, const Group& g) {
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const UttInfo info = ws_at<UttInfo>(a.ws, a.L.off_utt)[item >> 1];
    double* nll_out = ws_at<double>(a.ws, a.L.off_nll);
    const int b = item >> 1;
    const int dir = item & 1;  // 0 alpha, 1 beta
    const int T = info.T, U = info.U;
    const int64_t start = info.start;
    const int64_t D = a.D;
    const int lane = g.tid & 31;
    const unsigned char* lp = static_cast<const unsigned char*>(a.lp);
    const int32_t* tg = a.targets + info.toff;

    // labels of my pairs and their skip transitions
    int cls[P];
    bool has_label[P], skip[P];
    bool bad = false;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int j = g.tid * P + p;
        if (dir == 0) {  // (blank 2j, label 2j+1 = l_j)
            has_label[p] = j < U;
            cls[p] = has_label[p] ? tg[j] : 0;
            skip[p] = j >= 1 && j < U && cls[p] != tg[j - 1];
        } else {  // (label 2j-1 = l_{j-1}, blank 2j)
            has_label[p] = j >= 1 && j <= U;
            cls[p] = has_label[p] ? tg[j - 1] : 0;
            skip[p] = j >= 1 && j < U && cls[p] != tg[j];
        }
        if (has_label[p] && (cls[p] < 0 || (int64_t)cls[p] >= D)) bad = true;
    }
    if constexpr (CTA) {
        bad = __syncthreads_or(bad);
    } else {
        bad = __any_sync(0xffffffffu, bad);
    }
    if (bad) {
        if (g.tid == 0) {
            set_status(ctrl, CTC_PACKED_DEV_LABEL_OUT_OF_RANGE);
            if (dir == 0) {
                nll_out[b] = __longlong_as_double(0x7ff8000000000000ll);
                if (a.reduction == CTC_PACKED_NONE) a.loss[b] = __int_as_float(0x7fc00000);
            }
        }
        group_sync<CTA>();
        return;
    }

    const int SS = g.n * P + 1;  // words per ring slot: P label words per thread, then the blank
    auto row_of = [&](int k) -> int64_t { return dir == 0 ? start + k : start + (T - 1 - k); };
    auto issue = [&](int k) {
        if (k < T) {
            const int64_t rowD = row_of(k) * D;
            uint32_t* slot = g.ring + (k % kRing) * SS;
#pragma unroll
            for (int p = 0; p < P; ++p)
                if (has_label[p]) gather_word<DT>(slot + p * g.n + g.tid, lp, a.lp_bytes, rowD + cls[p]);
            if (g.tid == 0) gather_word<DT>(slot + g.n * P, lp, a.lp_bytes, rowD + a.blank);
        }
        cp_async_commit();
    };
    float lpl[P];
    float lpb;
    auto consume = [&](int k) {
        const int64_t rowD = row_of(k) * D;
        const uint32_t* slot = g.ring + (k % kRing) * SS;
        lpb = gathered_log2<DT>(slot[g.n * P], lp, rowD + a.blank);
#pragma unroll
        for (int p = 0; p < P; ++p)
            lpl[p] = has_label[p] ? gathered_log2<DT>(slot[p * g.n + g.tid], lp, rowD + cls[p]) : kNeg;
    };

    float* store_base = ws_at<float>(a.ws, dir == 0 ? a.L.off_alpha : a.L.off_beta);
    int32_t* off_base = ws_at<int32_t>(a.ws, dir == 0 ? a.L.off_aoff : a.L.off_boff);
    const int j0 = g.tid * P;
    const bool store_me = j0 <= U;
    auto store_row = [&](int64_t row, const float (&x)[P], const float (&y)[P]) {
        if (!store_me) return;
        float* dst = store_base + row * a.L.pitch + 2 * j0;
        if constexpr (P == 1) {
            *reinterpret_cast<float2*>(dst) = make_float2(x[0], y[0]);
        } else {
#pragma unroll
            for (int p = 0; p < P; p += 2)
                *reinterpret_cast<float4*>(dst + 2 * p) = make_float4(x[p], y[p], x[p + 1], y[p + 1]);
        }
    };

    // prologue: kRing-1 frames in flight
#pragma unroll 1
    for (int k = 0; k < kRing - 1; ++k) issue(k);

    float vb[P], vl[P];  // post-emission values, base 2, minus the running offset
    int acc_off = 0, delta_prev = 0;
    float m_last = kNeg, m_before = kNeg;  // group maxima of the two previous frames (warp mode)

    // frame of step 0
    cp_async_wait<kRing - 2>();
    group_sync<CTA>();
    consume(0);
    {
        float x[P], y[P];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int j = j0 + p;
            if (dir == 0) {
                vb[p] = j == 0 ? lpb : kNeg;
                vl[p] = (j == 0 && U >= 1) ? lpl[p] : kNeg;
                x[p] = j == 0 ? 0.0f : kNeg;  // pre-emission: log2(1) for the two start states
                y[p] = (j == 0 && U >= 1) ? 0.0f : kNeg;
            } else {
                vb[p] = j == U ? lpb : kNeg;
                vl[p] = (j == U && U >= 1) ? lpl[p] : kNeg;
                x[p] = vl[p];
                y[p] = vb[p];
            }
        }
        const int64_t row = row_of(0);
        if (dir == 0) {
            store_row(row, x, y);
        } else {
            store_row(row, vl, vb);
        }
        if (g.tid == 0) off_base[row] = 0;
        float m = kNeg;
#pragma unroll
        for (int p = 0; p < P; ++p) m = fmaxf(m, fmaxf(vb[p], vl[p]));
        publish_max<CTA>(g, 0, m);
        if constexpr (!CTA) m_last = warp_max(m);
        if constexpr (CTA) {
            if (dir == 0 && lane == 31) g.halo[0 * g.nw + g.warp] = vl[P - 1];
            if (dir == 1 && lane == 0) g.halo[0 * g.nw + g.warp] = vl[0];
        }
    }
    issue(kRing - 1);

#pragma unroll 1
    for (int i = 1; i < T; ++i) {
        cp_async_wait<kRing - 2>();
        group_sync<CTA>();
        consume(i);
        // the state just below (alpha) or above (beta) my pairs, from the previous frame
        float nb;
        if (dir == 0) {
            nb = __shfl_up_sync(0xffffffffu, vl[P - 1], 1);
            if (lane == 0) {
                nb = kNeg;
                if constexpr (CTA) {
                    if (g.warp > 0) nb = g.halo[((i - 1) & 1) * g.nw + g.warp - 1];
                }
            }
        } else {
            nb = __shfl_down_sync(0xffffffffu, vl[0], 1);
            if (lane == 31) {
                nb = kNeg;
                if constexpr (CTA) {
                    if (g.warp < g.nw - 1) nb = g.halo[((i - 1) & 1) * g.nw + g.warp + 1];
                }
            }
        }
        // offset of this frame from the exact maximum two frames back
        float m2 = kNeg;
        if (i >= 2) {
            if constexpr (CTA) {
                const float v = lane < g.nw ? g.maxima[((i - 2) & 3) * g.nw + lane] : kNeg;
                m2 = warp_max(v);
            } else {
                m2 = m_before;
            }
        }
        int delta = 0;
        if (m2 > kNegHalf) delta = min(max(__float2int_rn(m2) - delta_prev, -(1 << 20)), 1 << 20);
        const float fd = (float)delta;

        float nbv[P], nlv[P];
        if (dir == 0) {
            float pb[P], pl[P];
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const float prev = p ? vl[p - 1] : nb;
                pb[p] = lse2(vb[p], prev) - fd;
                pl[p] = lse3(vl[p], vb[p], skip[p] ? prev : kNeg) - fd;
                nbv[p] = pb[p] + lpb;
                nlv[p] = pl[p] + lpl[p];
            }
            store_row(row_of(i), pb, pl);
        } else {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const float next = (p < P - 1) ? vl[p + 1] : nb;
                nbv[p] = lse2(vb[p], next) - fd + lpb;
                nlv[p] = lse3(vl[p], vb[p], skip[p] ? next : kNeg) - fd + lpl[p];
            }
            store_row(row_of(i), nlv, nbv);
        }
        float m = kNeg;
#pragma unroll
        for (int p = 0; p < P; ++p) {
            vb[p] = nbv[p];
            vl[p] = nlv[p];
            m = fmaxf(m, fmaxf(vb[p], vl[p]));
        }
        acc_off += delta;
        delta_prev = delta;
        if (g.tid == 0) off_base[row_of(i)] = acc_off;
        if constexpr (CTA) {
            if (dir == 0 && lane == 31) g.halo[(i & 1) * g.nw + g.warp] = vl[P - 1];
            if (dir == 1 && lane == 0) g.halo[(i & 1) * g.nw + g.warp] = vl[0];
            publish_max<CTA>(g, i & 3, m);
        } else {
            m_before = m_last;
            m_last = warp_max(m);
        }
        issue(i + kRing - 1);
    }

    if (dir == 0) {
        // the paths end in the last blank (pair U) or the last label (pair U-1)
        if (g.tid == 0) {
            g.fin[0] = kNeg;
            g.fin[1] = kNeg;
        }
        group_sync<CTA>();
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int j = j0 + p;
            if (j == U) g.fin[0] = vb[p];
            if (U >= 1 && j == U - 1) g.fin[1] = vl[p];
        }
        group_sync<CTA>();
        if (g.tid == 0) {
            const float x = lse2(g.fin[0], g.fin[1]);
            double v;
            if (isnan(x)) {
                v = (double)x;
            } else if (x <= kNegHalf) {
                v = __longlong_as_double(0x7ff0000000000000ll);  // no path: +inf
            } else {
                v = -((double)acc_off + (double)x) * kLn2D;
            }
            nll_out[b] = v;
            if (a.reduction == CTC_PACKED_NONE) {
                float out = (float)v;
                if (a.zero_infinity && isinf(v)) out = 0.0f;
                a.loss[b] = out;
            }
        }
    }
    cp_async_wait<0>();
    group_sync<CTA>();
}

// Label metadata the backward needs, one warp per utterance: for each target
// position whether it is the first occurrence of its class (then it owns the
// class's posterior sum), the next position with the same class, and whether
// the id equals the blank (then its posterior joins the blank column).
__device__ void run_label_item(const ChainArgs& a, int b, int lane) {
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    const UttInfo info = utt[b];
    const int U = info.U;
    const int32_t* tg = a.targets + info.toff;
    int32_t* nxt = ws_at<int32_t>(a.ws, a.L.off_nxt) + info.moff;
    int32_t* rank = ws_at<int32_t>(a.ws, a.L.off_rank) + info.moff;
    int32_t* owner = ws_at<int32_t>(a.ws, a.L.off_owner) + info.moff;
    bool bad = false;
    int running = 0;
    for (int j0 = 0; j0 < U; j0 += 32) {
        const int j = j0 + lane;
        bool first = false, is_blank = false;
        int nx = -1, c = 0;
        if (j < U) {
            c = tg[j];
            if (c < 0 || c >= a.D) bad = true;
            is_blank = c == a.blank;
            if (!is_blank) {
                first = true;
                for (int k = j - 1; k >= 0; --k)
                    if (tg[k] == c) {
                        first = false;
                        break;
                    }
                for (int k = j + 1; k < U; ++k)
                    if (tg[k] == c) {
                        nx = k;
                        break;
                    }
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, first);
        const int r = running + __popc(m & ((1u << lane) - 1u));
        if (j < U) {
            nxt[j] = nx;
            rank[j] = first ? r : (is_blank ? -2 : -1);
            if (first) owner[r] = c;
        }
        running += __popc(m);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        owner[running] = a.blank;
        utt[b].n_owners = running + 1;
        utt[b].labels_ok = bad ? 0 : 1;
        if (bad) set_status(ctrl, CTC_PACKED_DEV_LABEL_OUT_OF_RANGE);
    }
}

}  // namespace

template <int P, int DT>
__global__ void __launch_bounds__(1024, 1) chain_kernel(ChainArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_item;
    __shared__ int s_last;
    __shared__ double s_red[32];
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const int32_t* queue = ws_at<int32_t>(a.ws, a.L.off_queue);
    const int NT = blockDim.x, NW = NT >> 5;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t* ring = reinterpret_cast<uint32_t*>(smem_raw);
    const int ring_words = kRing * (NT * P + NW);
    float* halo = reinterpret_cast<float*>(ring + ring_words);
    float* maxima = halo + 2 * NW;
    float* fin = maxima + 4 * NW;  // 2 per warp
    const int n_big = ctrl->n_big, n_small = ctrl->n_small, n_lab = ctrl->n_lab;

    // 1. multi-warp chains, longest first, one at a time per CTA
    Group cg{tid, NT, warp, NW, ring, halo, maxima, fin};
    for (;;) {
        if (tid == 0) s_item = (int)atomicAdd(&ctrl->big_head, 1u);
        __syncthreads();
        const int k = s_item;
        __syncthreads();
        if (k >= n_big) break;
        run_chain_item<P, DT, true>(a, queue[k], cg);
    }
    // 2. single-warp chains, each warp on its own
    Group wg{lane, 32, warp, NW, ring + warp * kRing * (32 * P + 1), halo, maxima, fin + 2 * warp};
    for (;;) {
        int k = 0;
        if (lane == 0) k = (int)atomicAdd(&ctrl->small_head, 1u);
        k = __shfl_sync(0xffffffffu, k, 0);
        if (k >= n_small) break;
        run_chain_item<P, DT, false>(a, queue[n_big + k], wg);
    }
    // 3. label metadata for the backward
    for (;;) {
        int k = 0;
        if (lane == 0) k = (int)atomicAdd(&ctrl->lab_head, 1u);
        k = __shfl_sync(0xffffffffu, k, 0);
        if (k >= n_lab) break;
        run_label_item(a, queue[2 * a.L.B + 1 + k], lane);
    }

    // 4. the last CTA to finish reduces the losses (fixed order: deterministic)
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(&ctrl->done_ctas, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last || a.reduction == CTC_PACKED_NONE) return;
    __threadfence();
    const double* nll = ws_at<double>(a.ws, a.L.off_nll);
    const int B = a.L.B;
    double acc = 0.0;
    for (int b = tid; b < B; b += NT) {
        double v = __ldcg(nll + b);
        if (a.zero_infinity && isinf(v) && v > 0) v = 0.0;
        if (a.reduction == CTC_PACKED_MEAN) v /= (double)max(a.target_lengths[b], 1);
        acc += v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) s_red[warp] = acc;
    __syncthreads();
    if (tid == 0) {
        double total = 0.0;
        for (int w = 0; w < NW; ++w) total += s_red[w];
        if (a.reduction == CTC_PACKED_MEAN) total = B > 0 ? total / (double)B : __longlong_as_double(0x7ff8000000000000ll);
        a.loss[0] = (float)total;
    }
}

#define CTCP_INSTANTIATE_CHAIN(P, DT) template __global__ void chain_kernel<P, DT>(ChainArgs);
CTCP_INSTANTIATE_CHAIN(1, 0)
CTCP_INSTANTIATE_CHAIN(1, 1)
CTCP_INSTANTIATE_CHAIN(1, 2)
CTCP_INSTANTIATE_CHAIN(2, 0)
CTCP_INSTANTIATE_CHAIN(2, 1)
CTCP_INSTANTIATE_CHAIN(2, 2)
CTCP_INSTANTIATE_CHAIN(4, 0)
CTCP_INSTANTIATE_CHAIN(4, 1)
CTCP_INSTANTIATE_CHAIN(4, 2)
CTCP_INSTANTIATE_CHAIN(8, 0)
CTCP_INSTANTIATE_CHAIN(8, 1)
CTCP_INSTANTIATE_CHAIN(8, 2)

int chain_pairs_per_thread(int max_target_len) { return pairs_for_max_u(max_target_len); }

int chain_warps(int max_target_len, int P) {
    const int pairs = max_target_len + 1;
    int nw = (pairs + 32 * P - 1) / (32 * P);
    return nw < 1 ? 1 : (nw > 32 ? 32 : nw);
}

static size_t chain_smem_bytes(int P, int nw) {
    const int nt = 32 * nw;
    return sizeof(uint32_t) * (size_t)kRing * (nt * P + nw) + sizeof(float) * (size_t)(2 * nw + 4 * nw + 2 * nw);
}

template <int P, int DT>
static cudaError_t launch_chain_t(const ChainArgs& a, int nw, cudaStream_t s) {
    static int configured_smem = -1;
    const size_t smem = chain_smem_bytes(P, nw);
    cudaError_t e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((int)smem > configured_smem) {
        e = cudaFuncSetAttribute(chain_kernel<P, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured_smem = (int)smem;
    }
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_kernel<P, DT>, 32 * nw, smem)) !=
        cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    // persistent grid: enough CTAs for every item, never more than fit at once
    long long want = 2ll * a.L.B;
    long long grid = (long long)sms * per_sm;
    if (want < grid) grid = want > 0 ? want : 1;
    chain_kernel<P, DT><<<(unsigned)grid, 32 * nw, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_chain(const ChainArgs& a, int P, int nw, int dtype, cudaStream_t s) {
#define CTCP_CASE(PP, DD) \
    if (P == PP && dtype == DD) return launch_chain_t<PP, DD>(a, nw, s);
    CTCP_CASE(1, 0) CTCP_CASE(1, 1) CTCP_CASE(1, 2)
    CTCP_CASE(2, 0) CTCP_CASE(2, 1) CTCP_CASE(2, 2)
    CTCP_CASE(4, 0) CTCP_CASE(4, 1) CTCP_CASE(4, 2)
    CTCP_CASE(8, 0) CTCP_CASE(8, 1) CTCP_CASE(8, 2)
#undef CTCP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace ctcp
