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
constexpr int kPostThreads = 256;
constexpr int kPostRows = 2;  // rows a warp of the class-sum pass walks together
constexpr int kUnroll = 4;                   // 16-byte chunks in flight per lane
constexpr int kBatchChunks = 32 * kUnroll;   // chunks a warp streams per batch
constexpr int kGroupShift = 21;             // offset group of pair j: (j * gp_mul) >> kGroupShift

// Entries of a warp's per-batch tables: the batches of the widest row (4-byte
// elements, shifted by up to 15 bytes), one more for the end mark, and slack.
__host__ __device__ constexpr int batch_slots(int D) {
    return (int)(((4ll * D + 32) / 16 + kBatchChunks - 1) / kBatchChunks) + 4;
}

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

}  // namespace

// Class sums of every row.  A warp takes kPostRows consecutive rows at a
// time and walks their states together, so each round trip to memory serves
// all of them.  For a covered row with a nonzero scale, each distinct class
// of its utterance (the blank last) gets one entry (class, -scale * sum of
// its states' posteriors); the header holds the entry count, the scale and
// whether the row is covered.
__global__ void __launch_bounds__(kPostThreads) post_kernel(GradArgs a) {
    extern __shared__ __align__(16) float post_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ulen = (int)align_up((size_t)a.L.max_U + 1, 4);
    float* gam = post_smem + (size_t)warp * kPostRows * ulen;  // label posteriors of the rows, [row][j]
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    // a stored row is [the per-warp offsets, owo ints][the state pairs, pitch ints]
    const int* __restrict__ alpha = ws_at<int>(a.ws, a.L.off_alpha);
    const int* __restrict__ beta = ws_at<int>(a.ws, a.L.off_beta);
    const LabelRec* __restrict__ lbl = ws_at<LabelRec>(a.ws, a.L.off_lbl);
    RowHead* head = ws_at<RowHead>(a.ws, a.L.off_head);
    int2* ent = ws_at<int2>(a.ws, a.L.off_ent);
    const uint32_t gp_mul = a.gp_mul;  // j / gpairs == (j * gp_mul) >> kGroupShift for every pair j
    pdl_wait();     // the forward's stored rows and metadata
    pdl_trigger();  // persistent grid: every block is already resident
    const bool ready = ctrl->grad_ready != 0;
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.L.T_total > 0 && !ready)
        set_status(ctrl, CTC_PACKED_DEV_NO_GRAD_STATE);
    const int B = a.L.B;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t n_blocks = (a.L.T_total + kPostRows - 1) / kPostRows;

    for (int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp; blk < n_blocks; blk += warps) {
        const int64_t r0 = blk * kPostRows;
        // per row: its utterance, scale and the constants of its posteriors
        int U[kPostRows], moff[kPostRows], toff[kPostRows], kint[kPostRows], nown[kPostRows];
        float scale[kPostRows], cfrac[kPostRows];
        bool live[kPostRows], covered[kPostRows];
        int jmax = -1;
        {
            int b = find_utterance(a.cu, B, r0);
#pragma unroll
            for (int r = 0; r < kPostRows; ++r) {
                const int64_t row = r0 + r;
                covered[r] = false;
                scale[r] = 0.0f;
                U[r] = 0;
                moff[r] = toff[r] = kint[r] = nown[r] = 0;
                cfrac[r] = 0.0f;
                if (row < a.L.T_total) {
                    while (b + 1 < B && (int64_t)a.cu[b + 1] <= row) ++b;  // rows ascend: walk forward
                    if (b >= 0) {
                        const UttInfo u = utt[b];
                        const int64_t t = row - u.start;
                        covered[r] = ready && u.valid && u.labels_ok && t >= 0 && t < u.T;
                        if (covered[r]) {
                            if (a.reduction == CTC_PACKED_NONE) {
                                scale[r] = a.grad_loss[b];
                            } else if (a.reduction == CTC_PACKED_SUM) {
                                scale[r] = a.grad_loss[0];
                            } else if (a.reduction == CTC_PACKED_MEAN) {
                                scale[r] = __fdiv_rn(a.grad_loss[0], (float)B * (float)max(u.U, 1));
                            } else if (a.reduction == CTC_PACKED_MEAN_BATCH) {
                                scale[r] = __fdiv_rn(a.grad_loss[0], (float)B);
                            } else {  // mean_volume
                                scale[r] = __fdiv_rn(a.grad_loss[0], (float)ctrl->tl_total);
                            }
                            if (a.zero_infinity && u.nll_inf) scale[r] = 0.0f;
                            // an infinite nll (no alignment, zero_infinity off) leaves the row unspecified
                            kint[r] = u.kint;
                            cfrac[r] = u.cfrac;
                            U[r] = u.U;
                            moff[r] = u.moff;
                            toff[r] = u.toff;
                            nown[r] = u.n_owners;
                        }
                    }
                }
                live[r] = covered[r] && scale[r] != 0.0f;
                if (live[r]) jmax = max(jmax, U[r]);
            }
        }
        // 1. posteriors of every state pair of the rows
        float blank_sum[kPostRows];
#pragma unroll
        for (int r = 0; r < kPostRows; ++r) blank_sum[r] = 0.0f;
        for (int j = lane; j <= jmax; j += 32) {
            const uint32_t ga = ((uint32_t)j * gp_mul) >> kGroupShift;
            const uint32_t gb = ((uint32_t)(j + 1) * gp_mul) >> kGroupShift;
            int2 av[kPostRows], bv[kPostRows];
            int bl[kPostRows], oa[kPostRows], ob0[kPostRows], ob1[kPostRows], rk[kPostRows];
#pragma unroll
            for (int r = 0; r < kPostRows; ++r) {
                const bool on = live[r] && j <= U[r];
                const bool lab = live[r] && j < U[r];
                const int64_t row = r0 + r;
                const int* ar = alpha + row * a.L.spitch;
                const int* br = beta + row * a.L.spitch;
                av[r] = on ? *reinterpret_cast<const int2*>(ar + a.L.owo + 2 * j) : make_int2(kFixZero, kFixZero);
                bv[r] = on ? *reinterpret_cast<const int2*>(br + a.L.owo + 2 * j) : make_int2(kFixZero, kFixZero);
                bl[r] = lab ? br[a.L.owo + 2 * j + 2] : kFixZero;
                oa[r] = on ? ar[ga] : 0;
                ob0[r] = on ? br[ga] : 0;
                ob1[r] = lab ? br[gb] : 0;
                rk[r] = lab ? lbl[moff[r] + j].rank : -1;
            }
#pragma unroll
            for (int r = 0; r < kPostRows; ++r) {
                blank_sum[r] += posterior(av[r].x, bv[r].y, oa[r] + ob0[r] + kint[r], cfrac[r]);
                const float gl = posterior(av[r].y, bl[r], oa[r] + ob1[r] + kint[r], cfrac[r]);
                if (live[r] && j < U[r]) gam[r * ulen + j] = gl;
                if (rk[r] == -2) blank_sum[r] += gl;
            }
        }
#pragma unroll
        for (int r = 0; r < kPostRows; ++r) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) blank_sum[r] += __shfl_xor_sync(0xffffffffu, blank_sum[r], o);
        }
        __syncwarp();
        // 2. each distinct class, summed by its first occurrence in target order
        for (int j = lane; j < jmax; j += 32) {
#pragma unroll
            for (int r = 0; r < kPostRows; ++r) {
                if (!(live[r] && j < U[r])) continue;
                const LabelRec lr = lbl[moff[r] + j];
                const int kind = lr.rank;
                if (kind >= 0) {
                    const LabelRec* lb = lbl + moff[r];
                    float sum = gam[r * ulen + j];
                    for (int jj = lr.next; jj >= 0; jj = lb[jj].next) sum += gam[r * ulen + jj];
                    ent[(r0 + r) * a.L.ecap + kind] = make_int2(a.targets[toff[r] + j], __float_as_int(-scale[r] * sum));
                }
            }
        }
        if (lane < kPostRows) {
#pragma unroll
            for (int r = 0; r < kPostRows; ++r) {
                if (r != lane || r0 + r >= a.L.T_total) continue;
                if (live[r])
                    ent[(r0 + r) * a.L.ecap + nown[r] - 1] = make_int2(a.blank, __float_as_int(-scale[r] * blank_sum[r]));
                head[r0 + r] = RowHead{live[r] ? nown[r] : 0, covered[r] ? scale[r] : 0.0f, covered[r] ? 1 : 0, 0};
            }
        }
        __syncwarp();
    }
}

template <int DT>
__global__ void __launch_bounds__(kMaxWarpsPerBlock * 32, 2) grad_kernel(GradArgs a) {
    constexpr int E = Elem<DT>::bytes;
    constexpr int V = 16 / E;  // elements per 16-byte chunk
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int K = a.rows_per_tile;   // rows per group
    const int cap = a.entry_cap;     // corrections a group can hold
    // this warp's slice: row scales, corrections (packed row/class, value), the batch tile
    unsigned char* ws = smem_raw + (size_t)warp * a.warp_smem;
    float* row_scale = reinterpret_cast<float*>(ws);  // K entries, NaN-free: 0 when not covered
    int* row_cov = reinterpret_cast<int*>(ws + align_up(4 * (size_t)K, 16));
    float* row_bias = reinterpret_cast<float*>(ws + 2 * align_up(4 * (size_t)K, 16));  // exponent bias of each row
    int* e_key = reinterpret_cast<int*>(ws + 3 * align_up(4 * (size_t)K, 16));
    float* e_val = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(e_key) + align_up(4 * (size_t)cap, 16));
    float* ptile = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(e_val) + align_up(4 * (size_t)cap, 16));
    uint32_t* pmark = reinterpret_cast<uint32_t*>(ptile + kBatchChunks * 8);  // kBatchChunks / 32 words
    // a row's class sums bucketed by batch: bstart[b] .. bstart[b + 1] in skey / sval
    int* bstart = reinterpret_cast<int*>(pmark + 4);
    const int nslot = batch_slots(a.D);
    int* bfill = bstart + nslot;
    int* skey = bfill + nslot;
    float* sval = reinterpret_cast<float*>(skey + align_up((size_t)cap, 4));

    const RowHead* __restrict__ head = ws_at<RowHead>(a.ws, a.L.off_head);
    const int2* __restrict__ ent = ws_at<int2>(a.ws, a.L.off_ent);
    const int D = a.D;
    const uintptr_t lp0 = reinterpret_cast<uintptr_t>(a.lp);
    const uintptr_t gr0 = reinterpret_cast<uintptr_t>(a.grad);
    const int64_t n_groups = a.n_tiles;
    const int wpb = blockDim.x >> 5;
    const int64_t warps = (int64_t)gridDim.x * wpb;

    for (int i = lane; i < kBatchChunks * V; i += 32) ptile[i] = 0.0f;
    if (lane < kBatchChunks / 32) pmark[lane] = 0u;
    __syncwarp();
    pdl_wait();     // the class sums of the pass before
    pdl_trigger();  // persistent grid: every block is already resident
    // logits input: exp(lp) = exp(z - lse) = 2^(z log2 e - lse log2 e)
    const bool logits = ws_at<Control>(a.ws, a.L.off_ctrl)->logits != 0;
    const float* __restrict__ lse = ws_at<float>(a.ws, a.L.off_lse);

    if (K == 1 && a.congruent) {
        // One row per warp task, lp and grad congruent modulo 16.  The batches
        // of a warp's rows form one continuous stream: the next batch, the
        // next row's first one included, is always in flight while the current
        // one computes, so a row's setup (header, class sums) waits on no
        // empty pipe.  Chunk q of a row covers grad bytes [qb + 16q, +16); the
        // ragged end chunks are read whole and stored element by element.
        const int64_t T = a.L.T_total;
        const uintptr_t lp_end = lp0 + (uintptr_t)T * D * E;
        struct RowGeo {
            uintptr_t g0, g1, qb, lpq;
            int pshift, nq, nb;
        };
        auto geo = [&](int64_t row) {
            RowGeo r;
            r.g0 = gr0 + (uintptr_t)(row * D * E);
            r.g1 = r.g0 + (uintptr_t)D * E;
            r.qb = r.g0 & ~uintptr_t(15);
            r.pshift = (int)((r.g0 - r.qb) / E);
            r.nq = (int)((((r.g1 + 15) & ~uintptr_t(15)) - r.qb) / 16);
            r.nb = (r.nq + kBatchChunks - 1) / kBatchChunks;
            r.lpq = r.qb + (lp0 + (uintptr_t)(row * D * E) - r.g0);
            return r;
        };
        auto load_batch = [&](const RowGeo& g, int bi, uint4 (&dst)[kUnroll]) {
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int q = bi * kBatchChunks + k * 32 + lane;
                const uintptr_t c = g.lpq + (uintptr_t)q * 16;
                if (q < g.nq && c >= lp0 && c + 16 <= lp_end) dst[k] = ld_stream(reinterpret_cast<const void*>(c));
            }
        };
        int64_t row = (int64_t)blockIdx.x * wpb + warp;
        if (row >= T) return;
        RowGeo g = geo(row);
        uint4 cur[kUnroll], nxt[kUnroll];
        load_batch(g, 0, cur);
        for (;;) {
            // the row's header and class sums, bucketed by batch
            const RowHead h = head[row];
            const int2* er = ent + row * a.L.ecap;
            const int count = h.count;
            const bool cov = h.covered != 0;
            const float s = h.scale;
            const float bias = logits ? -lse[row] * kLog2e : 0.0f;
            for (int i = lane; i <= g.nb; i += 32) bfill[i] = 0;
            __syncwarp();
            for (int e = lane; e < count; e += 32) atomicAdd(&bfill[(er[e].x + g.pshift) / (kBatchChunks * V)], 1);
            __syncwarp();
            {
                int run = 0;
                for (int base = 0; base <= g.nb; base += 32) {
                    const int i = base + lane;
                    const int c = i < g.nb ? bfill[i] : 0;
                    int x = c;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= o) x += y;
                    }
                    if (i <= g.nb) bstart[i] = run + x - c;
                    run += __shfl_sync(0xffffffffu, x, 31);
                }
            }
            __syncwarp();
            for (int i = lane; i < g.nb; i += 32) bfill[i] = bstart[i];
            __syncwarp();
            for (int e = lane; e < count; e += 32) {
                const int2 v = er[e];
                const int pos = atomicAdd(&bfill[(v.x + g.pshift) / (kBatchChunks * V)], 1);
                skey[pos] = v.x;
                sval[pos] = __int_as_float(v.y);
            }
            __syncwarp();

            const int64_t nrow = row + warps;
            RowGeo gn = g;
            if (nrow < T) gn = geo(nrow);
            // the whole row is requested from DRAM at once, while its first
            // batch is already in flight (measured: fetching further ahead, a
            // row or a few batches, is slower)
            if (lane == 0) {
                const uintptr_t lo = lp0 + (uintptr_t)(row * D * E);
                prefetch_l2(lo, lo + (uintptr_t)D * E);
            }
            for (int bi = 0; bi < g.nb; ++bi) {
                if (bi + 1 < g.nb) {
                    load_batch(g, bi + 1, nxt);
                } else if (nrow < T) {
                    load_batch(gn, 0, nxt);
                }
                const int q0 = bi * kBatchChunks;
                for (int e = bstart[bi] + lane; e < bstart[bi + 1]; e += 32) {
                    const int idx = skey[e] + g.pshift - q0 * V;
                    ptile[idx] = sval[e];
                    atomicOr(&pmark[idx / (32 * V)], 1u << ((idx / V) & 31));
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < kUnroll; ++k) {
                    const int q = q0 + k * 32 + lane;
                    if (q >= g.nq) continue;
                    const int ql = k * 32 + lane;
                    const bool marked = (pmark[k] >> lane) & 1u;
                    const uintptr_t c0 = g.qb + (uintptr_t)q * 16;
                    const uintptr_t cl = g.lpq + (uintptr_t)q * 16;
                    float pn[V];
#pragma unroll
                    for (int i = 0; i < V; ++i) pn[i] = 0.0f;
                    if (marked) {
#pragma unroll
                        for (int i = 0; i < V; i += 4) {
                            const float4 v = reinterpret_cast<const float4*>(ptile + ql * V)[i / 4];
                            pn[i] = v.x;
                            pn[i + 1] = v.y;
                            pn[i + 2] = v.z;
                            pn[i + 3] = v.w;
                            reinterpret_cast<float4*>(ptile + ql * V)[i / 4] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                    if (c0 >= g.g0 && c0 + 16 <= g.g1) {
                        *reinterpret_cast<uint4*>(c0) = cov ? chunk_grad<DT>(cur[k], s, pn, bias) : make_uint4(0u, 0u, 0u, 0u);
                    } else if (cl >= lp0 && cl + 16 <= lp_end) {
                        // a ragged end chunk, read whole: store only the row's elements
                        const uint4 o = cov ? chunk_grad<DT>(cur[k], s, pn, bias) : make_uint4(0u, 0u, 0u, 0u);
                        const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                        for (int i = 0; i < V; ++i) {
                            const uintptr_t ad = c0 + (uintptr_t)i * E;
                            if (ad >= g.g0 && ad < g.g1) {
                                if constexpr (E == 4) {
                                    store_elem<DT>(ad, w[i]);
                                } else {
                                    store_elem<DT>(ad, (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu));
                                }
                            }
                        }
                    } else {
                        // a ragged chunk at an end of the lp buffer: element by element
                        const uintptr_t lo = c0 > g.g0 ? c0 : g.g0;
                        const uintptr_t hi = c0 + 16 < g.g1 ? c0 + 16 : g.g1;
                        for (uintptr_t ad = lo; ad < hi; ad += E) {
                            const float x = bits_to_float<DT>(load_elem<DT>(cl + (ad - c0)));
                            const int i = (int)((ad - c0) / E);
                            float pk = 0.0f;  // pn[i], selected without dynamic indexing
#pragma unroll
                            for (int ii = 0; ii < V; ++ii) pk = ii == i ? pn[ii] : pk;
                            const float gv = cov ? fmaf(s, fast_ex2(fmaf(x, kLog2e, bias)), pk) : 0.0f;
                            store_elem<DT>(ad, pack1<DT>(gv));
                        }
                    }
                }
                __syncwarp();
                if (lane < kBatchChunks / 32) pmark[lane] = 0u;
                __syncwarp();
#pragma unroll
                for (int k = 0; k < kUnroll; ++k) cur[k] = nxt[k];
            }
            if (nrow >= T) break;
            row = nrow;
            g = gn;
        }
        return;
    }
    for (int64_t grp = (int64_t)blockIdx.x * wpb + warp; grp < n_groups; grp += warps) {
        const int64_t r0 = grp * K;
        const int nrows = (int)min((int64_t)K, a.L.T_total - r0);

        // the next group's class sums start their way into L2
        {
            const int64_t nr0 = (grp + warps) * K;
            const int64_t nrows_next = nr0 < a.L.T_total ? min((int64_t)K, a.L.T_total - nr0) : 0;
            const int64_t bytes = nrows_next * (int64_t)a.L.ecap * 8;
            for (int64_t off = (int64_t)lane * 128; off < bytes; off += 32 * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(ent + nr0 * a.L.ecap) + off));
        }
        // 1. the group's rows: scale, coverage and class sums (key = row in group * D + class)
        int count = 0;  // corrections so far (warp-uniform)
        for (int rr = 0; rr < nrows; ++rr) {
            const RowHead h = head[r0 + rr];
            if (lane == 0) {
                row_scale[rr] = h.scale;
                row_cov[rr] = h.covered;
                row_bias[rr] = logits ? -lse[r0 + rr] * kLog2e : 0.0f;
            }
            const int2* er = ent + (r0 + rr) * a.L.ecap;
            for (int e = lane; e < h.count; e += 32) {
                const int2 v = er[e];
                e_key[count + e] = rr * D + v.x;
                e_val[count + e] = __int_as_float(v.y);
            }
            count += h.count;
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
            const float bias = row_bias[0];
            const int nb = (nq + kBatchChunks - 1) / kBatchChunks;
            // bucket the class sums by batch, once per row
            for (int i = lane; i <= nb; i += 32) bfill[i] = 0;
            __syncwarp();
            for (int e = lane; e < count; e += 32) atomicAdd(&bfill[(e_key[e] + pshift) / (kBatchChunks * V)], 1);
            __syncwarp();
            {
                int run = 0;
                for (int base = 0; base <= nb; base += 32) {
                    const int i = base + lane;
                    const int c = i < nb ? bfill[i] : 0;
                    int x = c;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= o) x += y;
                    }
                    if (i <= nb) bstart[i] = run + x - c;
                    run += __shfl_sync(0xffffffffu, x, 31);
                }
            }
            __syncwarp();
            for (int i = lane; i < nb; i += 32) bfill[i] = bstart[i];
            __syncwarp();
            for (int e = lane; e < count; e += 32) {
                const int f = e_key[e];
                const int pos = atomicAdd(&bfill[(f + pshift) / (kBatchChunks * V)], 1);
                skey[pos] = f;
                sval[pos] = e_val[e];
            }
            __syncwarp();

            auto load_batch = [&](int q0, uint4 (&dst)[kUnroll]) {
#pragma unroll
                for (int k = 0; k < kUnroll; ++k) {
                    const int q = q0 + k * 32 + lane;
                    if (cov && q >= qf0 && q < qf1) dst[k] = ld_stream(reinterpret_cast<const void*>(lpq + (uintptr_t)q * 16));
                }
            };
            uint4 cur[kUnroll], nxt[kUnroll];
            load_batch(0, cur);
            for (int bi = 0; bi < nb; ++bi) {
                const int q0 = bi * kBatchChunks;
                if (bi + 1 < nb) load_batch(q0 + kBatchChunks, nxt);  // in flight while this batch computes
                for (int e = bstart[bi] + lane; e < bstart[bi + 1]; e += 32) {
                    const int idx = skey[e] + pshift - q0 * V;
                    ptile[idx] = sval[e];
                    atomicOr(&pmark[idx / (32 * V)], 1u << ((idx / V) & 31));
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
                        float pn[V];
#pragma unroll
                        for (int i = 0; i < V; ++i) pn[i] = 0.0f;
                        if (marked) {
#pragma unroll
                            for (int i = 0; i < V; i += 4) {
                                const float4 v = reinterpret_cast<const float4*>(ptile + ql * V)[i / 4];
                                pn[i] = v.x;
                                pn[i + 1] = v.y;
                                pn[i + 2] = v.z;
                                pn[i + 3] = v.w;
                                reinterpret_cast<float4*>(ptile + ql * V)[i / 4] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
                        *reinterpret_cast<uint4*>(c0) = cov ? chunk_grad<DT>(cur[k], s, pn, bias) : make_uint4(0u, 0u, 0u, 0u);
                    } else {
                        // the ragged first / last chunk of the row
                        const uintptr_t lo = c0 > g0 ? c0 : g0;
                        const uintptr_t hi = c0 + 16 < g1 ? c0 + 16 : g1;
                        for (uintptr_t ad = lo; ad < hi; ad += E) {
                            const size_t f = (ad - g0) / E;
                            const float x = bits_to_float<DT>(load_elem<DT>(a0 + f * E));
                            const float pk = marked ? ptile[ql * V + (int)(f + pshift) - q * V] : 0.0f;
                            const float gv = cov ? fmaf(s, fast_ex2(fmaf(x, kLog2e, bias)), pk) : 0.0f;
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
#pragma unroll
                for (int k = 0; k < kUnroll; ++k) cur[k] = nxt[k];
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
                        const float s = row_scale[r], bias = row_bias[r];
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
                            out[i] = fmaf(s, fast_ex2(fmaf(bits_to_float<DT>(bits), kLog2e, bias)), pv[i]);
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
                        const float gv =
                            row_cov[r] ? fmaf(row_scale[r], fast_ex2(fmaf(x, kLog2e, row_bias[r])), pk) : 0.0f;
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
    return launch_pdl(grad_kernel<DT>, dim3((unsigned)grid), dim3(wpb * 32), smem, s, a);
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
    warp_smem = 3 * align_up(4 * (size_t)k, 16) + 2 * align_up(4 * (size_t)entry_cap, 16) +
                4 * (size_t)kBatchChunks * 8 + 4 * (kBatchChunks / 32) +
                4 * 2 * (size_t)batch_slots(D) + 2 * 4 * align_up((size_t)entry_cap, 4);
    warp_smem = align_up(warp_smem, 16);
}

uint32_t grad_group_multiplier(const Layout& L) {
    const uint32_t m = ((1u << kGroupShift) + (uint32_t)L.gpairs - 1) / (uint32_t)L.gpairs;
    for (uint32_t j = 0; j <= (uint32_t)L.max_U + 1; ++j)
        if (((j * m) >> kGroupShift) != j / (uint32_t)L.gpairs) return 0;
    return m;
}

cudaError_t launch_post(const GradArgs& a, cudaStream_t s) {
    if (a.L.T_total == 0) return cudaSuccess;
    // as many warps per block (up to 8) as 200 KB of shared memory hold
    const size_t warp_smem = sizeof(float) * kPostRows * align_up((size_t)a.L.max_U + 1, 4);
    int wpb = (int)(200 * 1024 / warp_smem);
    wpb = wpb < 1 ? 1 : (wpb > kPostThreads / 32 ? kPostThreads / 32 : wpb);
    const size_t smem = (size_t)wpb * warp_smem;
    cudaError_t e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(post_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, post_kernel, 32 * wpb, smem)) != cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)sms * per_sm;
    const long long blocks = (a.L.T_total + kPostRows - 1) / kPostRows;
    const long long want = (blocks + wpb - 1) / wpb;
    if (want < grid) grid = want;
    return launch_pdl(post_kernel, dim3((unsigned)grid), dim3(32 * wpb), smem, s, a);
}

cudaError_t launch_grad(const GradArgs& a, int dtype, cudaStream_t s) {
    if (dtype == 0) return launch_grad_t<0>(a, s);
    if (dtype == 1) return launch_grad_t<1>(a, s);
    if (dtype == 2) return launch_grad_t<2>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace ctcp
