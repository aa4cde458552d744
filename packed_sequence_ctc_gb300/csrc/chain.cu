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
// backward program, after the forward).  Lane l of a chain warp holds P
// consecutive *state pairs*:
//   alpha pair j = (blank 2j, label 2j+1),   beta pair j = (label 2j-1, blank 2j),
// so a frame step needs only the state just below (alpha) or above (beta) the
// lane's pairs: one warp shuffle.
//
// Ghost lanes.  A long target spreads over several warps of a CTA.  Each
// warp owns (32 - G) * P pairs; its G extra lanes at the edge facing its
// neighbour (below for alpha, above for beta) shadow the neighbour's G * P
// edge pairs.  The shadow copies are exact right after a halo exchange and
// go wrong one pair per frame from the outer edge inward, so the owned pairs
// stay exact for G * P frames: the warps exchange their edges through shared
// memory, under one named barrier, only every G * P frames, and run the
// frames in between on shuffles alone.  Outside the target range (the lower
// shadow of the first warp, the upper one of the last) the states are zero
// and stay exactly zero.
//
// Emissions come from the emission matrix (emit.cu), whose entries pair a
// label's emission with the frame's blank: every frame a lane copies its
// first pair's entry (16 bytes, label and blank) and the label halves of
// its other pairs into its slice of the warp's shared-memory ring, R frames
// ahead.  No lane reads another lane's slice, so no warp sync is needed.
//
// Arithmetic: the recursion runs on probabilities in extended range (a float
// mantissa and an int32 binary exponent per state, see ctc_common.cuh):
// alpha_t(s) = (alpha_{t-1}(s) + alpha_{t-1}(s-1) + [skip] alpha_{t-1}(s-2)) * p_t(s),
// i.e. only multiply-adds and integer exponent arithmetic on the critical
// path, no exp or log, no cross-warp normalisation.
//
// What is stored for the backward, one int32 per state holding m * 2^k
// exactly up to a 19-bit mantissa (enc_state in ctc_common.cuh), k relative
// to a per-(frame, warp) integer offset (the largest exponent among the
// warp's owned states, stored per frame in aoff / boff): alpha rows hold the
// value *before* the frame's emission, alpha_t(s) / p_t(s), so the backward
// needs no log-probability gather; beta rows hold beta_t(s).  A row is
// encoded and stored one frame late, so that work overlaps the next frame's
// dependent chain.
#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

template <int P, int G_>
struct ChainShape {
    static constexpr int G = G_;                 // shadow lanes per warp
    static constexpr int GP = group_pairs(P, G); // pairs a warp owns
    static constexpr int F = G * P;              // frames between halo exchanges (8, 8, 4, 4)
    static constexpr int R = F == 8 ? 8 : 4;     // emission frames in flight per warp
    // extended values per lane and frame in the ring: (label 0, blank), the
    // other labels, padded to 16 bytes
    static constexpr int LW = 2 * ((P + 2) / 2);
    static constexpr int XW = G * P * 2;      // extended values one warp sends per exchange
    // One-pair chains stage a block's encoded rows in shared memory and write
    // them out together after the block; the others store each row as it is
    // made (their rings leave no room for a stage at 31 warps).
    static constexpr bool kStaged = P == 1;
    static constexpr int kStageInts = kStaged ? F * 32 * 2 * P : 0;  // per warp
    static_assert(F <= 8, "between renormalisations a mantissa grows at most 12x a frame");
    static_assert(R % F == 0, "a block of frames maps onto consecutive ring slots");
};

__device__ __forceinline__ void bar_named(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool bar_named_or(int id, int n, bool v) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((int)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
// 8- and 16-byte async copies global -> shared.
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

struct ItemCtx {
    int w;     // this warp's index among the item's warps
    int nw;    // warps running the item (1: a single-warp item, no exchanges)
    XP* ring;  // this warp's emission ring
    XP* xch;   // halo exchange buffers, [2][nw][XW]
    XP* fin;   // 2 extended values shared by the item's warps
    int* stage;  // this warp's encoded rows of one block of frames (one-pair chains)
};

// One chain (DIR 0 alpha, 1 beta) of utterance b, run by warp c.w of c.nw.
//
// Frame 0 is the initialisation; frames 1.. run in blocks of F: each
// frame is one recursion step on shuffles alone, the row of the frame
// before is encoded and stored on the side, and the emissions of the frame
// R - 1 ahead are requested.  After a block the states are renormalised
// (between renormalisations a mantissa grows at most 12x a frame) and the
// warps of a multi-warp item exchange their edges.
// CKPT: the checkpoint policy (store_rows > 1) is compiled as a variant of
// its own, so that the default (every row or none) keeps the plain loop.
template <int P, int G, int DIR, bool CKPT, bool STORE>
__device__ void run_chain(const ChainArgs& a, int b, const ItemCtx& c) {
    using S = ChainShape<P, G>;
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const UttInfo info = ws_at<UttInfo>(a.ws, a.L.off_utt)[b];
    double* nll_out = ws_at<double>(a.ws, a.L.off_nll);
    const int T = info.T, U = info.U;
    const int lane = threadIdx.x & 31;
    const bool multi = c.nw > 1;
    const int nthreads = 32 * c.nw;
    const int32_t* tg = a.targets + info.toff;
    const XP zero{0.0f, kEZero};

    // my pairs: owned lanes in pair order, shadow lanes at the edge
    const bool own = DIR == 0 ? lane >= S::G : lane < 32 - S::G;
    const int j0 = DIR == 0 ? c.w * S::GP + (lane - S::G) * P : c.w * S::GP + lane * P;
    bool has_label[P], skip[P];
    int wl[P];  // emission-row entry of my label state (U: the zero emission)
    bool bad = false;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int j = j0 + p;
        if (DIR == 0) {  // (blank 2j, label 2j+1 = l_j)
            has_label[p] = j >= 0 && j < U;
            wl[p] = has_label[p] ? j : U;
            skip[p] = j >= 1 && j < U && tg[j] != tg[j - 1];
        } else {  // (label 2j-1 = l_{j-1}, blank 2j)
            has_label[p] = j >= 1 && j <= U;
            wl[p] = has_label[p] ? j - 1 : U;
            skip[p] = j >= 1 && j < U && tg[j - 1] != tg[j];
        }
        if (own && has_label[p]) {
            const int cl = tg[wl[p]];
            if (cl < 0 || cl >= a.D) bad = true;
        }
    }
    if (c.w == 0 && lane == 0) {
        c.fin[0] = zero;
        c.fin[1] = zero;
    }
    bad = multi ? bar_named_or(1, nthreads, bad) : __any_sync(0xffffffffu, bad);
    if (bad) {
        if (DIR == 0 && c.w == 0 && lane == 0) {
            set_status(ctrl, CTC_PACKED_DEV_LABEL_OUT_OF_RANGE);
            nll_out[b] = __longlong_as_double(0x7ff8000000000000ll);
            if (a.reduction == CTC_PACKED_NONE) a.loss[b] = __int_as_float(0x7fc00000);
        }
        return;
    }

    // emission stream: frame k is row start + k (alpha) or start + T - 1 - k
    // (beta); the matrix has kEmPad >= R rows of padding at both ends, so
    // frames up to R - 1 past the utterance are read without a check
    const XP2* em = ws_at<XP2>(a.ws, em_base(a.L));
    const int64_t row0 = DIR == 0 ? (int64_t)info.start : (int64_t)info.start + T - 1;
    const int64_t estep = DIR == 0 ? (int64_t)a.L.epitch : -(int64_t)a.L.epitch;
    const XP2* src0[P];  // my entries in frame 0's row
#pragma unroll
    for (int p = 0; p < P; ++p) src0[p] = em + row0 * a.L.epitch + wl[p];
    // ring slot of frame k: (k - 1) mod R; lane l's values are LW consecutive XP
    const uint32_t ring_lane = smem_addr(c.ring) + (uint32_t)(lane * S::LW) * 8u;
    constexpr uint32_t kSlotBytes = 32u * S::LW * 8u;
    // frame k into ring slot `slot`; each address is formed from frame 0's, so
    // no register that a copy in flight still reads is written over
    auto request = [&](uint32_t slot, int k) {
        const uint32_t dst = ring_lane + slot * kSlotBytes;
        const int64_t off = (int64_t)k * estep;
        cp_async16(dst, src0[0] + off);
#pragma unroll
        for (int p = 1; p < P; ++p) cp_async8(dst + 8u * (p + 1), &src0[p][off].l);
        cp_async_commit();
    };
    auto emissions = [&](uint32_t slot, XP (&el)[P], XP& eb) {
        const XP* e = reinterpret_cast<const XP*>(c.ring) + slot * 32 * S::LW + lane * S::LW;
        el[0] = e[0];
        eb = e[1];
#pragma unroll
        for (int p = 1; p < P; ++p) el[p] = e[p + 1];
    };

    // stored rows, written one frame late: row k of the chain (frame k) is
    // packed row row0 + k (alpha) or row0 - k (beta)
    const bool store_me = own && j0 <= U;
    int* const st_base = ws_at<int>(a.ws, DIR == 0 ? a.L.off_alpha : a.L.off_beta);
    // a stored row is [the per-warp offsets, owo ints][the state pairs, pitch ints]
    int* st = st_base + row0 * a.L.spitch + a.L.owo + 2 * max(j0, 0);
    const intptr_t st_step = (DIR == 0 ? 1 : -1) * (intptr_t)a.L.spitch;
    int32_t* const off_base = st_base + row0 * a.L.spitch + c.w;
    int32_t* offp = off_base;
    const intptr_t off_step = st_step;
    // the warp's own pairs [p0, p0 + np) are contiguous in the row and, in the
    // stage, from lane `lane0` on; written in 16-byte chunks of two pairs
    // (an odd count also writes pair U + 1, which the row's pitch holds and
    // no reader uses)
    const int p0 = c.w * S::GP, np = min(S::GP, U + 1 - p0), nch = (np + 1) >> 1;
    const int lane0 = DIR == 0 ? S::G : 0;
    const uint32_t ch_mul = (65536u + (uint32_t)nch - 1) / (uint32_t)max(nch, 1);  // c / nch for c < 256
    int a_hold = 0;  // lane q: the offset of the block's row q
    // alpha rows: (blank, label) sums before the emission; beta: (label, blank) after it
    float rx[P], ry[P];
    int ex[P], ey[P];
    auto flush_row = [&](int slot) {
        int emax = kEZero;
#pragma unroll
        for (int p = 0; p < P; ++p) emax = max(emax, max(ex[p], ey[p]));
        const int A = __reduce_max_sync(0xffffffffu, own ? emax : kEZero);
        int x[P], y[P];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            x[p] = enc_state(rx[p], ex[p], A);
            y[p] = enc_state(ry[p], ey[p], A);
        }
        if constexpr (S::kStaged) {
            reinterpret_cast<int2*>(c.stage)[slot * 32 + lane] = make_int2(x[0], y[0]);
            if (lane == slot) a_hold = A;
        } else {
            if (store_me) {
#pragma unroll
                for (int p = 0; p < P; p += 2)
                    *reinterpret_cast<int4*>(st + 2 * p) = make_int4(x[p], y[p], x[p + 1], y[p + 1]);
            }
            if (lane == 0) *offp = A;
            st += st_step;
            offp += off_step;
        }
    };
    // Checkpoint policy (store_rows = K > 1): only rows whose absolute index
    // is a multiple of K are kept, written straight to their place (no stage);
    // the backward recomputes the rows in between from them.
    auto flush_ckpt = [&](int k) {  // the row of chain frame k, if it is a checkpoint
        const int64_t row = row0 + (DIR == 0 ? (int64_t)k : -(int64_t)k);
        if ((row & (int64_t)(a.store_rows - 1)) != 0) return;  // the same for every lane
        int emax = kEZero;
#pragma unroll
        for (int p = 0; p < P; ++p) emax = max(emax, max(ex[p], ey[p]));
        const int A = __reduce_max_sync(0xffffffffu, own ? emax : kEZero);
        int* rp = st_base + row * a.L.spitch;
        if (store_me) {
#pragma unroll
            for (int p = 0; p < P; ++p)
                *reinterpret_cast<int2*>(rp + a.L.owo + 2 * (j0 + p)) =
                    make_int2(enc_state(rx[p], ex[p], A), enc_state(ry[p], ey[p], A));
        }
        if (lane == 0) rp[c.w] = A;
    };
    // rows k0 .. k0 + n - 1 of the chain, staged in slots 0 .. n - 1: the
    // warp's segments as 16-byte chunks spread over all lanes, and the offsets
    auto write_rows = [&](int k0, int n) {
        if constexpr (S::kStaged) {
            __syncwarp();
            const int total = n * nch;
            for (int cq = lane; cq < total; cq += 32) {
                const int r = (int)(((uint32_t)cq * ch_mul) >> 16), k = cq - r * nch;
                const int4 v = reinterpret_cast<const int4*>(c.stage + r * 64 + 2 * lane0)[k];
                const int64_t row = row0 + (DIR == 0 ? (int64_t)(k0 + r) : -(int64_t)(k0 + r));
                reinterpret_cast<int4*>(st_base + row * a.L.spitch + a.L.owo + 2 * p0)[k] = v;
            }
            if (lane < n) off_base[(intptr_t)(k0 + lane) * off_step] = a_hold;
            __syncwarp();
        }
    };

    XP vb[P], vl[P];  // alpha (blank 2j, label 2j+1) / beta (label 2j-1, blank 2j)
#pragma unroll
    for (int p = 0; p < P; ++p) vb[p] = vl[p] = zero;
    // one recursion step with this frame's emissions.  The shuffle hands lane 0
    // (alpha) / lane 31 (beta) its own state: those lanes shadow pairs that
    // are either outside the target (zero, and zero feeds zero) or
    // overwritten at the next exchange.
    auto step = [&](const XP (&el)[P], const XP& eb) {
        XP nb;
        {
            const XP mine = DIR == 0 ? vl[P - 1] : vl[0];
            nb.m = DIR == 0 ? __shfl_up_sync(0xffffffffu, mine.m, 1) : __shfl_down_sync(0xffffffffu, mine.m, 1);
            nb.e = DIR == 0 ? __shfl_up_sync(0xffffffffu, mine.e, 1) : __shfl_down_sync(0xffffffffu, mine.e, 1);
        }
        float Sb[P], Sl[P];
        int Eb[P], El[P];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const XP o = DIR == 0 ? (p ? vl[p - 1] : nb) : (p < P - 1 ? vl[p + 1] : nb);
            xp_sum3(vl[p], vb[p], skip[p] ? o : zero, Sl[p], El[p]);
            xp_sum2(vb[p], o, Sb[p], Eb[p]);
        }
#pragma unroll
        for (int p = 0; p < P; ++p) {
            vl[p] = XP{Sl[p] * el[p].m, El[p] + el[p].e};
            vb[p] = XP{Sb[p] * eb.m, Eb[p] + eb.e};
            if (DIR == 0) {
                rx[p] = Sb[p];
                ex[p] = Eb[p];
                ry[p] = Sl[p];
                ey[p] = El[p];
            } else {
                rx[p] = vl[p].m;
                ex[p] = vl[p].e;
                ry[p] = vb[p].m;
                ey[p] = vb[p].e;
            }
        }
    };
    auto renormalise = [&]() {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            vb[p] = xp_norm(vb[p].m, vb[p].e);
            vl[p] = xp_norm(vl[p].m, vl[p].e);
        }
    };
    // halo exchange e: alpha sends its top shadowed lanes up, beta its bottom ones down
    auto exchange = [&](int e) {
        XP* buf = c.xch + (e & 1) * (c.nw * S::XW);
        const int qs = DIR == 0 ? lane - (32 - S::G) : lane;
        if (qs >= 0 && qs < S::G) {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                buf[c.w * S::XW + (qs * P + p) * 2] = vb[p];
                buf[c.w * S::XW + (qs * P + p) * 2 + 1] = vl[p];
            }
        }
        bar_named(1, nthreads);
        const int src = DIR == 0 ? c.w - 1 : c.w + 1;
        const int qr = DIR == 0 ? lane : lane - (32 - S::G);
        if (src >= 0 && src < c.nw && qr >= 0 && qr < S::G) {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                vb[p] = buf[src * S::XW + (qr * P + p) * 2];
                vl[p] = buf[src * S::XW + (qr * P + p) * 2 + 1];
            }
        }
    };

    // prologue: frames 0 .. R-2 requested (frame k into slot (k - 1) mod R)
#pragma unroll
    for (int k = 0; k < S::R - 1; ++k) request((uint32_t)((k + S::R - 1) & (S::R - 1)), k);

    // frame 0
    {
        cp_async_wait<S::R - 2>();
        XP el[P], eb;
        emissions(S::R - 1, el, eb);
        request(S::R - 2, S::R - 1);
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int j = j0 + p;
            if (DIR == 0) {
                vb[p] = j == 0 ? xp_norm(eb.m, eb.e) : zero;
                vl[p] = (j == 0 && U >= 1) ? xp_norm(el[p].m, el[p].e) : zero;
                // before the first emission the start states hold 1
                rx[p] = j == 0 ? 1.0f : 0.0f;
                ex[p] = j == 0 ? 0 : kEZero;
                ry[p] = (j == 0 && U >= 1) ? 1.0f : 0.0f;
                ey[p] = (j == 0 && U >= 1) ? 0 : kEZero;
            } else {
                vb[p] = j == U ? xp_norm(eb.m, eb.e) : zero;
                vl[p] = (j == U && U >= 1) ? xp_norm(el[p].m, el[p].e) : zero;
                rx[p] = vl[p].m;
                ex[p] = vl[p].e;
                ry[p] = vb[p].m;
                ey[p] = vb[p].e;
            }
        }
    }

    // full blocks: frames i0 .. i0+F-1, i0 = 1 mod F, in slots base .. base+F-1;
    // the request made at frame i goes to frame i-1's slot
    int i0 = 1;
#pragma unroll 1
    for (; i0 + S::F - 1 < T; i0 += S::F) {
        const uint32_t base = (uint32_t)((i0 - 1) & (S::R - 1));
#pragma unroll
        for (int q = 0; q < S::F; ++q) {
            cp_async_wait<S::R - 2>();
            XP el[P], eb;
            emissions(base + q, el, eb);
            request((base + q + S::R - 1) & (S::R - 1), i0 + q + S::R - 1);
            if (CKPT) {
                flush_ckpt(i0 + q - 1);
            } else if (STORE) {
                flush_row(q);  // frame i0 + q - 1
            }
            step(el, eb);
        }
        renormalise();
        if (multi) exchange((i0 - 1) / S::F);
        if (!CKPT && STORE) write_rows(i0 - 1, S::F);
    }
    // the last frames (fewer than F: no exchange needed)
#pragma unroll 1
    for (int i = i0; i < T; ++i) {
        cp_async_wait<S::R - 2>();
        XP el[P], eb;
        const uint32_t slot = (uint32_t)((i - 1) & (S::R - 1));
        emissions(slot, el, eb);
        request((slot + S::R - 1) & (S::R - 1), i + S::R - 1);
        if (CKPT) {
            flush_ckpt(i - 1);
        } else if (STORE) {
            flush_row(i - i0);  // frame i - 1
        }
        step(el, eb);
    }
    if (CKPT) {
        flush_ckpt(T - 1);
    } else if (STORE) {
        flush_row(T - i0);  // frame T - 1 (T >= 1 for every queued item)
        write_rows(i0 - 1, T - i0 + 1);
    }
    cp_async_wait<0>();
    renormalise();

    if (DIR == 0) {
        // the paths end in the last blank (pair U) or the last label (pair U-1)
        if (own) {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int j = j0 + p;
                if (j == U) c.fin[0] = vb[p];
                if (U >= 1 && j == U - 1) c.fin[1] = vl[p];
            }
        }
        if (multi) {
            bar_named(1, nthreads);
        } else {
            __syncwarp();
        }
        if (c.w == 0 && lane == 0) {
            const XP f0 = c.fin[0], f1 = c.fin[1];
            double v;
            UttInfo* uw = ws_at<UttInfo>(a.ws, a.L.off_utt) + b;
            int kint = 0, ninf = 0;
            float cfrac = __int_as_float(0x7fc00000);  // the backward's posterior factor, NaN unless nll is finite
            if (info.has_nan) {
                v = __longlong_as_double(0x7ff8000000000000ll);
            } else if (f0.m == 0.0f && f1.m == 0.0f) {
                v = __longlong_as_double(0x7ff0000000000000ll);  // no path: +inf
                ninf = 1;
            } else {
                const int Em = max(f0.e, f1.e);
                const double sum = (double)f0.m * exp2((double)(max(f0.e - Em, -1100))) +
                                   (double)f1.m * exp2((double)(max(f1.e - Em, -1100)));
                const double nl2 = -((double)Em + log2(sum));  // nll in bits
                v = nl2 * kLn2D;
                const double kf = floor(nl2);
                kint = (int)fmin(fmax(kf, -1.0e9), 1.0e9);
                cfrac = (float)exp2(nl2 - kf);
            }
            uw->kint = kint;
            uw->cfrac = cfrac;
            uw->nll_inf = ninf;
            nll_out[b] = v;
            if (a.reduction == CTC_PACKED_NONE) {
                float out = (float)v;
                if (a.zero_infinity && isinf(v)) out = 0.0f;
                a.loss[b] = out;
            }
        }
    }
}

template <int P, int G, bool CKPT>
__device__ __forceinline__ void run_item(const ChainArgs& a, int item, const ItemCtx& c) {
    if (CKPT || a.store_rows) {
        if (item & 1) {
            run_chain<P, G, 1, CKPT, true>(a, item >> 1, c);
        } else {
            run_chain<P, G, 0, CKPT, true>(a, item >> 1, c);
        }
    } else {
        if (item & 1) {
            run_chain<P, G, 1, CKPT, false>(a, item >> 1, c);
        } else {
            run_chain<P, G, 0, CKPT, false>(a, item >> 1, c);
        }
    }
}

}  // namespace

// MAXT: the most threads a CTA launches with.  An item of up to 8 warps runs
// under a 256-thread bound, which leaves the compiler room for ~120
// registers a thread instead of 64 (measured: 13 us faster on the 8193-class
// workload's 8-warp chains).
// CKPT: the chains keep only checkpoint rows (store_rows > 1), a kernel of
// its own so that the default one holds only the plain loop.
template <int P, int G, int MAXT, bool CKPT>
__global__ void __launch_bounds__(MAXT, 1) chain_kernel(ChainArgs a) {
    using S = ChainShape<P, G>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_item;
    __shared__ int s_last;
    __shared__ double s_red[32];
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const int32_t* queue = ws_at<int32_t>(a.ws, a.L.off_queue);
    const UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    pdl_wait();     // queue, metadata and emission matrix from the earlier kernels
    pdl_trigger();  // persistent grid: every CTA is already resident
    const int NT = blockDim.x, NW = NT >> 5;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    XP* rings = reinterpret_cast<XP*>(smem_raw);
    XP* xch = rings + NW * S::R * 32 * S::LW;
    XP* fins = xch + 2 * NW * S::XW;
    XP* my_ring = rings + warp * S::R * 32 * S::LW;
    // stages after the 2 * NW fin values, on a 16-byte boundary
    int* my_stage = reinterpret_cast<int*>(fins + 2 * NW) + warp * S::kStageInts;
    const int n_big = ctrl->n_big, n_small = ctrl->n_small;

    // 1. multi-warp chains, longest first, one at a time per CTA
    for (;;) {
        if (tid == 0) s_item = (int)atomicAdd(&ctrl->big_head, 1u);
        __syncthreads();
        const int k = s_item;
        __syncthreads();
        if (k >= n_big) break;
        const int item = queue[k];
        const int U = utt[item >> 1].U;
        const int nw = min(NW, (U + 1 + S::GP - 1) / S::GP);
        if (warp < nw) run_item<P, G, CKPT>(a, item, ItemCtx{warp, nw, my_ring, xch, fins, my_stage});
    }
    // 2. single-warp chains, each warp on its own
    for (;;) {
        int k = 0;
        if (lane == 0) k = (int)atomicAdd(&ctrl->small_head, 1u);
        k = __shfl_sync(0xffffffffu, k, 0);
        if (k >= n_small) break;
        run_item<P, G, CKPT>(a, queue[n_big + k], ItemCtx{0, 1, my_ring, xch, fins + 2 * warp, my_stage});
    }
    // 3. (the label analysis of the backward runs in the emission gather's kernel)
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
        if (a.reduction == CTC_PACKED_MEAN || a.reduction == CTC_PACKED_MEAN_BATCH)
            total = B > 0 ? total / (double)B : __longlong_as_double(0x7ff8000000000000ll);
        if (a.reduction == CTC_PACKED_MEAN_VOLUME) total = total / (double)ctrl->tl_total;  // x / 0: inf or NaN
        a.loss[0] = (float)total;
    }
}

template __global__ void chain_kernel<1, 8, 256, false>(ChainArgs);
template __global__ void chain_kernel<1, 8, 512, false>(ChainArgs);
template __global__ void chain_kernel<2, 4, 512, false>(ChainArgs);
template __global__ void chain_kernel<2, 2, 512, false>(ChainArgs);
template __global__ void chain_kernel<2, 2, 1024, false>(ChainArgs);
template __global__ void chain_kernel<4, 1, 1024, false>(ChainArgs);
template __global__ void chain_kernel<1, 8, 256, true>(ChainArgs);
template __global__ void chain_kernel<1, 8, 512, true>(ChainArgs);
template __global__ void chain_kernel<2, 4, 512, true>(ChainArgs);
template __global__ void chain_kernel<2, 2, 512, true>(ChainArgs);
template __global__ void chain_kernel<2, 2, 1024, true>(ChainArgs);
template __global__ void chain_kernel<4, 1, 1024, true>(ChainArgs);

template <int P, int G, int MAXT, bool CKPT>
static cudaError_t launch_chain_c(const ChainArgs& a, cudaStream_t s) {
    using S = ChainShape<P, G>;
    const int nw = a.L.nwo;  // warps for the longest possible target
    const size_t smem = sizeof(XP) * ((size_t)nw * S::R * 32 * S::LW + 2 * (size_t)nw * S::XW + 2 * (size_t)nw) +
                        sizeof(int) * (size_t)nw * S::kStageInts;
    cudaError_t e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    // set on every call (on the current device): a cached value could go
    // stale between host threads launching with different sizes
    e = cudaFuncSetAttribute(chain_kernel<P, G, MAXT, CKPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_kernel<P, G, MAXT, CKPT>, 32 * nw, smem)) !=
        cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    // persistent grid: enough CTAs for every item, never more than fit at once
    long long want = 2ll * a.L.B;
    long long grid = (long long)sms * per_sm;
    if (want < grid) grid = want > 0 ? want : 1;
    return launch_pdl(chain_kernel<P, G, MAXT, CKPT>, dim3((unsigned)grid), dim3(32 * nw), smem, s, a);
}

template <int P, int G, int MAXT>
static cudaError_t launch_chain_t(const ChainArgs& a, cudaStream_t s) {
    return a.store_rows > 1 ? launch_chain_c<P, G, MAXT, true>(a, s) : launch_chain_c<P, G, MAXT, false>(a, s);
}

cudaError_t launch_chain(const ChainArgs& a, cudaStream_t s) {
    // the smallest thread bound that holds the chain's warps: fewer threads
    // a CTA, more registers a thread
    int P, G;
    chain_shape_for_max_u(a.L.max_U, P, G);
    if (P == 1) return a.L.nwo <= 8 ? launch_chain_t<1, 8, 256>(a, s) : launch_chain_t<1, 8, 512>(a, s);
    if (P == 2 && G == 4) return launch_chain_t<2, 4, 512>(a, s);
    if (P == 2) return a.L.nwo <= 16 ? launch_chain_t<2, 2, 512>(a, s) : launch_chain_t<2, 2, 1024>(a, s);
    return launch_chain_t<4, 1, 1024>(a, s);
}

}  // namespace ctcp
