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
// Arithmetic: the recursion runs on probabilities in extended range (a float
// mantissa and an int32 binary exponent per state, see ctc_common.cuh):
// alpha_t(s) = (alpha_{t-1}(s) + alpha_{t-1}(s-1) + [skip] alpha_{t-1}(s-2)) * p_t(s),
// i.e. only multiply-adds and integer exponent arithmetic on the critical
// path, no exp or log, no cross-warp normalisation.
//
// What is stored for the backward, as int32 fixed-point log2 values with 19
// fraction bits relative to a per-(frame, warp) integer offset (the warp's
// largest exponent, stored per frame in aoff / boff): alpha rows hold the
// value *before* the frame's emission, alpha_t(s) / p_t(s), so the backward
// needs no log-probability gather; beta rows hold beta_t(s).  The posterior
// is then an exact integer sum plus one ex2.
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
    float* halo;     // [2][nw] extended values (m, e)   (CTA mode)
    float* fin;      // 2 extended values private to the group
};

template <bool CTA>
__device__ __forceinline__ void group_sync() {
    if constexpr (CTA) {
        __syncthreads();
    } else {
        __syncwarp();
    }
}

template <int DT>
__device__ __forceinline__ uintptr_t word_of(uintptr_t addr) {
    if constexpr (DT == 0) {
        return addr;
    } else {
        return addr & ~uintptr_t(3);
    }
}

// Copy the 4-byte word holding element `addr` into the ring slot `dst`.  The
// buffer starts 4-byte aligned, so the word never starts before it; a word
// that would run past its end copies only the element's 2 bytes (cp.async
// zero-fills the rest).  `live` false copies nothing (the address is then a
// valid one that is not read).
template <int DT>
__device__ __forceinline__ void gather(uint32_t dst, uintptr_t addr, uintptr_t hi, bool live) {
    const uintptr_t w = word_of<DT>(addr);
    int n = 4;
    if constexpr (DT != 0) n = (w + 4 <= hi) ? 4 : 2;
    n = live ? n : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(w), "r"(n) : "memory");
}

template <int P, int DT, bool CTA>
__device__ void run_chain_item(const ChainArgs& a, int item, const Group& g) {
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const UttInfo info = ws_at<UttInfo>(a.ws, a.L.off_utt)[item >> 1];
    double* nll_out = ws_at<double>(a.ws, a.L.off_nll);
    const int b = item >> 1;
    const int dir = item & 1;  // 0 alpha, 1 beta
    const int T = info.T, U = info.U;
    const int lane = g.tid & 31;
    const int32_t* tg = a.targets + info.toff;
    constexpr int E = Elem<DT>::bytes;

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
        if (has_label[p] && (cls[p] < 0 || cls[p] >= a.D)) bad = true;
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

    // gather streams: frame 0 is row start (alpha) or row start + T - 1 (beta)
    const uintptr_t buf_lo = reinterpret_cast<uintptr_t>(a.lp);
    const uintptr_t buf_hi = buf_lo + (uintptr_t)a.lp_bytes;
    const int64_t row0 = dir == 0 ? (int64_t)info.start : (int64_t)info.start + T - 1;
    const intptr_t step_bytes = (dir == 0 ? 1 : -1) * (intptr_t)a.D * E;
    const int d_odd = (E == 2) ? (a.D & 1) : 0;
    uintptr_t gnext[P], gfirst[P];
    int half0[P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
        gfirst[p] = gnext[p] = buf_lo + (uintptr_t)((row0 * a.D + cls[p]) * E);
        half0[p] = (int)((gfirst[p] >> 1) & 1);
    }
    const uintptr_t bfirst = buf_lo + (uintptr_t)((row0 * a.D + a.blank) * E);
    uintptr_t bnext = bfirst;
    const int bhalf0 = (int)((bfirst >> 1) & 1);

    const int SS = g.n * P + 1;  // words per ring slot: P label words per thread, then the blank
    const uint32_t ring_s = smem_addr(g.ring);
    auto issue = [&](int k) {
        const bool live = k < T;
        const uint32_t slot = ring_s + (uint32_t)((k & (kRing - 1)) * SS) * 4u;
#pragma unroll
        for (int p = 0; p < P; ++p) {
            gather<DT>(slot + (uint32_t)(p * g.n + g.tid) * 4u, live ? gnext[p] : gfirst[p], buf_hi,
                       live && has_label[p]);
            gnext[p] += live ? step_bytes : 0;
        }
        if (g.tid == 0) gather<DT>(slot + (uint32_t)(g.n * P) * 4u, live ? bnext : bfirst, buf_hi, live);
        bnext += live ? step_bytes : 0;
        cp_async_commit();
    };
    // emissions of step k as extended probabilities; a NaN log probability is remembered
    bool saw_nan = false;
    auto consume = [&](int k, XP& eb, XP (&el)[P]) {
        const uint32_t* slot = g.ring + (k & (kRing - 1)) * SS;
        const int flip = d_odd & k;  // with D odd a 2-byte element changes halves every frame
        const float lb = word_to_float<DT>(slot[g.n * P], bhalf0 ^ flip);
        saw_nan |= lb != lb;
        eb = xp_from_log(lb);
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const float ll = word_to_float<DT>(slot[p * g.n + g.tid], half0[p] ^ flip);
            saw_nan |= has_label[p] && ll != ll;
            el[p] = has_label[p] ? xp_from_log(ll) : XP{0.0f, kEZero};
        }
    };

    const int j0 = g.tid * P;
    const bool store_me = j0 <= U;
    int* st = ws_at<int>(a.ws, dir == 0 ? a.L.off_alpha : a.L.off_beta) + row0 * a.L.pitch + 2 * j0;
    const intptr_t st_step = (dir == 0 ? 1 : -1) * (intptr_t)a.L.pitch;
    int32_t* offp = ws_at<int32_t>(a.ws, dir == 0 ? a.L.off_aoff : a.L.off_boff) + row0 * a.L.nwo +
                    (CTA ? g.warp : 0);
    const intptr_t off_step = (dir == 0 ? 1 : -1) * (intptr_t)a.L.nwo;
    auto store_row = [&](const int (&x)[P], const int (&y)[P], int A) {
        if (store_me) {
            if constexpr (P == 1) {
                *reinterpret_cast<int2*>(st) = make_int2(x[0], y[0]);
            } else {
#pragma unroll
                for (int p = 0; p < P; p += 2)
                    *reinterpret_cast<int4*>(st + 2 * p) = make_int4(x[p], y[p], x[p + 1], y[p + 1]);
            }
        }
        if (lane == 0) *offp = A;
        st += st_step;
        offp += off_step;
    };
    XP* halo = reinterpret_cast<XP*>(g.halo);
    const XP zero{0.0f, kEZero};

    // prologue: kRing-1 frames in flight
#pragma unroll 1
    for (int k = 0; k < kRing - 1; ++k) issue(k);

    XP vb[P], vl[P];  // alpha (blank 2j, label 2j+1) / beta (label 2j-1, blank 2j), extended probabilities
    XP eb_cur, el_cur[P], eb_nxt, el_nxt[P];

    // step 0 (frames 0 and 1 have landed)
    cp_async_wait<kRing - 3>();
    group_sync<CTA>();
    consume(0, eb_cur, el_cur);
    consume(1, eb_nxt, el_nxt);
    {
        int x[P], y[P];
        int emax = kEZero;
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int j = j0 + p;
            if (dir == 0) {
                vb[p] = j == 0 ? eb_cur : zero;
                vl[p] = (j == 0 && U >= 1) ? el_cur[p] : zero;
            } else {
                vb[p] = j == U ? eb_cur : zero;
                vl[p] = (j == U && U >= 1) ? el_cur[p] : zero;
            }
            vb[p] = xp_norm(vb[p].m, vb[p].e);
            vl[p] = xp_norm(vl[p].m, vl[p].e);
            emax = max(emax, max(vb[p].e, vl[p].e));
        }
        if constexpr (CTA) {
            if (dir == 0 && lane == 31) halo[g.warp] = vl[P - 1];
            if (dir == 1 && lane == 0) halo[g.warp] = vl[0];
        }
        const int A = dir == 0 ? 0 : __reduce_max_sync(0xffffffffu, emax);
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int j = j0 + p;
            if (dir == 0) {  // before the emission the two start states have probability 1
                x[p] = j == 0 ? 0 : kFixZero;
                y[p] = (j == 0 && U >= 1) ? 0 : kFixZero;
            } else {
                x[p] = fix_log2(vl[p].m, vl[p].e, A);
                y[p] = fix_log2(vb[p].m, vb[p].e, A);
            }
        }
        store_row(x, y, A);
    }
    issue(kRing - 1);

#pragma unroll 1
    for (int i = 1; i < T; ++i) {
        cp_async_wait<kRing - 3>();  // frames i and i+1 have landed
        group_sync<CTA>();
        eb_cur = eb_nxt;
#pragma unroll
        for (int p = 0; p < P; ++p) el_cur[p] = el_nxt[p];
        // the label state just below (alpha) or above (beta) my pairs, previous frame
        XP nb;
        {
            const int src = dir == 0 ? max(g.warp - 1, 0) : min(g.warp + 1, g.nw - 1);
            const XP h = CTA ? halo[((i - 1) & 1) * g.nw + src] : zero;
            const bool edge = dir == 0 ? (lane == 0) : (lane == 31);
            const bool has_nb = CTA && (dir == 0 ? g.warp > 0 : g.warp < g.nw - 1);
            const XP mine = dir == 0 ? vl[P - 1] : vl[0];
            nb.m = dir == 0 ? __shfl_up_sync(0xffffffffu, mine.m, 1) : __shfl_down_sync(0xffffffffu, mine.m, 1);
            nb.e = dir == 0 ? __shfl_up_sync(0xffffffffu, mine.e, 1) : __shfl_down_sync(0xffffffffu, mine.e, 1);
            if (edge) nb = has_nb ? h : zero;
        }
        float Sb[P], Sl[P];
        int Eb[P], El[P];
        if (dir == 0) {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const XP prev = p ? vl[p - 1] : nb;
                xp_sum3(vl[p], vb[p], skip[p] ? prev : zero, Sl[p], El[p]);
                xp_sum2(vb[p], prev, Sb[p], Eb[p]);
            }
        } else {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const XP next = (p < P - 1) ? vl[p + 1] : nb;
                xp_sum3(vl[p], vb[p], skip[p] ? next : zero, Sl[p], El[p]);
                xp_sum2(vb[p], next, Sb[p], Eb[p]);
            }
        }
#pragma unroll
        for (int p = 0; p < P; ++p) {
            vl[p] = xp_norm(Sl[p] * el_cur[p].m, El[p] + el_cur[p].e);
            vb[p] = xp_norm(Sb[p] * eb_cur.m, Eb[p] + eb_cur.e);
        }
        if constexpr (CTA) {  // the critical value first: the neighbour warp waits for it
            if (dir == 0 && lane == 31) halo[(i & 1) * g.nw + g.warp] = vl[P - 1];
            if (dir == 1 && lane == 0) halo[(i & 1) * g.nw + g.warp] = vl[0];
        }
        // off the critical path: the next frame's emissions, the stored rows, the next gather
        consume(i + 1, eb_nxt, el_nxt);
        int emax = kEZero;
#pragma unroll
        for (int p = 0; p < P; ++p) emax = dir == 0 ? max(emax, max(Eb[p], El[p])) : max(emax, max(vb[p].e, vl[p].e));
        const int A = __reduce_max_sync(0xffffffffu, emax);
        int x[P], y[P];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            if (dir == 0) {  // alpha rows: before the emission
                x[p] = fix_log2(Sb[p], Eb[p], A);
                y[p] = fix_log2(Sl[p], El[p], A);
            } else {
                x[p] = fix_log2(vl[p].m, vl[p].e, A);
                y[p] = fix_log2(vb[p].m, vb[p].e, A);
            }
        }
        store_row(x, y, A);
        issue(i + kRing - 1);
    }

    if (dir == 0) {
        // the paths end in the last blank (pair U) or the last label (pair U-1)
        XP* fin = reinterpret_cast<XP*>(g.fin);
        if (g.tid == 0) {
            fin[0] = XP{0.0f, kEZero};
            fin[1] = XP{0.0f, kEZero};
        }
        group_sync<CTA>();
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int j = j0 + p;
            if (j == U) fin[0] = vb[p];
            if (U >= 1 && j == U - 1) fin[1] = vl[p];
        }
        bool any_nan;
        if constexpr (CTA) {
            any_nan = __syncthreads_or(saw_nan);
        } else {
            any_nan = __any_sync(0xffffffffu, saw_nan);
            __syncwarp();
        }
        if (g.tid == 0) {
            const XP f0 = fin[0], f1 = fin[1];
            double v;
            if (any_nan) {
                v = __longlong_as_double(0x7ff8000000000000ll);
            } else if (f0.m == 0.0f && f1.m == 0.0f) {
                v = __longlong_as_double(0x7ff0000000000000ll);  // no path: +inf
            } else {
                const int Em = max(f0.e, f1.e);
                const double s = (double)f0.m * exp2((double)(max(f0.e - Em, -1100))) +
                                 (double)f1.m * exp2((double)(max(f1.e - Em, -1100)));
                v = -((double)Em + log2(s)) * kLn2D;
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

// A multi-warp chain item, split by role.  Consumer warps (the first nwc)
// hold the state pairs and run the recursion; producer warps gather each
// frame's label and blank words kRawFrames-1 frames ahead with cp.async
// (a raw ring), turn them into extended-range emissions one frame ahead of
// use (a converted ring) and leave the consumers nothing but the
// recursion, the halo exchange and the stores.  One CTA barrier per frame
// orders both rings.
constexpr int kRawFrames = 16;
constexpr int kConvFrames = 2;

template <int P, int DT>
__device__ void run_chain_item_split(const ChainArgs& a, int item, int nwc, unsigned char* smem) {
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const UttInfo info = ws_at<UttInfo>(a.ws, a.L.off_utt)[item >> 1];
    double* nll_out = ws_at<double>(a.ws, a.L.off_nll);
    const int b = item >> 1;
    const int dir = item & 1;  // 0 alpha, 1 beta
    const int T = info.T, U = info.U;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NC = 32 * nwc;                 // consumer threads
    const int NP = (int)blockDim.x - NC;     // producer threads
    const bool consumer = tid < NC;
    const int ptid = tid - NC;
    const int32_t* tg = a.targets + info.toff;
    constexpr int E = Elem<DT>::bytes;
    const int W = a.L.max_U + 1;  // words per frame in the rings: labels 0..U-1, the blank at U
    uint32_t* raw = reinterpret_cast<uint32_t*>(smem);
    XP* conv = reinterpret_cast<XP*>(smem + sizeof(uint32_t) * kRawFrames * W);
    XP* halo = conv + kConvFrames * W;  // [2][nwc]
    XP* fin = halo + 2 * 32;

    // consumers: labels of the pairs and their skip transitions
    bool has_label[P], skip[P];
    bool bad = false;
    const int j0 = consumer ? tid * P : 0;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int j = j0 + p;
        has_label[p] = false;
        skip[p] = false;
        if (consumer) {
            if (dir == 0) {  // (blank 2j, label 2j+1 = l_j)
                has_label[p] = j < U;
                skip[p] = j >= 1 && j < U && tg[j] != tg[j - 1];
            } else {  // (label 2j-1 = l_{j-1}, blank 2j)
                has_label[p] = j >= 1 && j <= U;
                skip[p] = j >= 1 && j < U && tg[j - 1] != tg[j];
            }
        }
    }
    // producers: the words they gather, and a range check of every label
    for (int w = consumer ? U + 1 : ptid; w < U; w += NP) {
        const int c = tg[w];
        if (c < 0 || c >= a.D) bad = true;
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        if (tid == 0) {
            set_status(ctrl, CTC_PACKED_DEV_LABEL_OUT_OF_RANGE);
            if (dir == 0) {
                nll_out[b] = __longlong_as_double(0x7ff8000000000000ll);
                if (a.reduction == CTC_PACKED_NONE) a.loss[b] = __int_as_float(0x7fc00000);
            }
        }
        __syncthreads();
        return;
    }

    // producer streams: frame k is row start + k (alpha) or start + T - 1 - k (beta).  A
    // producer thread owns the words w = ptid and ptid + NP (at most two; the blank is word U)
    const uintptr_t buf_lo = reinterpret_cast<uintptr_t>(a.lp);
    const uintptr_t buf_hi = buf_lo + (uintptr_t)a.lp_bytes;
    const int64_t row0 = dir == 0 ? (int64_t)info.start : (int64_t)info.start + T - 1;
    const intptr_t step_bytes = (dir == 0 ? 1 : -1) * (intptr_t)a.D * E;
    const int d_odd = (E == 2) ? (a.D & 1) : 0;
    const uint32_t raw_s = smem_addr(raw);
    bool saw_nan = false;
    bool own[2];
    uintptr_t gfirst[2], gnext[2];
    int half0[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int w = ptid + q * NP;
        own[q] = !consumer && w <= U;
        const int c = own[q] ? (w < U ? tg[w] : a.blank) : a.blank;
        gfirst[q] = gnext[q] = buf_lo + (uintptr_t)((row0 * a.D + c) * E);
        half0[q] = (int)((gfirst[q] >> 1) & 1);
    }
    auto issue_raw = [&](int k) {
        if (!consumer) {
            const bool live = k < T;
            const uint32_t slot = raw_s + (uint32_t)((k & (kRawFrames - 1)) * W) * 4u;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                if (own[q]) gather<DT>(slot + (uint32_t)(ptid + q * NP) * 4u, live ? gnext[q] : gfirst[q], buf_hi, live);
                gnext[q] += live ? step_bytes : 0;
            }
            cp_async_commit();
        }
    };
    auto convert = [&](int k) {  // raw frame k -> converted ring
        if (!consumer && k < T) {
            const uint32_t* rs = raw + (k & (kRawFrames - 1)) * W;
            XP* cs = conv + (k % kConvFrames) * W;
            const int flip = d_odd & k;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                if (own[q]) {
                    const int w = ptid + q * NP;
                    const float x = word_to_float<DT>(rs[w], half0[q] ^ flip);
                    saw_nan |= x != x;
                    cs[w] = xp_from_log(x);
                }
            }
        }
    };

    const bool store_me = consumer && j0 <= U;
    int* st = ws_at<int>(a.ws, dir == 0 ? a.L.off_alpha : a.L.off_beta) + row0 * a.L.pitch + 2 * j0;
    const intptr_t st_step = (dir == 0 ? 1 : -1) * (intptr_t)a.L.pitch;
    int32_t* offp = ws_at<int32_t>(a.ws, dir == 0 ? a.L.off_aoff : a.L.off_boff) + row0 * a.L.nwo + warp;
    const intptr_t off_step = (dir == 0 ? 1 : -1) * (intptr_t)a.L.nwo;
    auto store_row = [&](const int (&x)[P], const int (&y)[P], int A) {
        if (store_me) {
            if constexpr (P == 1) {
                *reinterpret_cast<int2*>(st) = make_int2(x[0], y[0]);
            } else {
#pragma unroll
                for (int p = 0; p < P; p += 2)
                    *reinterpret_cast<int4*>(st + 2 * p) = make_int4(x[p], y[p], x[p + 1], y[p + 1]);
            }
        }
        if (lane == 0) *offp = A;
        st += st_step;
        offp += off_step;
    };
    const XP zero{0.0f, kEZero};
    // emissions of frame k for my pairs, from the converted ring
    auto emissions = [&](int k, XP& eb, XP (&el)[P]) {
        const XP* cs = conv + (k % kConvFrames) * W;
        eb = cs[U];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int j = j0 + p;
            const int w = dir == 0 ? j : j - 1;
            el[p] = has_label[p] ? cs[w] : zero;
        }
    };

    // prologue: raw frames 0 .. kRawFrames-2 in flight, frames 0 .. kConvFrames-2 converted
#pragma unroll 1
    for (int k = 0; k < kRawFrames - 1; ++k) issue_raw(k);
    if (!consumer) {
        cp_async_wait<kRawFrames - kConvFrames>();
        for (int k = 0; k < kConvFrames - 1; ++k) convert(k);
    }

    XP vb[P], vl[P];
#pragma unroll 1
    for (int i = 0; i < T; ++i) {
        __syncthreads();
        if (!consumer) {
            // producers: frame i + kConvFrames - 1 into the converted ring, frame i + kRawFrames - 1 requested
            cp_async_wait<kRawFrames - kConvFrames - 1>();
            convert(i + kConvFrames - 1);
            issue_raw(i + kRawFrames - 1);
            continue;
        }
        XP eb, el[P];
        emissions(i, eb, el);
        if (i == 0) {
            int x[P], y[P];
            int emax = kEZero;
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int j = j0 + p;
                if (dir == 0) {
                    vb[p] = j == 0 ? eb : zero;
                    vl[p] = (j == 0 && U >= 1) ? el[p] : zero;
                } else {
                    vb[p] = j == U ? eb : zero;
                    vl[p] = (j == U && U >= 1) ? el[p] : zero;
                }
                vb[p] = xp_norm(vb[p].m, vb[p].e);
                vl[p] = xp_norm(vl[p].m, vl[p].e);
                emax = max(emax, max(vb[p].e, vl[p].e));
            }
            if (dir == 0 && lane == 31) halo[warp] = vl[P - 1];
            if (dir == 1 && lane == 0) halo[warp] = vl[0];
            const int A = dir == 0 ? 0 : __reduce_max_sync(0xffffffffu, emax);
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int j = j0 + p;
                if (dir == 0) {
                    x[p] = j == 0 ? 0 : kFixZero;
                    y[p] = (j == 0 && U >= 1) ? 0 : kFixZero;
                } else {
                    x[p] = fix_log2(vl[p].m, vl[p].e, A);
                    y[p] = fix_log2(vb[p].m, vb[p].e, A);
                }
            }
            store_row(x, y, A);
            continue;
        }
        // the label state just below (alpha) or above (beta) my pairs, previous frame
        XP nb;
        {
            const int src = dir == 0 ? max(warp - 1, 0) : min(warp + 1, nwc - 1);
            const XP h = halo[((i - 1) & 1) * nwc + src];
            const bool edge = dir == 0 ? (lane == 0) : (lane == 31);
            const bool has_nb = dir == 0 ? warp > 0 : warp < nwc - 1;
            const XP mine = dir == 0 ? vl[P - 1] : vl[0];
            nb.m = dir == 0 ? __shfl_up_sync(0xffffffffu, mine.m, 1) : __shfl_down_sync(0xffffffffu, mine.m, 1);
            nb.e = dir == 0 ? __shfl_up_sync(0xffffffffu, mine.e, 1) : __shfl_down_sync(0xffffffffu, mine.e, 1);
            if (edge) nb = has_nb ? h : zero;
        }
        float Sb[P], Sl[P];
        int Eb[P], El[P];
        if (dir == 0) {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const XP prev = p ? vl[p - 1] : nb;
                xp_sum3(vl[p], vb[p], skip[p] ? prev : zero, Sl[p], El[p]);
                xp_sum2(vb[p], prev, Sb[p], Eb[p]);
            }
        } else {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const XP next = (p < P - 1) ? vl[p + 1] : nb;
                xp_sum3(vl[p], vb[p], skip[p] ? next : zero, Sl[p], El[p]);
                xp_sum2(vb[p], next, Sb[p], Eb[p]);
            }
        }
#pragma unroll
        for (int p = 0; p < P; ++p) {
            vl[p] = xp_norm(Sl[p] * el[p].m, El[p] + el[p].e);
            vb[p] = xp_norm(Sb[p] * eb.m, Eb[p] + eb.e);
        }
        if (dir == 0 && lane == 31) halo[(i & 1) * nwc + warp] = vl[P - 1];
        if (dir == 1 && lane == 0) halo[(i & 1) * nwc + warp] = vl[0];
        int emax = kEZero;
#pragma unroll
        for (int p = 0; p < P; ++p) emax = dir == 0 ? max(emax, max(Eb[p], El[p])) : max(emax, max(vb[p].e, vl[p].e));
        const int A = __reduce_max_sync(0xffffffffu, emax);
        int x[P], y[P];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            if (dir == 0) {  // alpha rows: before the emission
                x[p] = fix_log2(Sb[p], Eb[p], A);
                y[p] = fix_log2(Sl[p], El[p], A);
            } else {
                x[p] = fix_log2(vl[p].m, vl[p].e, A);
                y[p] = fix_log2(vb[p].m, vb[p].e, A);
            }
        }
        store_row(x, y, A);
    }

    const bool any_nan = __syncthreads_or(saw_nan);
    if (dir == 0) {
        // the paths end in the last blank (pair U) or the last label (pair U-1)
        if (tid == 0) {
            fin[0] = zero;
            fin[1] = zero;
        }
        __syncthreads();
        if (consumer) {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int j = j0 + p;
                if (j == U) fin[0] = vb[p];
                if (U >= 1 && j == U - 1) fin[1] = vl[p];
            }
        }
        __syncthreads();
        if (tid == 0) {
            const XP f0 = fin[0], f1 = fin[1];
            double v;
            if (any_nan) {
                v = __longlong_as_double(0x7ff8000000000000ll);
            } else if (f0.m == 0.0f && f1.m == 0.0f) {
                v = __longlong_as_double(0x7ff0000000000000ll);  // no path: +inf
            } else {
                const int Em = max(f0.e, f1.e);
                const double sum = (double)f0.m * exp2((double)(max(f0.e - Em, -1100))) +
                                   (double)f1.m * exp2((double)(max(f1.e - Em, -1100)));
                v = -((double)Em + log2(sum)) * kLn2D;
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
    __syncthreads();
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
    float* fin = halo + 4 * NW;  // 2 extended values per warp
    const int n_big = ctrl->n_big, n_small = ctrl->n_small, n_lab = ctrl->n_lab;

    // 1. multi-warp chains, longest first, one at a time per CTA
    for (;;) {
        if (tid == 0) s_item = (int)atomicAdd(&ctrl->big_head, 1u);
        __syncthreads();
        const int k = s_item;
        __syncthreads();
        if (k >= n_big) break;
        if (P == 1 && a.consumer_warps < NW) {
            run_chain_item_split<P, DT>(a, queue[k], a.consumer_warps, smem_raw);
        } else {  // every warp holds pairs and gathers its own columns
            Group cg{tid, NT, warp, NW, ring, halo, fin};
            run_chain_item<P, DT, true>(a, queue[k], cg);
        }
    }
    // 2. single-warp chains, each warp on its own
    Group wg{lane, 32, warp, NW, ring + warp * kRing * (32 * P + 1), halo, fin + 4 * warp};
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

int chain_pairs_per_thread(int max_target_len) { return pairs_for_max_u(max_target_len); }

int chain_warps(int max_target_len, int P) {
    const int pairs = max_target_len + 1;
    int nw = (pairs + 32 * P - 1) / (32 * P);
    return nw < 1 ? 1 : (nw > 30 ? 30 : nw);
}

static size_t chain_smem_bytes(int P, int nw, int max_u) {
    const int nt = 32 * nw;
    const size_t warp_mode = sizeof(uint32_t) * (size_t)kRing * (nt * P + nw) + sizeof(float) * (size_t)(4 * nw + 4 * nw);
    const size_t W = (size_t)max_u + 1;
    const size_t split = P == 1 ? sizeof(uint32_t) * kRawFrames * W + sizeof(XP) * (kConvFrames * W + 2 * 32 + 2) : 0;
    return warp_mode > split ? warp_mode : split;
}

// Producer warps a chain CTA gets: enough that each producer thread owns at
// most two of the max_U + 1 columns, when consumers and producers fit 32 warps.
static int producer_warps(int P, int nwc, int max_u) {
    if (P != 1) return 0;
    const int nwp = (max_u + 1 + 63) / 64;
    return nwc + nwp <= 32 ? nwp : 0;
}

template <int P, int DT>
static cudaError_t launch_chain_t(const ChainArgs& a0, int nwc, cudaStream_t s) {
    ChainArgs a = a0;
    a.consumer_warps = nwc;
    const int nw = nwc + producer_warps(P, nwc, a.L.max_U);
    static int configured_smem = -1;
    const size_t smem = chain_smem_bytes(P, nw, a.L.max_U);
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
#undef CTCP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace ctcp
