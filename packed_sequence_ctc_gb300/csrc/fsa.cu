// Full-sum loss over a generic FSA on the packed layout: the topology the
// CTC kernels build into their recursion, given instead as an edge list.
//
// Page "feat(asr): native CTC loss kernel over sequence-packed log
// probabilities", ctc_loss.py, module docstring: the packed CTC loss follows
// RETURNN's packed full-sum loss over a generic FSA edge list (scores
// addressed in the token-flat buffer through per-sequence start offsets,
// posteriors scattered back into a buffer of the same layout, the gradient
// exp(log_probs) - posterior masked per frame); it differs by building the
// CTC topology into the recursion.  This file is that generic form.
//
// Sequence b owns states [state_offsets[b], state_offsets[b+1]) of the start
// and final weight arrays (log weights, -inf: none) and edges
// [edge_offsets[b], edge_offsets[b+1]) of (from, to, label) with a log
// weight each, state ids local to the sequence; every edge consumes one
// frame.  With lp the sequence's rows:
//   alpha_0(s) = start(s),  alpha_{t+1}(s') = logsumexp_{e=(s,s',c,w)} alpha_t(s) + w + lp[t, c]
//   Z = logsumexp_s alpha_T(s) + final(s),  loss = -Z
//   beta_T(s) = final(s),   beta_t(s) = logsumexp_{e=(s,s',c,w)} w + lp[t, c] + beta_{t+1}(s')
//   grad[t, c] = scale * (exp(lp[t, c]) - sum_{e with label c} exp(alpha_t(s) + w + lp[t, c] + beta_{t+1}(s') - Z))
//
// The recursions carry every value in extended range, as the CTC chain
// does: a float mantissa and an int exponent (exp of a log weight or log
// probability via xp_from_log).  An edge's term is the product of three such
// values and a sum aligns its terms to the largest exponent, so a frame needs
// no shift, no exp and no log; Z keeps its exponent, and an occupancy is a
// product divided by Z, formed directly as a float.  Every sum runs in a
// fixed order, so results are bitwise reproducible:
//   index    one CTA per sequence, once per forward: the edges sorted stably
//            (counting sort; ties keep the edge order) by destination, by
//            source and by label, as per-state and per-label lists; the
//            sequence's distinct labels (at most max_labels) in increasing
//            order, and each edge's slot among them.
//   chain    (the forward call) 2B CTAs: CTA b runs sequence b's forward
//            recursion, CTA B + b its backward recursion at the same time.
//            A thread per state (or a few): alpha_{t+1}(s') is the sum over
//            the state's incoming edges in list order, beta_t(s) over its
//            outgoing edges.  The words holding the next frame's label
//            values are copied ahead and converted to extended range during
//            the frame by label threads (warps of their own after the state
//            threads when they fit the CTA), each converting the words it
//            copied; one barrier per frame.  Every alpha_t and beta_t row is
//            stored (8 bytes a state), and the backward recursion also keeps
//            each frame's label values.
//   post     (the backward call) a CTA per row at a time over a contiguous
//            range of rows: the row's alpha_t, beta_{t+1} and label values
//            copied into shared memory (the next row's copies in flight
//            meanwhile), then each label's class sum over its contiguous
//            range of edges in label order, each occupancy formed as it is
//            summed (short lists by a thread, long ones by a warp); the dense
//            rows are written by the CTC path's all-SM gradient stream from
//            the rows' class sums.
#include <cstdint>

#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

constexpr int kIdxThreads = 256;      // threads of the index kernel
constexpr int kFsaMaxThreads = 512;   // threads of a recursion CTA (states per thread <= 8); the
                                      // recursions are declared for one CTA an SM: left free, the
                                      // compiler trades registers for occupancy (40 with spills),
                                      // and one CTA's frame chain ran 1.9 times slower
constexpr int kFsaSmemBudget = 200 * 1024;  // shared memory of a recursion CTA, edge lists included
constexpr int kFsaSmemLimit = 224 * 1024;   // its per-frame buffers alone (larger plans are rejected)
constexpr int kShortList = 8;         // label lists up to this long are summed by one thread, longer by a warp

// Workspace of the FSA path.  Per sequence: log Z (double), Z in extended
// range, and the number of distinct labels (-1: the sequence was rejected);
// per frame: the forward and backward values of every state in extended
// range and the frame's label values; per row: the class-sum header and sums
// read by the gradient stream; per state: offsets of its incoming and
// outgoing edge lists; per edge: the records of both lists, each edge's
// position in label order and its record at that position.
struct FsaLayout {
    size_t off_z, off_nlab, off_zx, off_alpha, off_beta, off_lx, off_head, off_ent;
    size_t off_inoff, off_outoff, off_rin, off_rout, off_rpos, off_lpos, off_tmp, off_labs, off_laboff, total;
    int cap;       // class sums a row can hold: min(max_labels, D)
    int E_total;   // edges of all sequences
};
__host__ __device__ inline FsaLayout fsa_layout(int64_t T_total, int32_t B, int32_t S_total, int32_t E_total,
                                                int32_t max_states, int32_t max_labels, int32_t D) {
    FsaLayout L{};
    L.cap = max_labels < D ? max_labels : D;
    L.E_total = E_total;
    const size_t Bn = (size_t)(B > 0 ? B : 1), cap = (size_t)(L.cap > 0 ? L.cap : 1);
    size_t o = 256;  // the status word sits at offset 0, as in the CTC workspace
    L.off_z = o;      o = align_up(o + sizeof(double) * Bn, 256);
    L.off_nlab = o;   o = align_up(o + sizeof(int32_t) * Bn, 256);
    L.off_zx = o;     o = align_up(o + 8 * Bn, 256);
    L.off_alpha = o;  o = align_up(o + 8 * (size_t)T_total * (size_t)max_states, 256);
    L.off_beta = o;   o = align_up(o + 8 * (size_t)T_total * (size_t)max_states, 256);
    L.off_lx = o;     o = align_up(o + 8 * (size_t)T_total * cap, 256);
    // per row: a header and the row's class sums, in the format the dense
    // gradient stream of the CTC path reads
    L.off_head = o;   o = align_up(o + sizeof(RowHead) * (size_t)T_total, 256);
    L.off_ent = o;    o = align_up(o + 8 * (size_t)T_total * cap, 256);
    L.off_inoff = o;  o = align_up(o + sizeof(int32_t) * ((size_t)S_total + Bn), 256);
    L.off_outoff = o; o = align_up(o + sizeof(int32_t) * ((size_t)S_total + Bn), 256);
    L.off_rin = o;    o = align_up(o + sizeof(int4) * (size_t)E_total, 256);
    L.off_rout = o;   o = align_up(o + sizeof(int4) * (size_t)E_total, 256);
    L.off_rpos = o;   o = align_up(o + sizeof(int4) * (size_t)E_total, 256);  // records in label order
    L.off_lpos = o;   o = align_up(o + sizeof(int32_t) * (size_t)E_total, 256);  // position in label order
    L.off_tmp = o;    o = align_up(o + sizeof(int32_t) * (size_t)E_total, 256);
    L.off_labs = o;   o = align_up(o + sizeof(int32_t) * Bn * cap, 256);
    L.off_laboff = o; o = align_up(o + sizeof(int32_t) * Bn * (cap + 1), 256);
    L.total = o;
    return L;
}

struct FsaArgs {
    const void* lp;
    int64_t T_total;
    int D;
    const int32_t* cu;
    const int32_t* lengths;
    int B;
    const int32_t* state_offsets;
    const float* start_weight;
    const float* final_weight;
    const int32_t* edge_offsets;
    const int32_t* edges;  // (from, to, label) per edge
    const float* edge_weight;
    int max_states;
    int max_labels;
    int S_total;  // entries of the start / final weight arrays
    int E_total;  // edges
    int zero_infinity;
    float* loss;
    const float* grad_loss;
    void* grad;
    void* ws;
    int ecap_smem;  // a recursion CTA keeps a sequence's edge lists in shared memory up to this many edges
    // a recursion CTA's threads: [0, nst) hold states; [lt0, lt0 + nlt) copy
    // and convert the label values (its own warps after the state threads
    // when they fit the CTA, else the state threads themselves)
    int nst, lt0, nlt;
    FsaLayout L;
};

template <int DT>
__device__ __forceinline__ float lp_at(const void* lp, int64_t idx) {
    if constexpr (DT == 0) {
        return reinterpret_cast<const float*>(lp)[idx];
    } else {
        return bits_to_float<DT>(reinterpret_cast<const unsigned short*>(lp)[idx]);
    }
}

// Checks sequence b's sizes and edges; returns false (and flags the status)
// when the sequence cannot be run.
__device__ bool fsa_check(const FsaArgs& a, int b, int S, int e0, int E, int64_t start, int T) {
    Control* ctrl = ws_at<Control>(a.ws, 0);
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    const int64_t span = (int64_t)a.cu[b + 1] - start;
    const int s0 = a.state_offsets[b];
    if (threadIdx.x == 0) {
        if (S < 1 || S > a.max_states || E < 0 || s0 < 0 || (int64_t)s0 + S > a.S_total || e0 < 0 ||
            (int64_t)e0 + E > a.E_total)
            atomicOr(&s_bad, 1);
        if (start < 0 || span < 0 || (int64_t)a.cu[b + 1] > a.T_total || T < 0 || T > span) atomicOr(&s_bad, 4);
    }
    __syncthreads();
    if (s_bad == 0) {  // the edge range is known to lie inside the edge array
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int* ed = a.edges + 3 * (size_t)(e0 + e);
            if (ed[0] < 0 || ed[0] >= S || ed[1] < 0 || ed[1] >= S) atomicOr(&s_bad, 1);
            if (ed[2] < 0 || ed[2] >= a.D) atomicOr(&s_bad, 2);
        }
    }
    __syncthreads();
    const int bad = s_bad;
    if (threadIdx.x == 0 && bad) {
        set_status(ctrl, (bad & 1 ? CTC_PACKED_DEV_BAD_FSA : 0u) | (bad & 2 ? CTC_PACKED_DEV_LABEL_OUT_OF_RANGE : 0u) |
                             (bad & 4 ? CTC_PACKED_DEV_BAD_LENGTH : 0u));
    }
    return bad == 0;
}

// Exclusive scan of one value per thread over the CTA; the CTA total goes to
// *total.
__device__ int fsa_block_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    const int prefix = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
    *total = s_warp[nw - 1];
    __syncthreads();
    return prefix;
}

// The contiguous segment [*b0, *b1) of K entries that this thread scans in
// turn around one block-wide scan of the segments' totals (a few barriers,
// not a block scan per blockDim.x entries).
__device__ __forceinline__ void scan_segment(int K, int* b0, int* b1) {
    const int seg = (K + (int)blockDim.x - 1) / (int)blockDim.x;
    *b0 = min((int)threadIdx.x * seg, K);
    *b1 = min(*b0 + seg, K);
}

// cnt[0 .. K) becomes the exclusive prefix of itself (also written to
// off_out[0 .. K] when given, off_out[K] = the total); returns the total.
// (The block scan's first barrier also orders every thread's earlier reads
// of cnt before these writes.)
__device__ int scan_counts(int* cnt, int K, int* s_warp, int* off_out) {
    int b0, b1;
    scan_segment(K, &b0, &b1);
    int local = 0;
    for (int k = b0; k < b1; ++k) local += cnt[k];
    int total;
    int run = fsa_block_scan(local, s_warp, &total);
    for (int k = b0; k < b1; ++k) {
        const int v = cnt[k];
        cnt[k] = run;
        if (off_out != nullptr) off_out[k] = run;
        run += v;
    }
    if (off_out != nullptr && threadIdx.x == 0) off_out[K] = total;
    __syncthreads();
    return total;
}

// Places edge e at cursor[key(e)]++ in edge order (a stable counting sort's
// last pass): the CTA walks the edges one warp at a time; inside a warp the
// lanes with equal keys take consecutive slots in lane order.
template <typename KeyF>
__device__ void place_stable(int E, KeyF key, int* cursor, int* out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int c0 = 0; c0 < E; c0 += blockDim.x) {
        for (int w = 0; w < nw; ++w) {
            if (warp == w) {
                const int e = c0 + threadIdx.x;
                const bool on = e < E;
                const int k = on ? key(e) : -1;
                const unsigned peers = __match_any_sync(0xffffffffu, k);
                const int leader = __ffs(peers) - 1;
                int base = 0;
                if (on && lane == leader) {
                    base = cursor[k];
                    cursor[k] = base + __popc(peers);
                }
                base = __shfl_sync(0xffffffffu, base, leader);
                if (on) out[base + __popc(peers & ((1u << lane) - 1u))] = e;
            }
            __syncthreads();
        }
    }
}

// 8-byte loads and stores of an extended value (its arrays are 8-byte aligned).
__device__ __forceinline__ XP ld_xp(const XP* p) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    return XP{__uint_as_float(v.x), (int)v.y};
}
__device__ __forceinline__ void st_xp(XP* p, XP x) {
    *reinterpret_cast<uint2*>(p) = make_uint2(__float_as_uint(x.m), (unsigned)x.e);
}

// exp(v) in extended range; a NaN stays in the mantissa, so every sum it
// enters is NaN.
__device__ __forceinline__ XP xp_exp(float v) {
    XP r = xp_from_log(v);
    if (v != v) r.m = v;
    return r;
}

// Product of three extended values.  A zero product takes the zero exponent,
// so that no sum aligns on it.
__device__ __forceinline__ XP xp_mul3(XP a, XP b, XP c) {
    XP r;
    r.m = a.m * b.m * c.m;
    r.e = r.m > 0.0f ? a.e + b.e + c.e : kEZero;
    return r;
}

// 2^k as a float for any k: 0 below 2^-126, 2^127 above.
__device__ __forceinline__ float pow2_any(int k) { return __int_as_float(min(max(127 + k, 0), 254) << 23); }

// Running sum S * 2^E of extended values in a fixed order: the sum and each
// new term are aligned to the larger exponent (a term 2^126 below it drops
// out).  S stays finite: every term's mantissa is below 8.
struct XSum {
    float S = 0.0f;
    int E = kEZero;
    __device__ __forceinline__ void add(XP x) {
        const int E2 = max(E, x.e);
        S = fmaf(S, pow2_nonpos(E - E2), x.m * pow2_nonpos(x.e - E2));
        E = E2;
    }
};

// The sum of a state's held terms (zero where it holds fewer): all aligned
// at once to their largest exponent and added in list order, as the first
// value of its running sum.
template <int N>
__device__ __forceinline__ XSum xsum_held(const XP (&t)[N]) {
    int E = t[0].e;
#pragma unroll
    for (int j = 1; j < N; ++j) E = max(E, t[j].e);
    float S = t[0].m * pow2_nonpos(t[0].e - E);
#pragma unroll
    for (int j = 1; j < N; ++j) S = fmaf(t[j].m, pow2_nonpos(t[j].e - E), S);
    XSum r;
    r.S = S;
    r.E = E;
    return r;
}

// Sum over the CTA of every thread's partial sum: the lanes by a fixed
// shuffle tree, then the warps in order (every thread gets the result).
__device__ __forceinline__ XSum block_xsum(XSum a, XP* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a.add(XP{__shfl_xor_sync(0xffffffffu, a.S, o), __shfl_xor_sync(0xffffffffu, a.E, o)});
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = XP{a.S, a.E};
    __syncthreads();
    XSum r;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r.add(red[i]);
    __syncthreads();
    return r;
}

}  // namespace

// Sorted edge lists of sequence b (see the file comment).  A sequence that
// fails its checks, or has more distinct labels than max_labels, gets a NaN
// loss and nlab = -1: the recursions skip it and its rows stay zero.
__global__ void __launch_bounds__(kIdxThreads) fsa_index_kernel(FsaArgs a) {
    extern __shared__ __align__(16) int idx_smem[];
    __shared__ int s_warp[32];
    const int b = blockIdx.x;
    const int s0 = a.state_offsets[b], S = a.state_offsets[b + 1] - s0;
    const int e0 = a.edge_offsets[b], E = a.edge_offsets[b + 1] - e0;
    const int64_t start = a.cu[b];
    const int T = a.lengths[b];
    int* nlab_out = ws_at<int32_t>(a.ws, a.L.off_nlab);
    double* z_out = ws_at<double>(a.ws, a.L.off_z);
    auto reject = [&]() {
        if (threadIdx.x == 0) {
            nlab_out[b] = -1;
            z_out[b] = __longlong_as_double(0x7ff8000000000000ll);
            a.loss[b] = __int_as_float(0x7fc00000);
        }
    };
    if (!fsa_check(a, b, S, e0, E, start, T)) {
        reject();
        return;
    }
    const int D = a.D, cap = a.L.cap;
    int* cnt = idx_smem;         // max(S, D) counters
    int* slot = idx_smem + (S > D ? S : D);  // label -> slot among the distinct labels, D entries
    const int* ed = a.edges + 3 * (size_t)e0;
    const float* ew = a.edge_weight + e0;
    int* tmp = ws_at<int32_t>(a.ws, a.L.off_tmp) + e0;

    // 1. labels: counts, the distinct ones in increasing order, their lists
    for (int c = threadIdx.x; c < D; c += blockDim.x) cnt[c] = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) atomicAdd(&cnt[ed[3 * e + 2]], 1);
    __syncthreads();
    int nlab = 0;
    {
        int b0, b1;
        scan_segment(D, &b0, &b1);
        int local = 0;
        for (int c = b0; c < b1; ++c) local += cnt[c] > 0 ? 1 : 0;
        int run = fsa_block_scan(local, s_warp, &nlab);
        for (int c = b0; c < b1; ++c) {
            slot[c] = run;
            run += cnt[c] > 0 ? 1 : 0;
        }
        __syncthreads();  // slots are read across the segments below
    }
    if (nlab > cap) {
        if (threadIdx.x == 0) set_status(ws_at<Control>(a.ws, 0), CTC_PACKED_DEV_BAD_FSA);
        reject();
        return;
    }
    int* labs = ws_at<int32_t>(a.ws, a.L.off_labs) + (size_t)b * cap;
    int* laboff = ws_at<int32_t>(a.ws, a.L.off_laboff) + (size_t)b * (cap + 1);
    for (int c = threadIdx.x; c < D; c += blockDim.x)
        if (cnt[c] > 0) labs[slot[c]] = c;
    scan_counts(cnt, D, s_warp, nullptr);  // cnt[c]: first list position of label c
    // the distinct labels' list offsets: label c's list starts at cnt[c]
    for (int i = threadIdx.x; i < nlab; i += blockDim.x) laboff[i] = cnt[labs[i]];
    if (threadIdx.x == 0) laboff[nlab] = E;
    __syncthreads();
    // edge ids in label order into tmp, then each edge's position in that
    // order (where the backward writes its occupancy, so that a label's
    // occupancies are one contiguous range)
    int* lpos = ws_at<int32_t>(a.ws, a.L.off_lpos) + e0;
    place_stable(E, [&](int e) { return ed[3 * e + 2]; }, cnt, tmp);
    for (int k = threadIdx.x; k < E; k += blockDim.x) lpos[tmp[k]] = k;
    __syncthreads();

    // 2. incoming lists (by destination): records (from, label slot, exp of
    //    the weight in extended range: mantissa bits, exponent)
    int* inoff = ws_at<int32_t>(a.ws, a.L.off_inoff) + s0 + b;
    for (int s = threadIdx.x; s < S; s += blockDim.x) cnt[s] = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) atomicAdd(&cnt[ed[3 * e + 1]], 1);
    __syncthreads();
    scan_counts(cnt, S, s_warp, inoff);
    place_stable(E, [&](int e) { return ed[3 * e + 1]; }, cnt, tmp);
    int4* rin = ws_at<int4>(a.ws, a.L.off_rin) + e0;
    for (int k = threadIdx.x; k < E; k += blockDim.x) {
        const int e = tmp[k];
        const XP w = xp_exp(ew[e]);
        rin[k] = make_int4(ed[3 * e], slot[ed[3 * e + 2]], __float_as_int(w.m), w.e);
    }
    __syncthreads();

    // 3. outgoing lists (by source): records (to, label slot, log weight,
    //    the edge's position in label order); and at each position in label
    //    order the edge's record (from, to, label slot, log weight)
    int* outoff = ws_at<int32_t>(a.ws, a.L.off_outoff) + s0 + b;
    for (int s = threadIdx.x; s < S; s += blockDim.x) cnt[s] = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) atomicAdd(&cnt[ed[3 * e]], 1);
    __syncthreads();
    scan_counts(cnt, S, s_warp, outoff);
    place_stable(E, [&](int e) { return ed[3 * e]; }, cnt, tmp);
    int4* rout = ws_at<int4>(a.ws, a.L.off_rout) + e0;
    int4* rpos = ws_at<int4>(a.ws, a.L.off_rpos) + e0;
    for (int k = threadIdx.x; k < E; k += blockDim.x) {
        const int e = tmp[k];
        rout[k] = make_int4(ed[3 * e + 1], slot[ed[3 * e + 2]], __float_as_int(ew[e]), lpos[e]);
        rpos[lpos[e]] = make_int4(ed[3 * e], ed[3 * e + 1], slot[ed[3 * e + 2]], __float_as_int(ew[e]));
    }
    if (threadIdx.x == 0) nlab_out[b] = nlab;
}

// Frames of label words (and, backward, stored alpha rows) a recursion CTA
// keeps in flight, ring - 1 ahead of the frame it computes: 4, or 2 for
// sequences of more than 4 states a thread (their rows would not fit).
__host__ __device__ constexpr int fsa_ring(int per) { return per > 4 ? 2 : 4; }

// Shared-memory plan of a recursion CTA (see FsaArgs::ecap_smem): the
// sequence's edge lists when it has at most ecap_smem edges, then the
// per-frame buffers.
struct FsaSmem {
    int4* rec;        // edge records of the list (incoming or outgoing), ecap_smem
    int* off;         // list offsets per state, Smax + 1
    XP* val;          // alpha or beta of two frames, 2 * Smax
    XP* lpx;          // exp of the label values of two frames, 2 * cap
    uint32_t* ring;   // words holding the label values of `ring` frames, ring * cap
    int* labs;        // the distinct labels, cap
};
__host__ __device__ inline size_t fsa_smem_plan(int ecap, int Smax, int cap, int ring_frames, unsigned char* base,
                                                FsaSmem* out) {
    size_t o = 0;
    auto take = [&](size_t bytes, size_t align) {
        o = align_up(o, align);
        const size_t at = o;
        o += bytes;
        return at;
    };
    const size_t rec = take(16 * (size_t)ecap, 16);
    const size_t off = take(4 * ((size_t)Smax + 1), 4);
    const size_t val = take(16 * (size_t)Smax, 8);
    const size_t lpx = take(16 * (size_t)cap, 8);
    const size_t ring = take(4 * (size_t)ring_frames * cap, 4);
    const size_t labs = take(4 * (size_t)cap, 4);
    if (out != nullptr) {
        out->rec = reinterpret_cast<int4*>(base + rec);
        out->off = reinterpret_cast<int*>(base + off);
        out->val = reinterpret_cast<XP*>(base + val);
        out->lpx = reinterpret_cast<XP*>(base + lpx);
        out->ring = reinterpret_cast<uint32_t*>(base + ring);
        out->labs = reinterpret_cast<int*>(base + labs);
    }
    return align_up(o, 16);
}

namespace {

// Starts the copy of the aligned 32-bit word that holds element idx of the
// log probabilities into *dst (row_flip and the label's parity say which
// half is the element).
// The buffer starts 4-byte aligned; only its last element of a 2-byte type
// can end a word that would reach past the buffer, and that one is read
// directly into the word's low half.
template <int DT>
__device__ __forceinline__ void fetch_word(uint32_t* dst, const void* lp, int64_t idx, uintptr_t lp_end) {
    constexpr int E = DT == 0 ? 4 : 2;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(lp) + (uintptr_t)idx * E;
    const uintptr_t w = addr & ~uintptr_t(3);
    if (w + 4 <= lp_end) {
        cp_async4(smem_addr(dst), reinterpret_cast<const void*>(w));
    } else {
        *dst = (uint32_t)*reinterpret_cast<const unsigned short*>(addr);
    }
}

}  // namespace

// Edges of a state held in registers across the frames (the first RE of
// its list; a CTC lattice has at most three per state), and where the rest
// of its list lies.
template <int PER, int RE>
struct EdgeRegs {
    int peer[PER][RE];   // the other state of each edge (source forward, destination backward)
    int slot[PER][RE];   // its label's slot among the sequence's distinct labels
    XP w[PER][RE];       // exp of its log weight
    int n[PER];          // edges held (at most RE)
    int k0[PER], k1[PER];  // the rest of the list: entries [k0, k1)
};

// Forward records hold the weight in extended range, backward ones the log
// weight.
template <bool BACKWARD, int PER, int RE>
__device__ __forceinline__ void load_edge_regs(EdgeRegs<PER, RE>& er, const int* off, const int4* rec, int S,
                                               int nst) {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int s = (int)threadIdx.x < nst ? (int)threadIdx.x + k * nst : S;  // label threads hold none
        int b0 = 0, b1 = 0;
        if (s < S) {
            b0 = off[s];
            b1 = off[s + 1];
        }
        const int n = min(b1 - b0, RE);
        er.n[k] = n;
        er.k0[k] = b0 + n;
        er.k1[k] = b1;
#pragma unroll
        for (int j = 0; j < RE; ++j) {
            const int4 r = j < n ? rec[b0 + j] : make_int4(0, 0, 0, 0);
            er.peer[k][j] = r.x;
            er.slot[k][j] = r.y;
            er.w[k][j] = BACKWARD ? xp_exp(__int_as_float(r.z)) : XP{__int_as_float(r.z), r.w};
        }
    }
}

// Which half of its 32-bit word holds a label's element of a 2-byte type in
// row `row`: the parity of the element's position (row * D + label) plus
// the buffer's own; `par` is the row-independent part (base ^ label).
__device__ __forceinline__ int row_flip(int64_t row, int D) { return (int)(row & (int64_t)D) & 1; }

// A label thread's labels: li, li + nlt, ... of the sequence's nlab; the
// first two are held in registers across the frames (each label's byte
// offset in a row and the parity of its element's half in a 32-bit word),
// the rest are read from shared memory each frame.
template <int DT>
struct LabelLane {
    int li, nlt, nlab;
    int n;               // labels held (0, 1 or 2)
    uint32_t off[2];     // byte offset of label li + j * nlt in a row
    int par[2];          // parity of its element's half (2-byte types)
};
template <int DT>
__device__ __forceinline__ LabelLane<DT> label_lane(const int* labs, int nlab, int li, int nlt, int base_half) {
    constexpr int E = DT == 0 ? 4 : 2;
    LabelLane<DT> L;
    L.li = li;
    L.nlt = nlt;
    L.nlab = nlab;
    L.n = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = li + j * nlt;
        const bool on = (unsigned)li < (unsigned)nlt && i < nlab;
        const int c = on ? labs[i] : 0;
        L.off[j] = (uint32_t)c * E;
        L.par[j] = (base_half ^ c) & 1;
        L.n += on ? 1 : 0;
    }
    return L;
}

// Starts the copies of the words holding the thread's labels of row `row`.
// Only the buffer's last row can hold an element whose word would reach
// past the buffer.
template <int DT>
__device__ __forceinline__ void issue_row(uint32_t* dst, const void* lp, int64_t row, int D, int64_t T_total,
                                          const int* labs, uintptr_t lp_end, const LabelLane<DT>& L) {
    constexpr int E = DT == 0 ? 4 : 2;
    if (L.n == 0) return;
    if (DT == 0 || row + 1 < T_total) {
        const uintptr_t rp = reinterpret_cast<uintptr_t>(lp) + (uintptr_t)(row * (int64_t)D) * E;
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (j < L.n)
                cp_async4(smem_addr(dst + L.li + j * L.nlt), reinterpret_cast<const void*>((rp + L.off[j]) & ~uintptr_t(3)));
        for (int i = L.li + 2 * L.nlt; i < L.nlab; i += L.nlt)
            cp_async4(smem_addr(dst + i), reinterpret_cast<const void*>((rp + (uintptr_t)labs[i] * E) & ~uintptr_t(3)));
    } else {
        for (int i = L.li; i < L.nlab; i += L.nlt) fetch_word<DT>(dst + i, lp, row * (int64_t)D + labs[i], lp_end);
    }
}

// The thread's label values of a frame in extended range, into dst (each
// label thread converts the labels whose words it copied, so its own wait
// for the copies suffices).
template <int DT>
__device__ __forceinline__ void convert_row(XP* dst, const uint32_t* lw, const int* labs, int flip, int base_half,
                                            const LabelLane<DT>& L) {
    if (L.n == 0) return;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = L.li + j * L.nlt;
        if (j < L.n) st_xp(dst + i, xp_exp(word_to_float<DT>(lw[i], L.par[j] ^ flip)));
    }
    for (int i = L.li + 2 * L.nlt; i < L.nlab; i += L.nlt)
        st_xp(dst + i, xp_exp(word_to_float<DT>(lw[i], ((base_half ^ labs[i]) & 1) ^ flip)));
}

// The same, also keeping the values in the workspace row gdst (the frame's
// label values, read by the backward's occupancies).
template <int DT>
__device__ __forceinline__ void convert_row_keep(XP* dst, XP* gdst, const uint32_t* lw, const int* labs, int flip,
                                                 int base_half, const LabelLane<DT>& L) {
    if (L.n == 0) return;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = L.li + j * L.nlt;
        if (j < L.n) {
            const XP v = xp_exp(word_to_float<DT>(lw[i], L.par[j] ^ flip));
            st_xp(dst + i, v);
            st_xp(gdst + i, v);
        }
    }
    for (int i = L.li + 2 * L.nlt; i < L.nlab; i += L.nlt) {
        const XP v = xp_exp(word_to_float<DT>(lw[i], ((base_half ^ labs[i]) & 1) ^ flip));
        st_xp(dst + i, v);
        st_xp(gdst + i, v);
    }
}

// Forward recursion of sequence b (a CTA of fsa_chain_kernel).
template <int DT, int PER>
__device__ __forceinline__ void fsa_alpha_body(const FsaArgs& a, int b) {
    constexpr int RE = PER <= 2 ? 3 : (PER == 4 ? 2 : 1);
    constexpr int RING = fsa_ring(PER);
    extern __shared__ __align__(16) unsigned char fsa_smem[];
    __shared__ XP red[kFsaMaxThreads / 32];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int nst = a.nst, li = tid - a.lt0, nlt = a.nlt;  // state threads; this label thread
    const int nlab = ws_at<int32_t>(a.ws, a.L.off_nlab)[b];
    if (nlab < 0) return;  // rejected by the index pass (NaN loss written there)
    const int s0 = a.state_offsets[b], S = a.state_offsets[b + 1] - s0;
    const int e0 = a.edge_offsets[b], E = a.edge_offsets[b + 1] - e0;
    const int64_t start = a.cu[b];
    const int T = a.lengths[b];
    const int Smax = a.max_states, cap = a.L.cap, D = a.D;
    FsaSmem sm;
    fsa_smem_plan(a.ecap_smem, Smax, cap, RING, fsa_smem, &sm);
    const int* inoff_g = ws_at<int32_t>(a.ws, a.L.off_inoff) + s0 + b;
    const int4* rin_g = ws_at<int4>(a.ws, a.L.off_rin) + e0;
    const int* labs_g = ws_at<int32_t>(a.ws, a.L.off_labs) + (size_t)b * cap;
    XP* alpha_rows = ws_at<XP>(a.ws, a.L.off_alpha);
    const uintptr_t lp0 = reinterpret_cast<uintptr_t>(a.lp);
    const uintptr_t lp_end = lp0 + (uintptr_t)(a.T_total * (int64_t)D * (DT == 0 ? 4 : 2));
    const int base_half = (int)((lp0 >> 1) & 1);

    // the sequence's incoming lists into shared memory when they fit
    const bool local = E <= a.ecap_smem;
    if (local) {
        for (int k = tid; k < E; k += nt) sm.rec[k] = rin_g[k];
        for (int s = tid; s <= S; s += nt) sm.off[s] = inoff_g[s];
    }
    const int4* rin = local ? sm.rec : rin_g;
    const int* inoff = local ? sm.off : inoff_g;
    // the label threads load, copy and convert their own labels (no barrier
    // between): label words of frames 0 .. RING - 2 in flight
    if ((unsigned)li < (unsigned)nlt)
        for (int i = li; i < nlab; i += nlt) sm.labs[i] = labs_g[i];
    const LabelLane<DT> ll = label_lane<DT>(sm.labs, nlab, li, nlt, base_half);
    auto issue = [&](int f) {
        if (f < T) issue_row<DT>(sm.ring + (f % RING) * cap, a.lp, start + f, D, a.T_total, sm.labs, lp_end, ll);
        cp_async_commit();
    };
    for (int f = 0; f < RING - 1; ++f) issue(f);
    for (int s = tid; s < S; s += nt) st_xp(sm.val + s, xp_exp(a.start_weight[s0 + s]));
    cp_async_wait<RING - 2>();
    if (T > 0) convert_row<DT>(sm.lpx, sm.ring, sm.labs, row_flip(start, D), base_half, ll);
    __syncthreads();
    EdgeRegs<PER, RE> er;
    load_edge_regs<false>(er, inoff, rin, S, nst);
    bool nan_seen = false;  // a NaN sum: the loss is NaN
    int p = 0;
    XP* row = alpha_rows + start * (int64_t)Smax;  // frame t's stored row
    for (int t = 0; t < T; ++t, row += Smax) {
        issue(t + RING - 1);
        const XP* alp = sm.val + p * Smax;
        XP* alq = sm.val + (p ^ 1) * Smax;
        const XP* lx = sm.lpx + (t & 1) * cap;  // the frame's label values
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int s = tid + k * nst;
            if (tid < nst && s < S) {
                st_xp(row + s, ld_xp(alp + s));  // alpha_t, read by the backward
                // alpha_{t+1}(s) = sum over the incoming list, in order, of
                // alpha_t(from) x exp(weight) x exp(lp[t, label])
                XP hold[RE];
#pragma unroll
                for (int j = 0; j < RE; ++j)
                    hold[j] = j < er.n[k] ? xp_mul3(ld_xp(alp + er.peer[k][j]), er.w[k][j], ld_xp(lx + er.slot[k][j]))
                                          : XP{0.0f, kEZero};
                XSum acc = xsum_held(hold);
                for (int kk = er.k0[k]; kk < er.k1[k]; ++kk) {
                    const int4 r = rin[kk];
                    acc.add(xp_mul3(ld_xp(alp + r.x), XP{__int_as_float(r.z), r.w}, ld_xp(lx + r.y)));
                }
                nan_seen |= acc.S != acc.S;
                st_xp(alq + s, xp_norm(acc.S, acc.E));
            }
        }
        cp_async_wait<RING - 2>();
        if (t + 1 < T)
            convert_row<DT>(sm.lpx + ((t + 1) & 1) * cap, sm.ring + ((t + 1) % RING) * cap, sm.labs,
                            row_flip(start + t + 1, D), base_half, ll);
        __syncthreads();
        p ^= 1;
    }
    cp_async_wait<0>();
    // Z = sum over the states of alpha_T(s) x exp(final(s))
    XSum zs;
    for (int s = tid; s < S; s += nt)
        zs.add(xp_mul3(ld_xp(sm.val + p * Smax + s), xp_exp(a.final_weight[s0 + s]), XP{1.0f, 0}));
    nan_seen |= zs.S != zs.S;
    const XSum z = block_xsum(zs, red);
    const bool any_nan = __syncthreads_or(nan_seen) != 0;
    if (tid == 0) {
        const XP zx = any_nan ? XP{0.0f, kEZero} : xp_norm(z.S, z.E);
        double lz;
        if (any_nan)
            lz = __longlong_as_double(0x7ff8000000000000ll);
        else if (zx.m == 0.0f)
            lz = -INFINITY;
        else
            lz = log((double)zx.m) + (double)zx.e * 0.69314718055994530942;
        ws_at<double>(a.ws, a.L.off_z)[b] = lz;
        st_xp(ws_at<XP>(a.ws, a.L.off_zx) + b, zx);
        float l = (float)-lz;
        if (a.zero_infinity && lz == -INFINITY) l = 0.0f;
        a.loss[b] = l;
    }
}

// Backward recursion of sequence b (a CTA of fsa_chain_kernel, beside the
// forward recursion): beta_t(s) over the state's outgoing edges in list
// order, from beta_T(s) = exp(final(s)) down; every beta_t row and every
// frame's label values are kept for the backward call's occupancies.
template <int DT, int PER>
__device__ __forceinline__ void fsa_beta_body(const FsaArgs& a, int b) {
    constexpr int RE = PER <= 2 ? 3 : (PER == 4 ? 2 : 1);
    constexpr int RING = fsa_ring(PER);
    extern __shared__ __align__(16) unsigned char fsa_smem[];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int nst = a.nst, li = tid - a.lt0, nlt = a.nlt;  // state threads; this label thread
    const int nlab = ws_at<int32_t>(a.ws, a.L.off_nlab)[b];
    if (nlab < 0) return;  // rejected by the index pass
    const int s0 = a.state_offsets[b], S = a.state_offsets[b + 1] - s0;
    const int e0 = a.edge_offsets[b], E = a.edge_offsets[b + 1] - e0;
    const int64_t start = a.cu[b];
    const int T = a.lengths[b];
    const int Smax = a.max_states, cap = a.L.cap, D = a.D;
    FsaSmem sm;
    fsa_smem_plan(a.ecap_smem, Smax, cap, RING, fsa_smem, &sm);
    const int* outoff_g = ws_at<int32_t>(a.ws, a.L.off_outoff) + s0 + b;
    const int4* rout_g = ws_at<int4>(a.ws, a.L.off_rout) + e0;
    const int* labs_g = ws_at<int32_t>(a.ws, a.L.off_labs) + (size_t)b * cap;
    XP* beta_rows = ws_at<XP>(a.ws, a.L.off_beta);
    XP* lx_rows = ws_at<XP>(a.ws, a.L.off_lx);
    const uintptr_t lp0 = reinterpret_cast<uintptr_t>(a.lp);
    const uintptr_t lp_end = lp0 + (uintptr_t)(a.T_total * (int64_t)D * (DT == 0 ? 4 : 2));
    const int base_half = (int)((lp0 >> 1) & 1);

    // the sequence's outgoing lists into shared memory when they fit
    const bool local = E <= a.ecap_smem;
    if (local) {
        for (int k = tid; k < E; k += nt) sm.rec[k] = rout_g[k];
        for (int s = tid; s <= S; s += nt) sm.off[s] = outoff_g[s];
    }
    const int4* rout = local ? sm.rec : rout_g;
    const int* outoff = local ? sm.off : outoff_g;
    // the label threads load, copy and convert their own labels (no barrier
    // between): label words of frames T - 1 .. T - RING + 1 in flight
    if ((unsigned)li < (unsigned)nlt)
        for (int i = li; i < nlab; i += nlt) sm.labs[i] = labs_g[i];
    const LabelLane<DT> ll = label_lane<DT>(sm.labs, nlab, li, nlt, base_half);
    auto issue = [&](int f) {
        if (f >= 0) issue_row<DT>(sm.ring + (f % RING) * cap, a.lp, start + f, D, a.T_total, sm.labs, lp_end, ll);
        cp_async_commit();
    };
    for (int j = 0; j < RING - 1; ++j) issue(T - 1 - j);
    for (int s = tid; s < S; s += nt) st_xp(sm.val + s, xp_exp(a.final_weight[s0 + s]));
    cp_async_wait<RING - 2>();
    if (T > 0)
        convert_row_keep<DT>(sm.lpx + ((T - 1) & 1) * cap, lx_rows + (start + T - 1) * (int64_t)cap,
                             sm.ring + ((T - 1) % RING) * cap, sm.labs, row_flip(start + T - 1, D), base_half, ll);
    __syncthreads();
    EdgeRegs<PER, RE> er;
    load_edge_regs<true>(er, outoff, rout, S, nst);
    int p = 0;
    for (int t = T - 1; t >= 0; --t) {
        issue(t - (RING - 1));
        const XP* bep = sm.val + p * Smax;  // beta_{t+1}
        XP* beq = sm.val + (p ^ 1) * Smax;
        const XP* lx = sm.lpx + (t & 1) * cap;  // the frame's label values
        XP* row = beta_rows + (start + t) * (int64_t)Smax;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int s = tid + k * nst;
            if (tid < nst && s < S) {
                // beta_t(s) = sum over the outgoing list, in order, of
                // exp(weight) x exp(lp[t, label]) x beta_{t+1}(to)
                XP hold[RE];
#pragma unroll
                for (int j = 0; j < RE; ++j)
                    hold[j] = j < er.n[k] ? xp_mul3(er.w[k][j], ld_xp(lx + er.slot[k][j]), ld_xp(bep + er.peer[k][j]))
                                          : XP{0.0f, kEZero};
                XSum acc = xsum_held(hold);
                for (int kk = er.k0[k]; kk < er.k1[k]; ++kk) {
                    const int4 r = rout[kk];
                    acc.add(xp_mul3(xp_exp(__int_as_float(r.z)), ld_xp(lx + r.y), ld_xp(bep + r.x)));
                }
                const XP v = xp_norm(acc.S, acc.E);
                st_xp(beq + s, v);
                st_xp(row + s, v);  // beta_t, read by the backward
            }
        }
        cp_async_wait<RING - 2>();
        if (t > 0)
            convert_row_keep<DT>(sm.lpx + ((t - 1) & 1) * cap, lx_rows + (start + t - 1) * (int64_t)cap,
                                 sm.ring + ((t - 1) % RING) * cap, sm.labs, row_flip(start + t - 1, D), base_half, ll);
        __syncthreads();
        p ^= 1;
    }
    cp_async_wait<0>();
}

// The recursions of the forward call: CTA b < B runs sequence b's forward
// recursion, CTA B + b its backward recursion at the same time.
template <int DT, int PER>
__global__ void __launch_bounds__(kFsaMaxThreads, 1) fsa_chain_kernel(FsaArgs a) {
    if ((int)blockIdx.x < a.B) {
        fsa_alpha_body<DT, PER>(a, (int)blockIdx.x);
    } else {
        fsa_beta_body<DT, PER>(a, (int)blockIdx.x - a.B);
    }
}

// Occupancies and class sums of each row, from the rows both recursions
// kept: edge e = (from, to, label, weight) at frame t has occupancy
//   alpha_t(from) x exp(weight) x exp(lp[t, label]) x beta_{t+1}(to) / Z,
// beta_T(to) = exp(final(to)); each label's edges are a contiguous range in
// label order, summed in that order (up to kShortList by one thread; longer
// ones by a warp: four lane-strided partial sums, then a fixed shuffle tree),
// and written as the row's class sums (class, -scale * occupancy) with the
// row's header.  The dense rows are written afterwards by the all-SM
// gradient stream.  A CTA takes a contiguous range of rows.
constexpr int kFsaPostThreads = 128;
constexpr int kFsaPostBudget = 36 * 1024;  // shared memory a CTA aims at (several CTAs an SM)
// The sequence whose rows start at or before `row` (the last b with
// cu[b] <= row; -1 before the first), by binary search.
__device__ __forceinline__ int fsa_seq_of_row(const int32_t* cu, int B, int64_t row) {
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
__device__ __forceinline__ XP ldg_xp(const XP* p) {
    const int2 v = __ldg(reinterpret_cast<const int2*>(p));
    return XP{__int_as_float(v.x), v.y};
}
// Its shared memory: two stages of a row's alpha_t and beta_{t+1} (Smax
// each) and label values (cap), the next row's copied in while the current
// one is summed; the sequence's labels, label offsets and long lists (cap);
// then the sequence's edge records in label order when it has at most
// a.ecap_smem edges.
__host__ __device__ inline size_t fsa_post_stage_bytes(int Smax, int cap) { return 16 * (size_t)Smax + 8 * (size_t)cap; }
__host__ __device__ inline size_t fsa_post_smem(int Smax, int cap, int ecap) {
    return 2 * fsa_post_stage_bytes(Smax, cap) + 4 * (size_t)cap + 4 * ((size_t)cap + 1) + 4 * (size_t)cap + 16 +
           16 * (size_t)ecap;
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__global__ void __launch_bounds__(kFsaPostThreads) fsa_post_kernel(FsaArgs a) {
    extern __shared__ __align__(16) unsigned char fsa_smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = kFsaPostThreads / 32;
    const int64_t T_total = a.T_total;
    const int64_t per = (T_total + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = (int64_t)blockIdx.x * per;
    const int64_t r1 = r0 + per < T_total ? r0 + per : T_total;
    const int cap = a.L.cap, Smax = a.max_states;
    // stage q: alpha_t, beta_{t+1} (exp(final) at the last frame), the frame's label values
    const size_t stage_bytes = fsa_post_stage_bytes(Smax, cap);
    auto stage_al = [&](int q) { return reinterpret_cast<XP*>(fsa_smem + q * stage_bytes); };
    auto stage_bn = [&](int q) { return stage_al(q) + Smax; };
    auto stage_lx = [&](int q) { return stage_al(q) + 2 * Smax; };
    int* const slabs = reinterpret_cast<int*>(fsa_smem + 2 * stage_bytes);
    int* const sloff = slabs + cap;
    int* const slong = sloff + cap + 1;  // the labels whose lists a warp sums
    int4* const srp = reinterpret_cast<int4*>(fsa_smem + align_up(2 * stage_bytes + 12 * (size_t)cap + 4, 16));
    __shared__ int s_nlong;
    const int32_t* nlab_all = ws_at<int32_t>(a.ws, a.L.off_nlab);
    const double* z_all = ws_at<double>(a.ws, a.L.off_z);
    const XP* zx_all = ws_at<XP>(a.ws, a.L.off_zx);
    const XP* alpha_rows = ws_at<XP>(a.ws, a.L.off_alpha);
    const XP* beta_rows = ws_at<XP>(a.ws, a.L.off_beta);
    const XP* lx_rows = ws_at<XP>(a.ws, a.L.off_lx);
    RowHead* head = ws_at<RowHead>(a.ws, a.L.off_head);
    int2* ent = ws_at<int2>(a.ws, a.L.off_ent);
    // the sequence whose labels, offsets and records are held
    int cur = -1, nlab = -1, s0 = 0, S = 0, T = 0, e0 = 0, nlong = 0;
    int q = 0;          // the stage of the current row
    bool have = false;  // the current row's copies were started by the row before
    int64_t start = 0;
    float scale = 0.0f, izm = 1.0f;
    XP zx{0.0f, 0};
    const int4* rpos = nullptr;
    int b = r0 < r1 ? fsa_seq_of_row(a.cu, a.B, r0) : -1;  // then walked forward: rows only grow
    for (int64_t row = r0; row < r1; ++row) {
        while (b + 1 < a.B && (int64_t)a.cu[b + 1] <= row) ++b;
        if (b < 0) continue;
        if (b != cur) {
            __syncthreads();  // every read of the previous sequence's data is done
            cur = b;
            nlab = nlab_all[b];
            if (nlab < 0) continue;  // rejected: its rows keep zero headers
            s0 = a.state_offsets[b];
            S = a.state_offsets[b + 1] - s0;
            e0 = a.edge_offsets[b];
            const int E = a.edge_offsets[b + 1] - e0;
            start = a.cu[b];
            T = a.lengths[b];
            const double lz = z_all[b];
            scale = a.grad_loss[b];
            if (!(lz > -INFINITY)) scale = 0.0f;  // no path: zero rows (defined only with zero_infinity)
            zx = ldg_xp(zx_all + b);
            izm = 1.0f / zx.m;
            const int* labs_g = ws_at<int32_t>(a.ws, a.L.off_labs) + (size_t)b * cap;
            const int* laboff_g = ws_at<int32_t>(a.ws, a.L.off_laboff) + (size_t)b * (cap + 1);
            if (tid == 0) s_nlong = 0;
            __syncthreads();
            for (int i = tid; i < nlab; i += kFsaPostThreads) slabs[i] = labs_g[i];
            for (int i = tid; i <= nlab; i += kFsaPostThreads) sloff[i] = laboff_g[i];
            // (any order: each long list is summed by one warp)
            for (int i = tid; i < nlab; i += kFsaPostThreads)
                if (laboff_g[i + 1] - laboff_g[i] > kShortList) slong[atomicAdd(&s_nlong, 1)] = i;
            const int4* rpos_g = ws_at<int4>(a.ws, a.L.off_rpos) + e0;
            if (E <= a.ecap_smem) {
                for (int k = tid; k < E; k += kFsaPostThreads) srp[k] = rpos_g[k];
                rpos = srp;
            } else {
                rpos = rpos_g;
            }
        }
        const int64_t t = row - start;
        if (nlab < 0 || t < 0 || t >= T) continue;  // a rejected sequence, or a row outside its frames: zero
        if (scale == 0.0f) {
            // no occupancy is read: the row is scale * exp(lp) with no class sums
            if (tid == 0) head[row] = RowHead{0, scale, 1, 0};
            continue;
        }
        // the row's values, staged: copied into stage q (unless the row
        // before already started that), and the next row of the sequence
        // copied into the other stage meanwhile
        __syncthreads();  // every read of the other stage (the row before) is done
        nlong = s_nlong;
        const bool last = t + 1 == T;
        auto copy_row = [&](int64_t rw, int qq) {
            const XP* al = alpha_rows + rw * Smax;
            const XP* bn = beta_rows + (rw + 1) * Smax;
            const XP* lx = lx_rows + rw * cap;
            const bool lst = rw - start + 1 == T;
            XP* dal = stage_al(qq);
            XP* dbn = stage_bn(qq);
            XP* dlx = stage_lx(qq);
            for (int st = tid; st < S; st += kFsaPostThreads) {
                cp_async8(smem_addr(dal + st), al + st);
                if (!lst) cp_async8(smem_addr(dbn + st), bn + st);
            }
            for (int i = tid; i < nlab; i += kFsaPostThreads) cp_async8(smem_addr(dlx + i), lx + i);
            cp_async_commit();
        };
        if (!have) copy_row(row, q);
        const bool next = row + 1 < r1 && t + 1 < T;  // the same sequence: the same scale, nothing skipped
        if (next) {
            copy_row(row + 1, q ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        if (last)
            for (int st = tid; st < S; st += kFsaPostThreads) stage_bn(q)[st] = xp_exp(__ldg(a.final_weight + s0 + st));
        __syncthreads();
        const XP* sal = stage_al(q);
        const XP* sbn = stage_bn(q);
        const XP* slx = stage_lx(q);
        // the occupancy of the edge at label-order position k
        auto occ = [&](int k) -> float {
            const int4 r = rpos[k];
            const XP as = sal[r.x];
            const float gm = as.m * izm;
            const int ge = as.e - zx.e;
            const XP x = xp_mul3(xp_exp(__int_as_float(r.w)), slx[r.z], sbn[r.y]);
            return x.m * gm * pow2_any(x.e + ge);
        };
        // short lists: a thread each, in order (a plain loop: unrolled to
        // kShortList with predicates it issued every step for lists of two or
        // three edges).  With fewer long lists than warps and few labels, the
        // warps that sum the long lists take no short ones (a CTC lattice's
        // blank list is then the longest single sum of the row); with many
        // labels every thread takes short lists.
        const int lw = nlong < nw && nlab <= 2 * (kFsaPostThreads - 32 * nlong) ? nlong : 0;
        for (int i = tid - 32 * lw; i < nlab; i += kFsaPostThreads - 32 * lw) {
            if (i < 0) break;
            const int k0 = sloff[i], k1 = sloff[i + 1];
            if (k1 - k0 > kShortList) continue;
            float P = 0.0f;
            for (int k = k0; k < k1; ++k) P += occ(k);
            ent[row * cap + i] = make_int2(slabs[i], __float_as_int(-scale * P));
        }
        // long lists: a warp each, lane l summing entries l, l + 32, l + 64,
        // l + 96 of each block of 128 in four partial sums, combined in a
        // fixed order, then a fixed shuffle tree
        for (int h = warp; h < nlong; h += nw) {
            const int i = slong[h];
            const int k0 = sloff[i], k1 = sloff[i + 1];
            float P0 = 0.0f, P1 = 0.0f, P2 = 0.0f, P3 = 0.0f;
            int k = k0 + lane;
            for (; k + 96 < k1; k += 128) {
                P0 += occ(k);
                P1 += occ(k + 32);
                P2 += occ(k + 64);
                P3 += occ(k + 96);
            }
            for (; k < k1; k += 32) P0 += occ(k);
            float P = (P0 + P1) + (P2 + P3);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) P += __shfl_xor_sync(0xffffffffu, P, o);
            if (lane == 0) ent[row * cap + i] = make_int2(slabs[i], __float_as_int(-scale * P));
        }
        if (tid == 0) head[row] = RowHead{nlab, scale, 1, 0};
        have = next;
        q ^= 1;
    }
}

// Every row's header starts as "not covered, no class sums"; the backward
// then fills the rows of the sequences it runs.
__global__ void fsa_head_init_kernel(FsaArgs a) {
    RowHead* head = ws_at<RowHead>(a.ws, a.L.off_head);
    for (int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; row < a.T_total;
         row += (int64_t)gridDim.x * blockDim.x)
        head[row] = RowHead{0, 0.0f, 0, 0};
}

}  // namespace ctcp

using namespace ctcp;

namespace {

bool fsa_valid_dtype(int d) { return d == CTC_PACKED_F32 || d == CTC_PACKED_BF16 || d == CTC_PACKED_F16; }

// Threads of a recursion CTA: a thread per state of the largest sequence, in
// whole warps, between 64 and 512 (at most 8 states a thread).
int recursion_threads(int max_states) {
    int nt = (max_states + 31) / 32 * 32;
    if (nt < 64) nt = 64;
    if (nt > kFsaMaxThreads) nt = kFsaMaxThreads;
    return nt;
}

// Label threads of a recursion CTA: warps of their own after the nst state
// threads, one per 64 labels (a sequence's distinct labels, at most
// min(max_labels, D)), as many as fit the CTA's 512 threads; none when not
// one fits (the state threads then copy and convert the labels).  Sets
// a.nst, a.lt0, a.nlt and returns the CTA's threads.
int recursion_geometry(FsaArgs& a, int max_states) {
    const int nst = recursion_threads(max_states);
    int nlw = (a.L.cap + 63) / 64;
    if (nlw > (kFsaMaxThreads - nst) / 32) nlw = (kFsaMaxThreads - nst) / 32;
    a.nst = nst;
    if (nlw < 1) {
        a.lt0 = 0;
        a.nlt = nst;
        return nst;
    }
    a.lt0 = nst;
    a.nlt = 32 * nlw;
    return nst + 32 * nlw;
}

// Ring depth of the recursions for sequences of up to max_states states.
int ring_for(int max_states) {
    const int nt = recursion_threads(max_states);
    return fsa_ring((max_states + nt - 1) / nt);
}

// A recursion CTA's per-frame buffers, and the row kernel's two stages of
// a row, each within a CTA's shared memory: max_states and max_labels bound
// them together.
bool fsa_plan_fits(int max_states, int max_labels, int D) {
    const int cap = max_labels < D ? max_labels : D;
    return fsa_smem_plan(0, max_states, cap, ring_for(max_states), nullptr, nullptr) <= (size_t)kFsaSmemLimit &&
           fsa_post_smem(max_states, cap, 0) <= (size_t)kFsaSmemLimit;
}

ctc_packed_status fsa_check_args(const void* log_probs, int dtype, int64_t T_total, int32_t D, const int32_t* cu,
                                 const int32_t* lengths, int32_t B, const int32_t* so, const float* sw,
                                 const float* fw, int32_t S_total, const int32_t* eo, const int32_t* edges,
                                 const float* ew, int32_t E_total, int32_t max_states, int32_t max_labels,
                                 const void* ws, size_t ws_bytes) {
    if (!fsa_valid_dtype(dtype) || T_total < 0 || B < 0 || D < 1 || S_total < 0 || E_total < 0)
        return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (max_labels < 1) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (D > kFsaMaxD || T_total > INT32_MAX || max_states < 1 || max_states > kFsaMaxStates ||
        !fsa_plan_fits(max_states, max_labels, D))
        return CTC_PACKED_ERR_UNSUPPORTED;
    if (cu == nullptr || so == nullptr || eo == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (B > 0 && (lengths == nullptr || sw == nullptr || fw == nullptr)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (E_total > 0 && (edges == nullptr || ew == nullptr)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (T_total > 0 && log_probs == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    // 4-byte alignment for every dtype: the recursions copy aligned 4-byte words
    if (reinterpret_cast<uintptr_t>(log_probs) % 4 != 0) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (ws == nullptr || reinterpret_cast<uintptr_t>(ws) % 256 != 0) return CTC_PACKED_ERR_WORKSPACE;
    if (ws_bytes < fsa_layout(T_total, B, S_total, E_total, max_states, max_labels, D).total)
        return CTC_PACKED_ERR_WORKSPACE;
    return CTC_PACKED_OK;
}

// A plain launch (no early start): these kernels read what the kernel before
// them on the stream wrote without a programmatic wait.
template <typename K>
cudaError_t launch_fsa(K kernel, unsigned grid, int threads, size_t smem, cudaStream_t s, const FsaArgs& a) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, threads, smem, s>>>(a);
    return cudaGetLastError();
}

// Edges of one sequence a recursion CTA keeps in shared memory (a 16-byte
// record each): four times the batch's mean per sequence (at least 1024), at
// most what the budget leaves after the per-frame buffers and at most the
// batch's edges, so that CTAs of ordinary sequences share an SM.  A sequence
// with more edges reads its lists from the workspace.
int smem_edges(int B, int E_total, int max_states, int cap) {
    const size_t fixed = fsa_smem_plan(0, max_states, cap, ring_for(max_states), nullptr, nullptr);
    if (fixed + 64 >= (size_t)kFsaSmemBudget) return 0;
    size_t e = ((size_t)kFsaSmemBudget - fixed - 64) / 16;
    size_t want = 4 * (((size_t)E_total + (size_t)B - 1) / (size_t)(B > 0 ? B : 1));
    if (want < 1024) want = 1024;
    if (e > want) e = want;
    if (e > (size_t)E_total) e = (size_t)E_total;
    return (int)e;
}

// Both recursions with PER states a thread (2B CTAs: forward, then
// backward): the smallest of 1, 2, 4, 8 that covers max_states with the
// a.nst state threads (nt threads in all, the label warps included).
template <int DT>
cudaError_t launch_recursions(int max_states, int B, int nt, size_t smem, cudaStream_t s, const FsaArgs& a) {
    const int per = (max_states + a.nst - 1) / a.nst;
    const unsigned grid = 2u * (unsigned)B;
    if (per <= 1) return launch_fsa(fsa_chain_kernel<DT, 1>, grid, nt, smem, s, a);
    if (per <= 2) return launch_fsa(fsa_chain_kernel<DT, 2>, grid, nt, smem, s, a);
    if (per <= 4) return launch_fsa(fsa_chain_kernel<DT, 4>, grid, nt, smem, s, a);
    return launch_fsa(fsa_chain_kernel<DT, 8>, grid, nt, smem, s, a);
}

FsaArgs make_fsa_args(const void* log_probs, int64_t T_total, int32_t D, const int32_t* cu, const int32_t* lengths,
                      int32_t B, const int32_t* so, const float* sw, const float* fw, int32_t S_total,
                      const int32_t* eo, const int32_t* edges, const float* ew, int32_t E_total, int32_t max_states,
                      int32_t max_labels, int zero_infinity, void* ws) {
    FsaArgs a{};
    a.lp = log_probs;
    a.T_total = T_total;
    a.D = D;
    a.cu = cu;
    a.lengths = lengths;
    a.B = B;
    a.state_offsets = so;
    a.start_weight = sw;
    a.final_weight = fw;
    a.edge_offsets = eo;
    a.edges = edges;
    a.edge_weight = ew;
    a.max_states = max_states;
    a.max_labels = max_labels;
    a.S_total = S_total;
    a.E_total = E_total;
    a.zero_infinity = zero_infinity ? 1 : 0;
    a.ws = ws;
    a.L = fsa_layout(T_total, B, S_total, E_total, max_states, max_labels, D);
    return a;
}

}  // namespace

extern "C" {

size_t ctc_packed_fsa_workspace_size(int64_t T_total, int32_t B, int32_t num_states, int32_t num_edges,
                                     int32_t max_states, int32_t max_labels, int32_t D) {
    if (T_total < 0 || B < 0 || num_states < 0 || num_edges < 0 || max_states < 1 || max_states > kFsaMaxStates ||
        T_total > INT32_MAX || max_labels < 1 || D < 1 || D > kFsaMaxD || !fsa_plan_fits(max_states, max_labels, D))
        return 0;
    return fsa_layout(T_total, B, num_states, num_edges, max_states, max_labels, D).total;
}

ctc_packed_status ctc_packed_fsa_forward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                                         const int32_t* cu_seqlens, const int32_t* lengths, int32_t B,
                                         const int32_t* state_offsets, const float* start_weight,
                                         const float* final_weight, int32_t num_states, const int32_t* edge_offsets,
                                         const int32_t* edges, const float* edge_weight, int32_t num_edges,
                                         int32_t max_states, int32_t max_labels, int zero_infinity, float* loss,
                                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    const ctc_packed_status st =
        fsa_check_args(log_probs, dtype, T_total, D, cu_seqlens, lengths, B, state_offsets, start_weight,
                       final_weight, num_states, edge_offsets, edges, edge_weight, num_edges, max_states, max_labels,
                       workspace, workspace_bytes);
    if (st != CTC_PACKED_OK) return st;
    if (B > 0 && loss == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    // the control block (status word, and the input mode the gradient stream
    // reads: log probabilities) is cleared on the stream before any kernel
    if (cudaMemsetAsync(workspace, 0, sizeof(Control), stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    if (B == 0) return CTC_PACKED_OK;
    FsaArgs a = make_fsa_args(log_probs, T_total, D, cu_seqlens, lengths, B, state_offsets, start_weight,
                              final_weight, num_states, edge_offsets, edges, edge_weight, num_edges, max_states,
                              max_labels, zero_infinity, workspace);
    a.loss = loss;
    // 1. per sequence: the sorted edge lists
    const size_t ismem = sizeof(int) * ((size_t)(max_states > D ? max_states : D) + (size_t)D);
    if (launch_fsa(fsa_index_kernel, (unsigned)B, kIdxThreads, ismem, stream, a) != cudaSuccess)
        return CTC_PACKED_ERR_CUDA;
    // 2. per sequence: the forward recursion (the loss) and, beside it, the
    //    backward recursion (beta rows and label values for the gradient)
    const int nt = recursion_geometry(a, max_states);
    a.ecap_smem = smem_edges(B, num_edges, max_states, a.L.cap);
    const size_t smem = fsa_smem_plan(a.ecap_smem, max_states, a.L.cap, ring_for(max_states), nullptr, nullptr);
    const cudaError_t e = dtype == CTC_PACKED_F32    ? launch_recursions<0>(max_states, B, nt, smem, stream, a)
                          : dtype == CTC_PACKED_BF16 ? launch_recursions<1>(max_states, B, nt, smem, stream, a)
                                                     : launch_recursions<2>(max_states, B, nt, smem, stream, a);
    return e == cudaSuccess ? CTC_PACKED_OK : CTC_PACKED_ERR_CUDA;
}

ctc_packed_status ctc_packed_fsa_backward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                                          const int32_t* cu_seqlens, const int32_t* lengths, int32_t B,
                                          const int32_t* state_offsets, const float* start_weight,
                                          const float* final_weight, int32_t num_states,
                                          const int32_t* edge_offsets, const int32_t* edges,
                                          const float* edge_weight, int32_t num_edges, int32_t max_states,
                                          int32_t max_labels, int zero_infinity, const float* grad_loss,
                                          void* workspace, size_t workspace_bytes, void* grad_log_probs,
                                          cudaStream_t stream) {
    const ctc_packed_status st =
        fsa_check_args(log_probs, dtype, T_total, D, cu_seqlens, lengths, B, state_offsets, start_weight,
                       final_weight, num_states, edge_offsets, edges, edge_weight, num_edges, max_states, max_labels,
                       workspace, workspace_bytes);
    if (st != CTC_PACKED_OK) return st;
    if (T_total == 0) return CTC_PACKED_OK;
    if (grad_log_probs == nullptr || (B > 0 && grad_loss == nullptr)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    const int eb = dtype == CTC_PACKED_F32 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(grad_log_probs) % eb != 0) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(grad_log_probs), l0 = reinterpret_cast<uintptr_t>(log_probs);
    const uintptr_t nbytes = (uintptr_t)(T_total * (int64_t)D * eb);
    if (g0 < l0 + nbytes && l0 < g0 + nbytes) return CTC_PACKED_ERR_INVALID_ARGUMENT;  // overlap
    FsaArgs a = make_fsa_args(log_probs, T_total, D, cu_seqlens, lengths, B, state_offsets, start_weight,
                              final_weight, num_states, edge_offsets, edges, edge_weight, num_edges, max_states,
                              max_labels, zero_infinity, workspace);
    a.grad_loss = grad_loss;
    a.grad = grad_log_probs;
    // 1. every row header "not covered"
    const long long hgrid = (T_total + 255) / 256;
    if (launch_fsa(fsa_head_init_kernel, (unsigned)(hgrid < 4096 ? hgrid : 4096), 256, 0, stream, a) != cudaSuccess)
        return CTC_PACKED_ERR_CUDA;
    // 2. per row: the edge occupancies from the forward's kept rows, each
    //    row's class sums and header (a contiguous range of rows a CTA)
    if (B > 0) {
        // the row staging, and the sequence's edge records up to a share of
        // an SM's shared memory that leaves room for several CTAs
        const size_t fixed = fsa_post_smem(max_states, a.L.cap, 0);
        const size_t room = fixed < (size_t)kFsaPostBudget ? ((size_t)kFsaPostBudget - fixed) / 16 : 0;
        a.ecap_smem = (int)(room < (size_t)num_edges ? room : (size_t)num_edges);
        const size_t smem = fsa_post_smem(max_states, a.L.cap, a.ecap_smem);
        int dev = 0, sms = 0, per_sm = 0;
        if (cudaFuncSetAttribute(fsa_post_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess ||
            cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fsa_post_kernel, kFsaPostThreads, smem) !=
                cudaSuccess)
            return CTC_PACKED_ERR_CUDA;
        long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);
        if (grid > T_total) grid = T_total;
        if (launch_fsa(fsa_post_kernel, (unsigned)grid, kFsaPostThreads, smem, stream, a) != cudaSuccess)
            return CTC_PACKED_ERR_CUDA;
    }
    // 3. the dense rows, scale * exp(lp) + class sums, by the CTC path's
    //    all-SM gradient stream over this workspace's headers and sums
    GradArgs ga{};
    ga.L.T_total = T_total;
    ga.L.B = B;
    ga.L.D = D;
    ga.L.ecap = a.L.cap;
    ga.L.off_ctrl = 0;
    ga.L.off_head = a.L.off_head;
    ga.L.off_ent = a.L.off_ent;
    ga.L.off_lse = 0;  // not read: the control block says log probabilities
    ga.ws = workspace;
    ga.lp = log_probs;
    ga.grad = grad_log_probs;
    ga.D = D;
    int k = 1, cap = 1;
    size_t wsm = 0;
    grad_geometry(ga.L, D, k, cap, wsm);
    ga.rows_per_tile = k;
    ga.entry_cap = cap;
    ga.warp_smem = wsm;
    ga.n_tiles = (T_total + k - 1) / k;
    ga.congruent = ((g0 ^ l0) & 15u) == 0 ? 1 : 0;
    return launch_grad(ga, (int)dtype, stream) == cudaSuccess ? CTC_PACKED_OK : CTC_PACKED_ERR_CUDA;
}

}  // extern "C"
