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
// One CTA per sequence walks its frames; the states' values sit in shared
// memory in float32 log space and each frame's log-sum-exp over the edges
// into a state is two passes over the edges: an atomic maximum (on an
// order-preserving integer key), then an atomic sum of exp(v - max).  The
// shared-memory atomics make the summation order, and so the last bits,
// run-dependent (as the page's own label scatter is).  The forward stores
// alpha_t of every frame in the workspace; the backward runs beta, forms the
// edge occupancies, sums them per class in a shared row of D values and
// writes each gradient row densely, in the log probabilities' dtype.
#include <cstdint>

#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

constexpr int kFsaThreads = 256;
// Edges a thread keeps in registers (its edges tid, tid + 256, ...): their
// ids, weight and the label values of this frame and the next, which load
// while the frame's barriers run.  A sequence's further edges are read from
// memory each frame.
constexpr int kFsaRegEdges = 4;

// Workspace of the FSA path: status header, log Z per sequence (double),
// each frame's forward values relative to the frame's own offset (float)
// and that offset (double).
struct FsaLayout {
    size_t off_z, off_coff, off_alpha, off_head, off_ent, total;
    int cap;  // class sums a row can hold: min(max_labels, D)
};
__host__ __device__ inline FsaLayout fsa_layout(int64_t T_total, int32_t B, int32_t max_states, int32_t max_labels,
                                                int32_t D) {
    FsaLayout L{};
    L.cap = max_labels < D ? max_labels : D;
    size_t o = 256;  // the status word sits at offset 0, as in the CTC workspace
    L.off_z = o;
    o = align_up(o + sizeof(double) * (size_t)(B > 0 ? B : 1), 256);
    L.off_coff = o;
    o = align_up(o + sizeof(double) * (size_t)T_total, 256);
    L.off_alpha = o;
    o = align_up(o + sizeof(float) * (size_t)T_total * (size_t)max_states, 256);
    // per row: a header and the row's class sums, in the format the dense
    // gradient stream of the CTC path reads
    L.off_head = o;
    o = align_up(o + sizeof(RowHead) * (size_t)T_total, 256);
    L.off_ent = o;
    o = align_up(o + 8 * (size_t)T_total * (size_t)(L.cap > 0 ? L.cap : 1), 256);
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
    FsaLayout L;
};

// Order-preserving map of a float onto a signed int (and back), so that an
// integer atomic maximum is a float maximum.
__device__ __forceinline__ int fkey(float f) {
    const int b = __float_as_int(f);
    return b >= 0 ? b : b ^ 0x7fffffff;
}
__device__ __forceinline__ float fdekey(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

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
__device__ bool fsa_check(const FsaArgs& a, int b, int S, int e0, int E, int64_t start, int T, bool& bad_label) {
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
    bad_label = bad != 0;
    return bad == 0;
}

// Block-wide maximum of v[0 .. n).
__device__ float block_max(const float* v, int n, float* red) {
    float m = -INFINITY;
    for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, v[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = -INFINITY;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    __syncthreads();
    return m;
}

// Shifts v[0 .. n) down by its maximum (when finite) and returns the shift:
// the recursions keep every frame's values near 0, so their float32 rounding
// stays relative to the frame, and carry the shifts in double.
__device__ float renormalise(float* v, int n, float* red) {
    const float m = block_max(v, n, red);
    if (m > -INFINITY && m < INFINITY) {
        for (int i = threadIdx.x; i < n; i += blockDim.x) v[i] -= m;
        __syncthreads();
        return m;
    }
    return 0.0f;
}

// Block-wide logsumexp of v[0 .. n) (one value per thread slot, strided).
__device__ float block_lse(const float* v, const float* w, int n, float* red) {
    float m = -INFINITY;
    for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, v[i] + w[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = -INFINITY;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    __syncthreads();
    float s = 0.0f;
    if (m > -INFINITY)
        for (int i = threadIdx.x; i < n; i += blockDim.x) s += expf(v[i] + w[i] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    s = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    __syncthreads();
    return m > -INFINITY ? m + logf(s) : -INFINITY;
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kFsaThreads) fsa_forward_kernel(FsaArgs a) {
    extern __shared__ __align__(16) float fsa_smem[];
    __shared__ float red[kFsaThreads / 32];
    const int b = blockIdx.x;
    const int s0 = a.state_offsets[b], S = a.state_offsets[b + 1] - s0;
    const int e0 = a.edge_offsets[b], E = a.edge_offsets[b + 1] - e0;
    const int64_t start = a.cu[b];
    const int T = a.lengths[b];
    double* z_out = ws_at<double>(a.ws, a.L.off_z);
    double* coff = ws_at<double>(a.ws, a.L.off_coff);
    bool bad = false;
    if (!fsa_check(a, b, S, e0, E, start, T, bad)) {
        if (threadIdx.x == 0) {
            z_out[b] = __longlong_as_double(0x7ff8000000000000ll);
            a.loss[b] = __int_as_float(0x7fc00000);
        }
        return;
    }
    float* al = fsa_smem;                                   // alpha_t
    int* mk = reinterpret_cast<int*>(fsa_smem + a.max_states);  // max key per state
    float* sm = fsa_smem + 2 * a.max_states;                // sum per state
    float* alpha_rows = ws_at<float>(a.ws, a.L.off_alpha);
    int efr[kFsaRegEdges], eto[kFsaRegEdges], elab[kFsaRegEdges];
    float ew[kFsaRegEdges], lpc[kFsaRegEdges], lpn[kFsaRegEdges], ev[kFsaRegEdges];
#pragma unroll
    for (int k = 0; k < kFsaRegEdges; ++k) {
        const int e = threadIdx.x + k * kFsaThreads;
        const bool on = e < E;
        const int* ed = a.edges + 3 * (size_t)(e0 + (on ? e : 0));
        efr[k] = on ? ed[0] : 0;
        eto[k] = on ? ed[1] : 0;
        elab[k] = on ? ed[2] : 0;
        ew[k] = on ? a.edge_weight[e0 + e] : -INFINITY;  // an absent edge never contributes
        lpc[k] = (on && T > 0) ? lp_at<DT>(a.lp, start * (int64_t)a.D + elab[k]) : 0.0f;
        lpn[k] = 0.0f;
    }
    const int e_reg = kFsaRegEdges * kFsaThreads;  // edges from here on are read each frame
    for (int s = threadIdx.x; s < S; s += blockDim.x) al[s] = a.start_weight[s0 + s];
    __syncthreads();
    double C = renormalise(al, S, red);  // alpha_t = al + C
    bool nan_seen = false;               // a NaN edge value: the loss is NaN
    for (int t = 0; t < T; ++t) {
        float* row = alpha_rows + (start + t) * (int64_t)a.max_states;
        if (threadIdx.x == 0) coff[start + t] = C;
        for (int s = threadIdx.x; s < S; s += blockDim.x) {
            row[s] = al[s];
            mk[s] = fkey(-INFINITY);
            sm[s] = 0.0f;
        }
        __syncthreads();
        const int64_t lrow = (start + t) * (int64_t)a.D;
#pragma unroll
        for (int k = 0; k < kFsaRegEdges; ++k) {
            ev[k] = al[efr[k]] + ew[k] + lpc[k];
            nan_seen |= ev[k] != ev[k];
            if (ev[k] > -INFINITY) atomicMax(&mk[eto[k]], fkey(ev[k]));
        }
        for (int e = e_reg + threadIdx.x; e < E; e += blockDim.x) {
            const int* ed = a.edges + 3 * (size_t)(e0 + e);
            const float v = al[ed[0]] + a.edge_weight[e0 + e] + lp_at<DT>(a.lp, lrow + ed[2]);
            nan_seen |= v != v;
            if (v > -INFINITY) atomicMax(&mk[ed[1]], fkey(v));
        }
        if (t + 1 < T) {  // the next frame's label values, in flight across the barriers
#pragma unroll
            for (int k = 0; k < kFsaRegEdges; ++k)
                if (threadIdx.x + k * kFsaThreads < E) lpn[k] = lp_at<DT>(a.lp, lrow + a.D + elab[k]);
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kFsaRegEdges; ++k)
            if (ev[k] > -INFINITY) atomicAdd(&sm[eto[k]], expf(ev[k] - fdekey(mk[eto[k]])));
        for (int e = e_reg + threadIdx.x; e < E; e += blockDim.x) {
            const int* ed = a.edges + 3 * (size_t)(e0 + e);
            const float v = al[ed[0]] + a.edge_weight[e0 + e] + lp_at<DT>(a.lp, lrow + ed[2]);
            if (v > -INFINITY) atomicAdd(&sm[ed[1]], expf(v - fdekey(mk[ed[1]])));
        }
        __syncthreads();
        for (int s = threadIdx.x; s < S; s += blockDim.x)
            al[s] = sm[s] > 0.0f ? fdekey(mk[s]) + logf(sm[s]) : (sm[s] != sm[s] ? sm[s] : -INFINITY);
        __syncthreads();
        C += renormalise(al, S, red);
#pragma unroll
        for (int k = 0; k < kFsaRegEdges; ++k) lpc[k] = lpn[k];
    }
    const float zr = block_lse(al, a.final_weight + s0, S, red);
    const bool any_nan = __syncthreads_or(nan_seen) != 0;
    if (threadIdx.x == 0) {
        const double Z = any_nan ? __longlong_as_double(0x7ff8000000000000ll)
                                 : (zr > -INFINITY ? C + (double)zr : (double)zr);
        z_out[b] = Z;
        float l = (float)-Z;
        if (a.zero_infinity && Z == -INFINITY) l = 0.0f;
        a.loss[b] = l;
    }
}

template <int DT>
__global__ void __launch_bounds__(kFsaThreads) fsa_backward_kernel(FsaArgs a) {
    extern __shared__ __align__(16) float fsa_smem[];
    __shared__ float red[kFsaThreads / 32];
    __shared__ int s_nlab;
    const int b = blockIdx.x;
    const int s0 = a.state_offsets[b], S = a.state_offsets[b + 1] - s0;
    const int e0 = a.edge_offsets[b], E = a.edge_offsets[b + 1] - e0;
    const int64_t start = a.cu[b];
    const int T = a.lengths[b];
    const double Z = ws_at<double>(a.ws, a.L.off_z)[b];
    const double* coff = ws_at<double>(a.ws, a.L.off_coff);
    bool bad = false;
    if (!fsa_check(a, b, S, e0, E, start, T, bad)) return;  // the rows keep zero headers: zero gradient
    float scale = a.grad_loss[b];
    if (!(Z > -INFINITY)) scale = 0.0f;  // no path: zero rows (defined only with zero_infinity)
    float* be = fsa_smem;                                   // beta_{t+1}
    int* mk = reinterpret_cast<int*>(fsa_smem + a.max_states);
    float* sm = fsa_smem + 2 * a.max_states;
    float* P = fsa_smem + 3 * a.max_states;                 // class occupancies of the frame, D values
    int* labs = reinterpret_cast<int*>(P + a.D);            // the sequence's distinct labels, cap entries
    const int cap = a.L.cap;
    const float* alpha_rows = ws_at<float>(a.ws, a.L.off_alpha);
    RowHead* head = ws_at<RowHead>(a.ws, a.L.off_head);
    int2* ent = ws_at<int2>(a.ws, a.L.off_ent);
    // the distinct labels of the edges, found once: P serves as the marker row
    int* mark = reinterpret_cast<int*>(P);
    for (int c = threadIdx.x; c < a.D; c += blockDim.x) mark[c] = 0;
    if (threadIdx.x == 0) s_nlab = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int c = a.edges[3 * (size_t)(e0 + e) + 2];
        if (atomicExch(&mark[c], 1) == 0) {
            const int i = atomicAdd(&s_nlab, 1);
            if (i < cap) labs[i] = c;
        }
    }
    __syncthreads();
    const int nlab = s_nlab;
    if (nlab > cap) {  // more distinct labels than max_labels: the rows keep zero headers
        if (threadIdx.x == 0) set_status(ws_at<Control>(a.ws, 0), CTC_PACKED_DEV_BAD_FSA);
        return;
    }
    int efr[kFsaRegEdges], eto[kFsaRegEdges], elab[kFsaRegEdges];
    float ew[kFsaRegEdges], lpc[kFsaRegEdges], lpn[kFsaRegEdges], ac[kFsaRegEdges], an[kFsaRegEdges];
    float ev[kFsaRegEdges];
#pragma unroll
    for (int k = 0; k < kFsaRegEdges; ++k) {
        const int e = threadIdx.x + k * kFsaThreads;
        const bool on = e < E;
        const int* ed = a.edges + 3 * (size_t)(e0 + (on ? e : 0));
        efr[k] = on ? ed[0] : 0;
        eto[k] = on ? ed[1] : 0;
        elab[k] = on ? ed[2] : 0;
        ew[k] = on ? a.edge_weight[e0 + e] : -INFINITY;  // an absent edge never contributes
        // this frame's label value and forward value at the edge's origin
        lpc[k] = (on && T > 0) ? lp_at<DT>(a.lp, (start + T - 1) * (int64_t)a.D + elab[k]) : 0.0f;
        ac[k] = (on && T > 0) ? alpha_rows[(start + T - 1) * (int64_t)a.max_states + efr[k]] : 0.0f;
        lpn[k] = an[k] = 0.0f;
    }
    const int e_reg = kFsaRegEdges * kFsaThreads;  // edges from here on are read each frame
    for (int s = threadIdx.x; s < S; s += blockDim.x) be[s] = a.final_weight[s0 + s];
    __syncthreads();
    double Dn = renormalise(be, S, red);  // beta_{t+1} = be + Dn
    for (int t = T - 1; t >= 0; --t) {
        // occupancy exponent: alpha row + edge + beta, plus this constant
        const float K = scale != 0.0f ? (float)(coff[start + t] + Dn - Z) : 0.0f;
        for (int s = threadIdx.x; s < S; s += blockDim.x) {
            mk[s] = fkey(-INFINITY);
            sm[s] = 0.0f;
        }
        for (int i = threadIdx.x; i < nlab; i += blockDim.x) P[labs[i]] = 0.0f;
        __syncthreads();
        const int64_t lrow = (start + t) * (int64_t)a.D;
        const float* arow = alpha_rows + (start + t) * (int64_t)a.max_states;
#pragma unroll
        for (int k = 0; k < kFsaRegEdges; ++k) {
            ev[k] = ew[k] + lpc[k] + be[eto[k]];
            if (ev[k] > -INFINITY) atomicMax(&mk[efr[k]], fkey(ev[k]));
        }
        for (int e = e_reg + threadIdx.x; e < E; e += blockDim.x) {
            const int* ed = a.edges + 3 * (size_t)(e0 + e);
            const float v = a.edge_weight[e0 + e] + lp_at<DT>(a.lp, lrow + ed[2]) + be[ed[1]];
            if (v > -INFINITY) atomicMax(&mk[ed[0]], fkey(v));
        }
        if (t > 0) {  // the previous frame's label and forward values, in flight across the barriers
#pragma unroll
            for (int k = 0; k < kFsaRegEdges; ++k) {
                if (threadIdx.x + k * kFsaThreads < E) {
                    lpn[k] = lp_at<DT>(a.lp, lrow - a.D + elab[k]);
                    an[k] = arow[efr[k] - a.max_states];
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kFsaRegEdges; ++k) {
            if (ev[k] > -INFINITY) {
                atomicAdd(&sm[efr[k]], expf(ev[k] - fdekey(mk[efr[k]])));
                if (scale != 0.0f) {
                    const float occ = expf(ac[k] + ev[k] + K);
                    if (occ > 0.0f) atomicAdd(&P[elab[k]], occ);
                }
            }
        }
        for (int e = e_reg + threadIdx.x; e < E; e += blockDim.x) {
            const int* ed = a.edges + 3 * (size_t)(e0 + e);
            const float v = a.edge_weight[e0 + e] + lp_at<DT>(a.lp, lrow + ed[2]) + be[ed[1]];
            if (v > -INFINITY) {
                atomicAdd(&sm[ed[0]], expf(v - fdekey(mk[ed[0]])));
                if (scale != 0.0f) {
                    const float occ = expf(arow[ed[0]] + v + K);
                    if (occ > 0.0f) atomicAdd(&P[ed[2]], occ);
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kFsaRegEdges; ++k) {
            lpc[k] = lpn[k];
            ac[k] = an[k];
        }
        // the row's class sums (class, -scale * occupancy) and header; the
        // dense rows are written afterwards by the all-SM gradient stream
        const int64_t row = start + t;
        const int n = scale != 0.0f ? nlab : 0;
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            ent[row * cap + i] = make_int2(labs[i], __float_as_int(-scale * P[labs[i]]));
        if (threadIdx.x == 0) head[row] = RowHead{n, scale, 1, 0};
        for (int s = threadIdx.x; s < S; s += blockDim.x)
            be[s] = sm[s] > 0.0f ? fdekey(mk[s]) + logf(sm[s]) : (sm[s] != sm[s] ? sm[s] : -INFINITY);
        __syncthreads();
        Dn += renormalise(be, S, red);
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

ctc_packed_status fsa_check_args(const void* log_probs, int dtype, int64_t T_total, int32_t D, const int32_t* cu,
                                 const int32_t* lengths, int32_t B, const int32_t* so, const float* sw,
                                 const float* fw, int32_t S_total, const int32_t* eo, const int32_t* edges,
                                 const float* ew, int32_t E_total, int32_t max_states, int32_t max_labels,
                                 const void* ws, size_t ws_bytes) {
    if (!fsa_valid_dtype(dtype) || T_total < 0 || B < 0 || D < 1 || S_total < 0 || E_total < 0)
        return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (max_labels < 1) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (D > kFsaMaxD || T_total > INT32_MAX || max_states < 1 || max_states > kFsaMaxStates)
        return CTC_PACKED_ERR_UNSUPPORTED;
    if (cu == nullptr || so == nullptr || eo == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (B > 0 && (lengths == nullptr || sw == nullptr || fw == nullptr)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (E_total > 0 && (edges == nullptr || ew == nullptr)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (T_total > 0 && log_probs == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(log_probs) % (dtype == CTC_PACKED_F32 ? 4 : 2) != 0)
        return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (ws == nullptr || reinterpret_cast<uintptr_t>(ws) % 256 != 0) return CTC_PACKED_ERR_WORKSPACE;
    if (ws_bytes < fsa_layout(T_total, B, max_states, max_labels, D).total) return CTC_PACKED_ERR_WORKSPACE;
    return CTC_PACKED_OK;
}

// A plain launch (no early start): these kernels read what the kernel before
// them on the stream wrote without a programmatic wait.
template <typename K>
cudaError_t launch_fsa(K kernel, unsigned grid, size_t smem, cudaStream_t s, const FsaArgs& a) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kFsaThreads, smem, s>>>(a);
    return cudaGetLastError();
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
    a.L = fsa_layout(T_total, B, max_states, max_labels, D);
    return a;
}

}  // namespace

extern "C" {

size_t ctc_packed_fsa_workspace_size(int64_t T_total, int32_t B, int32_t max_states, int32_t max_labels, int32_t D) {
    if (T_total < 0 || B < 0 || max_states < 1 || max_states > kFsaMaxStates || T_total > INT32_MAX ||
        max_labels < 1 || D < 1 || D > kFsaMaxD)
        return 0;
    return fsa_layout(T_total, B, max_states, max_labels, D).total;
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
    const size_t smem = sizeof(float) * 3 * (size_t)max_states;
    cudaError_t e = dtype == CTC_PACKED_F32    ? launch_fsa(fsa_forward_kernel<0>, (unsigned)B, smem, stream, a)
                    : dtype == CTC_PACKED_BF16 ? launch_fsa(fsa_forward_kernel<1>, (unsigned)B, smem, stream, a)
                                               : launch_fsa(fsa_forward_kernel<2>, (unsigned)B, smem, stream, a);
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
    const long long hgrid = (T_total + kFsaThreads - 1) / kFsaThreads;
    if (launch_fsa(fsa_head_init_kernel, (unsigned)(hgrid < 4096 ? hgrid : 4096), 0, stream, a) != cudaSuccess)
        return CTC_PACKED_ERR_CUDA;
    // 2. per sequence: beta, edge occupancies, each row's class sums and header
    if (B > 0) {
        const size_t smem = sizeof(float) * (3 * (size_t)max_states + (size_t)D) + sizeof(int) * (size_t)a.L.cap;
        const cudaError_t e =
            dtype == CTC_PACKED_F32    ? launch_fsa(fsa_backward_kernel<0>, (unsigned)B, smem, stream, a)
            : dtype == CTC_PACKED_BF16 ? launch_fsa(fsa_backward_kernel<1>, (unsigned)B, smem, stream, a)
                                       : launch_fsa(fsa_backward_kernel<2>, (unsigned)B, smem, stream, a);
        if (e != cudaSuccess) return CTC_PACKED_ERR_CUDA;
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
