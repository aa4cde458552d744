// Shared definitions of the packed CTC kernels: workspace layout, the
// extended-range probability arithmetic of the recursions, the stored state
// encoding, element conversions and the async-copy primitives.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ctc_packed.h"

namespace ctcp {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr double kLog2eD = 1.4426950408889634074;
constexpr double kLn2D = 0.69314718055994530942;
constexpr int kMaxD = 1 << 20;        // classes of the CTC path; rows are streamed in batches
constexpr int kFsaMaxD = 16384;       // classes of the FSA path (its backward sums a frame in a shared row of D)
constexpr int kFsaMaxStates = 4096;  // states of one FSA sequence (shared-memory rows)
constexpr int kMaxTargetLen = 3839;   // 4 state pairs per lane, 31 own lanes in each of 32 warps
constexpr long long kSpinLimit = 1ll << 26;  // bounded waits give up after this many polls

// Control block at the start of the workspace.
struct Control {
    uint32_t status;      // OR of CTC_PACKED_DEV_* bits
    uint32_t big_head;    // next multi-warp chain item
    uint32_t small_head;  // next single-warp chain item
    uint32_t done_ctas;   // CTAs of the chain kernel that have finished
    uint32_t grad_ready;  // 1 once a forward has stored what the backward needs
    int32_t n_big, n_small, n_lab;
    uint32_t logits;      // 1: the forward took logits, normalised each row, and kept its log-sum-exp
    int32_t tl_total;     // sum of the target lengths (negative ones as 0): mean_volume's divisor
    uint32_t ckpt;        // the forward kept every state row (1) or only those at multiples of ckpt
    uint32_t pad[5];
};
static_assert(sizeof(Control) == 64, "control block is 64 bytes");

// Per-utterance metadata written by the prep kernel.
struct UttInfo {
    int32_t start;      // first row
    int32_t T;          // frames
    int32_t U;          // target length (0 when invalid)
    int32_t toff;       // first target id in the concatenated targets
    int32_t moff;       // first slot of this utterance in the label-metadata arrays
    int32_t valid;      // metadata well formed
    int32_t labels_ok;  // every target id in [0, D) (set by the label analysis)
    int32_t n_owners;   // distinct non-blank target classes + 1 (the blank group)
    int32_t has_nan;    // a label or blank log probability of the utterance is NaN (set by the emission gather)
    // nll * log2(e) = kint + log2(cfrac), cfrac in [1, 2), and whether nll is +inf (set by the alpha chain)
    int32_t kint;
    float cfrac;
    int32_t nll_inf;
    int32_t pad;
};

// Label record of target position j of an utterance (written by the label
// analysis): rank >= 0 for the first occurrence of a class (its index among
// the utterance's distinct classes), -1 for a later occurrence, -2 for a
// target id equal to the blank; next: the next position with the same class
// (-1: none); cls: the class.
struct LabelRec {
    int32_t rank, next, cls, pad;
};

// Per-row header of the backward's class sums (written by the posterior pass).
struct RowHead {
    int32_t count;    // class-sum entries of the row
    float scale;      // upstream gradient factor of the row's utterance (0 when not covered)
    int32_t covered;  // the row belongs to a well-formed utterance's frames
    int32_t pad;
};

// Byte offsets of every array inside the caller's workspace.
struct Layout {
    int64_t T_total;
    int32_t B, max_U, D, pitch;  // pitch: ints per stored state row (>= 2 * (max_U + 1))
    int32_t ecap;                // distinct classes a target can have: min(max_U + 1, D)
    int32_t gpairs;              // state pairs a chain warp owns (its offset group)
    int32_t nwo;                 // per-frame offsets stored per chain row (one per offset group)
    int32_t epitch;              // entries per row of the emission matrix (max_U + 1)
    int32_t owo;                 // per-frame offsets at the head of a stored row: nwo rounded up to 4
    int32_t spitch;              // ints per stored row: owo offsets, then pitch state ints
    int64_t lab_cap;             // label-metadata slots: B * max_U + B
    size_t off_ctrl, off_utt, off_queue, off_nll, off_alpha, off_beta;
    size_t off_lbl, off_em, off_head, off_ent, off_lse;
    size_t loss_only_total;      // a loss-only forward uses the arrays up to here only
    size_t total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Rows of padding before and after the emission matrix: a chain prefetches
// up to this many frames past either end of its utterance without a bounds
// check (those rows are never consumed).
constexpr int kEmPad = 8;

// The shape of a chain: the state pairs (blank, label) each lane holds (P)
// and the lanes of each warp that shadow the neighbouring warp's edge pairs
// (G), so that the warp runs G * P frames between two halo exchanges.  A
// warp owns group_pairs(P, G) pairs and at most 32 warps run a chain.
__host__ __device__ constexpr int group_pairs(int P, int G) { return (32 - G) * P; }
// The shape for a target bound:
//   one pair per lane, 8 shadow lanes, up to 16 warps (a chain CTA of at
//     most 512 threads keeps 128 registers a thread);
//   two pairs, 4 shadow lanes (8 frames an exchange), up to 16 warps;
//   two pairs, 2 shadow lanes (4 frames), up to 32 warps (an 8-frame ring of
//     32 warps would not fit shared memory);
//   four pairs, 1 shadow lane.
// (Measured: with one pair on the 8193-class workload 8 shadow lanes beat 4,
// 2 and 16; with two pairs on the long-form workload 4 shadow lanes took the
// forward from 0.910 to 0.853 ms against 2.)
__host__ __device__ inline void chain_shape_for_max_u(int max_u, int& P, int& G) {
    const int pairs = max_u + 1;
    if (pairs <= group_pairs(1, 8) * 16) {
        P = 1;
        G = 8;
    } else if (pairs <= group_pairs(2, 4) * 16) {
        P = 2;
        G = 4;
    } else if (pairs <= group_pairs(2, 2) * 32) {
        P = 2;
        G = 2;
    } else {
        P = 4;
        G = 1;
    }
}
__host__ __device__ inline int pairs_for_max_u(int max_u) {
    int P, G;
    chain_shape_for_max_u(max_u, P, G);
    return P;
}

__host__ __device__ inline Layout make_layout(int64_t T_total, int32_t B, int32_t max_U, int32_t D) {
    Layout L{};
    L.T_total = T_total;
    L.B = B;
    L.max_U = max_U;
    L.D = D;
    // a row holds 2 ints per state pair; a lane stores its P pairs as one
    // aligned vector, so the pitch is a multiple of 2P ints (and of 4)
    int P, G;
    chain_shape_for_max_u(max_U, P, G);
    L.pitch = (int32_t)align_up((size_t)(2 * (max_U + 1)), (size_t)(2 * P > 4 ? 2 * P : 4));
    L.ecap = (max_U + 1) < D ? (max_U + 1) : D;
    L.gpairs = group_pairs(P, G);
    {
        const int pairs = max_U + 1;
        const int nw = (pairs + L.gpairs - 1) / L.gpairs;
        L.nwo = nw < 1 ? 1 : nw;
    }
    L.owo = (L.nwo + 3) / 4 * 4;
    L.spitch = L.owo + L.pitch;
    L.epitch = max_U + 1;  // (label, blank) entries, then (zero, blank)
    L.lab_cap = (int64_t)B * max_U + B;
    size_t o = 0;
    L.off_ctrl = o;   o = align_up(o + sizeof(Control), 256);
    L.off_utt = o;    o = align_up(o + sizeof(UttInfo) * (size_t)B, 256);
    L.off_queue = o;  o = align_up(o + sizeof(int32_t) * (3 * (size_t)B + 1), 256);
    L.off_nll = o;    o = align_up(o + sizeof(double) * (size_t)B, 256);
    L.off_em = o;     o = align_up(o + 16 * (size_t)(T_total + 2 * kEmPad) * (size_t)L.epitch, 256);
    L.off_lse = o;    o = align_up(o + sizeof(float) * (size_t)T_total, 256);
    L.loss_only_total = o;
    // what only the backward reads: the stored rows, label records, class sums
    L.off_alpha = o;  o = align_up(o + sizeof(int32_t) * (size_t)T_total * (size_t)L.spitch, 256);
    L.off_beta = o;   o = align_up(o + sizeof(int32_t) * (size_t)T_total * (size_t)L.spitch, 256);
    L.off_lbl = o;    o = align_up(o + sizeof(int4) * (size_t)L.lab_cap, 256);
    L.off_head = o;   o = align_up(o + sizeof(RowHead) * (size_t)T_total, 256);
    L.off_ent = o;    o = align_up(o + 8 * (size_t)T_total * (size_t)L.ecap, 256);
    L.total = o;
    return L;
}

template <typename T>
__host__ __device__ inline T* ws_at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<unsigned char*>(ws) + off);
}
template <typename T>
__host__ __device__ inline const T* ws_at(const void* ws, size_t off) {
    return reinterpret_cast<const T*>(static_cast<const unsigned char*>(ws) + off);
}
// Row 0 of the emission matrix (after its leading padding).
__host__ __device__ inline size_t em_base(const Layout& L) { return L.off_em + 16 * (size_t)kEmPad * (size_t)L.epitch; }

// Element types: 0 float32, 1 bfloat16, 2 float16.
template <int DT>
struct Elem {
    static constexpr int bytes = DT == 0 ? 4 : 2;
};

// ---------------------------------------------------------------- arithmetic

__device__ __forceinline__ float fast_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// ------------------------------------------- extended-range probabilities
//
// The recursions run on probabilities, not logs: a state is m * 2^e with a
// float mantissa m in [1, 2) (0 for an unreachable state) and its own int32
// binary exponent e, so no state ever under- or overflows and the chain needs
// no exp/log at all -- only multiply-adds and integer exponent arithmetic,
// rounded to nearest (unbiased).  An emission p = exp(lp) enters as
// (mp, ep) with lp * log2(e) split exactly into an integer and a fraction;
// the ex2 approximation of the fraction acts as a ~1e-7 relative perturbation
// of that one input probability, shared bit for bit by the forward and the
// backward chain.  (A log-space float32 recursion instead accumulates the
// bias of the fast log2 near 1 on every step: ~2e-5 on the posteriors of a
// 2000-frame utterance.)

constexpr int kEZero = -(1 << 29);    // exponent of an unreachable state (m = 0)
constexpr int kEZeroEm = -(1 << 24);  // exponent of a zero emission: a recursion adds emission
                                      // exponents over a few frames between renormalisations
constexpr float kL2eHi = 1.4426950216293335f;     // float(log2 e)
constexpr float kL2eLo = 1.9259629911783890e-8f;  // log2 e - kL2eHi

struct XP {
    float m;  // mantissa, 0 for probability 0
    int e;    // binary exponent
};
// One entry of the emission matrix: a label's emission and the frame's blank
// emission side by side, so one 16-byte copy brings a lane both.
struct __align__(16) XP2 {
    XP l, b;
};

// exp(lp) in extended form.  lp * log2 e = yh + yl exactly (FMA), then
// exp(lp) = 2^floor(yh) * 2^((yh - floor(yh)) + yl), the mantissa in (1-2^-23, 2].
__device__ __forceinline__ XP xp_from_log(float lp) {
    const float yh = lp * kL2eHi;
    const float yl = fmaf(lp, kL2eLo, fmaf(lp, kL2eHi, -yh));
    const float fl = floorf(yh);
    XP r;
    r.m = fast_ex2((yh - fl) + yl);
    r.e = (int)fminf(fl, 16777216.0f);  // log probabilities above 2^24 saturate (no overflow downstream)
    if (!(yh > -3.0e7f)) {  // exp(lp) == 0: lp = -inf, below any representable probability, or NaN
        r.m = 0.0f;         // (callers flag a NaN separately)
        r.e = kEZeroEm;
    }
    return r;
}

// 2^k for k <= 0, flushed to 0 below 2^-126 (an exact power of two).
__device__ __forceinline__ float pow2_nonpos(int k) { return __int_as_float(max(127 + k, 0) << 23); }

// (m, e) with m rescaled into [1, 2); 0 becomes (0, kEZero).  m is a finite
// non-negative normal number or 0 (a sum of normalised mantissas times an
// emission mantissa never leaves [1, 12)).
__device__ __forceinline__ XP xp_norm(float m, int e) {
    const int bits = __float_as_int(m);
    XP r;
    r.m = bits == 0 ? 0.0f : __int_as_float((bits & 0x007fffff) | 0x3f800000);
    r.e = bits == 0 ? kEZero : e + ((bits >> 23) - 127);
    return r;
}

// Sum of two / three extended values, as an unnormalised (S, E): S in [0, 6).
__device__ __forceinline__ void xp_sum2(XP a, XP b, float& S, int& E) {
    E = max(a.e, b.e);
    S = fmaf(a.m, pow2_nonpos(a.e - E), b.m * pow2_nonpos(b.e - E));
}
__device__ __forceinline__ void xp_sum3(XP a, XP b, XP c, float& S, int& E) {
    E = max(a.e, max(b.e, c.e));
    S = fmaf(a.m, pow2_nonpos(a.e - E), fmaf(b.m, pow2_nonpos(b.e - E), c.m * pow2_nonpos(c.e - E)));
}

// Stored form of a state for the backward: the value S * 2^(E - A), relative
// to a per-(frame, warp) integer offset A, as one int32 that holds it
// exactly up to rounding: the top 13 bits are the signed binary exponent k,
// the low kFixFrac = 19 bits the mantissa fraction (rounded to nearest), so
// v = k * 2^19 + frac19 and the value is (1 + frac19 / 2^19) * 2^k.  The int
// order follows the value order.  Built from the float's own bits (no log):
// (bits + 8) >> 4 is the float's biased exponent and top 19 mantissa bits,
// rounded, with a carry moving into the exponent.  S may be any finite
// non-negative float, normalised or not.  A state more than 2^3800 below the
// offset is stored as zero (a posterior can only be understated by it).
constexpr int kFixFrac = 19;
constexpr int kFixZero = (int)0x80000000;  // probability 0
__device__ __forceinline__ int enc_state(float S, int E, int A) {
    const int d = E - A;
    const int v = ((__float_as_int(S) + 8) >> 4) + ((d - 127) << kFixFrac);
    return (S > 0.0f && d >= -3800) ? v : kFixZero;
}

// ------------------------------------------------------------- conversions

// The value of element `half` (0 low, 1 high) of a 32-bit word in dtype DT.
template <int DT>
__device__ __forceinline__ float word_to_float(uint32_t w, int half) {
    if constexpr (DT == 0) {
        return __uint_as_float(w);
    } else if constexpr (DT == 1) {
        return __uint_as_float(half ? (w & 0xffff0000u) : (w << 16));
    } else {
        unsigned short h = half ? (unsigned short)(w >> 16) : (unsigned short)(w & 0xffffu);
        return __half2float(__ushort_as_half(h));
    }
}
template <int DT>
__device__ __forceinline__ float bits_to_float(uint32_t bits) {  // bits of one element in the low part
    if constexpr (DT == 0) {
        return __uint_as_float(bits);
    } else if constexpr (DT == 1) {
        return __uint_as_float(bits << 16);
    } else {
        return __half2float(__ushort_as_half((unsigned short)bits));
    }
}
// Round-to-nearest-even conversion of two floats into one packed word.
template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (DT == 1) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}
template <int DT>
__device__ __forceinline__ uint32_t pack1(float x) {  // one element in the low bits
    if constexpr (DT == 0) {
        return __float_as_uint(x);
    } else if constexpr (DT == 1) {
        __nv_bfloat16 v = __float2bfloat16_rn(x);
        return (uint32_t)(*reinterpret_cast<unsigned short*>(&v));
    } else {
        __half v = __float2half_rn(x);
        return (uint32_t)(*reinterpret_cast<unsigned short*>(&v));
    }
}

// ------------------------------------------------------- async-copy helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Returns true once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Bulk copy global -> shared (both 16-byte aligned, size a multiple of 16),
// completion reported on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ------------------------------------------------- dense gradient chunks

// Asks L2 to fetch bytes [lo, hi) ahead of use, rounded inward to 16 bytes
// (a bulk prefetch is a hint: it holds no register and completes nothing).
__device__ __forceinline__ void prefetch_l2(uintptr_t lo, uintptr_t hi) {
    lo = (lo + 15) & ~uintptr_t(15);
    hi &= ~uintptr_t(15);
    if (hi > lo)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"((uint32_t)(hi - lo)) : "memory");
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

// Gradient of one whole 16-byte chunk: s * exp(lp) + pn element by element,
// pn the chunk's negated class sums (zero where none), in pairs on the
// paired fp32 pipes, rounded once into the chunk's dtype.  exp(lp) is
// 2^(x log2 e + bias): bias = 0 for log probabilities, -lse log2 e for a row
// of logits (then exp(lp) is the row's softmax); x log2 e + 0 rounds as the
// product alone, so log-probability rows are unchanged by the bias.
template <int DT>
__device__ __forceinline__ uint4 chunk_grad(uint4 in, float s, const float (&pn)[16 / Elem<DT>::bytes], float bias) {
    const float2 l2e = make_float2(kLog2e, kLog2e), s2 = make_float2(s, s), b2 = make_float2(bias, bias);
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    if constexpr (DT == 0) {
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
            const float2 t = __ffma2_rn(make_float2(__uint_as_float(w[i]), __uint_as_float(w[i + 1])), l2e, b2);
            const float2 r = __ffma2_rn(s2, make_float2(fast_ex2(t.x), fast_ex2(t.y)), make_float2(pn[i], pn[i + 1]));
            o[i] = r.x;
            o[i + 1] = r.y;
        }
        return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]), __float_as_uint(o[3]));
    } else {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 x;
            if constexpr (DT == 1) {  // bfloat16: the high half is already a float
                x = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
            } else {
                x = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            }
            const float2 t = __ffma2_rn(x, l2e, b2);
            const float2 r =
                __ffma2_rn(s2, make_float2(fast_ex2(t.x), fast_ex2(t.y)), make_float2(pn[2 * i], pn[2 * i + 1]));
            o[i] = pack2<DT>(r.x, r.y);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
}


// s * exp(lp) of a whole 16-byte chunk, element by element in pairs,
// rounded once into the chunk's dtype: the gradient of a chunk that holds no
// class sum.
template <int DT>
__device__ __forceinline__ uint4 chunk_scaled(uint4 in, float s, float bias) {
    const float2 l2e = make_float2(kLog2e, kLog2e), s2 = make_float2(s, s), b2 = make_float2(bias, bias);
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    if constexpr (DT == 0) {
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
            const float2 t = __ffma2_rn(make_float2(__uint_as_float(w[i]), __uint_as_float(w[i + 1])), l2e, b2);
            const float2 r = __fmul2_rn(s2, make_float2(fast_ex2(t.x), fast_ex2(t.y)));
            o[i] = r.x;
            o[i + 1] = r.y;
        }
        return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]), __float_as_uint(o[3]));
    } else {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 x;
            if constexpr (DT == 1) {
                x = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
            } else {
                x = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            }
            const float2 t = __ffma2_rn(x, l2e, b2);
            const float2 r = __fmul2_rn(s2, make_float2(fast_ex2(t.x), fast_ex2(t.y)));
            o[i] = pack2<DT>(r.x, r.y);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__device__ __forceinline__ void set_status(Control* ctrl, uint32_t bits) { atomicOr(&ctrl->status, bits); }

// ------------------------------------------------ programmatic dependent launch
//
// Every kernel is launched with programmatic stream serialization, so it can
// be scheduled while the kernel before it on the stream drains.  pdl_wait()
// blocks until that kernel has completed and its writes are visible (a no-op
// when launched without the attribute); it comes before anything that reads
// what the stream's earlier work wrote.  pdl_trigger() lets the next kernel's
// blocks be scheduled from now on; only kernels whose blocks are all resident
// from the start (persistent grids, one-CTA kernels) call it early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace ctcp
