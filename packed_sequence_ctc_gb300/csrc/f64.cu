// Float64 path of the packed CTC loss: float64 log probabilities (or logits)
// in, a float64 loss and gradient out, on the same packed layout as the other
// dtypes (token-flat rows, cu_seqlens, concatenated targets) and with no
// padded tensor.
//
// Page "feat(asr): native CTC loss kernel over sequence-packed log
// probabilities": ctc.py ``forward_packed`` keeps float64 inputs on a path of
// their own at float64 precision (its Triton kernels take float32, bfloat16
// and float16 only), and test_ctc_loss.py ``test_float64_takes_padded_path``
// holds that path to 1e-10.  The recursion and gradient are the ones of
// ctc_loss.py (``_alpha_kernel``, ``_beta_grad_kernel``): alpha over the
// extended label sequence, beta from the last frame (here in the forward
// call, beside alpha, where the page recomputes it in the backward), and
// grad[t, c] = scale * (exp(lp[t, c]) - sum_{s: l(s) = c} gamma_t(s)) with
// gamma_t(s) = alpha_t(s) beta_t(s) / Z.
//
// Arithmetic.  A probability is carried in extended range: a 62-bit integer
// mantissa (its leading one at bit 61) and an int exponent (zero: m = 0).
// The recursions then take no exp, log or float64 operation per state and
// frame, which matters on a part whose float64 rate is a small fraction of
// its integer and float32 rates: a sum shifts its terms to the largest
// exponent and adds them, a product takes the high 62 bits of the mantissa
// product and adds the exponents, and each emission exp(lp[t, c]) is
// converted once, in a parallel gather.  Every step keeps 62 bits, so the
// loss and gradient keep float64's digits over thousands of frames.  The
// posteriors go to fixed point (units of 2^-62) for the class sums, which
// are then exact integer sums.
//
// Kernels, in stream order.  Forward:
//   prep    one CTA: utterance checks, target offsets, the losses of
//           utterances without frames
//   lse     (logits) one warp per row: the row's log-sum-exp
//   emit    one warp per row: exp(lp[t, c]) of the row's labels and blank
//           (Tang's table-driven exp in float64, see x_from_log)
//   chain   one CTA per utterance and recursion, a thread per state (or per
//           few), one barrier per frame: the alpha recursion (every alpha
//           row stored, Z and the nll per utterance) and, when the
//           gradient's state is kept, the beta recursion at the same time on
//           CTAs of its own (the label analysis, distinct classes in target
//           order, then every beta row stored)
//   reduce  one CTA: the reduced loss in a fixed summation order
// Backward:
//   post    a small CTA per row at a time: the row's posteriors from the
//           two stored rows, summed per distinct class (exact integer sums),
//           as gradient entries
//   grad    one warp per row: scale * exp(lp) for every class (a table-driven
//           exp, see exp_table), then each class sum rewrites its element,
//           scale * exp(lp) - scale * P
// Every sum runs in a fixed order, so results are bitwise reproducible.
#include <cmath>
#include <cstdint>

#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

constexpr int kZeroE = -(1 << 30);  // exponent of zero; values below 2^kZeroE flush to zero
constexpr int kRowWarps = 8;        // warps (rows) per CTA of the row kernels
constexpr int kMaxChainThreads = 1024;
// Frames of a recursion's emissions in flight through shared memory, RING - 1
// ahead of the frame computed: 4 up to 2048 states a CTA; larger CTAs load
// one frame ahead into registers (their rings would not fit).
__host__ __device__ constexpr int f64_ring(int per) { return per <= 2 ? 4 : 0; }

// Extended-range value m * 2^(e - 61): m an integer with its leading one at
// bit 61 (62 significant bits, carried on the integer pipes: this part's
// float64 pipe is narrow), or zero (m = 0, e = kZeroE).  NaN and infinite
// inputs are flagged apart (the utterance's loss is NaN).
struct X64 {
    unsigned long long m;
    int e;
};
constexpr unsigned long long kXOne = 1ull << 61;  // the mantissa of 1

// Emission entry of the workspace (16 bytes).
struct EmX {
    unsigned long long m;
    int32_t e, pad;
};

// Per-utterance record of the float64 path (64 bytes).
struct F64Utt {
    int32_t start, T, U, toff;
    int32_t valid;      // cu_seqlens, lengths and target length well formed
    int32_t labels_ok;  // every target id in [0, D) (cleared by the alpha recursion)
    int32_t has_nan;    // a label or blank log probability of the utterance is NaN
    int32_t nll_inf;    // no alignment: Z = 0
    int32_t ncls;       // distinct classes of the target, the blank included (label analysis)
    int32_t ze;
    int32_t bfirst;     // first target position whose id is the blank, -1: none (label analysis)
    int32_t pad1;
    double nll, zm;     // nll, and Z = zm * 2^ze
};
static_assert(sizeof(F64Utt) == 64, "utterance record is 64 bytes");

struct F64Layout {
    int64_t T_total;
    int32_t B, max_U, D;
    int32_t Ep;    // emission entries per row: max_U labels, then the blank
    int32_t Sp;    // stored alpha states per row: 2 max_U + 1, padded to even
    int32_t ecap;  // class sums a row can hold: min(max_U + 1, D)
    size_t off_ctrl, off_utt, off_lse, off_em, loss_only_total, off_am, off_ae, off_bm, off_bx, off_lrec, off_cls,
        off_ent, total;
};

__host__ __device__ inline F64Layout f64_layout(int64_t T, int32_t B, int32_t max_U, int32_t D) {
    F64Layout L{};
    L.T_total = T;
    L.B = B;
    L.max_U = max_U;
    L.D = D;
    L.Ep = max_U + 1;
    L.Sp = 2 * max_U + 2;
    L.ecap = L.Ep < D ? L.Ep : D;
    size_t o = 0;
    L.off_ctrl = o; o = align_up(o + sizeof(Control), 256);
    L.off_utt = o;  o = align_up(o + sizeof(F64Utt) * (size_t)B, 256);
    L.off_lse = o;  o = align_up(o + sizeof(double) * (size_t)T, 256);
    L.off_em = o;   o = align_up(o + sizeof(EmX) * (size_t)T * (size_t)L.Ep, 256);
    L.loss_only_total = o;
    // what only the backward reads
    L.off_am = o;   o = align_up(o + sizeof(double) * (size_t)T * (size_t)L.Sp, 256);
    L.off_ae = o;   o = align_up(o + sizeof(int32_t) * (size_t)T * (size_t)L.Sp, 256);
    // beta_t(s) before frame t's emission, every row (the beta recursion)
    L.off_bm = o;   o = align_up(o + sizeof(double) * (size_t)T * (size_t)L.Sp, 256);
    L.off_bx = o;   o = align_up(o + sizeof(int32_t) * (size_t)T * (size_t)L.Sp, 256);
    // per target position: the rank of a first occurrence (-1 otherwise) and
    // the next position with the same class (-1: none)
    L.off_lrec = o; o = align_up(o + sizeof(int2) * (size_t)B * (size_t)L.Ep, 256);
    L.off_cls = o;  o = align_up(o + sizeof(int32_t) * (size_t)B * (size_t)L.Ep, 256);
    L.off_ent = o;  o = align_up(o + sizeof(double) * (size_t)T * (size_t)L.ecap, 256);
    L.total = o;
    return L;
}

struct F64Args {
    F64Layout L;
    void* ws;
    const double* lp;
    double* grad;
    const int32_t* cu;
    const int32_t* lengths;
    const int32_t* targets;
    const int32_t* target_lengths;
    double* loss;
    const double* grad_loss;
    int D, blank, reduction, zero_infinity, need_grad, logits;
};

// ------------------------------------------------------------ extended range

__device__ __forceinline__ X64 x_zero() { return X64{0ull, kZeroE}; }

// m * 2^(e - 61) (m < 2^64) with m's leading one moved to bit 61; exponents
// below kZeroE give zero, above 2^30 saturate.
__device__ __forceinline__ X64 x_norm(unsigned long long m, long long e) {
    if (m == 0) return x_zero();
    const int sh = __clzll((long long)m) - 2;
    const unsigned long long mm = sh >= 0 ? m << sh : m >> -sh;
    const long long ne = e - sh;
    if (ne <= kZeroE) return x_zero();
    return X64{mm, (int)min(ne, (long long)(1 << 30))};
}

// a + b + c: each mantissa shifted to the largest exponent (bits below the
// 62nd drop out), summed (below 3 * 2^62), renormalised.
__device__ __forceinline__ X64 x_add3(X64 a, X64 b, X64 c) {
    const int E = max(a.e, max(b.e, c.e));
    auto aligned = [&](X64 x) {
        const long long d = (long long)E - x.e;
        return d < 62 ? x.m >> d : 0ull;
    };
    return x_norm(aligned(a) + aligned(b) + aligned(c), E);
}

// a * b: the 124-bit product of the mantissas, its leading 62 bits (the
// high word moved up by 2 or 3 with the low word's top bits).
__device__ __forceinline__ X64 x_mul(X64 a, X64 b) {
    const unsigned long long hi = __umul64hi(a.m, b.m), lo = a.m * b.m;
    if (hi == 0) return x_zero();  // a zero factor: normalised products are at least 2^122
    const int s = __clzll((long long)hi) - 2;  // 2 or 3
    const long long e = (long long)a.e + b.e + 3 - s;
    if (e <= kZeroE) return x_zero();
    return X64{(hi << s) | (lo >> (64 - s)), (int)min(e, (long long)(1 << 30))};
}

// A positive normal float64 v times 2^k in extended range, by v's bits.
__device__ __forceinline__ X64 x_of_double(double v, long long k) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(v);
    const long long e = (long long)(u >> 52) - 1023 + k;
    if (e <= kZeroE) return x_zero();
    return X64{((u & 0xfffffffffffffull) | (1ull << 52)) << 9, (int)min(e, (long long)(1 << 30))};
}

// The mantissa of a nonzero extended value as a float64 in [1, 2).
__device__ __forceinline__ double x_mantissa(X64 x) { return __ull2double_rn(x.m) * 0x1p-61; }

// exp(x) in extended range by Tang's table-driven method (P. T. P. Tang,
// ACM TOMS 15(2), 1989) in float64: n = round(x * 64 / ln2) by the
// 1.5 * 2^52 rounding constant, r = x - n ln2/64 by two fused multiply-adds
// (ln2/64 as a float64 and its remainder), |r| <= ln2/128; exp(r) - 1 by its
// Taylor polynomial to r^5 (the next term is below 2^-53 of the result);
// exp(x) = 2^(n >> 6) * T[n & 63] * (1 + p), T[j] = 2^(j/64) from a table the
// caller fills.  About ten float64 operations, within about one unit in the
// last place, the mantissa taken by its bits and the exponent kept apart (no
// underflow).  -inf gives zero, and so do NaN and +inf (the caller flags
// those).
constexpr double kLn2o64D = 0.010830424696249145;     // ln 2 / 64, rounded
constexpr double kLn2o64LoD = 3.623510646634843e-19;   // ln 2 / 64 minus the above
constexpr double k64oLn2D = 92.332482616893656;
__device__ __forceinline__ X64 x_from_log(double x, const double* T) {
    if (!(x > -1.0e9) || !(x < INFINITY)) return x_zero();  // below 2^kZeroE (or NaN, +-inf)
    if (x > 1.0e9) x = 1.0e9;                                // saturates (see x_of_double)
    const double t = fma(x, k64oLn2D, 0x1.8p52);
    const long long n = __double_as_longlong(t) - __double_as_longlong(0x1.8p52);
    const double nd = t - 0x1.8p52;
    const double r = fma(-nd, kLn2o64LoD, fma(-nd, kLn2o64D, x));
    double q = fma(r, 1.0 / 120.0, 1.0 / 24.0);
    q = fma(r, q, 1.0 / 6.0);
    q = fma(r, q, 0.5);
    const double p = fma(r * r, q, r);
    const double tj = T[n & 63];
    return x_of_double(fma(tj, p, tj), n >> 6);
}

// ln 2 / 64 in units of 2^-53: kLn2o64Hi + kLn2o64Lo / 2^11 (within 2^-12
// of a unit).
constexpr long long kLn2o64Hi = 97551793252583ll;
constexpr long long kLn2o64Lo = 1511;

// exp(x) by Tang's table-driven method (P. T. P. Tang, "Table-driven
// implementation of the exponential function in IEEE floating-point
// arithmetic", ACM TOMS 15(2), 1989), shaped for a part with a narrow float64
// pipe: one float64 operation an element, the reduction on the integer pipe.
// x = (64 k + j) ln2/64 + r, with n = 64 k + j = round(x * 64/ln2) taken in
// float32 from x's fixed-point form below: a rounding off by one only leaves
// |r| < ln2/64.  x and n ln2/64
// are formed as 64-bit integers in units of 2^-53 (x's bits below 2^-53
// drop out), so their difference R is r * 2^53 to within a unit.  Then
// exp(r) = 1 + s, s = r + q, q = r^2/2 + r^3/6 + r^4/24 in float32 from R's
// leading bits: |q| < 6e-5, so float32 rounds it to within 4e-12, and the
// dropped r^5/120 is below 1.3e-12.  q joins R (rounded to 2^-40), and the
// sum S, |S| < 2^47, is added to the bit pattern of 0.75, which in [0.5, 1)
// moves by one per 2^-53: that is 0.75 + s exactly.  Finally exp(x) =
// 2^k * T[j] * (1 + s) = fma(T[j], 0.75 + s, T[j] / 4), with T[j] =
// 2^(j/64) from a table the caller fills (shared memory), the quarter and
// 2^k taken on the exponent field.  A table c * 2^(j/64) gives c * exp(x) (the caller keeps
// c * exp(x) a normal number).  The relative error is below about 1e-11;
// the gradient it feeds is held to 1e-10.  |x| >= 512, NaN and infinities
// take the library exp, times T[0] (the test is on the exponent field).
__device__ __forceinline__ double exp_table(double x, const double* T) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(x);
    const int ex = (int)(u >> 52 & 0x7ff);
    if (ex >= 1023 + 9) return T[0] * exp(x);  // T[0]: the table's own factor
    // x * 2^53: the significand (implicit bit included) moved by ex - 1022
    // bits, at most 9 to the left (62 bits in all): moved 10 left, then
    // 1032 - ex right
    const unsigned long long sig = ((u & 0xfffffffffffffull) | (1ull << 52)) << 10;
    long long X = (long long)(sig >> min(1032 - ex, 63));
    if (u >> 63) X = -X;
    // n from X's high word (|x| < 2^-21 gives 0, as it should)
    const int n = __float2int_rn((float)(int)(X >> 32) * (92.332482616893656f * 0x1p-21f));  // 64 / ln 2
    const long long R = X - ((long long)n * kLn2o64Hi + (((long long)n * kLn2o64Lo + 1024) >> 11));
    // r in float32 from R's bits down to 2^-37 (|R| < 2^47: 31 bits)
    const float rf = (float)(int)(R >> 16) * 0x1p-37f;
    const float q = rf * rf * fmaf(rf, fmaf(rf, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f);  // >= 0
    // q in units of 2^-40 (below 2^27: one conversion), then 2^-53
    const long long S = R + ((long long)__float2int_rn(q * 0x1p40f) << 13);
    // 0.75 + s by its bits: in [0.5, 1) a float64's bit pattern moves by one
    // per 2^-53, so adding S to 0.75's pattern is exact; then
    // T[j] (1 + s) = fma(T[j], 0.75 + s, T[j] / 4), the quarter by the
    // exponent field (exact)
    const double s75 = __longlong_as_double(0x3FE8000000000000ll + S);
    const double t = T[n & 63];
    const double t4 = __longlong_as_double(__double_as_longlong(t) - (2ll << 52));
    const double y = fma(t, s75, t4);  // in [0.98, 2.03) times the table's factor
    return __longlong_as_double(__double_as_longlong(y) + ((long long)(n >> 6) << 52));
}

// Fills the 64-entry table of exp_table (2^(j/64)); the caller synchronises.
__device__ __forceinline__ void fill_exp_table(double* T) {
    if (threadIdx.x < 64) T[threadIdx.x] = exp2((double)threadIdx.x * (1.0 / 64.0));
}

__device__ __forceinline__ X64 ld_em(const EmX* p) {
    const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(p);
    return X64{v.x, (int)(long long)v.y};
}

// 16-byte async copy global -> shared.
__device__ __forceinline__ void cp_async_n16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// ------------------------------------------------------------ helpers

__device__ __forceinline__ int f64_utterance_of_row(const int32_t* cu, int B, int64_t row) {
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

// Upstream gradient factor of utterance b under the call's reduction.
__device__ __forceinline__ double f64_scale(const F64Args& a, const F64Utt& u, int b, int tl_total) {
    double s;
    if (a.reduction == CTC_PACKED_NONE) {
        s = a.grad_loss[b];
    } else if (a.reduction == CTC_PACKED_SUM) {
        s = a.grad_loss[0];
    } else if (a.reduction == CTC_PACKED_MEAN) {
        s = a.grad_loss[0] / ((double)a.L.B * (double)max(u.U, 1));
    } else if (a.reduction == CTC_PACKED_MEAN_BATCH) {
        s = a.grad_loss[0] / (double)a.L.B;
    } else {
        s = a.grad_loss[0] / (double)tl_total;
    }
    if (a.zero_infinity && u.nll_inf) s = 0.0;
    return s;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exclusive scan of one value per thread over the CTA (blockDim a multiple
// of 32); the CTA total goes to *total.
__device__ int f64_block_scan(int v, int* s_warp, int* total) {
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

}  // namespace

// ------------------------------------------------------------ forward kernels

__global__ void __launch_bounds__(1024) f64_prep_kernel(F64Args a) {
    __shared__ int s_warp[32];
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    F64Utt* utt = ws_at<F64Utt>(a.ws, a.L.off_utt);
    const int B = a.L.B, tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) {
        *ctrl = Control{};
        ctrl->grad_ready = a.need_grad ? 1u : 0u;
        ctrl->logits = a.logits ? 1u : 0u;
        ctrl->ckpt = 1;
    }
    __syncthreads();
    uint32_t bad_bits = 0;
    int toff_base = 0;
    for (int base = 0; base < B; base += nt) {
        const int b = base + tid;
        int T = 0, uraw = 0, c0 = 0, valid = 0;
        if (b < B) {
            c0 = a.cu[b];
            const int c1 = a.cu[b + 1];
            T = a.lengths[b];
            uraw = a.target_lengths[b];
            uint32_t bits = 0;
            if (uraw < 0) bits |= CTC_PACKED_DEV_NEGATIVE_TARGET_LENGTH;
            if (uraw > a.L.max_U) bits |= CTC_PACKED_DEV_TARGET_LENGTH_EXCEEDS_MAX;
            if (c0 < 0 || c1 < c0 || (int64_t)c1 > a.L.T_total) bits |= CTC_PACKED_DEV_BAD_CU_SEQLENS;
            if (T < 0 || (int64_t)T > (int64_t)c1 - (int64_t)c0) bits |= CTC_PACKED_DEV_BAD_LENGTH;
            bad_bits |= bits;
            valid = bits == 0;
        }
        int total;
        const int toff = toff_base + f64_block_scan(b < B ? max(uraw, 0) : 0, s_warp, &total);
        if (b < B) {
            F64Utt u{};
            u.start = c0;
            u.T = valid ? T : 0;
            u.U = valid ? uraw : 0;
            u.toff = toff;
            u.valid = valid;
            u.labels_ok = 1;
            u.nll_inf = (valid && T == 0 && uraw > 0) ? 1 : 0;
            u.ze = kZeroE;
            // utterances without a recursion get their loss here
            const double v = !valid ? __longlong_as_double(0x7ff8000000000000ll)
                                    : (T == 0 ? (uraw == 0 ? 0.0 : __longlong_as_double(0x7ff0000000000000ll)) : 0.0);
            u.nll = v;
            utt[b] = u;
            if ((!valid || T == 0) && a.reduction == CTC_PACKED_NONE)
                a.loss[b] = (a.zero_infinity && isinf(v)) ? 0.0 : v;
        }
        toff_base += total;
    }
    if (bad_bits) atomicOr(&ctrl->status, bad_bits);
    if (tid == 0) ctrl->tl_total = toff_base;
}

// Row log-sum-exp of logits: max, then the sum of exp(z - max).  A NaN or
// +inf logit gives NaN, a row of -inf gives -inf.
__global__ void __launch_bounds__(kRowWarps * 32) f64_lse_kernel(F64Args a) {
    __shared__ double s_exp[64];
    fill_exp_table(s_exp);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    double* lse = ws_at<double>(a.ws, a.L.off_lse);
    const int D = a.D;
    const int64_t warps = (int64_t)gridDim.x * kRowWarps;
    for (int64_t row = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5); row < a.L.T_total; row += warps) {
        const double* z = a.lp + row * D;
        double m = -INFINITY;
        bool bad = false;
        for (int c = lane; c < D; c += 32) {
            const double v = __ldg(z + c);
            bad |= (v != v) || v == INFINITY;
            m = fmax(m, v);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, o));
        bad = __any_sync(0xffffffffu, bad);
        double s = 0.0;
        if (!bad && m > -INFINITY)
            for (int c = lane; c < D; c += 32) s += exp_table(__ldg(z + c) - m, s_exp);
        s = warp_sum(s);
        if (lane == 0)
            lse[row] = bad ? __longlong_as_double(0x7ff8000000000000ll) : (m == -INFINITY ? m : m + log(s));
    }
}

// exp(lp[t, c]) in extended range for the U labels of the row's utterance
// and its blank (entry U).  A label outside [0, D) gets zero here; the
// recursion rejects the utterance.
__global__ void __launch_bounds__(kRowWarps * 32) f64_emit_kernel(F64Args a) {
    __shared__ double s_exp[64];
    fill_exp_table(s_exp);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    F64Utt* utt = ws_at<F64Utt>(a.ws, a.L.off_utt);
    EmX* em = ws_at<EmX>(a.ws, a.L.off_em);
    const double* lse = ws_at<double>(a.ws, a.L.off_lse);
    const int D = a.D, Ep = a.L.Ep;
    const int64_t warps = (int64_t)gridDim.x * kRowWarps;
    for (int64_t row = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5); row < a.L.T_total; row += warps) {
        const int b = f64_utterance_of_row(a.cu, a.L.B, row);
        if (b < 0) continue;
        const F64Utt u = utt[b];
        const int64_t t = row - u.start;
        if (!u.valid || t < 0 || t >= u.T) continue;
        const double sh = a.logits ? lse[row] : 0.0;
        const double* x = a.lp + row * D;
        EmX* out = em + row * Ep;
        bool nan = false;
        for (int k = lane; k <= u.U; k += 32) {
            const int c = k < u.U ? a.targets[u.toff + k] : a.blank;
            X64 v = x_zero();
            if (c >= 0 && c < D) {
                const double y = __ldg(x + c) - sh;
                nan |= !(y < INFINITY);  // NaN or +inf: the utterance's loss is NaN
                v = x_from_log(y, s_exp);
            }
            *reinterpret_cast<ulonglong2*>(out + k) = make_ulonglong2(v.m, (unsigned long long)(long long)v.e);
        }
        if (__any_sync(0xffffffffu, nan) && lane == 0) atomicOr(&utt[b].has_nan, 1);
    }
}

// Forward recursion of one utterance: thread i holds states i, i + nt, ...
// (PER of them); the previous frame's values sit in shared memory, double
// buffered, so one barrier per frame separates a frame's writes from the
// next frame's reads.  The next frame's emissions load during the current
// frame.
template <int PER>
__device__ __forceinline__ void f64_alpha_chain(const F64Args& a, int b) {
    constexpr int RING = f64_ring(PER);
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_bad;
    const int tid = threadIdx.x, nt = blockDim.x;
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    F64Utt* utt = ws_at<F64Utt>(a.ws, a.L.off_utt);
    const F64Utt u = utt[b];
    if (!u.valid || u.T == 0) return;
    const int U = u.U, S = 2 * U + 1, T = u.T, Ep = a.L.Ep, Sp = a.L.Sp;
    const int cap = PER * nt;
    unsigned long long* const mbuf = reinterpret_cast<unsigned long long*>(smem);  // two buffers of cap mantissas
    int* const ebuf = reinterpret_cast<int*>(mbuf + 2 * cap);      // two buffers of cap exponents
    EmX* const ring = reinterpret_cast<EmX*>(ebuf + 2 * cap);      // RING frames of the states' emissions
    if (tid == 0) s_bad = 0;
    __syncthreads();
    const int32_t* tg = a.targets + u.toff;
    int ent[PER];
    bool skip[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int s = tid + k * nt;
        ent[k] = U;
        skip[k] = false;
        if (s < S && (s & 1)) {
            const int j = s >> 1;
            const int c = tg[j];
            if (c < 0 || c >= a.D) s_bad = 1;
            ent[k] = j;
            skip[k] = j >= 1 && c != tg[j - 1];
        }
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            set_status(ctrl, CTC_PACKED_DEV_LABEL_OUT_OF_RANGE);
            const double nan = __longlong_as_double(0x7ff8000000000000ll);
            utt[b].labels_ok = 0;
            utt[b].nll = nan;
            if (a.reduction == CTC_PACKED_NONE) a.loss[b] = nan;
        }
        return;
    }
    const EmX* em = ws_at<EmX>(a.ws, a.L.off_em) + (size_t)u.start * Ep;
    unsigned long long* am = ws_at<unsigned long long>(a.ws, a.L.off_am) + (size_t)u.start * Sp;
    int32_t* ae = ws_at<int32_t>(a.ws, a.L.off_ae) + (size_t)u.start * Sp;
    const bool store = a.need_grad != 0;

    X64 nx[PER];
    // frame 0: the first blank and the first label
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int s = tid + k * nt;
        X64 v = x_zero();
        if (s < S && s <= 1) v = ld_em(em + ent[k]);
        if (s < S) {
            mbuf[s] = v.m;
            ebuf[s] = v.e;
            if (store) {
                am[s] = v.m;
                ae[s] = v.e;
            }
        }
        if (RING == 0) nx[k] = (s < S && T > 1) ? ld_em(em + Ep + ent[k]) : x_zero();
    }
    // the states' emissions of frame f into ring slot f % RING (each thread
    // copies and later reads its own states' entries)
    auto issue = [&](int f) {
        if (f < T) {
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int s = tid + k * nt;
                if (s < S) cp_async_n16(ring + (f % (RING > 0 ? RING : 1)) * cap + s, em + (size_t)f * Ep + ent[k]);
            }
        }
        cp_async_commit();
    };
    if (RING > 0)
        for (int f = 1; f < RING; ++f) issue(f);
    __syncthreads();
    int p = 0;
    for (int t = 1; t < T; ++t) {
        X64 e_t[PER];
        if constexpr (RING > 0) {
            issue(t + RING - 1);
            cp_async_wait<RING - 1>();  // frame t's entries have landed
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int s = tid + k * nt;
                e_t[k] = s < S ? ld_em(ring + (t % RING) * cap + s) : x_zero();
            }
        } else {
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                e_t[k] = nx[k];
                const int s = tid + k * nt;
                if (s < S && t + 1 < T) nx[k] = ld_em(em + (size_t)(t + 1) * Ep + ent[k]);
            }
        }
        const unsigned long long* mp = mbuf + p * cap;
        const int* ep = ebuf + p * cap;
        unsigned long long* mq = mbuf + (p ^ 1) * cap;
        int* eq = ebuf + (p ^ 1) * cap;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int s = tid + k * nt;
            if (s < S) {
                const X64 v0{mp[s], ep[s]};
                const X64 v1 = s >= 1 ? X64{mp[s - 1], ep[s - 1]} : x_zero();
                const X64 v2 = skip[k] ? X64{mp[s - 2], ep[s - 2]} : x_zero();
                const X64 r = x_mul(x_add3(v0, v1, v2), e_t[k]);
                mq[s] = r.m;
                eq[s] = r.e;
                if (store) {
                    am[(size_t)t * Sp + s] = r.m;
                    ae[(size_t)t * Sp + s] = r.e;
                }
            }
        }
        __syncthreads();
        p ^= 1;
    }
    if (RING > 0) cp_async_wait<0>();
    if (tid == 0) {
        const unsigned long long* mp = mbuf + p * cap;
        const int* ep = ebuf + p * cap;
        const X64 last{mp[S - 1], ep[S - 1]};
        const X64 prev = S >= 2 ? X64{mp[S - 2], ep[S - 2]} : x_zero();
        const X64 z = x_add3(last, prev, x_zero());
        const bool has_nan = u.has_nan != 0;  // written by the emission gather
        double v, zm = 0.0;
        int inf = 0;
        if (has_nan) {
            v = __longlong_as_double(0x7ff8000000000000ll);
        } else if (z.m == 0) {
            v = __longlong_as_double(0x7ff0000000000000ll);
            inf = 1;
        } else {
            zm = x_mantissa(z);
            v = -(log(zm) + (double)z.e * kLn2D);
        }
        utt[b].nll = v;
        utt[b].zm = zm;
        utt[b].ze = z.e;
        utt[b].nll_inf = inf;
        if (a.reduction == CTC_PACKED_NONE) a.loss[b] = (a.zero_infinity && inf) ? 0.0 : v;
    }
}

// Backward recursion of one utterance from its last frame, run by the
// forward call beside the alpha recursion (on CTAs of its own).  beta_t(s)
// excludes frame t's emission; g_t(s) = beta_t(s) * exp(lp[t, l(s)]) is what
// frame t - 1 reads:
//   beta_{T-1}(s) = 1 for the last two states,
//   beta_t(s) = g_{t+1}(s) + g_{t+1}(s + 1) + [l(s + 2) != l(s)] g_{t+1}(s + 2).
// Every beta row is stored for the backward's posteriors; g is double
// buffered in shared memory, one barrier per frame.  First the label
// analysis the class sums use: first occurrences ranked in target order,
// links to the next occurrence, labels equal to the blank joining its class
// (in shared memory that the recursion reuses afterwards).
template <int PER>
__device__ __forceinline__ void f64_beta_chain(const F64Args& a, int b) {
    constexpr int RING = f64_ring(PER);
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_warp[32];
    __shared__ int s_bfirst, s_bad;
    const int tid = threadIdx.x, nt = blockDim.x;
    F64Utt* utt = ws_at<F64Utt>(a.ws, a.L.off_utt);
    const F64Utt u = utt[b];
    if (!u.valid || u.T == 0) return;
    const int U = u.U, S = 2 * U + 1, T = u.T, Ep = a.L.Ep, Sp = a.L.Sp;
    const int cap = PER * nt;

    // 1. label analysis
    int* const lab = reinterpret_cast<int*>(smem);  // the target
    int* const nxt = lab + U;                       // next position of the same class, -1: none
    int* const rnk = nxt + U;                       // rank of a first occurrence, -1 otherwise
    if (tid == 0) {
        s_bfirst = -1;
        s_bad = 0;
    }
    __syncthreads();
    for (int j = tid; j < U; j += nt) {
        const int c = a.targets[u.toff + j];
        lab[j] = c;
        if (c < 0 || c >= a.D) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) return;  // the alpha recursion reports it
    int running = 0;
    for (int j0 = 0; j0 < U; j0 += nt) {
        const int j = j0 + tid;
        bool first = false;
        if (j < U) {
            const int c = lab[j];
            first = true;
            for (int k = 0; k < j; ++k)
                if (lab[k] == c) {
                    first = false;
                    break;
                }
            int nx = -1;
            for (int k = j + 1; k < U; ++k)
                if (lab[k] == c) {
                    nx = k;
                    break;
                }
            nxt[j] = nx;
            if (c == a.blank) {
                if (first) s_bfirst = j;
                first = false;
            }
        }
        int total;
        const int pre = f64_block_scan(first ? 1 : 0, s_warp, &total);
        if (j < U) rnk[j] = first ? running + pre : -1;
        running += total;
    }
    const int ncls = running + 1;
    int32_t* cls = ws_at<int32_t>(a.ws, a.L.off_cls) + (size_t)b * Ep;
    int2* lrec = ws_at<int2>(a.ws, a.L.off_lrec) + (size_t)b * Ep;
    for (int j = tid; j < U; j += nt) {
        if (rnk[j] >= 0) cls[rnk[j]] = lab[j];
        lrec[j] = make_int2(rnk[j], nxt[j]);
    }
    if (tid == 0) {
        cls[ncls - 1] = a.blank;
        utt[b].ncls = ncls;
        utt[b].bfirst = s_bfirst;
    }
    int eidx[PER];
    bool skip2[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int s = tid + k * nt;
        eidx[k] = (s & 1) ? (s >> 1) : U;
        skip2[k] = (s & 1) && s + 2 < S && lab[(s + 2) >> 1] != lab[s >> 1];
    }
    __syncthreads();  // the label arrays are read: their shared memory goes to the recursion

    // 2. the recursion
    unsigned long long* const gbm = reinterpret_cast<unsigned long long*>(smem);  // two buffers of cap mantissas
    int* const gbe = reinterpret_cast<int*>(gbm + 2 * cap);                         // two buffers of cap exponents
    EmX* const ring = reinterpret_cast<EmX*>(gbe + 2 * cap);  // RING frames of the states' emissions
    const EmX* em = ws_at<EmX>(a.ws, a.L.off_em) + (size_t)u.start * Ep;
    unsigned long long* bm = ws_at<unsigned long long>(a.ws, a.L.off_bm) + (size_t)u.start * Sp;
    int32_t* bx = ws_at<int32_t>(a.ws, a.L.off_bx) + (size_t)u.start * Sp;
    // frame f's emissions into ring slot f % RING (each thread copies and
    // later reads its own states' entries)
    auto issue = [&](int f) {
        if (f >= 0) {
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int s = tid + k * nt;
                if (s < S) cp_async_n16(ring + (f % (RING > 0 ? RING : 1)) * cap + s, em + (size_t)f * Ep + eidx[k]);
            }
        }
        cp_async_commit();
    };
    X64 nx[PER];  // without a ring: the next frame's emissions, loaded a frame ahead
    if constexpr (RING > 0) {
        for (int j = 0; j < RING - 1; ++j) issue(T - 1 - j);
    } else {
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int s = tid + k * nt;
            nx[k] = s < S ? ld_em(em + (size_t)(T - 1) * Ep + eidx[k]) : x_zero();
        }
    }
    int p = 0;  // g of frame t + 1 is in buffer p
    for (int t = T - 1; t >= 0; --t) {
        X64 e_t[PER];
        if constexpr (RING > 0) {
            issue(t - (RING - 1));
            cp_async_wait<RING - 1>();  // frame t's entries have landed
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int s = tid + k * nt;
                e_t[k] = s < S ? ld_em(ring + (t % RING) * cap + s) : x_zero();
            }
        } else {
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                e_t[k] = nx[k];
                const int s = tid + k * nt;
                if (s < S && t > 0) nx[k] = ld_em(em + (size_t)(t - 1) * Ep + eidx[k]);
            }
        }
        const unsigned long long* gmp = gbm + p * cap;
        const int* gep = gbe + p * cap;
        unsigned long long* gmq = gbm + (p ^ 1) * cap;
        int* geq = gbe + (p ^ 1) * cap;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int s = tid + k * nt;
            if (s < S) {
                X64 be;
                if (t == T - 1) {
                    be = s >= S - 2 ? X64{kXOne, 0} : x_zero();
                } else {
                    const X64 v0{gmp[s], gep[s]};
                    const X64 v1 = s + 1 < S ? X64{gmp[s + 1], gep[s + 1]} : x_zero();
                    const X64 v2 = skip2[k] ? X64{gmp[s + 2], gep[s + 2]} : x_zero();
                    be = x_add3(v0, v1, v2);
                }
                const X64 g = x_mul(be, e_t[k]);
                gmq[s] = g.m;
                geq[s] = g.e;
                bm[(size_t)t * Sp + s] = be.m;
                bx[(size_t)t * Sp + s] = be.e;
            }
        }
        __syncthreads();
        p ^= 1;
    }
    if (RING > 0) cp_async_wait<0>();
}

// The recursions of the forward call: CTA b < B runs utterance b's alpha
// recursion; with the gradient's state kept, CTA B + b runs its beta
// recursion at the same time.
template <int PER>
__global__ void __launch_bounds__(kMaxChainThreads, 1) f64_chain_kernel(F64Args a) {
    if ((int)blockIdx.x < a.L.B) {
        f64_alpha_chain<PER>(a, (int)blockIdx.x);
    } else {
        f64_beta_chain<PER>(a, (int)blockIdx.x - a.L.B);
    }
}

// The reduced loss (sum, mean, mean_batch, mean_volume) in a fixed order.
__global__ void __launch_bounds__(256) f64_reduce_kernel(F64Args a) {
    __shared__ double s_red[8];
    const F64Utt* utt = ws_at<F64Utt>(a.ws, a.L.off_utt);
    const Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const int B = a.L.B, tid = threadIdx.x;
    double acc = 0.0;
    for (int b = tid; b < B; b += 256) {
        double v = utt[b].nll;
        if (a.zero_infinity && isinf(v) && v > 0) v = 0.0;
        if (a.reduction == CTC_PACKED_MEAN) v /= (double)max(a.target_lengths[b], 1);
        acc += v;
    }
    acc = warp_sum(acc);
    if ((tid & 31) == 0) s_red[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
        double total = 0.0;
        for (int w = 0; w < 8; ++w) total += s_red[w];
        if (a.reduction == CTC_PACKED_MEAN || a.reduction == CTC_PACKED_MEAN_BATCH)
            total = B > 0 ? total / (double)B : __longlong_as_double(0x7ff8000000000000ll);
        if (a.reduction == CTC_PACKED_MEAN_VOLUME) total = total / (double)ctrl->tl_total;
        a.loss[0] = total;
    }
}

// ------------------------------------------------------------ backward kernels

// A posterior (an extended value in [0, 2)) in fixed point, units of 2^-62:
// its mantissa moved by its exponent (bits below 2^-62, about 2e-19, drop
// out).  Class sums of such values are exact integer sums, the same in any
// order, and convert to float64 once.
__device__ __forceinline__ long long post_fixed(X64 x) {
    if (x.m == 0) return 0;
    // m 2^(e - 61) times 2^62; a posterior is at most 1 (e <= 0), and the
    // shift is capped at 1 for the undefined rows of an utterance without a
    // path (Z = 0 and no zero_infinity)
    const long long sh = min((long long)x.e + 1, 1ll);
    return (long long)(sh >= 0 ? x.m << sh : (sh > -64 ? x.m >> -sh : 0ull));
}
// The posterior a * b * c (alpha, beta, 1 / Z) in the same fixed point,
// without normalising the products: the high word of a.m * b.m (below
// 2^60), the high word of that times c.m (below 2^58), moved by the
// exponent sum: a.m b.m c.m 2^(ea + eb + ec - 183) = p 2^(ea + eb + ec - 55)
// with p the second high word, times 2^62.
__device__ __forceinline__ long long post_fixed3(X64 a, X64 b, X64 c) {
    const unsigned long long p = __umul64hi(__umul64hi(a.m, b.m), c.m);
    if (p == 0) return 0;
    // a posterior of at most 1 needs a shift of at most 7 (p >= 2^55); the
    // cap keeps the shift defined on the undefined rows of an utterance
    // without a path
    const long long sh = min((long long)a.e + b.e + c.e + 7, 7ll);
    return (long long)(sh >= 0 ? p << sh : (sh > -64 ? p >> -sh : 0ull));
}

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Posteriors and class sums of each row, from the rows both recursions
// stored: gamma_t(s) = alpha_t(s) beta_t(s) / Z in fixed point (post_fixed3),
// summed per distinct class in exact integer arithmetic (so in any order and
// the same as any other order), each sum written as its gradient entry
// -scale * P: a first occurrence's thread sums its class's label states along
// the next-occurrence links; the blank class is the CTA's sum of the blank
// states plus the labels equal to the blank.  One CTA per row at a time, over
// a contiguous range of rows (mostly of one utterance, whose links are loaded
// once).  Rows without class sums (outside every utterance, a malformed or
// unaligned one, scale 0) are left to the dense pass.  Small CTAs, so that an
// SM holds many rows in flight: each row's loads wait on DRAM, then its
// class sums on two barriers (measured on the 8193-class workload: 226 us
// with 256 threads a CTA).
constexpr int kPostThreads = 64;
constexpr int kPostUnroll = 4;  // states a thread loads at once
__global__ void __launch_bounds__(kPostThreads) f64_post_kernel(F64Args a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int Uc = a.L.max_U > 0 ? a.L.max_U : 1;
    long long* const gam = reinterpret_cast<long long*>(smem);  // label-state posteriors of the row
    int2* const lr = reinterpret_cast<int2*>(gam + Uc);         // the utterance's (rank, next) links
    __shared__ long long s_wsum[kPostThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x, nw = nt >> 5;
    const Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const F64Utt* utt = ws_at<F64Utt>(a.ws, a.L.off_utt);
    if (ctrl->grad_ready == 0) return;  // the dense pass reports it
    const int tl_total = ctrl->tl_total;
    const int64_t T_total = a.L.T_total;
    const int64_t per = (T_total + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = (int64_t)blockIdx.x * per;
    const int64_t r1 = r0 + per < T_total ? r0 + per : T_total;
    const int Sp = a.L.Sp;
    const unsigned long long* am_all = ws_at<unsigned long long>(a.ws, a.L.off_am);
    const int32_t* ae_all = ws_at<int32_t>(a.ws, a.L.off_ae);
    const unsigned long long* bm_all = ws_at<unsigned long long>(a.ws, a.L.off_bm);
    const int32_t* bx_all = ws_at<int32_t>(a.ws, a.L.off_bx);
    double* ent = ws_at<double>(a.ws, a.L.off_ent);
    const double qnan = __longlong_as_double(0x7ff8000000000000ll);
    // the utterance whose record, scale, 1 / Z and links are held (rows of a
    // CTA's range mostly belong to one)
    int cur = -1;
    F64Utt u{};
    double scale = 0.0;
    X64 izx = x_zero();
    for (int64_t row = r0; row < r1; ++row) {
        const int b = f64_utterance_of_row(a.cu, a.L.B, row);
        if (b < 0) continue;
        if (b != cur) {
            __syncthreads();  // every read of the previous links is done
            u = utt[b];
            cur = b;
            if (!u.valid || !u.labels_ok) continue;
            scale = f64_scale(a, u, b, tl_total);
            izx = x_of_double(1.0 / u.zm, -(long long)u.ze);  // 1 / Z
            const int2* lg = ws_at<int2>(a.ws, a.L.off_lrec) + (size_t)b * a.L.Ep;
            for (int j = tid; j < u.U; j += nt) lr[j] = lg[j];
        }
        const int64_t t = row - u.start;
        if (!u.valid || !u.labels_ok || t < 0 || t >= u.T || scale == 0.0) continue;
        const int U = u.U, S = 2 * U + 1;
        const bool nan_utt = u.has_nan != 0;
        const unsigned long long* am = am_all + row * Sp;
        const int32_t* ae = ae_all + row * Sp;
        const unsigned long long* bm = bm_all + row * Sp;
        const int32_t* bx = bx_all + row * Sp;
        long long bpart = 0;
        // the posterior alpha * beta / Z (at most 1) in fixed point,
        // kPostUnroll states a thread at a time (their loads in flight
        // together); NaN entries: see entry
        for (int s0 = tid; s0 < S; s0 += kPostUnroll * nt) {
            X64 av[kPostUnroll], bv[kPostUnroll];
#pragma unroll
            for (int q = 0; q < kPostUnroll; ++q) {
                const int s = s0 + q * nt;
                av[q] = x_zero();
                bv[q] = x_zero();
                if (s < S) {
                    av[q] = X64{__ldg(am + s), __ldg(ae + s)};
                    bv[q] = X64{__ldg(bm + s), __ldg(bx + s)};
                }
            }
#pragma unroll
            for (int q = 0; q < kPostUnroll; ++q) {
                const int s = s0 + q * nt;
                if (s < S) {
                    const long long g = nan_utt ? 0 : post_fixed3(av[q], bv[q], izx);
                    if (s & 1) {
                        gam[s >> 1] = g;
                    } else {
                        bpart += g;
                    }
                }
            }
        }
        bpart = warp_sum_ll(bpart);
        if (lane == 0) s_wsum[warp] = bpart;
        __syncthreads();
        // a class sum P (fixed point) as its gradient entry -scale * P
        const double nscale = -scale * 0x1p-62;
        auto entry = [&](long long P) { return nan_utt ? qnan : nscale * __ll2double_rn(P); };
        double* er = ent + row * a.L.ecap;
        for (int j = tid; j < U; j += nt) {
            const int r = lr[j].x;
            if (r < 0) continue;
            long long P = gam[j];
            for (int jj = lr[j].y; jj >= 0; jj = lr[jj].y) P += gam[jj];
            er[r] = entry(P);
        }
        if (tid == 0) {
            long long P = 0;
            for (int w = 0; w < nw; ++w) P += s_wsum[w];
            for (int jj = u.bfirst; jj >= 0; jj = lr[jj].y) P += gam[jj];
            er[u.ncls - 1] = entry(P);
        }
        __syncthreads();  // gam and s_wsum are free for the next row
    }
}

// scale * exp(x[c] - sh) for the lane's elements c of a row: with FOLDED the
// table T already holds scale * 2^(j/64); without SHIFT the row is not
// shifted.
template <bool SHIFT, bool FOLDED>
__device__ __forceinline__ void dense_row(double* g, const double* x, int D, int lane, double sh, double scale,
                                          const double* T) {
    auto f = [&](double v) {
        if (SHIFT) v -= sh;
        return FOLDED ? exp_table(v, T) : scale * exp_table(v, T);
    };
    int c = lane;
    for (; c + 96 < D; c += 128) {
        const double x0 = __ldg(x + c), x1 = __ldg(x + c + 32), x2 = __ldg(x + c + 64), x3 = __ldg(x + c + 96);
        g[c] = f(x0);
        g[c + 32] = f(x1);
        g[c + 64] = f(x2);
        g[c + 96] = f(x3);
    }
    for (; c < D; c += 32) g[c] = f(__ldg(x + c));
}

// The dense gradient: one warp per row.  A row outside every utterance's
// frames (or of a malformed utterance, or after a loss-only forward) is 0.
__global__ void __launch_bounds__(kRowWarps * 32) f64_grad_kernel(F64Args a) {
    __shared__ double s_exp[64];
    __shared__ double s_sexp[kRowWarps][64];  // per warp: scale * 2^(j/64) of its current row
    fill_exp_table(s_exp);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    double* sexp = s_sexp[threadIdx.x >> 5];
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    const F64Utt* utt = ws_at<F64Utt>(a.ws, a.L.off_utt);
    const double* lse = ws_at<double>(a.ws, a.L.off_lse);
    const double* ent = ws_at<double>(a.ws, a.L.off_ent);
    const int32_t* cls = ws_at<int32_t>(a.ws, a.L.off_cls);
    const bool ready = ctrl->grad_ready != 0;
    const bool logits = ctrl->logits != 0;
    const int tl_total = ctrl->tl_total;
    const int D = a.D;
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.L.T_total > 0 && !ready)
        set_status(ctrl, CTC_PACKED_DEV_NO_GRAD_STATE);
    const int64_t warps = (int64_t)gridDim.x * kRowWarps;
    for (int64_t row = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5); row < a.L.T_total; row += warps) {
        const int b = f64_utterance_of_row(a.cu, a.L.B, row);
        double* g = a.grad + row * D;
        const double* x = a.lp + row * D;
        bool covered = false;
        F64Utt u{};
        if (b >= 0) {
            u = utt[b];
            const int64_t t = row - u.start;
            covered = ready && u.valid && u.labels_ok && t >= 0 && t < u.T;
        }
        if (!covered) {
            for (int c = lane; c < D; c += 32) g[c] = 0.0;
            continue;
        }
        const double scale = f64_scale(a, u, b, tl_total);
        const double sh = logits ? lse[row] : 0.0;
        // scale * exp(x) = exp_table(x) on the table scale * 2^(j/64) when
        // every result stays a normal number (2^-200 <= |scale| <= 2^200 and
        // the table's |x| < 512): one multiply a table entry, not an element
        const int se = (int)((unsigned long long)__double_as_longlong(scale) >> 52 & 0x7ff);
        const bool folded = se >= 1023 - 200 && se <= 1023 + 200;
        __syncwarp();
        sexp[lane] = scale * s_exp[lane];
        sexp[lane + 32] = scale * s_exp[lane + 32];
        __syncwarp();
        auto sexp_of = [&](double v) { return folded ? exp_table(v, sexp) : scale * exp_table(v, s_exp); };
        // the dense pass, its row-uniform choices taken once: log
        // probabilities need no shift (a float64 subtraction an element)
        if (logits)
            folded ? dense_row<true, true>(g, x, D, lane, sh, scale, sexp) : dense_row<true, false>(g, x, D, lane, sh, scale, s_exp);
        else
            folded ? dense_row<false, true>(g, x, D, lane, sh, scale, sexp) : dense_row<false, false>(g, x, D, lane, sh, scale, s_exp);
        if (scale != 0.0) {
            __syncwarp();  // the dense stores land before the class sums rewrite their elements
            const double* er = ent + row * a.L.ecap;
            const int32_t* cl = cls + (size_t)b * a.L.Ep;
            for (int k = lane; k < u.ncls; k += 32) {
                const int cc = cl[k];
                g[cc] = sexp_of(__ldg(x + cc) - sh) + er[k];
            }
        }
    }
}

}  // namespace ctcp

using namespace ctcp;

namespace {

bool f64_valid_reduction(int r) {
    return r == CTC_PACKED_NONE || r == CTC_PACKED_SUM || r == CTC_PACKED_MEAN || r == CTC_PACKED_MEAN_BATCH ||
           r == CTC_PACKED_MEAN_VOLUME;
}

ctc_packed_status f64_check(const double* log_probs, int64_t T_total, int32_t D, const int32_t* cu,
                            const int32_t* lengths, const int32_t* targets, const int32_t* target_lengths, int32_t B,
                            int32_t max_target_len, int32_t blank, int reduction, const void* ws, size_t ws_bytes,
                            bool loss_only) {
    if (!f64_valid_reduction(reduction)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (T_total < 0 || B < 0 || max_target_len < 0 || D < 1) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (blank < 0 || blank >= D) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (D > kMaxD || max_target_len > kMaxTargetLen || T_total > INT32_MAX) return CTC_PACKED_ERR_UNSUPPORTED;
    if (cu == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (B > 0 && (lengths == nullptr || target_lengths == nullptr)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (B > 0 && max_target_len > 0 && targets == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (T_total > 0 && log_probs == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(log_probs) % 8 != 0) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (ws == nullptr || reinterpret_cast<uintptr_t>(ws) % 256 != 0) return CTC_PACKED_ERR_WORKSPACE;
    const F64Layout L = f64_layout(T_total, B, max_target_len, D);
    if (ws_bytes < (loss_only ? L.loss_only_total : L.total)) return CTC_PACKED_ERR_WORKSPACE;
    return CTC_PACKED_OK;
}

F64Args f64_args(const double* log_probs, int64_t T_total, int32_t D, const int32_t* cu, const int32_t* lengths,
                 const int32_t* targets, const int32_t* target_lengths, int32_t B, int32_t max_target_len,
                 int32_t blank, int zero_infinity, int reduction, void* ws) {
    F64Args a{};
    a.L = f64_layout(T_total, B, max_target_len, D);
    a.ws = ws;
    a.lp = log_probs;
    a.cu = cu;
    a.lengths = lengths;
    a.targets = targets;
    a.target_lengths = target_lengths;
    a.D = D;
    a.blank = blank;
    a.reduction = reduction;
    a.zero_infinity = zero_infinity ? 1 : 0;
    return a;
}

// States per thread of the recursion CTAs and their thread count: at most
// 1024 threads, each holding 1, 2, 4 or 8 states.
void chain_shape(int max_U, int& per, int& nt) {
    const int S = 2 * max_U + 1;
    per = 1;
    while (per * kMaxChainThreads < S) per <<= 1;
    const int need = (S + per - 1) / per;
    nt = (need + 31) / 32 * 32;
}

template <typename K>
cudaError_t launch_chain_kernel(K kernel, unsigned grid, int nt, size_t smem, cudaStream_t s, const F64Args& a) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, nt, smem, s>>>(a);
    return cudaGetLastError();
}

// Persistent grid of one of the row kernels.
template <typename K>
cudaError_t launch_rows(K kernel, int64_t rows, cudaStream_t s, const F64Args& a) {
    if (rows <= 0) return cudaSuccess;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kRowWarps * 32, 0)) != cudaSuccess)
        return e;
    if (per_sm < 1) per_sm = 1;
    long long grid = (long long)sms * per_sm;
    const long long want = (rows + kRowWarps - 1) / kRowWarps;
    if (want < grid) grid = want;
    kernel<<<(unsigned)grid, kRowWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

// The posterior / class-sum kernel: a grid of the SMs times the CTAs an SM
// holds, each over a contiguous range of rows.
cudaError_t launch_post(int64_t rows, int32_t max_U, cudaStream_t s, const F64Args& a) {
    if (rows <= 0) return cudaSuccess;
    const size_t smem = (size_t)(max_U > 0 ? max_U : 1) * (sizeof(long long) + sizeof(int2));
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(f64_post_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f64_post_kernel, kPostThreads, smem)) !=
        cudaSuccess)
        return e;
    if (per_sm < 1) per_sm = 1;
    long long grid = (long long)sms * per_sm;
    if (rows < grid) grid = rows;
    f64_post_kernel<<<(unsigned)grid, kPostThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

namespace ctcp {

size_t f64_workspace_bytes(int64_t T_total, int32_t B, int32_t max_target_len, int32_t D, bool loss_only) {
    const F64Layout L = f64_layout(T_total, B, max_target_len, D);
    return loss_only ? L.loss_only_total : L.total;
}

}  // namespace ctcp

extern "C" {

ctc_packed_status ctc_packed_forward_f64(const double* log_probs, int64_t T_total, int32_t D,
                                         const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* targets,
                                         const int32_t* target_lengths, int32_t B, int32_t max_target_len,
                                         int32_t blank, int zero_infinity, ctc_packed_reduction reduction,
                                         double* loss, void* workspace, size_t workspace_bytes, unsigned flags,
                                         cudaStream_t stream) {
    if ((flags & ~(CTC_PACKED_FLAG_LOSS_ONLY | CTC_PACKED_FLAG_LOGITS)) != 0) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    const bool loss_only = (flags & CTC_PACKED_FLAG_LOSS_ONLY) != 0;
    const ctc_packed_status st = f64_check(log_probs, T_total, D, cu_seqlens, lengths, targets, target_lengths, B,
                                           max_target_len, blank, (int)reduction, workspace, workspace_bytes,
                                           loss_only);
    if (st != CTC_PACKED_OK) return st;
    if (loss == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    F64Args a = f64_args(log_probs, T_total, D, cu_seqlens, lengths, targets, target_lengths, B, max_target_len,
                         blank, zero_infinity, (int)reduction, workspace);
    a.loss = loss;
    a.need_grad = loss_only ? 0 : 1;
    a.logits = (flags & CTC_PACKED_FLAG_LOGITS) != 0 ? 1 : 0;
    f64_prep_kernel<<<1, 1024, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    if (a.logits && launch_rows(f64_lse_kernel, T_total, stream, a) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    if (launch_rows(f64_emit_kernel, T_total, stream, a) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    if (B > 0) {
        int per = 1, nt = 32;
        chain_shape(max_target_len, per, nt);
        const size_t cap = (size_t)per * nt;
        // both recursions: two buffers of state values and the emission ring;
        // the beta CTAs first hold their label analysis in the same memory
        size_t smem = 2 * cap * (sizeof(double) + sizeof(int)) + (size_t)f64_ring(per) * cap * sizeof(EmX);
        const size_t labels = 3 * sizeof(int) * (size_t)max_target_len;
        if (a.need_grad && labels > smem) smem = labels;
        // with the gradient's state kept, the beta recursions run beside the alpha ones
        const unsigned grid = (unsigned)B * (a.need_grad ? 2u : 1u);
        cudaError_t e;
        switch (per) {
            case 1: e = launch_chain_kernel(f64_chain_kernel<1>, grid, nt, smem, stream, a); break;
            case 2: e = launch_chain_kernel(f64_chain_kernel<2>, grid, nt, smem, stream, a); break;
            case 4: e = launch_chain_kernel(f64_chain_kernel<4>, grid, nt, smem, stream, a); break;
            default: e = launch_chain_kernel(f64_chain_kernel<8>, grid, nt, smem, stream, a); break;
        }
        if (e != cudaSuccess) return CTC_PACKED_ERR_CUDA;
        if (reduction != CTC_PACKED_NONE) {
            f64_reduce_kernel<<<1, 256, 0, stream>>>(a);
            if (cudaGetLastError() != cudaSuccess) return CTC_PACKED_ERR_CUDA;
        }
    } else if (reduction != CTC_PACKED_NONE) {
        f64_reduce_kernel<<<1, 256, 0, stream>>>(a);
        if (cudaGetLastError() != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    }
    return CTC_PACKED_OK;
}

ctc_packed_status ctc_packed_backward_f64(const double* log_probs, int64_t T_total, int32_t D,
                                          const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* targets,
                                          const int32_t* target_lengths, int32_t B, int32_t max_target_len,
                                          int32_t blank, int zero_infinity, ctc_packed_reduction reduction,
                                          const double* grad_loss, void* workspace, size_t workspace_bytes,
                                          double* grad_log_probs, cudaStream_t stream) {
    const ctc_packed_status st = f64_check(log_probs, T_total, D, cu_seqlens, lengths, targets, target_lengths, B,
                                           max_target_len, blank, (int)reduction, workspace, workspace_bytes, false);
    if (st != CTC_PACKED_OK) return st;
    if (grad_log_probs == nullptr || (B > 0 && grad_loss == nullptr)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(grad_log_probs) % 8 != 0) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(grad_log_probs), l0 = reinterpret_cast<uintptr_t>(log_probs);
    const uintptr_t nbytes = (uintptr_t)(T_total * (int64_t)D * 8);
    if (g0 < l0 + nbytes && l0 < g0 + nbytes) return CTC_PACKED_ERR_INVALID_ARGUMENT;  // overlap
    if (T_total == 0) return CTC_PACKED_OK;
    F64Args a = f64_args(log_probs, T_total, D, cu_seqlens, lengths, targets, target_lengths, B, max_target_len,
                         blank, zero_infinity, (int)reduction, workspace);
    a.grad = grad_log_probs;
    a.grad_loss = grad_loss;
    if (B > 0 && launch_post(T_total, max_target_len, stream, a) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    if (launch_rows(f64_grad_kernel, T_total, stream, a) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    return CTC_PACKED_OK;
}

}  // extern "C"
