// Prep kernel of the forward: per-utterance metadata, target offsets and the
// length-sorted work queue.  One CTA; no host synchronisation anywhere.
//
// Checks of page "feat(asr): native CTC loss kernel over sequence-packed log
// probabilities", ctc_loss.py ``packed_ctc_loss``: a negative target length
// and one beyond the targets width are errors, not impossible alignments.
// Here they set a status bit and give the utterance a NaN loss, because a
// kernel cannot raise.  ``_alpha_kernel``: an utterance without frames has
// loss 0 without targets and +inf with targets.
#include "ctc_common.cuh"
#include "ctc_kernels.h"

namespace ctcp {

namespace {

constexpr int kPrepThreads = 1024;
constexpr int kSortMax = 4096;

// Exclusive scan of one value per thread over the whole CTA; returns the
// prefix and writes the CTA total to *total.
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;  // inclusive prefix of warp totals
    }
    __syncthreads();
    int prefix = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
    *total = s_warp[(blockDim.x >> 5) - 1];
    __syncthreads();
    return prefix;
}

}  // namespace

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(PrepArgs a) {
    __shared__ int s_warp[32];
    __shared__ long long s_keys[kSortMax];
    Control* ctrl = ws_at<Control>(a.ws, a.L.off_ctrl);
    UttInfo* utt = ws_at<UttInfo>(a.ws, a.L.off_utt);
    int32_t* queue = ws_at<int32_t>(a.ws, a.L.off_queue);
    double* nll = ws_at<double>(a.ws, a.L.off_nll);
    const int B = a.L.B;
    const int tid = threadIdx.x, nt = blockDim.x;
    pdl_wait();     // the stream's earlier work may still use this workspace
    pdl_trigger();  // one CTA: the emission gather's blocks may queue up behind it

    if (tid == 0) {
        ctrl->status = 0;
        ctrl->big_head = 0;
        ctrl->small_head = 0;
        ctrl->done_ctas = 0;
        ctrl->grad_ready = a.need_grad ? 1u : 0u;
        ctrl->logits = a.logits ? 1u : 0u;
        ctrl->ckpt = (uint32_t)a.ckpt;
    }

    // 1. validate, and scan the target offsets (raw lengths) and the
    //    label-metadata offsets (valid lengths plus one blank slot each)
    uint32_t bad_bits = 0;
    int toff_base = 0, moff_base = 0;
    for (int base = 0; base < B; base += nt) {
        const int b = base + tid;
        int T = 0, U = 0, start = 0, valid = 0, uraw = 0;
        if (b < B) {
            const int c0 = a.cu[b], c1 = a.cu[b + 1];
            T = a.lengths[b];
            uraw = a.target_lengths[b];
            uint32_t bits = 0;
            if (uraw < 0) bits |= CTC_PACKED_DEV_NEGATIVE_TARGET_LENGTH;
            if (uraw > a.L.max_U) bits |= CTC_PACKED_DEV_TARGET_LENGTH_EXCEEDS_MAX;
            if (c0 < 0 || c1 < c0 || (int64_t)c1 > a.L.T_total) bits |= CTC_PACKED_DEV_BAD_CU_SEQLENS;
            if (T < 0 || (int64_t)T > (int64_t)c1 - (int64_t)c0) bits |= CTC_PACKED_DEV_BAD_LENGTH;
            bad_bits |= bits;
            valid = bits == 0;
            start = c0;
            U = valid ? uraw : 0;
        }
        int total_t, total_m;
        const int toff = toff_base + block_exclusive_scan(b < B ? max(uraw, 0) : 0, s_warp, &total_t);
        const int moff = moff_base + block_exclusive_scan(b < B ? U + 1 : 0, s_warp, &total_m);
        if (b < B) {
            UttInfo info;
            info.start = start;
            info.T = valid ? T : 0;
            info.U = U;
            info.toff = toff;
            info.moff = moff;
            info.valid = valid;
            info.labels_ok = 1;
            info.n_owners = 1;
            info.has_nan = 0;
            info.kint = 0;
            info.cfrac = 0.0f;
            info.nll_inf = (valid && T == 0 && U > 0) ? 1 : 0;
            info.pad = 0;
            utt[b] = info;
            // utterances that need no recursion get their loss here
            if (!valid || T == 0) {
                const double v = !valid ? __longlong_as_double(0x7ff8000000000000ll)
                                        : (U == 0 ? 0.0 : __longlong_as_double(0x7ff0000000000000ll));
                nll[b] = v;
                if (a.reduction == CTC_PACKED_NONE) {
                    float out = (float)v;
                    if (a.zero_infinity && isinf(v)) out = 0.0f;
                    a.loss[b] = out;
                }
            }
        }
        toff_base += total_t;
        moff_base += total_m;
    }
    if (bad_bits) atomicOr(&ctrl->status, bad_bits);
    if (tid == 0) ctrl->tl_total = toff_base;
    __syncthreads();

    // 2. order the utterances longest first (the serial chain of the longest
    //    one is the critical path), then split them into multi-warp and
    //    single-warp chain items
    const bool sorted = B <= kSortMax;
    if (sorted) {
        int n = 1;
        while (n < B) n <<= 1;
        for (int i = tid; i < n; i += nt) {
            if (i < B) {
                const UttInfo& u = utt[i];
                const int key = (u.valid && u.T > 0) ? u.T : -1;
                s_keys[i] = ((long long)(0x7fffffff - key) << 32) | (unsigned)i;
            } else {
                s_keys[i] = 0x7fffffffffffffffll;
            }
        }
        __syncthreads();
        for (int k = 2; k <= n; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = tid; i < n; i += nt) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const long long x = s_keys[i], y = s_keys[ixj];
                        const bool up = (i & k) == 0;
                        if ((x > y) == up) {
                            s_keys[i] = y;
                            s_keys[ixj] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
    }
    const int warp_pairs = a.group_pairs;  // pairs one chain warp owns
    int big_base = 0, small_base = 0, lab_base = 0;
    // first pass counts the big items, so the small ones can follow them
    int n_big = 0;
    for (int base = 0; base < B; base += nt) {
        const int i = base + tid;
        int is_big = 0;
        if (i < B) {
            const int b = sorted ? (int)(s_keys[i] & 0xffffffffll) : i;
            const UttInfo& u = utt[b];
            is_big = (u.valid && u.T > 0 && u.U + 1 > warp_pairs) ? 1 : 0;
        }
        int t;
        block_exclusive_scan(is_big, s_warp, &t);
        n_big += t;
    }
    const int per = a.need_grad ? 2 : 1;
    for (int base = 0; base < B; base += nt) {
        const int i = base + tid;
        int b = -1, is_big = 0, is_small = 0, is_lab = 0;
        if (i < B) {
            b = sorted ? (int)(s_keys[i] & 0xffffffffll) : i;
            const UttInfo& u = utt[b];
            const bool work = u.valid && u.T > 0;
            is_big = (work && u.U + 1 > warp_pairs) ? 1 : 0;
            is_small = (work && !is_big) ? 1 : 0;
            is_lab = (work && a.need_grad) ? 1 : 0;
        }
        int tb, ts, tl;
        const int pb = block_exclusive_scan(is_big, s_warp, &tb);
        const int ps = block_exclusive_scan(is_small, s_warp, &ts);
        const int pl = block_exclusive_scan(is_lab, s_warp, &tl);
        // items are (b << 1) | direction, direction 0 = alpha, 1 = beta
        if (is_big) {
            queue[(big_base + pb) * per] = b << 1;
            if (per == 2) queue[(big_base + pb) * per + 1] = (b << 1) | 1;
        }
        if (is_small) {
            queue[n_big * per + (small_base + ps) * per] = b << 1;
            if (per == 2) queue[n_big * per + (small_base + ps) * per + 1] = (b << 1) | 1;
        }
        big_base += tb;
        small_base += ts;
        lab_base += tl;
        if (is_lab) queue[2 * B + 1 + (lab_base - tl + pl)] = b;
    }
    if (tid == 0) {
        ctrl->n_big = big_base * per;
        ctrl->n_small = small_base * per;
        ctrl->n_lab = lab_base;
    }
}

}  // namespace ctcp
