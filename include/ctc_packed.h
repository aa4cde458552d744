/*
 * ctc_packed.h -- CTC loss and gradient over sequence-packed log probabilities
 * on NVIDIA GB300 (sm_103a).
 *
 * What is computed.  Page "feat(asr): native CTC loss kernel over
 * sequence-packed log probabilities" (NVIDIA-NeMo/Speech PR #16437), file
 * nemo/collections/asr/parts/triton/ctc_loss.py, module docstring and
 * packed_ctc_loss:
 *
 *   - The log probabilities of a batch are ONE token-flat (T_total, D) buffer:
 *     utterance b owns rows [cu_seqlens[b], cu_seqlens[b] + lengths[b]).  The
 *     padded (B, T, D) tensor and its padded gradient are never formed.
 *   - Per utterance the loss is the CTC negative log-likelihood over the
 *     extended label sequence (blank, l_1, blank, ..., l_U, blank), S = 2U+1
 *     states; the skip over a blank is allowed between two different target
 *     ids (a target id equal to the blank is a label like any other).
 *     An utterance that cannot be aligned has loss +inf, or 0 with
 *     zero_infinity, which also zeroes its gradient.  An utterance with no
 *     frames has loss 0 without targets and +inf with targets.
 *   - The gradient has the layout and dtype of log_probs: row t of utterance
 *     b is  scale_b * ( exp(lp[t, c]) - sum over states s with l'_s = c of
 *     posterior_t(s) ),  the gradient with respect to the logits when
 *     log_probs is a log_softmax output.  Rows outside every utterance are 0.
 *   - Reductions (file nemo/collections/asr/losses/ctc.py, forward_packed):
 *     NONE keeps the B losses, SUM adds them, MEAN divides each by
 *     max(target_length, 1) and averages over the B utterances; MEAN_BATCH
 *     and MEAN_VOLUME are the module's further reductions (see the enum).
 *   - The input may also be a model's unnormalised logits
 *     (CTC_PACKED_FLAG_LOGITS): log_softmax is then taken inside the path.
 *   - The same full-sum loss over a generic FSA edge list instead of the
 *     CTC lattice: ctc_packed_fsa_forward / ctc_packed_fsa_backward.
 *   - Inputs may be float32, bfloat16 or float16; all arithmetic is float32
 *     (offsets that keep the recursion accurate are integers, the
 *     per-utterance log-likelihood is assembled in float64).
 *
 * Conventions shared by every call:
 *   - All array arguments are DEVICE pointers owned by the caller.  The
 *     library allocates nothing and keeps no state between calls except what
 *     the caller's workspace holds.
 *   - Calls are asynchronous on `stream` and never synchronise with the
 *     host, so a forward + backward pair can be captured in a CUDA graph and
 *     replayed with new contents in the same buffers.  ctc_packed_read_status
 *     is the one call that waits.
 *   - Integer metadata is int32.  Row and element offsets are computed in
 *     64-bit inside the kernels.
 *   - Targets are CONCATENATED: utterance b's ids are
 *     targets[sum_{j<b} target_lengths[j] + i], i < target_lengths[b].  The
 *     buffer must hold sum(target_lengths) ints.
 *   - max_target_len is the caller's bound on every target_lengths[b] (the
 *     page sizes its states by the longest target, or by the targets width
 *     under graph capture).  Results do not depend on it; it only sizes the
 *     workspace and the kernels' state lanes.
 *
 * Errors.  Arguments that the host can check (null pointers, D < 1, blank
 * outside [0, D), unknown dtype or reduction, workspace too small, sizes the
 * kernels do not support) make the call return an error code before anything
 * is enqueued.  Errors that only the device can see set bits of a status
 * word in the workspace and give that utterance a NaN loss; they never trap:
 *   negative target length, target length above max_target_len, lengths[b]
 *   negative or longer than its cu_seqlens span, cu_seqlens decreasing or
 *   past T_total, a target id outside [0, D).
 */
#ifndef CTC_PACKED_H
#define CTC_PACKED_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CTC_PACKED_F32 = 0,  /* float32 log probabilities and gradient */
    CTC_PACKED_BF16 = 1, /* bfloat16 */
    CTC_PACKED_F16 = 2,  /* float16 */
    /* float64: sizes the workspace of ctc_packed_forward_f64 and
     * ctc_packed_backward_f64, whose loss and upstream gradient are float64
     * too; the entry points above reject it */
    CTC_PACKED_F64 = 3
} ctc_packed_dtype;

typedef enum {
    CTC_PACKED_NONE = 0,       /* loss has B entries */
    CTC_PACKED_SUM = 1,        /* loss has 1 entry: sum of the B losses */
    CTC_PACKED_MEAN = 2,       /* loss has 1 entry: mean over b of loss_b / max(U_b, 1) */
    /* NeMo's further reductions of the per-utterance losses (page
     * "feat(asr): native CTC loss kernel over sequence-packed log
     * probabilities", test_ctc_loss.py parametrizes both; the page does not
     * print their bodies, read as): */
    CTC_PACKED_MEAN_BATCH = 3, /* loss has 1 entry: (1/B) sum_b loss_b */
    CTC_PACKED_MEAN_VOLUME = 4 /* loss has 1 entry: sum_b loss_b / sum_b max(U_b, 0) */
} ctc_packed_reduction;

typedef enum {
    CTC_PACKED_OK = 0,
    CTC_PACKED_ERR_INVALID_ARGUMENT = 1, /* a host-checkable argument is wrong */
    CTC_PACKED_ERR_WORKSPACE = 2,        /* workspace NULL or smaller than ctc_packed_workspace_size */
    CTC_PACKED_ERR_CUDA = 3,             /* a CUDA runtime call failed (see cudaGetLastError) */
    CTC_PACKED_ERR_UNSUPPORTED = 4       /* sizes beyond what the kernels support (D > 1048576, max_target_len > 3839; FSA: D > 16384, or max_states and max_labels beyond shared memory) */
} ctc_packed_status;

/* Bits of the device status word (ctc_packed_read_status). */
#define CTC_PACKED_DEV_NEGATIVE_TARGET_LENGTH 0x1u
#define CTC_PACKED_DEV_TARGET_LENGTH_EXCEEDS_MAX 0x2u
#define CTC_PACKED_DEV_BAD_LENGTH 0x4u
#define CTC_PACKED_DEV_BAD_CU_SEQLENS 0x8u
#define CTC_PACKED_DEV_LABEL_OUT_OF_RANGE 0x10u
#define CTC_PACKED_DEV_WAIT_TIMEOUT 0x20u /* a bounded wait inside a kernel gave up */
#define CTC_PACKED_DEV_NO_GRAD_STATE 0x40u /* backward after a CTC_PACKED_FLAG_LOSS_ONLY forward: rows left zero */
#define CTC_PACKED_DEV_BAD_FSA 0x80u       /* FSA path: a sequence's states, edges or offsets out of range */

/* Flags of ctc_packed_forward. */
#define CTC_PACKED_FLAG_LOSS_ONLY 0x1u /* skip the work only the backward needs; ctc_packed_backward then fails */
/*
 * The (T_total, D) input holds a model's unnormalised logits z, not log
 * probabilities.  The forward takes log_softmax over each row itself: one
 * extra dense read of z computes each row's log-sum-exp lse[t] (kept in the
 * workspace), and the path then uses lp[t, c] = z[t, c] - lse[t] in float32,
 * so no normalised copy of the rows is ever written.  The following
 * ctc_packed_backward returns the gradient with respect to the logits,
 * scale * softmax(z)[t, c] - P[t, c] (the log_softmax backward is fused; it
 * is the identity on rows that sum to zero).  A row holding NaN or +inf gets
 * a NaN log_softmax, a row of -inf a NaN one too, as log_softmax gives.
 * Page "feat(asr): native CTC loss kernel over sequence-packed log
 * probabilities", ctc_loss.py: the path's input is log_softmax(logits) and
 * its gradient scale * exp(lp) - P is the gradient with respect to them.
 */
#define CTC_PACKED_FLAG_LOGITS 0x2u

/*
 * Bytes of device workspace a forward/backward pair with these sizes needs.
 * The workspace carries the per-utterance metadata, the work queue, the
 * stored forward (alpha) and backward (beta) state rows, their per-frame
 * offsets and the per-utterance log-likelihoods.  Returns 0 when the sizes
 * are invalid (negative) or unsupported.
 */
size_t ctc_packed_workspace_size(int64_t T_total, int32_t B, int32_t max_target_len, int32_t D,
                                 ctc_packed_dtype dtype);

/*
 * Bytes of workspace a forward with CTC_PACKED_FLAG_LOSS_ONLY needs (the
 * metadata, the work queue and the emission matrix: no state rows are
 * stored).  At most ctc_packed_workspace_size.  0 for invalid or
 * unsupported sizes.
 */
size_t ctc_packed_workspace_size_loss_only(int64_t T_total, int32_t B, int32_t max_target_len, int32_t D,
                                           ctc_packed_dtype dtype);

/*
 * Forward: per-utterance CTC loss, reduced as asked.
 *
 *   log_probs      (T_total, D) row-major, dtype `dtype`, device; 4-byte aligned.
 *   cu_seqlens     (B + 1) int32: utterance b's rows start at cu_seqlens[b];
 *                  cu_seqlens[B] <= T_total.
 *   lengths        (B) int32: frames of utterance b, at most its span
 *                  cu_seqlens[b+1] - cu_seqlens[b] (rows past it are a gap).
 *   targets        concatenated int32 target ids (see the header comment).
 *   target_lengths (B) int32, each in [0, max_target_len].
 *   blank          class index of the blank, in [0, D).
 *   loss           float32 device output: B entries for NONE, 1 otherwise.
 *   workspace      device buffer of at least ctc_packed_workspace_size bytes
 *                  (ctc_packed_workspace_size_loss_only with
 *                  CTC_PACKED_FLAG_LOSS_ONLY); pass the same one, unchanged,
 *                  to ctc_packed_backward.
 *   flags          0, or an OR of CTC_PACKED_FLAG_LOSS_ONLY and
 *                  CTC_PACKED_FLAG_LOGITS; other bits are invalid.
 */
ctc_packed_status ctc_packed_forward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                                     const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* targets,
                                     const int32_t* target_lengths, int32_t B, int32_t max_target_len,
                                     int32_t blank, int zero_infinity, ctc_packed_reduction reduction, float* loss,
                                     void* workspace, size_t workspace_bytes, unsigned flags, cudaStream_t stream);

/*
 * Backward: gradient of the reduced loss with respect to log_probs (with
 * respect to the logits after a forward with CTC_PACKED_FLAG_LOGITS).
 *
 * Same inputs as the forward that filled `workspace` (same values, same
 * buffers or copies of them).  grad_loss is the float32 upstream gradient of
 * the loss (B entries for NONE, 1 otherwise).  grad_log_probs receives
 * (T_total, D) values in `dtype` (rounded to nearest even from float32); it
 * may not overlap log_probs.  Every row is written: rows outside every
 * utterance get 0.  The backward only reads the workspace, except for the
 * status word.
 */
ctc_packed_status ctc_packed_backward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                                      const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* targets,
                                      const int32_t* target_lengths, int32_t B, int32_t max_target_len,
                                      int32_t blank, int zero_infinity, ctc_packed_reduction reduction,
                                      const float* grad_loss, void* workspace, size_t workspace_bytes,
                                      void* grad_log_probs, cudaStream_t stream);

/*
 * Forward and backward in one call, for callers that have the upstream
 * gradient `grad_loss` at hand when they ask for the loss (a training step
 * that reduces the loss and calls backward right away).  Page "feat(asr):
 * native CTC loss kernel over sequence-packed log probabilities",
 * ctc_loss.py ``_PackedCTCLoss``: its forward and backward run one after the
 * other; here one call enqueues both.
 *
 * Arguments are those of ctc_packed_forward and ctc_packed_backward
 * together; `flags` is 0 or CTC_PACKED_FLAG_LOGITS.  `loss` gets what
 * ctc_packed_forward writes and `grad_log_probs` what ctc_packed_backward
 * writes with the same inputs and grad_loss, bit for bit.  The workspace is
 * left as after ctc_packed_forward, so ctc_packed_backward may follow with
 * another grad_loss.
 */
ctc_packed_status ctc_packed_forward_backward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total,
                                              int32_t D, const int32_t* cu_seqlens, const int32_t* lengths,
                                              const int32_t* targets, const int32_t* target_lengths, int32_t B,
                                              int32_t max_target_len, int32_t blank, int zero_infinity,
                                              ctc_packed_reduction reduction, const float* grad_loss, float* loss,
                                              void* grad_log_probs, void* workspace, size_t workspace_bytes,
                                              unsigned flags, cudaStream_t stream);

/*
 * Float64 path: the forward and backward above for float64 log probabilities
 * (or logits with CTC_PACKED_FLAG_LOGITS), with a float64 loss, upstream
 * gradient and gradient; same layout, sizes, checks, device status bits,
 * reductions and flags as ctc_packed_forward / ctc_packed_backward.  The
 * workspace comes from ctc_packed_workspace_size(..., CTC_PACKED_F64) (or the
 * loss-only size) and is not interchangeable with the other dtypes' one.
 *   log_probs, grad_log_probs  8-byte aligned; not overlapping.
 *   loss                       float64 device output: B entries for NONE, 1 otherwise.
 *   grad_loss                  float64 device input: B entries for NONE, 1 otherwise.
 * Precision: probabilities are carried as a 62-bit integer mantissa with an
 * int exponent through both recursions, so no state underflows; the loss and
 * gradient agree with an exact float64 evaluation to about 1e-12 relative.
 * A NaN or +inf label or blank log probability gives the utterance a NaN
 * loss (and NaN class entries in its gradient rows).
 * Page "feat(asr): native CTC loss kernel over sequence-packed log
 * probabilities": ctc.py forward_packed serves float64 at float64 precision
 * on a path of its own, and test_ctc_loss.py test_float64_takes_padded_path
 * holds it to 1e-10; this path does the same without padding the batch.
 */
ctc_packed_status ctc_packed_forward_f64(const double* log_probs, int64_t T_total, int32_t D,
                                         const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* targets,
                                         const int32_t* target_lengths, int32_t B, int32_t max_target_len,
                                         int32_t blank, int zero_infinity, ctc_packed_reduction reduction,
                                         double* loss, void* workspace, size_t workspace_bytes, unsigned flags,
                                         cudaStream_t stream);
ctc_packed_status ctc_packed_backward_f64(const double* log_probs, int64_t T_total, int32_t D,
                                          const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* targets,
                                          const int32_t* target_lengths, int32_t B, int32_t max_target_len,
                                          int32_t blank, int zero_infinity, ctc_packed_reduction reduction,
                                          const double* grad_loss, void* workspace, size_t workspace_bytes,
                                          double* grad_log_probs, cudaStream_t stream);

/*
 * Copies the device status word of `workspace` (an OR of CTC_PACKED_DEV_*
 * bits, 0 when every utterance was well formed) into *device_status after
 * the work queued on `stream` so far has finished.  This call synchronises
 * the stream; do not call it during graph capture.
 */
ctc_packed_status ctc_packed_read_status(const void* workspace, uint32_t* device_status, cudaStream_t stream);

/*
 * Bytes of the fixed scratch array behind ctc_packed_forward_noalloc (32 MiB).
 * A batch fits when ctc_packed_workspace_size_loss_only(...) <= this value.
 */
#define CTC_PACKED_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * Loss-only forward for callers that cannot allocate device memory and so
 * cannot hand the library a workspace.  Examples: a plain C host with no
 * device allocator; a process whose device memory is reserved by another
 * framework's pool, where a new allocation could fail; a scoring loop
 * (validation, n-best rescoring) that must not stall on the device-wide
 * synchronisation that freeing memory brings.  The page "feat(asr): native
 * CTC loss kernel over sequence-packed log probabilities" has no counterpart:
 * its forward always allocates its own buffers.
 *
 * Arguments and the loss are those of ctc_packed_forward with
 * CTC_PACKED_FLAG_LOSS_ONLY; there is no workspace argument and no backward.
 * The scratch is an array of CTC_PACKED_NOALLOC_SCRATCH_BYTES in the memory of
 * each device, built into the library.  The function calls no allocator
 * (no cudaMalloc or cudaFree, nothing of a framework's).
 *
 *   - Size limit: a batch whose ctc_packed_workspace_size_loss_only exceeds
 *     CTC_PACKED_NOALLOC_SCRATCH_BYTES is rejected with
 *     CTC_PACKED_ERR_WORKSPACE before any CUDA call.  Sizes that are invalid
 *     or unsupported return the codes ctc_packed_forward would return.
 *   - Device: the call uses the scratch of the CURRENT device, and `stream`
 *     must belong to it.
 *   - Address look-up: every call asks the runtime for the scratch's device
 *     address on the current device (cudaGetSymbolAddress; nothing is cached,
 *     so a device reset leaves no stale address behind).  The first look-up
 *     on a device may load the library's device code there: make the first
 *     call on a device before any stream capture starts.  If the look-up
 *     fails, the call returns CTC_PACKED_ERR_CUDA and clears the CUDA error
 *     it left.
 *   - Memory: the array holds 32 MiB of device memory on every device where
 *     the library's device code is loaded, at the latest from the first call
 *     on that device.
 *   - Zeroing: nothing needs clearing by the caller.  The first kernel of
 *     every call resets, on `stream`, the counters and queue heads that must
 *     start at zero; the rest is written before it is read.
 *   - Overlap: all calls on one device share the one scratch.  Two calls whose
 *     GPU work can overlap (different streams without an ordering event,
 *     different host threads) race and give wrong losses.  Issue them on
 *     one stream, or order them with events.
 *   - Malformed inputs that only the device can see give that utterance a
 *     NaN loss, as in ctc_packed_forward.  The status word lives in the
 *     scratch and cannot be read by the caller.
 */
ctc_packed_status ctc_packed_forward_noalloc(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total,
                                             int32_t D, const int32_t* cu_seqlens, const int32_t* lengths,
                                             const int32_t* targets, const int32_t* target_lengths, int32_t B,
                                             int32_t max_target_len, int32_t blank, int zero_infinity,
                                             ctc_packed_reduction reduction, float* loss, cudaStream_t stream);

/*
 * Full-sum loss over a generic FSA on the same packed layout.
 *
 * Page "feat(asr): native CTC loss kernel over sequence-packed log
 * probabilities", ctc_loss.py, module docstring: the packed CTC loss follows
 * RETURNN's packed full-sum loss over a generic FSA edge list and differs by
 * building the CTC topology into its recursion.  These calls take the
 * topology as data instead.
 *
 * Sequence b (frames as in ctc_packed_forward: rows cu_seqlens[b] ..
 * cu_seqlens[b] + lengths[b]) owns:
 *   - states [state_offsets[b], state_offsets[b+1]) of start_weight and
 *     final_weight (num_states floats each, log weights, -inf: none);
 *     1 <= states of a sequence <= max_states <= 4096;
 *   - edges [edge_offsets[b], edge_offsets[b+1]) of `edges` (num_edges rows
 *     of int32 (from, to, label), states local to the sequence, label in
 *     [0, D <= 16384)) with a log weight each in edge_weight; max_labels
 *     bounds the distinct labels of one sequence's edges (more: the sequence
 *     is rejected like malformed data: status bit, NaN loss, zero rows).
 * Every edge consumes one frame.  The loss is -log of the sum over all paths
 * of lengths[b] edges of exp(start + edge weights + lp of the edges' labels
 * + final); +inf with no path (0 with zero_infinity).  The backward writes
 * scale_b * (exp(lp[t, c]) - sum of the occupancies of frame t's edges with
 * label c), scale_b = grad_loss[b] (0 for an infinite loss), and 0 on rows
 * outside every sequence; the page's gradient convention (the gradient with
 * respect to the logits of a log_softmax).  The recursions carry float32
 * mantissas with integer exponents (no underflow at any length); every sum
 * runs in a fixed order (each sequence's edges are sorted once per forward
 * into per-state and per-label lists), so results are bitwise reproducible.
 * max_states and max_labels together bound the kernels' shared memory: a
 * recursion's per-frame buffers (about 20 bytes a state and 36 a label; 28 a
 * label above 2048 states) and the backward's two stages of a row (32 bytes
 * a state and 28 a label) must each fit in 224 KB, else
 * CTC_PACKED_ERR_UNSUPPORTED (the workspace size is 0).
 *
 * All pointers are device memory; log_probs is 4-byte aligned for every
 * dtype.  Errors the host can see return before
 * anything is enqueued; malformed FSA data or lengths set the status word
 * (ctc_packed_read_status works on this workspace) and a NaN loss.  The
 * workspace holds the status word, each sequence's log-sum, its sorted edge
 * lists, every frame's forward and backward values and label values (the
 * forward runs both recursions of a sequence at the same time) and, after
 * the backward, each row's class sums; it is sized by
 * ctc_packed_fsa_workspace_size with the same num_states and num_edges as
 * the calls.  Pass it unchanged from the forward to the backward.  The
 * backward forms each row's edge occupancies and class sums from those
 * values, then writes the dense gradient rows with the CTC path's all-SM
 * gradient stream.
 */
size_t ctc_packed_fsa_workspace_size(int64_t T_total, int32_t B, int32_t num_states, int32_t num_edges,
                                     int32_t max_states, int32_t max_labels, int32_t D);
ctc_packed_status ctc_packed_fsa_forward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                                         const int32_t* cu_seqlens, const int32_t* lengths, int32_t B,
                                         const int32_t* state_offsets, const float* start_weight,
                                         const float* final_weight, int32_t num_states, const int32_t* edge_offsets,
                                         const int32_t* edges, const float* edge_weight, int32_t num_edges,
                                         int32_t max_states, int32_t max_labels, int zero_infinity, float* loss,
                                         void* workspace, size_t workspace_bytes, cudaStream_t stream);
ctc_packed_status ctc_packed_fsa_backward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                                          const int32_t* cu_seqlens, const int32_t* lengths, int32_t B,
                                          const int32_t* state_offsets, const float* start_weight,
                                          const float* final_weight, int32_t num_states,
                                          const int32_t* edge_offsets, const int32_t* edges,
                                          const float* edge_weight, int32_t num_edges, int32_t max_states,
                                          int32_t max_labels, int zero_infinity, const float* grad_loss,
                                          void* workspace, size_t workspace_bytes, void* grad_log_probs,
                                          cudaStream_t stream);

/* Human-readable name of a ctc_packed_status value (static storage). */
const char* ctc_packed_status_string(ctc_packed_status status);

#ifdef __cplusplus
}
#endif

#endif /* CTC_PACKED_H */
