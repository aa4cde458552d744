// Loss-only forward whose scratch memory is a fixed array compiled into the
// library, for callers that cannot supply a device workspace.
//
// Who needs it: code that must not allocate device memory at the point where
// it wants a loss.  Examples are a plain C host with no device allocator of
// its own; a process whose device memory is already reserved by another
// framework's memory pool, where a fresh allocation could fail; and a scoring
// loop (validation, n-best rescoring) that must not stall, since freeing
// device memory synchronises the whole device.  Such callers pass only their
// inputs and the loss buffer.
//
// The computation is the one of ctc_packed_forward with
// CTC_PACKED_FLAG_LOSS_ONLY; the same prep and chain kernels run, with this
// array as their workspace.
#include <cstdint>

#include "ctc_common.cuh"

// The scratch of ctc_packed_forward_noalloc: one per device (a __device__
// variable has one instance in each device's memory), 256-byte aligned as
// the workspace must be.
static __device__ __align__(256) unsigned char ctc_noalloc_scratch[CTC_PACKED_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch on the current device.  Looked up on every
// call (a cheap host-side query), so nothing cached can go stale; the first
// look-up on a device may load the library's device code there.
ctc_packed_status scratch_on_current_device(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, ctc_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();  // leave no error behind for the caller's next launch check
        return CTC_PACKED_ERR_CUDA;
    }
    *out = p;
    return CTC_PACKED_OK;
}

}  // namespace

extern "C" ctc_packed_status ctc_packed_forward_noalloc(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total,
                                                        int32_t D, const int32_t* cu_seqlens, const int32_t* lengths,
                                                        const int32_t* targets, const int32_t* target_lengths,
                                                        int32_t B, int32_t max_target_len, int32_t blank,
                                                        int zero_infinity, ctc_packed_reduction reduction,
                                                        float* loss, cudaStream_t stream) {
    // size check first, so an oversized call touches no device state
    const size_t need = ctc_packed_workspace_size_loss_only(T_total, B, max_target_len, D, dtype);
    if (need == 0) {
        const bool in_range = (dtype == CTC_PACKED_F32 || dtype == CTC_PACKED_BF16 || dtype == CTC_PACKED_F16) &&
                              T_total >= 0 && B >= 0 && max_target_len >= 0 && D >= 1;
        return in_range ? CTC_PACKED_ERR_UNSUPPORTED : CTC_PACKED_ERR_INVALID_ARGUMENT;
    }
    if (need > (size_t)CTC_PACKED_NOALLOC_SCRATCH_BYTES) return CTC_PACKED_ERR_WORKSPACE;
    void* scratch = nullptr;
    const ctc_packed_status st = scratch_on_current_device(&scratch);
    if (st != CTC_PACKED_OK) return st;
    // The prep kernel that opens the forward resets the control block (status
    // word, queue heads, CTA counter) on the stream before anything reads it;
    // every other scratch entry is written before it is read within the call.
    // So nothing needs clearing from the host, and one call leaves no state
    // that the next depends on.  A loss-only forward touches only the first
    // ctc_packed_workspace_size_loss_only bytes of a workspace.
    return ctc_packed_forward(log_probs, dtype, T_total, D, cu_seqlens, lengths, targets, target_lengths, B,
                              max_target_len, blank, zero_infinity, reduction, loss, scratch,
                              (size_t)CTC_PACKED_NOALLOC_SCRATCH_BYTES, CTC_PACKED_FLAG_LOSS_ONLY, stream);
}
