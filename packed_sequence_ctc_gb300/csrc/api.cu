// C-ABI entry points of the packed CTC library: host-side argument checks,
// workspace layout and kernel launches.  No host synchronisation except in
// ctc_packed_read_status.
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "ctc_common.cuh"
#include "ctc_kernels.h"

using namespace ctcp;

namespace {

int elem_bytes(ctc_packed_dtype d) { return d == CTC_PACKED_F32 ? 4 : 2; }

bool valid_dtype(int d) { return d == CTC_PACKED_F32 || d == CTC_PACKED_BF16 || d == CTC_PACKED_F16; }
bool valid_reduction(int r) {
    return r == CTC_PACKED_NONE || r == CTC_PACKED_SUM || r == CTC_PACKED_MEAN || r == CTC_PACKED_MEAN_BATCH ||
           r == CTC_PACKED_MEAN_VOLUME;
}

// Checks shared by forward and backward.  Returns CTC_PACKED_OK or the error.
ctc_packed_status check_common(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                               const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* target_lengths,
                               int32_t B, int32_t max_target_len, int32_t blank, int reduction,
                               const void* workspace, size_t workspace_bytes, bool loss_only = false) {
    if (!valid_dtype(dtype) || !valid_reduction(reduction)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (T_total < 0 || B < 0 || max_target_len < 0 || D < 1) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (blank < 0 || blank >= D) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (D > kMaxD || max_target_len > kMaxTargetLen || T_total > INT32_MAX) return CTC_PACKED_ERR_UNSUPPORTED;
    if (cu_seqlens == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (B > 0 && (lengths == nullptr || target_lengths == nullptr)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (T_total > 0 && log_probs == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    // 4-byte alignment even for 2-byte types: the label-column gathers fetch aligned 4-byte words
    if (reinterpret_cast<uintptr_t>(log_probs) % 4 != 0) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr) return CTC_PACKED_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return CTC_PACKED_ERR_WORKSPACE;
    const Layout L = make_layout(T_total, B, max_target_len, D);
    if (workspace_bytes < (loss_only ? L.loss_only_total : L.total)) return CTC_PACKED_ERR_WORKSPACE;
    return CTC_PACKED_OK;
}

// Rows of at least this many bytes take the bulk-copy gradient stream
// (stream.cu); narrower rows the class-sum pass plus the row-group stream
// (grad.cu), which packs several rows per warp.  Measured: 1025 bf16
// classes (2050-byte rows) 37.3 us by the two kernels against 39.1 us by
// the stream; 1025 fp32 classes (4100 bytes) 212 us against 170 us.
constexpr long long kStreamMinRowBytes = 4096;

// CTC_PACKED_STREAM=0 keeps every backward on the class-sum pass and the
// row-group stream, =1 sends every supported one through the bulk-copy
// stream; unset, the row width decides.
int stream_override() {
    const char* e = std::getenv("CTC_PACKED_STREAM");
    if (e == nullptr || e[0] == '\0') return -1;
    return e[0] == '0' ? 0 : 1;
}

// State-row policy: 1 keeps every frame's alpha and beta rows for the
// backward; K > 1 (a power of two) keeps only the rows at multiples of K and
// the backward recomputes the others (segpost.cu).  CTC_PACKED_CKPT=K
// overrides (1 or a power of two the recompute supports).
int checkpoint_interval(const Layout& L) {
    const int kmax = segpost_max_ckpt(L);
    const char* e = std::getenv("CTC_PACKED_CKPT");
    if (e != nullptr && e[0] != '\0') {
        const int k = std::atoi(e);
        if (k >= 2 && (k & (k - 1)) == 0 && k <= kmax) return k;
        return 1;
    }
    return 1;
}

// Fills `sa` for the bulk-copy stream; false when it cannot run this call
// (unaligned buffers, or one team's slots do not fit shared memory).
bool plan_stream(StreamArgs& sa, const Layout& L, const void* lp, void* grad, ctc_packed_dtype dtype, int32_t D,
                 const int32_t* cu, const int32_t* targets, const float* grad_loss, int32_t blank, int reduction, int zero_infinity,
                 void* workspace) {
    const uintptr_t l0 = reinterpret_cast<uintptr_t>(lp), g0 = reinterpret_cast<uintptr_t>(grad);
    if ((l0 & 15u) != 0 || (g0 & 15u) != 0) return false;
    sa = StreamArgs{};
    sa.L = L;
    sa.ws = workspace;
    sa.lp = lp;
    sa.grad = grad;
    sa.cu = cu;
    sa.targets = targets;
    sa.grad_loss = grad_loss;
    sa.D = D;
    sa.blank = blank;
    sa.reduction = reduction;
    sa.zero_infinity = zero_infinity ? 1 : 0;
    sa.elem_bytes = elem_bytes(dtype);
    sa.gp_mul = grad_group_multiplier(L);
    if (sa.gp_mul == 0) return false;
    return stream_plan(sa);
}

// The forward's kernels: prep, the logits' row log-sum-exp (logits input),
// the emission gather with the label analysis, the chains.
ctc_packed_status enqueue_forward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                                  const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* targets,
                                  const int32_t* target_lengths, int32_t B, int32_t max_target_len, int32_t blank,
                                  int zero_infinity, int reduction, float* loss, void* workspace, bool need_grad,
                                  bool logits, cudaStream_t stream) {
    const Layout L = make_layout(T_total, B, max_target_len, D);
    PrepArgs pa{};
    pa.L = L;
    pa.ws = workspace;
    pa.cu = cu_seqlens;
    pa.lengths = lengths;
    pa.target_lengths = target_lengths;
    pa.loss = loss;
    pa.reduction = reduction;
    pa.zero_infinity = zero_infinity ? 1 : 0;
    pa.need_grad = need_grad ? 1 : 0;
    pa.group_pairs = L.gpairs;
    pa.logits = logits ? 1 : 0;
    const int ckpt = checkpoint_interval(L);
    pa.ckpt = ckpt;
    if (launch_prep(pa, stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;

    ChainArgs ca{};
    ca.L = L;
    ca.ws = workspace;
    ca.lp = log_probs;
    ca.lp_bytes = T_total * (int64_t)D * elem_bytes(dtype);
    ca.cu = cu_seqlens;
    ca.targets = targets;
    ca.target_lengths = target_lengths;
    ca.loss = loss;
    ca.D = D;
    ca.blank = blank;
    ca.reduction = reduction;
    ca.zero_infinity = zero_infinity ? 1 : 0;
    ca.lse = nullptr;
    ca.store_rows = need_grad ? ckpt : 0;
    if (logits) {
        // one dense pass over the logits: each row's log-sum-exp
        if (launch_lse(ca, (int)dtype, stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
        ca.lse = ws_at<float>(workspace, L.off_lse);
    }
    if (launch_emit(ca, (int)dtype, stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    if (launch_chain(ca, stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    return CTC_PACKED_OK;
}

// Checks of the gradient arguments (backward and forward-backward calls).
ctc_packed_status check_grad_args(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D, int32_t B,
                                  int32_t max_target_len, const int32_t* targets, const float* grad_loss,
                                  const void* grad_log_probs) {
    if (grad_log_probs == nullptr || (B > 0 && grad_loss == nullptr)) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (B > 0 && max_target_len > 0 && targets == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    const int eb = elem_bytes(dtype);
    if (reinterpret_cast<uintptr_t>(grad_log_probs) % eb != 0) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(grad_log_probs), l0 = reinterpret_cast<uintptr_t>(log_probs);
    const uintptr_t nbytes = (uintptr_t)(T_total * (int64_t)D * eb);
    if (g0 < l0 + nbytes && l0 < g0 + nbytes) return CTC_PACKED_ERR_INVALID_ARGUMENT;  // overlap
    return CTC_PACKED_OK;
}

}  // namespace

extern "C" {

size_t ctc_packed_workspace_size(int64_t T_total, int32_t B, int32_t max_target_len, int32_t D,
                                 ctc_packed_dtype dtype) {
    if ((!valid_dtype(dtype) && dtype != CTC_PACKED_F64) || T_total < 0 || B < 0 || max_target_len < 0 || D < 1)
        return 0;
    if (D > kMaxD || max_target_len > kMaxTargetLen || T_total > INT32_MAX) return 0;
    if (dtype == CTC_PACKED_F64) return f64_workspace_bytes(T_total, B, max_target_len, D, false);
    return make_layout(T_total, B, max_target_len, D).total;
}

size_t ctc_packed_workspace_size_loss_only(int64_t T_total, int32_t B, int32_t max_target_len, int32_t D,
                                           ctc_packed_dtype dtype) {
    if ((!valid_dtype(dtype) && dtype != CTC_PACKED_F64) || T_total < 0 || B < 0 || max_target_len < 0 || D < 1)
        return 0;
    if (D > kMaxD || max_target_len > kMaxTargetLen || T_total > INT32_MAX) return 0;
    if (dtype == CTC_PACKED_F64) return f64_workspace_bytes(T_total, B, max_target_len, D, true);
    return make_layout(T_total, B, max_target_len, D).loss_only_total;
}

ctc_packed_status ctc_packed_forward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                                     const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* targets,
                                     const int32_t* target_lengths, int32_t B, int32_t max_target_len,
                                     int32_t blank, int zero_infinity, ctc_packed_reduction reduction, float* loss,
                                     void* workspace, size_t workspace_bytes, unsigned flags, cudaStream_t stream) {
    ctc_packed_status st = check_common(log_probs, dtype, T_total, D, cu_seqlens, lengths, target_lengths, B,
                                        max_target_len, blank, reduction, workspace, workspace_bytes,
                                        (flags & CTC_PACKED_FLAG_LOSS_ONLY) != 0);
    if (st != CTC_PACKED_OK) return st;
    if (loss == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (B > 0 && max_target_len > 0 && targets == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if ((flags & ~(CTC_PACKED_FLAG_LOSS_ONLY | CTC_PACKED_FLAG_LOGITS)) != 0) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    const bool logits = (flags & CTC_PACKED_FLAG_LOGITS) != 0;
    const bool need_grad = (flags & CTC_PACKED_FLAG_LOSS_ONLY) == 0;
    return enqueue_forward(log_probs, dtype, T_total, D, cu_seqlens, lengths, targets, target_lengths, B,
                           max_target_len, blank, zero_infinity, reduction, loss, workspace, need_grad, logits, stream);
}

ctc_packed_status ctc_packed_backward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total, int32_t D,
                                      const int32_t* cu_seqlens, const int32_t* lengths, const int32_t* targets,
                                      const int32_t* target_lengths, int32_t B, int32_t max_target_len,
                                      int32_t blank, int zero_infinity, ctc_packed_reduction reduction,
                                      const float* grad_loss, void* workspace, size_t workspace_bytes,
                                      void* grad_log_probs, cudaStream_t stream) {
    ctc_packed_status st = check_common(log_probs, dtype, T_total, D, cu_seqlens, lengths, target_lengths, B,
                                        max_target_len, blank, reduction, workspace, workspace_bytes);
    if (st != CTC_PACKED_OK) return st;
    if (T_total == 0) return CTC_PACKED_OK;
    st = check_grad_args(log_probs, dtype, T_total, D, B, max_target_len, targets, grad_loss, grad_log_probs);
    if (st != CTC_PACKED_OK) return st;
    const int eb = elem_bytes(dtype);
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(grad_log_probs), l0 = reinterpret_cast<uintptr_t>(log_probs);

    GradArgs ga{};
    ga.L = make_layout(T_total, B, max_target_len, D);
    ga.ws = workspace;
    ga.lp = log_probs;
    ga.grad = grad_log_probs;
    ga.cu = cu_seqlens;
    ga.targets = targets;
    ga.grad_loss = grad_loss;
    ga.D = D;
    ga.blank = blank;
    ga.reduction = reduction;
    ga.zero_infinity = zero_infinity ? 1 : 0;
    int k = 1, cap = 1;
    size_t wsm = 0;
    grad_geometry(ga.L, D, k, cap, wsm);
    ga.rows_per_tile = k;
    ga.entry_cap = cap;
    ga.warp_smem = wsm;
    ga.n_tiles = (T_total + k - 1) / k;
    ga.congruent = ((g0 ^ l0) & 15u) == 0 ? 1 : 0;
    ga.gp_mul = grad_group_multiplier(ga.L);
    if (ga.gp_mul == 0) return CTC_PACKED_ERR_UNSUPPORTED;
    ga.ckpt = checkpoint_interval(ga.L);
    if (ga.ckpt > 1) {
        // checkpoint rows only: class sums by recomputation, then the row-group stream
        if (launch_segpost(ga, stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
        if (launch_grad(ga, (int)dtype, stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
        return CTC_PACKED_OK;
    }
    const int ov = stream_override();
    if (ov != 0 && (ov == 1 || (long long)D * eb >= kStreamMinRowBytes)) {
        StreamArgs sa;
        if (plan_stream(sa, ga.L, log_probs, grad_log_probs, dtype, D, cu_seqlens, targets, grad_loss, blank, reduction,
                        zero_infinity, workspace)) {
            if (launch_stream(sa, (int)dtype, stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
            return CTC_PACKED_OK;
        }
    }
    if (launch_post(ga, stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    if (launch_grad(ga, (int)dtype, stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    return CTC_PACKED_OK;
}

ctc_packed_status ctc_packed_forward_backward(const void* log_probs, ctc_packed_dtype dtype, int64_t T_total,
                                              int32_t D, const int32_t* cu_seqlens, const int32_t* lengths,
                                              const int32_t* targets, const int32_t* target_lengths, int32_t B,
                                              int32_t max_target_len, int32_t blank, int zero_infinity,
                                              ctc_packed_reduction reduction, const float* grad_loss, float* loss,
                                              void* grad_log_probs, void* workspace, size_t workspace_bytes,
                                              unsigned flags, cudaStream_t stream) {
    ctc_packed_status st = check_common(log_probs, dtype, T_total, D, cu_seqlens, lengths, target_lengths, B,
                                        max_target_len, blank, reduction, workspace, workspace_bytes);
    if (st != CTC_PACKED_OK) return st;
    if (loss == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if ((flags & ~CTC_PACKED_FLAG_LOGITS) != 0) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    if (T_total > 0) {
        st = check_grad_args(log_probs, dtype, T_total, D, B, max_target_len, targets, grad_loss, grad_log_probs);
        if (st != CTC_PACKED_OK) return st;
    } else if (B > 0 && max_target_len > 0 && targets == nullptr) {
        return CTC_PACKED_ERR_INVALID_ARGUMENT;
    }
    // the forward's kernels, then the backward's, back to back on the stream
    st = enqueue_forward(log_probs, dtype, T_total, D, cu_seqlens, lengths, targets, target_lengths, B, max_target_len,
                         blank, zero_infinity, reduction, loss, workspace, true, (flags & CTC_PACKED_FLAG_LOGITS) != 0,
                         stream);
    if (st != CTC_PACKED_OK) return st;
    return ctc_packed_backward(log_probs, dtype, T_total, D, cu_seqlens, lengths, targets, target_lengths, B,
                               max_target_len, blank, zero_infinity, reduction, grad_loss, workspace, workspace_bytes,
                               grad_log_probs, stream);
}

ctc_packed_status ctc_packed_read_status(const void* workspace, uint32_t* device_status, cudaStream_t stream) {
    if (workspace == nullptr || device_status == nullptr) return CTC_PACKED_ERR_INVALID_ARGUMENT;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return CTC_PACKED_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return CTC_PACKED_ERR_CUDA;
    *device_status = v;
    return CTC_PACKED_OK;
}

const char* ctc_packed_status_string(ctc_packed_status status) {
    switch (status) {
        case CTC_PACKED_OK: return "ok";
        case CTC_PACKED_ERR_INVALID_ARGUMENT: return "invalid argument";
        case CTC_PACKED_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case CTC_PACKED_ERR_CUDA: return "CUDA runtime error";
        case CTC_PACKED_ERR_UNSUPPORTED: return "unsupported size (D > 1048576, max_target_len > 3839, or FSA D > 16384)";
    }
    return "unknown status";
}

}  // extern "C"

namespace ctcp {

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
    // one thread per utterance, in whole warps (64 to 1024): the kernel is a
    // chain of CTA barriers, which cost more the more warps take part
    int nt = (a.L.B + 31) / 32 * 32;
    nt = nt < 64 ? 64 : (nt > 1024 ? 1024 : nt);
    return launch_pdl(prep_kernel, dim3(1), dim3(nt), 0, s, a);
}

}  // namespace ctcp
