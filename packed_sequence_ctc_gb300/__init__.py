"""Packed-sequence CTC loss on GB300: Python binding of ``libctc_packed.so``.

The compute path is the C-ABI library declared in ``include/ctc_packed.h``
(CUDA kernels for sm_103a).  This module only marshals arguments: it turns
torch tensors into device pointers and the current CUDA stream into a
``cudaStream_t``.  There is no CPU or PyTorch fallback: if the library is
missing, every call raises.

Low-level functions carry the C names (``ctc_packed_forward`` ...).  On top
of them, ``packed_ctc_loss`` is an autograd-aware functional with the
semantics of page "feat(asr): native CTC loss kernel over sequence-packed log
probabilities", ctc_loss.py ``packed_ctc_loss`` and ctc.py ``forward_packed``,
except that the targets are concatenated rather than padded.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "load_library", "ctc_packed_workspace_size", "ctc_packed_forward", "ctc_packed_backward",
    "ctc_packed_read_status", "ctc_packed_status_string", "packed_ctc_loss", "PackedCTCLoss", "Workspace",
    "DTYPE_CODES", "REDUCTION_CODES", "DEVICE_STATUS_BITS", "CTCPackedError",
    "ctc_packed_forward_noalloc", "NOALLOC_SCRATCH_BYTES", "FLAG_LOSS_ONLY", "FLAG_LOGITS",
    "ctc_packed_fsa_workspace_size", "ctc_packed_fsa_forward", "ctc_packed_fsa_backward",
    "ctc_packed_forward_backward", "ctc_packed_workspace_size_loss_only", "WORKSPACE_DTYPE_CODES",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libctc_packed.so")

DTYPE_CODES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
# workspace sizes also exist for float64, whose calls are ctc_packed_forward_f64 / ctc_packed_backward_f64
WORKSPACE_DTYPE_CODES = {**DTYPE_CODES, torch.float64: 3}
REDUCTION_CODES = {"none": 0, "sum": 1, "mean": 2, "mean_batch": 3, "mean_volume": 4}
FLAG_LOSS_ONLY = 0x1
FLAG_LOGITS = 0x2  # the input rows are logits: log_softmax is taken inside, the gradient is w.r.t. the logits
NOALLOC_SCRATCH_BYTES = 32 << 20  # CTC_PACKED_NOALLOC_SCRATCH_BYTES
DEVICE_STATUS_BITS = {
    0x1: "target_lengths must not be negative",
    0x2: "target_lengths must not exceed the targets width (max_target_len)",
    0x4: "lengths must be non-negative and fit their cu_seqlens span",
    0x8: "cu_seqlens must be non-decreasing and end at or before T_total",
    0x10: "target ids must lie in [0, D)",
    0x20: "a bounded wait inside a kernel gave up",
    0x40: "backward after a loss-only forward",
    0x80: "FSA states, edges or offsets out of range",
}

_lib = None


class CTCPackedError(RuntimeError):
    """A call of the C library returned an error status."""


def load_library(path: Optional[str] = None):
    """Load ``libctc_packed.so`` (built by ``packed_sequence_ctc_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m packed_sequence_ctc_gb300.build` "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    vp, i64, i32, sz, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_uint
    lib.ctc_packed_workspace_size.argtypes = [i64, i32, i32, i32, ctypes.c_int]
    lib.ctc_packed_workspace_size.restype = sz
    lib.ctc_packed_workspace_size_loss_only.argtypes = [i64, i32, i32, i32, ctypes.c_int]
    lib.ctc_packed_workspace_size_loss_only.restype = sz
    lib.ctc_packed_forward.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp, vp, vp, i32, i32, i32, ctypes.c_int,
                                       ctypes.c_int, vp, vp, sz, u32, vp]
    lib.ctc_packed_forward.restype = ctypes.c_int
    lib.ctc_packed_backward.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp, vp, vp, i32, i32, i32, ctypes.c_int,
                                        ctypes.c_int, vp, vp, sz, vp, vp]
    lib.ctc_packed_backward.restype = ctypes.c_int
    lib.ctc_packed_forward_backward.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp, vp, vp, i32, i32, i32,
                                                ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, sz, u32, vp]
    lib.ctc_packed_forward_backward.restype = ctypes.c_int
    lib.ctc_packed_forward_f64.argtypes = [vp, i64, i32, vp, vp, vp, vp, i32, i32, i32, ctypes.c_int, ctypes.c_int,
                                           vp, vp, sz, u32, vp]
    lib.ctc_packed_forward_f64.restype = ctypes.c_int
    lib.ctc_packed_backward_f64.argtypes = [vp, i64, i32, vp, vp, vp, vp, i32, i32, i32, ctypes.c_int, ctypes.c_int,
                                            vp, vp, sz, vp, vp]
    lib.ctc_packed_backward_f64.restype = ctypes.c_int
    lib.ctc_packed_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.ctc_packed_read_status.restype = ctypes.c_int
    lib.ctc_packed_status_string.argtypes = [ctypes.c_int]
    lib.ctc_packed_status_string.restype = ctypes.c_char_p
    lib.ctc_packed_forward_noalloc.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp, vp, vp, i32, i32, i32,
                                               ctypes.c_int, ctypes.c_int, vp, vp]
    lib.ctc_packed_forward_noalloc.restype = ctypes.c_int
    lib.ctc_packed_fsa_workspace_size.argtypes = [i64, i32, i32, i32, i32, i32, i32]
    lib.ctc_packed_fsa_workspace_size.restype = sz
    lib.ctc_packed_fsa_forward.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp, i32, vp, vp, vp, i32, vp, vp, vp, i32,
                                           i32, i32, ctypes.c_int, vp, vp, sz, vp]
    lib.ctc_packed_fsa_forward.restype = ctypes.c_int
    lib.ctc_packed_fsa_backward.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp, i32, vp, vp, vp, i32, vp, vp, vp,
                                            i32, i32, i32, ctypes.c_int, vp, vp, sz, vp, vp]
    lib.ctc_packed_fsa_backward.restype = ctypes.c_int
    if path == LIB_PATH:
        _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int):
    if rc != 0:
        msg = load_library().ctc_packed_status_string(rc).decode()
        raise CTCPackedError(f"ctc_packed call failed: {msg} (status {rc})")


def ctc_packed_status_string(status: int) -> str:
    return load_library().ctc_packed_status_string(int(status)).decode()


def ctc_packed_workspace_size(T_total: int, B: int, max_target_len: int, D: int, dtype: torch.dtype) -> int:
    return int(load_library().ctc_packed_workspace_size(T_total, B, max_target_len, D, WORKSPACE_DTYPE_CODES[dtype]))


def ctc_packed_workspace_size_loss_only(T_total: int, B: int, max_target_len: int, D: int, dtype: torch.dtype) -> int:
    return int(load_library().ctc_packed_workspace_size_loss_only(T_total, B, max_target_len, D,
                                                                  WORKSPACE_DTYPE_CODES[dtype]))


def ctc_packed_forward(log_probs, cu_seqlens, lengths, targets, target_lengths, blank: int, zero_infinity: bool,
                       reduction: str, loss, workspace, max_target_len: int, flags: int = 0, stream=None):
    """Enqueue the forward on `stream` (default: torch's current stream).
    float64 log probabilities take ctc_packed_forward_f64 (`loss` float64)."""
    T_total, D = log_probs.shape
    B = lengths.numel()
    if log_probs.dtype == torch.float64:
        _check(load_library().ctc_packed_forward_f64(
            _ptr(log_probs), T_total, D, _ptr(cu_seqlens), _ptr(lengths), _ptr(targets) if targets.numel() else None,
            _ptr(target_lengths), B, max_target_len, blank, int(bool(zero_infinity)), REDUCTION_CODES[reduction],
            _ptr(loss), _ptr(workspace), workspace.numel(), flags, _stream(stream)))
        return
    _check(load_library().ctc_packed_forward(
        _ptr(log_probs), DTYPE_CODES[log_probs.dtype], T_total, D, _ptr(cu_seqlens), _ptr(lengths),
        _ptr(targets) if targets.numel() else None, _ptr(target_lengths), B, max_target_len, blank,
        int(bool(zero_infinity)), REDUCTION_CODES[reduction], _ptr(loss), _ptr(workspace), workspace.numel(),
        flags, _stream(stream)))


def ctc_packed_backward(log_probs, cu_seqlens, lengths, targets, target_lengths, blank: int, zero_infinity: bool,
                        reduction: str, grad_loss, workspace, grad_log_probs, max_target_len: int, stream=None):
    """Enqueue the backward on `stream` (default: torch's current stream).
    float64 log probabilities take ctc_packed_backward_f64 (`grad_loss` float64)."""
    T_total, D = log_probs.shape
    B = lengths.numel()
    if log_probs.dtype == torch.float64:
        _check(load_library().ctc_packed_backward_f64(
            _ptr(log_probs), T_total, D, _ptr(cu_seqlens), _ptr(lengths), _ptr(targets) if targets.numel() else None,
            _ptr(target_lengths), B, max_target_len, blank, int(bool(zero_infinity)), REDUCTION_CODES[reduction],
            _ptr(grad_loss), _ptr(workspace), workspace.numel(), _ptr(grad_log_probs), _stream(stream)))
        return
    _check(load_library().ctc_packed_backward(
        _ptr(log_probs), DTYPE_CODES[log_probs.dtype], T_total, D, _ptr(cu_seqlens), _ptr(lengths),
        _ptr(targets) if targets.numel() else None, _ptr(target_lengths), B, max_target_len, blank,
        int(bool(zero_infinity)), REDUCTION_CODES[reduction], _ptr(grad_loss), _ptr(workspace), workspace.numel(),
        _ptr(grad_log_probs), _stream(stream)))


def ctc_packed_forward_backward(log_probs, cu_seqlens, lengths, targets, target_lengths, blank: int,
                                zero_infinity: bool, reduction: str, grad_loss, loss, grad_log_probs, workspace,
                                max_target_len: int, flags: int = 0, stream=None):
    """Enqueue forward and backward in one call (bitwise equal to
    ctc_packed_forward followed by ctc_packed_backward).  float64 log
    probabilities run exactly those two calls (the float64 path has no
    single entry point)."""
    T_total, D = log_probs.shape
    B = lengths.numel()
    if log_probs.dtype == torch.float64:
        ctc_packed_forward(log_probs, cu_seqlens, lengths, targets, target_lengths, blank, zero_infinity, reduction,
                           loss, workspace, max_target_len, flags=flags, stream=stream)
        ctc_packed_backward(log_probs, cu_seqlens, lengths, targets, target_lengths, blank, zero_infinity, reduction,
                            grad_loss, workspace, grad_log_probs, max_target_len, stream=stream)
        return
    _check(load_library().ctc_packed_forward_backward(
        _ptr(log_probs), DTYPE_CODES[log_probs.dtype], T_total, D, _ptr(cu_seqlens), _ptr(lengths),
        _ptr(targets) if targets.numel() else None, _ptr(target_lengths), B, max_target_len, blank,
        int(bool(zero_infinity)), REDUCTION_CODES[reduction], _ptr(grad_loss), _ptr(loss), _ptr(grad_log_probs),
        _ptr(workspace), workspace.numel(), flags, _stream(stream)))


def ctc_packed_forward_noalloc(log_probs, cu_seqlens, lengths, targets, target_lengths, blank: int,
                               zero_infinity: bool, reduction: str, loss, max_target_len: int, stream=None):
    """Enqueue the loss-only forward that uses the library's own fixed scratch
    (for callers that cannot allocate a workspace; calls overlapping on the
    GPU race, see the C declaration).  The call runs on log_probs' device,
    whose scratch it uses; every tensor (and `stream`) must be on that
    device."""
    if log_probs.dtype not in DTYPE_CODES or log_probs.ndim != 2 or not log_probs.is_contiguous():
        raise TypeError("log_probs must be a contiguous (T_total, D) float32, bfloat16 or float16 tensor")
    dev = log_probs.device
    want = ((cu_seqlens, torch.int32, "cu_seqlens"), (lengths, torch.int32, "lengths"),
            (targets, torch.int32, "targets"), (target_lengths, torch.int32, "target_lengths"),
            (loss, torch.float32, "loss"))
    for t, dt, name in want:
        if t.dtype != dt or not t.is_contiguous() or t.device != dev:
            raise TypeError(f"{name} must be a contiguous {dt} tensor on {dev}")
    if stream is not None and getattr(stream, "device", dev) != dev:
        raise ValueError(f"stream must belong to {dev}")
    T_total, D = log_probs.shape
    B = lengths.numel()
    with torch.cuda.device(dev):
        _check(load_library().ctc_packed_forward_noalloc(
            _ptr(log_probs), DTYPE_CODES[log_probs.dtype], T_total, D, _ptr(cu_seqlens), _ptr(lengths),
            _ptr(targets) if targets.numel() else None, _ptr(target_lengths), B, max_target_len, blank,
            int(bool(zero_infinity)), REDUCTION_CODES[reduction], _ptr(loss), _stream(stream)))


def ctc_packed_fsa_workspace_size(T_total: int, B: int, num_states: int, num_edges: int, max_states: int,
                                  max_labels: int, D: int) -> int:
    """Workspace bytes of the FSA calls; num_states and num_edges are the
    totals over the batch (start_weight entries and edge rows)."""
    return int(load_library().ctc_packed_fsa_workspace_size(T_total, B, num_states, num_edges, max_states,
                                                            max_labels, D))


def _fsa_args(log_probs, cu_seqlens, lengths, fsa):
    """Marshal the FSA tensors: fsa = (state_offsets, start_weight,
    final_weight, edge_offsets, edges (E, 3) int32, edge_weight); each must
    be a contiguous tensor of that dtype on the log probabilities' device."""
    so, sw, fw, eo, ed, ew = fsa
    want = ((cu_seqlens, torch.int32, "cu_seqlens"), (lengths, torch.int32, "lengths"),
            (so, torch.int32, "state_offsets"), (sw, torch.float32, "start_weight"),
            (fw, torch.float32, "final_weight"), (eo, torch.int32, "edge_offsets"), (ed, torch.int32, "edges"),
            (ew, torch.float32, "edge_weight"))
    for t, dt, name in want:
        if t.dtype != dt or not t.is_contiguous() or t.device != log_probs.device:
            raise TypeError(f"{name} must be a contiguous {dt} tensor on {log_probs.device}")
    if ed.ndim != 2 or ed.shape[1] != 3:
        raise ValueError("edges must have shape (E, 3): from, to, label")
    if ew.numel() != ed.shape[0] or fw.numel() != sw.numel():
        raise ValueError("edge_weight needs one value per edge, final_weight one per start_weight entry")
    if so.numel() != lengths.numel() + 1 or eo.numel() != lengths.numel() + 1:
        raise ValueError("state_offsets and edge_offsets need B + 1 entries")
    T_total, D = log_probs.shape
    return (_ptr(log_probs), DTYPE_CODES[log_probs.dtype], T_total, D, _ptr(cu_seqlens), _ptr(lengths),
            lengths.numel(), _ptr(so), _ptr(sw), _ptr(fw), sw.numel(), _ptr(eo),
            _ptr(ed) if ed.numel() else None, _ptr(ew) if ew.numel() else None, ed.shape[0])


def ctc_packed_fsa_forward(log_probs, cu_seqlens, lengths, fsa, max_states: int, max_labels: int,
                           zero_infinity: bool, loss, workspace, stream=None):
    """Enqueue the FSA full-sum forward (per-sequence losses into `loss`)."""
    _check(load_library().ctc_packed_fsa_forward(
        *_fsa_args(log_probs, cu_seqlens, lengths, fsa), max_states, max_labels, int(bool(zero_infinity)),
        _ptr(loss), _ptr(workspace), workspace.numel(), _stream(stream)))


def ctc_packed_fsa_backward(log_probs, cu_seqlens, lengths, fsa, max_states: int, max_labels: int,
                            zero_infinity: bool, grad_loss, workspace, grad_log_probs, stream=None):
    """Enqueue the FSA full-sum backward (gradient rows into `grad_log_probs`)."""
    _check(load_library().ctc_packed_fsa_backward(
        *_fsa_args(log_probs, cu_seqlens, lengths, fsa), max_states, max_labels, int(bool(zero_infinity)),
        _ptr(grad_loss), _ptr(workspace), workspace.numel(), _ptr(grad_log_probs), _stream(stream)))


def ctc_packed_read_status(workspace, stream=None) -> int:
    """The device status word (waits for the stream)."""
    out = ctypes.c_uint32(0)
    _check(load_library().ctc_packed_read_status(_ptr(workspace), ctypes.byref(out), _stream(stream)))
    return int(out.value)


class Workspace:
    """A device workspace sized for a batch shape (reusable across calls)."""

    def __init__(self, T_total: int, B: int, max_target_len: int, D: int, dtype: torch.dtype, device=None):
        n = ctc_packed_workspace_size(T_total, B, max_target_len, D, dtype)
        if n == 0:
            raise CTCPackedError("unsupported workspace sizes")
        self.tensor = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
        self.shape = (T_total, B, max_target_len, D, dtype)


def _int32(t: torch.Tensor, device) -> torch.Tensor:
    return t.to(device=device, dtype=torch.int32).contiguous()


def _raise_on_status(status: int):
    if status:
        msgs = [m for bit, m in DEVICE_STATUS_BITS.items() if status & bit]
        raise ValueError("; ".join(msgs))


class PackedCTCLoss(torch.autograd.Function):
    """Autograd glue: forward and backward both run in the CUDA library."""

    @staticmethod
    def forward(ctx, log_probs, cu_seqlens, lengths, targets, target_lengths, blank, zero_infinity, reduction,
                max_target_len, check, logits=False):
        if log_probs.dtype not in WORKSPACE_DTYPE_CODES:
            raise TypeError(f"log_probs must be float32, bfloat16, float16 or float64, got {log_probs.dtype}.")
        if log_probs.ndim != 2 or not log_probs.is_cuda:
            raise ValueError("log_probs must be a (T_total, D) CUDA tensor")
        dev = log_probs.device
        log_probs = log_probs.contiguous()
        cu, ln, tg, tl = (_int32(x, dev) for x in (cu_seqlens, lengths, targets, target_lengths))
        B = ln.numel()
        T_total, D = log_probs.shape
        ws = Workspace(T_total, B, max_target_len, D, log_probs.dtype, dev).tensor
        loss_dtype = torch.float64 if log_probs.dtype == torch.float64 else torch.float32
        loss = torch.empty(B if reduction == "none" else 1, dtype=loss_dtype, device=dev)
        ctc_packed_forward(log_probs, cu, ln, tg, tl, blank, zero_infinity, reduction, loss, ws, max_target_len,
                           flags=FLAG_LOGITS if logits else 0)
        if check:
            _raise_on_status(ctc_packed_read_status(ws))
        ctx.save_for_backward(log_probs, cu, ln, tg, tl, ws)
        ctx.args = (blank, zero_infinity, reduction, max_target_len)
        return loss if reduction == "none" else loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        log_probs, cu, ln, tg, tl, ws = ctx.saved_tensors
        blank, zero_infinity, reduction, max_target_len = ctx.args
        g_dtype = torch.float64 if log_probs.dtype == torch.float64 else torch.float32
        g = grad_out.to(g_dtype).reshape(-1).contiguous()
        grad = torch.empty_like(log_probs)
        ctc_packed_backward(log_probs, cu, ln, tg, tl, blank, zero_infinity, reduction, g, ws, grad, max_target_len)
        return grad, None, None, None, None, None, None, None, None, None, None


def packed_ctc_loss(log_probs: torch.Tensor, cu_seqlens: torch.Tensor, lengths: torch.Tensor, targets: torch.Tensor,
                    target_lengths: torch.Tensor, *, blank: int, zero_infinity: bool = False, reduction: str = "none",
                    max_target_len: Optional[int] = None, check: Optional[bool] = None,
                    logits: bool = False) -> torch.Tensor:
    """CTC loss over token-flat log probabilities (targets concatenated).

    ``logits=True``: the rows are a model's unnormalised logits; the library
    takes log_softmax of each row itself (no normalised copy is written) and
    the gradient is with respect to the logits.

    ``max_target_len`` bounds every target length (the width of a padded
    targets buffer); when omitted it is read from ``target_lengths``, which
    synchronises with the device.  ``check`` (default: on unless a CUDA graph
    is being captured) reads the device status after the forward and raises
    ``ValueError`` for malformed lengths or target ids, as the page's host
    checks do.
    """
    if reduction not in REDUCTION_CODES:
        raise ValueError(f"unexpected reduction {reduction!r}")
    if not 0 <= blank < log_probs.shape[-1]:
        raise ValueError(f"blank must be a class index below {log_probs.shape[-1]}, got {blank}.")
    capturing = torch.cuda.is_available() and torch.cuda.is_current_stream_capturing()
    if max_target_len is None:
        if capturing:
            raise ValueError("max_target_len is required under graph capture")
        max_target_len = int(target_lengths.max()) if target_lengths.numel() else 0
        max_target_len = max(max_target_len, 0)
    if check is None:
        check = not capturing
    return PackedCTCLoss.apply(log_probs, cu_seqlens, lengths, targets, target_lengths, blank, zero_infinity,
                               reduction, max_target_len, check, logits)
