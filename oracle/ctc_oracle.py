"""Driver of the fp64 CTC oracle (``ctc_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The oracle is the plain, slow, float64 statement
of what the packed CTC loss computes; the tests compare the CUDA library
against it.  Only ``tests/``, the package's ``smoke()`` check and the CPU
baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA path and imports nothing from it.

Page "feat(asr): native CTC loss kernel over sequence-packed log
probabilities" (NVIDIA-NeMo/Speech PR #16437):

* ``nemo/collections/asr/parts/triton/ctc_loss.py``, ``packed_ctc_loss``
  docstring: the per-utterance loss has the semantics of
  ``torch.nn.functional.ctc_loss(reduction="none")`` -- ``inf`` for an
  utterance that cannot be aligned, or 0 with ``zero_infinity``, which also
  zeroes its gradient; float32 / bfloat16 / float16 inputs.
* same file, ``_PackedCTCLoss``: a frame outside every utterance gets a zero
  gradient; the gradient takes the dtype of the log probabilities.
* ``nemo/collections/asr/losses/ctc.py``, ``forward_packed``: reduction
  ``sum`` adds the losses; ``mean`` divides each loss by its target length
  clamped to at least 1 and averages over the batch; ``none`` keeps them.
  The module's own ``reduce`` then offers ``mean_batch`` and ``mean_volume``
  (the page's tests parametrize both; the page does not print their
  bodies).  Read here as the batch mean of the losses and as the sum of the
  losses over the sum of the target lengths.

Half-precision inputs are upcast exactly to float64 before anything else,
so the oracle sees the very values the kernels read.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ctc_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_ctc_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ctc_oracle.c`` with gcc into ``oracle/_ctc_oracle.so``."""
    with _lock:
        stale = not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB_PATH + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library and declare its entry points."""
    lib = ctypes.CDLL(path)
    i64p = ctypes.POINTER(ctypes.c_int64)
    f64p = ctypes.POINTER(ctypes.c_double)
    lib.ctc_oracle_batch.argtypes = [f64p, ctypes.c_int64, ctypes.c_int64, i64p, i64p, i64p, i64p,
                                     ctypes.c_int64, ctypes.c_int64, f64p, f64p, ctypes.c_int]
    lib.ctc_oracle_batch.restype = ctypes.c_int
    lib.ctc_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def max_threads() -> int:
    return int(_load().ctc_oracle_max_threads())


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor; .double() upcasts half types exactly
        return np.ascontiguousarray(x.detach().cpu().double().numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _as_i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def raw_nll_and_grad(log_probs, cu_seqlens, lengths, targets, target_lengths, blank: int,
                     need_grad: bool = True, threads: int = 0, lib=None) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """Per-utterance negative log-likelihood (``inf`` if infeasible) and the
    unit-scale gradient rows ``exp(lp) - P`` (zero outside every utterance)."""
    lp = _as_f64(log_probs)
    if lp.ndim != 2:
        raise ValueError("log_probs must be (T_total, D)")
    T_total, D = lp.shape
    cu = _as_i64(cu_seqlens)
    ln = _as_i64(lengths)
    tg = _as_i64(targets).reshape(-1)
    tl = _as_i64(target_lengths)
    B = int(ln.shape[0])
    nll = np.zeros(B, dtype=np.float64)
    grad = np.zeros((T_total, D), dtype=np.float64) if need_grad else None

    def p(a, t):
        return a.ctypes.data_as(ctypes.POINTER(t))

    rc = (lib or _load()).ctc_oracle_batch(
        p(lp, ctypes.c_double), T_total, D, p(cu, ctypes.c_int64), p(ln, ctypes.c_int64),
        p(tg if tg.size else np.zeros(1, np.int64), ctypes.c_int64), p(tl, ctypes.c_int64), B, int(blank),
        p(nll, ctypes.c_double), p(grad, ctypes.c_double) if grad is not None else None, int(threads))
    if rc != 0:
        raise MemoryError("oracle ran out of memory")
    return nll, grad


def utterance_scales(nll: np.ndarray, target_lengths, reduction: str, zero_infinity: bool,
                     grad_loss=None) -> np.ndarray:
    """The upstream gradient each utterance's rows are multiplied by."""
    tl = _as_i64(target_lengths)
    B = nll.shape[0]
    if reduction == "none":
        g = np.ones(B) if grad_loss is None else _as_f64(grad_loss).reshape(B)
        scale = g.copy()
    elif reduction == "sum":
        g = 1.0 if grad_loss is None else float(_as_f64(grad_loss).reshape(-1)[0])
        scale = np.full(B, g)
    elif reduction == "mean":
        g = 1.0 if grad_loss is None else float(_as_f64(grad_loss).reshape(-1)[0])
        scale = g / (B * np.maximum(tl, 1).astype(np.float64))
    elif reduction == "mean_batch":
        g = 1.0 if grad_loss is None else float(_as_f64(grad_loss).reshape(-1)[0])
        scale = np.full(B, g / B) if B else np.zeros(0)
    elif reduction == "mean_volume":
        g = 1.0 if grad_loss is None else float(_as_f64(grad_loss).reshape(-1)[0])
        with np.errstate(divide="ignore", invalid="ignore"):
            scale = np.full(B, np.float64(g) / np.float64(tl.sum()))
    else:
        raise ValueError(f"unknown reduction {reduction!r}")
    if zero_infinity:
        scale = np.where(np.isposinf(nll), 0.0, scale)
    return scale


def reduce_losses(nll: np.ndarray, target_lengths, reduction: str, zero_infinity: bool):
    """Apply zero_infinity and the reduction to the per-utterance losses."""
    tl = _as_i64(target_lengths)
    losses = np.where(np.isposinf(nll), 0.0, nll) if zero_infinity else nll.copy()
    if reduction == "none":
        return losses
    if reduction == "sum":
        return np.float64(losses.sum())
    if reduction == "mean":
        if losses.shape[0] == 0:
            return np.float64(np.nan)
        return np.float64((losses / np.maximum(tl, 1)).mean())
    if reduction == "mean_batch":
        if losses.shape[0] == 0:
            return np.float64(np.nan)
        return np.float64(losses.mean())
    if reduction == "mean_volume":
        with np.errstate(divide="ignore", invalid="ignore"):
            return np.float64(losses.sum()) / np.float64(tl.sum())
    raise ValueError(f"unknown reduction {reduction!r}")


def ctc_loss_packed(log_probs, cu_seqlens, lengths, targets, target_lengths, blank: int,
                    zero_infinity: bool = False, reduction: str = "none", grad_loss=None,
                    need_grad: bool = True, threads: int = 0):
    """Loss (after reduction) and gradient of the packed CTC loss in float64.

    Returns ``(loss, grad, nll)``: ``loss`` is a float64 scalar, or a ``(B,)``
    array for ``reduction="none"``; ``grad`` is ``(T_total, D)`` float64 (or
    None); ``nll`` holds the raw per-utterance losses.
    """
    nll, raw = raw_nll_and_grad(log_probs, cu_seqlens, lengths, targets, target_lengths, blank,
                                need_grad=need_grad, threads=threads)
    loss = reduce_losses(nll, target_lengths, reduction, zero_infinity)
    grad = None
    if need_grad:
        scale = utterance_scales(nll, target_lengths, reduction, zero_infinity, grad_loss)
        cu = _as_i64(cu_seqlens)
        ln = _as_i64(lengths)
        grad = np.zeros_like(raw)
        for b in range(nll.shape[0]):
            rows = slice(int(cu[b]), int(cu[b]) + int(ln[b]))
            if scale[b] != 0.0:
                grad[rows] = raw[rows] * scale[b]
            # a zero scale leaves exact zeros (zero_infinity zeroes the gradient)
    return loss, grad, nll


def log_softmax_rows(logits) -> np.ndarray:
    """Row-wise log_softmax in float64: ``z - max - log(sum(exp(z - max)))``
    over the class axis (a row of -inf stays NaN, as log_softmax gives)."""
    z = _as_f64(logits)
    if z.ndim != 2:
        raise ValueError("logits must be (T_total, D)")
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        m = z.max(axis=1, keepdims=True) if z.shape[1] else np.zeros((z.shape[0], 1))
        return z - m - np.log(np.exp(z - m).sum(axis=1, keepdims=True))


def ctc_loss_packed_logits(logits, cu_seqlens, lengths, targets, target_lengths, blank: int,
                           zero_infinity: bool = False, reduction: str = "none", grad_loss=None,
                           need_grad: bool = True, threads: int = 0):
    """The packed CTC loss of ``log_softmax(logits)`` and its gradient with
    respect to the logits, in float64.

    Page "feat(asr): native CTC loss kernel over sequence-packed log
    probabilities", ``ctc_loss.py``: the path's inputs are the log_softmax
    of a model's logits, and the gradient it returns, ``scale * exp(lp) - P``,
    is the gradient with respect to those logits (each row of
    ``exp(lp) - P`` sums to zero, so log_softmax's backward leaves it
    unchanged).  With ``lp = log_softmax(logits)`` that is
    ``scale * softmax(logits) - P``: the loss and gradient of
    ``ctc_loss_packed`` on the normalised rows.  Returns ``(loss, grad, nll)``
    as ``ctc_loss_packed`` does, ``grad`` with respect to the logits.
    """
    return ctc_loss_packed(log_softmax_rows(logits), cu_seqlens, lengths, targets, target_lengths, blank,
                           zero_infinity, reduction, grad_loss=grad_loss, need_grad=need_grad, threads=threads)


def oracle_batch(batch, grad_loss=None, need_grad: bool = True, threads: int = 0):
    """``ctc_loss_packed`` on a ``workloads.Batch``-like object."""
    return ctc_loss_packed(batch.log_probs, batch.cu_seqlens, batch.lengths, batch.targets, batch.target_lengths,
                           batch.blank, batch.zero_infinity, batch.reduction, grad_loss=grad_loss,
                           need_grad=need_grad, threads=threads)
