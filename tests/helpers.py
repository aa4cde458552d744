"""Shared helpers of the GPU tests: run a batch through the C-ABI and compare
with the fp64 oracle at the tolerances of the contract.

Tolerances (per element):
* loss: |gpu - oracle| <= 1e-4 * max(1, |oracle|), infinities must match;
* float32 gradient: 2e-5 absolute;
* bfloat16 / float16 gradient: one unit in the last place of the oracle value
  in that dtype, plus 1e-3 absolute (the oracle runs on the upcast half
  values, so both sides see the same inputs).
"""

from __future__ import annotations

import numpy as np
import torch

import packed_sequence_ctc_gb300 as pk

MANTISSA_BITS = {torch.float32: 23, torch.bfloat16: 7, torch.float16: 10}


def ulp(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    m, e = np.frexp(np.abs(ref))
    return np.ldexp(1.0, e - 1 - MANTISSA_BITS[dtype])


def grad_tolerance(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    if dtype == torch.float32:
        return np.full_like(ref, 2e-5)
    return ulp(ref, dtype) + 1e-3


def loss_close(gpu, ref) -> bool:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isinf(gpu) & np.isinf(ref) & (np.sign(gpu) == np.sign(ref))
    close = np.abs(gpu - ref) <= 1e-4 * np.maximum(1.0, np.abs(ref))
    return bool(np.all(both_inf | close))


def assert_loss_close(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not loss_close(gpu, ref):
        diff = np.abs(gpu - ref) / np.maximum(1.0, np.abs(ref))
        raise AssertionError(f"loss mismatch: max scaled diff {np.nanmax(diff)}\ngpu={gpu}\nref={ref}")


def assert_grad_close(gpu: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, rows=None):
    g = gpu.double().cpu().numpy()
    if rows is not None:
        g, ref = g[rows], ref[rows]
    tol = grad_tolerance(ref, dtype)
    bad = ~(np.abs(g - ref) <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.nanmax(np.abs(g - ref) - tol)
        raise AssertionError(f"{int(bad.sum())} gradient entries out of tolerance (worst excess {worst}); "
                             f"first {idx.tolist()}: gpu {g[bad][:5]} ref {ref[bad][:5]}")


def to_device(batch, device="cuda"):
    return {
        "log_probs": batch.log_probs.to(device).contiguous(),
        "cu": batch.cu_seqlens.to(device),
        "lengths": batch.lengths.to(device),
        "targets": batch.targets.to(device),
        "target_lengths": batch.target_lengths.to(device),
    }


def run_gpu(batch, grad_loss=None, max_target_len=None, need_grad=True, grad_offset_bytes=0, guard_bytes=64,
            device="cuda", log_probs=None, logits=False):
    """Forward + backward of `batch` through the C-ABI on the current stream.

    The gradient lands inside a larger buffer whose margins hold a sentinel,
    so writes outside [0, T_total*D) are caught.  ``logits=True`` passes the
    rows as logits (CTC_PACKED_FLAG_LOGITS).  Returns (loss, grad, status).
    """
    d = to_device(batch, device)
    lp = d["log_probs"] if log_probs is None else log_probs
    T_total, D = lp.shape
    B = batch.B
    mtl = batch.max_target_len if max_target_len is None else max_target_len
    ws = pk.Workspace(T_total, B, mtl, D, lp.dtype, device).tensor
    red = batch.reduction
    loss = torch.full((B if red == "none" else 1,), float("nan"), dtype=torch.float32, device=device)
    pk.ctc_packed_forward(lp, d["cu"], d["lengths"], d["targets"], d["target_lengths"], batch.blank,
                          batch.zero_infinity, red, loss, ws, mtl,
                          flags=(0 if need_grad else pk.FLAG_LOSS_ONLY) | (pk.FLAG_LOGITS if logits else 0))
    grad = None
    if need_grad:
        if grad_loss is None:
            grad_loss = torch.ones(B if red == "none" else 1, dtype=torch.float32)
        g_up = torch.as_tensor(grad_loss, dtype=torch.float32).reshape(-1).to(device)
        esz = lp.element_size()
        n = T_total * D * esz
        raw = torch.full((n + 2 * guard_bytes + 16,), 0xA5, dtype=torch.uint8, device=device)
        start = guard_bytes + grad_offset_bytes
        grad_view = raw[start: start + n].view(lp.dtype).view(T_total, D)
        pk.ctc_packed_backward(lp, d["cu"], d["lengths"], d["targets"], d["target_lengths"], batch.blank,
                               batch.zero_infinity, red, g_up, ws, grad_view, mtl)
        torch.cuda.synchronize()
        head = raw[:start].cpu()
        tail = raw[start + n:].cpu()
        assert bool((head == 0xA5).all()) and bool((tail == 0xA5).all()), "gradient write outside its buffer"
        grad = grad_view.clone()
    status = pk.ctc_packed_read_status(ws)
    out = loss.double().cpu().numpy()
    return (out if red == "none" else out[0]), grad, status


def run_gpu_fused(batch, grad_loss=None, max_target_len=None, guard_bytes=64, device="cuda", log_probs=None,
                  logits=False, workspace=None):
    """Forward and backward in one call (ctc_packed_forward_backward) on the
    current stream, the gradient inside a sentinel-guarded buffer like
    run_gpu.  Returns (loss, grad, status, workspace)."""
    d = to_device(batch, device)
    lp = d["log_probs"] if log_probs is None else log_probs
    T_total, D = lp.shape
    B = batch.B
    mtl = batch.max_target_len if max_target_len is None else max_target_len
    ws = pk.Workspace(T_total, B, mtl, D, lp.dtype, device).tensor if workspace is None else workspace
    red = batch.reduction
    loss = torch.full((B if red == "none" else 1,), float("nan"), dtype=torch.float32, device=device)
    if grad_loss is None:
        grad_loss = torch.ones(B if red == "none" else 1, dtype=torch.float32)
    g_up = torch.as_tensor(grad_loss, dtype=torch.float32).reshape(-1).to(device)
    n = T_total * D * lp.element_size()
    raw = torch.full((n + 2 * guard_bytes + 16,), 0xA5, dtype=torch.uint8, device=device)
    grad_view = raw[guard_bytes: guard_bytes + n].view(lp.dtype).view(T_total, D)
    pk.ctc_packed_forward_backward(lp, d["cu"], d["lengths"], d["targets"], d["target_lengths"], batch.blank,
                                   batch.zero_infinity, red, g_up, loss, grad_view, ws, mtl,
                                   flags=pk.FLAG_LOGITS if logits else 0)
    torch.cuda.synchronize()
    head = raw[:guard_bytes].cpu()
    tail = raw[guard_bytes + n:].cpu()
    assert bool((head == 0xA5).all()) and bool((tail == 0xA5).all()), "gradient write outside its buffer"
    status = pk.ctc_packed_read_status(ws)
    out = loss.double().cpu().numpy()
    return (out if red == "none" else out[0]), grad_view.clone(), status, ws
