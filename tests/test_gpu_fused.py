"""The forward-backward call (ctc_packed_forward_backward), through the C-ABI.

The call must give exactly what a forward followed by a backward gives: the
same losses and the same gradient bits, on every named workload and on the
edge cases of the page's test file (test_ctc_loss.py of "feat(asr): native
CTC loss kernel over sequence-packed log probabilities"), which are also
checked against the fp64 oracle.  Rows of at least 4 KB take the bulk-copy
gradient stream; CTC_PACKED_STREAM=1 sends narrow rows through it as well, so
the edge cases run there at small sizes too.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import packed_sequence_ctc_gb300 as pk
import workloads
from helpers import assert_grad_close, assert_loss_close, run_gpu, run_gpu_fused

pytestmark = pytest.mark.gpu


def _defined_rows(batch, nll):
    rows = np.zeros(batch.T_total, dtype=bool)
    for b in range(batch.B):
        s, e = int(batch.cu_seqlens[b]), int(batch.cu_seqlens[b + 1])
        if batch.zero_infinity or np.isfinite(nll[b]):
            rows[s:e] = True
    rows[int(batch.cu_seqlens[-1]):] = True
    return rows


def _same(batch, grad_loss=None, **kw):
    l1, g1, s1 = run_gpu(batch, grad_loss=grad_loss, **kw)
    l2, g2, s2, _ = run_gpu_fused(batch, grad_loss=grad_loss, **kw)
    assert s1 == s2
    assert np.array_equal(np.asarray(l1), np.asarray(l2), equal_nan=True)
    assert torch.equal(g1.view(torch.uint8) if g1.dtype != torch.float32 else g1.view(torch.int32),
                       g2.view(torch.uint8) if g2.dtype != torch.float32 else g2.view(torch.int32))
    return l2, g2, s2


@pytest.mark.parametrize("name", ["tiny", "conformer", "longform", "char", "largevocab"])
def test_fused_equals_forward_then_backward(cuda_device, name):
    batch = workloads.workload(name, device=cuda_device)
    g = torch.linspace(0.5, 1.5, batch.B) if batch.reduction == "none" else torch.tensor([0.75])
    _, _, status = _same(batch, grad_loss=g)
    assert status == 0


def _wide_cases():
    # rows of 2048 bf16 or 1024 fp32 elements take the bulk-copy gradient stream
    yield "repeats_blank_id", workloads.make_batch([90, 70, 33], [30, 20, 12], 2048, seed=3, repeat_prob=0.3,
                                                   redraw_infeasible=True, dtype=torch.bfloat16, blank=7,
                                                   label_low=0, label_high=40)
    yield "empty_and_zero_length", workloads.make_batch([40, 0, 25, 9], [0, 2, 5, 0], 1024, seed=5, blank=0,
                                                        dtype=torch.float32)
    yield "gaps", workloads.make_batch([30, 22, 41], [6, 5, 9], 1024, seed=8, gaps=[3, 0, 5], dtype=torch.float32)
    yield "infeasible", workloads.make_batch([6, 50], [5, 8], 2048, seed=9, targets=[[3, 3, 3, 3, 3], list(range(1, 9))],
                                            dtype=torch.float16)
    yield "infeasible_zero_inf", workloads.make_batch([6, 50], [5, 8], 2048, seed=9,
                                                     targets=[[3, 3, 3, 3, 3], list(range(1, 9))],
                                                     dtype=torch.float16, zero_infinity=True)


@pytest.mark.parametrize("reduction", ["none", "sum", "mean", "mean_batch", "mean_volume"])
@pytest.mark.parametrize("case", [c for c, _ in _wide_cases()])
def test_fused_wide_rows_match_oracle(cuda_device, case, reduction):
    batch = dict(_wide_cases())[case]
    batch.reduction = reduction
    g = torch.linspace(-1.0, 2.0, batch.B) if reduction == "none" else torch.tensor([1.7])
    loss, grad, _ = _same(batch, grad_loss=g)
    ref_loss, ref_grad, nll = oracle.oracle_batch(batch, grad_loss=g.double().numpy())
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, batch.log_probs.dtype, rows=_defined_rows(batch, nll))


@pytest.mark.parametrize("case", [c for c, _ in _wide_cases()])
def test_fused_narrow_rows_through_the_bulk_copy_stream(cuda_device, case, monkeypatch):
    monkeypatch.setenv("CTC_PACKED_STREAM", "1")
    batch = dict(_wide_cases())[case]
    # the same utterances with 9 classes: rows far below 4 KB
    small = workloads.make_batch(batch.lengths.tolist(), batch.target_lengths.tolist(), 9, seed=2,
                                 targets=None, label_high=8, repeat_prob=0.2, dtype=batch.log_probs.dtype,
                                 zero_infinity=batch.zero_infinity)
    loss, grad, _ = _same(small)
    ref_loss, ref_grad, nll = oracle.oracle_batch(small)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, small.log_probs.dtype, rows=_defined_rows(small, nll))


def test_fused_logits_input(cuda_device):
    batch = workloads.select_utterances(workloads.workload("largevocab", device=cuda_device), [0, 5, 9])
    z = workloads.unnormalised_logits(batch, seed=17)
    loss, grad, status, _ = run_gpu_fused(batch, log_probs=z.cuda().contiguous(), logits=True)
    l2, g2, s2 = run_gpu(batch, log_probs=z.cuda().contiguous(), logits=True)
    assert status == 0 and s2 == 0
    assert np.array_equal(loss, l2)
    assert torch.equal(grad.view(torch.int16), g2.view(torch.int16))
    ref_loss, ref_grad, _ = oracle.ctc_loss_packed_logits(z, batch.cu_seqlens, batch.lengths, batch.targets,
                                                          batch.target_lengths, batch.blank, batch.zero_infinity,
                                                          batch.reduction)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, batch.log_probs.dtype)


def test_backward_after_fused_call_reuses_the_workspace(cuda_device):
    batch = workloads.select_utterances(workloads.workload("largevocab", device=cuda_device), [1, 2, 3, 4])
    _, _, _, ws = run_gpu_fused(batch, grad_loss=torch.ones(4))
    g2 = torch.tensor([2.0, -1.0, 0.5, 3.0])
    d = {k: v.cuda() for k, v in (("cu", batch.cu_seqlens), ("ln", batch.lengths), ("tg", batch.targets),
                                  ("tl", batch.target_lengths))}
    lp = batch.log_probs.cuda().contiguous()
    grad = torch.empty_like(lp)
    pk.ctc_packed_backward(lp, d["cu"], d["ln"], d["tg"], d["tl"], batch.blank, batch.zero_infinity, "none",
                           g2.cuda(), ws, grad, batch.max_target_len)
    _, ref, _ = run_gpu(batch, grad_loss=g2)
    assert torch.equal(grad.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("bad,bit", [("label", 0x10), ("length", 0x4), ("negative", 0x1)])
def test_fused_malformed_input(cuda_device, bad, bit):
    batch = workloads.make_batch([80, 60], [12, 9], 1024, seed=1)
    if bad == "label":
        batch.targets = batch.targets.clone()
        batch.targets[1] = 1024
    elif bad == "length":
        batch.lengths = torch.tensor([81, 60], dtype=torch.int32)
    else:
        batch.target_lengths = torch.tensor([-1, 9], dtype=torch.int32)
        batch.targets = batch.targets[12:]
    loss, grad, status = _same(batch)
    assert status & bit
    assert math.isnan(loss[0]) and math.isfinite(loss[1])
    assert torch.all(grad[:80] == 0)


def test_fused_deterministic(cuda_device):
    batch = workloads.select_utterances(workloads.workload("largevocab", device=cuda_device), list(range(12)))
    l1, g1, _, _ = run_gpu_fused(batch)
    l2, g2, _, _ = run_gpu_fused(batch)
    assert np.array_equal(l1, l2)
    assert torch.equal(g1.view(torch.int16), g2.view(torch.int16))
