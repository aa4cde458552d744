"""The checkpoint policy of the state rows (CTC_PACKED_CKPT=K): the chains
keep only the rows whose index is a multiple of K and the backward
recomputes the others.  Page "feat(asr): native CTC loss kernel over
sequence-packed log probabilities", ctc_loss.py ``_PackedCTCLoss``: the
forward keeps the states the backward needs; keeping fewer and recomputing
is the other choice, measured slower here and so not the default.  The
results must still match the fp64 oracle at the contract's tolerances."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_grad_close, assert_loss_close, run_gpu

pytestmark = pytest.mark.gpu


def _defined_rows(batch, nll):
    rows = np.zeros(batch.T_total, dtype=bool)
    for b in range(batch.B):
        s, e = int(batch.cu_seqlens[b]), int(batch.cu_seqlens[b + 1])
        if batch.zero_infinity or np.isfinite(nll[b]):
            rows[s:e] = True
    rows[int(batch.cu_seqlens[-1]):] = True
    return rows


@pytest.mark.parametrize("K", [4, 8, 16])
@pytest.mark.parametrize("name", ["tiny", "conformer"])
def test_checkpointed_rows_match_the_oracle(cuda_device, monkeypatch, K, name):
    monkeypatch.setenv("CTC_PACKED_CKPT", str(K))
    batch = workloads.workload(name, device=cuda_device)
    loss, grad, status = run_gpu(batch)
    assert status == 0
    ref_loss, ref_grad, nll = oracle.oracle_batch(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, batch.log_probs.dtype, rows=_defined_rows(batch, nll))


@pytest.mark.parametrize("zero_infinity", [False, True])
def test_checkpointed_edge_cases(cuda_device, monkeypatch, zero_infinity):
    # spans shorter and longer than K, gaps, an empty target, an unalignable
    # utterance, repeats and a blank-id label
    monkeypatch.setenv("CTC_PACKED_CKPT", "8")
    batch = workloads.make_batch([3, 17, 0, 40, 9, 6], [1, 5, 0, 12, 0, 5], 11, seed=13, blank=4,
                                 targets=[[2], [1, 1, 3, 4, 4], [], [0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 1], [], [7, 7, 7, 7, 7]],
                                 gaps=[2, 0, 3, 1, 0, 4], zero_infinity=zero_infinity, reduction="mean")
    loss, grad, _ = run_gpu(batch)
    ref_loss, ref_grad, nll = oracle.oracle_batch(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32, rows=_defined_rows(batch, nll))


def test_checkpointed_large_vocabulary_sample(cuda_device, monkeypatch):
    monkeypatch.setenv("CTC_PACKED_CKPT", "8")
    batch = workloads.select_utterances(workloads.workload("largevocab", device=cuda_device), [0, 7, 33])
    loss, grad, status = run_gpu(batch)
    assert status == 0
    ref_loss, ref_grad, _ = oracle.oracle_batch(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, batch.log_probs.dtype)
