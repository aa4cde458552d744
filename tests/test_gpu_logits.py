"""GPU parity of the logits input form (CTC_PACKED_FLAG_LOGITS).

The forward takes each row's log_softmax itself (a dense log-sum-exp pass)
and the backward returns the gradient with respect to the logits.  Every
case compares with ``oracle.ctc_loss_packed_logits`` (fp64 log_softmax, then
the fp64 oracle) at the contract's tolerances: the three dtypes, both
gradient paths (one row per warp at a large vocabulary, several rows per
warp at a small one), the reductions with unalignable, empty and gapped
utterances, a NaN logit, and the autograd wrapper.
"""

import numpy as np
import pytest
import torch

import oracle
import packed_sequence_ctc_gb300 as pk
import workloads
from tests.helpers import assert_grad_close, assert_loss_close, run_gpu

pytestmark = pytest.mark.gpu


def _ref(batch, z, grad_loss=None):
    return oracle.ctc_loss_packed_logits(z, batch.cu_seqlens, batch.lengths, batch.targets, batch.target_lengths,
                                         batch.blank, batch.zero_infinity, batch.reduction, grad_loss=grad_loss)


def _defined_rows(batch, nll):
    rows = np.ones(batch.log_probs.shape[0], dtype=bool)
    cu, ln = batch.cu_seqlens.numpy(), batch.lengths.numpy()
    for b in range(batch.B):
        if not np.isfinite(nll[b]) and not batch.zero_infinity:
            rows[cu[b]:cu[b] + ln[b]] = False
    return rows


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_logits_match_the_oracle(cuda_device, dtype):
    batch = workloads.make_batch([130, 77, 301, 9, 64], [30, 12, 70, 3, 20], 37, dtype=dtype, seed=41,
                                 repeat_prob=0.2, redraw_infeasible=True, reduction="none")
    z = workloads.unnormalised_logits(batch, seed=5)
    gl = torch.tensor([0.5, 1.0, 2.0, -1.0, 0.25])
    loss, grad, status = run_gpu(batch, grad_loss=gl, log_probs=z.cuda(), logits=True)
    assert status == 0
    ref_loss, ref_grad, nll = _ref(batch, z, grad_loss=gl.numpy())
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype, rows=_defined_rows(batch, nll))


def test_large_vocabulary_rows(cuda_device):
    # D = 8193 bf16: rows are not 16-byte aligned; one row per gradient warp
    batch = workloads.make_batch([211, 180, 97], [40, 33, 20], 8193, dtype=torch.bfloat16, seed=8, sigma=3.0,
                                 label_high=8192, reduction="none")
    z = workloads.unnormalised_logits(batch, seed=6, offset=30.0)
    loss, grad, status = run_gpu(batch, log_probs=z.cuda(), logits=True)
    assert status == 0
    ref_loss, ref_grad, _ = _ref(batch, z)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.bfloat16)


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_small_vocabulary_reductions_and_degenerate_utterances(cuda_device, reduction):
    # D = 29: several rows per gradient warp; an empty utterance, an
    # unalignable one and a gap row
    batch = workloads.make_batch([60, 0, 45, 4, 33], [12, 2, 9, 6, 5], 29, dtype=torch.float16, seed=12,
                                 repeat_prob=0.3, reduction=reduction, zero_infinity=True, gaps=[0, 2, 0, 1, 3])
    z = workloads.unnormalised_logits(batch, seed=7)
    loss, grad, status = run_gpu(batch, log_probs=z.cuda(), logits=True)
    assert status == 0
    ref_loss, ref_grad, _ = _ref(batch, z)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float16)


def test_row_shift_of_the_logits(cuda_device):
    batch = workloads.make_batch([90, 70, 40], [20, 15, 8], 65, dtype=torch.float32, seed=3, reduction="sum")
    z = workloads.unnormalised_logits(batch, seed=1, offset=0.0)
    z2 = workloads.unnormalised_logits(batch, seed=2, offset=40.0)
    l1, g1, _ = run_gpu(batch, log_probs=z.cuda(), logits=True)
    l2, g2, _ = run_gpu(batch, log_probs=z2.cuda(), logits=True)
    assert_loss_close(l2, l1)
    assert torch.allclose(g1, g2, atol=2e-5, rtol=0)


def test_a_nan_logit_poisons_only_its_utterance(cuda_device):
    batch = workloads.make_batch([40, 50, 30], [8, 10, 6], 33, dtype=torch.float32, seed=4, reduction="none")
    z = workloads.unnormalised_logits(batch, seed=9)
    z[45, 7] = float("nan")  # a row of utterance 1
    loss, _, _ = run_gpu(batch, log_probs=z.cuda(), logits=True, need_grad=False)
    ref_loss, _, _ = _ref(batch, z)
    assert np.isnan(loss[1]) and np.isnan(ref_loss[1])
    assert_loss_close(loss[[0, 2]], ref_loss[[0, 2]])


def test_autograd_wrapper_with_logits(cuda_device):
    batch = workloads.make_batch([120, 96, 50], [25, 19, 11], 41, dtype=torch.bfloat16, seed=21, reduction="mean")
    z = workloads.unnormalised_logits(batch, seed=11).cuda().requires_grad_(True)
    loss = pk.packed_ctc_loss(z, batch.cu_seqlens.cuda(), batch.lengths.cuda(), batch.targets.cuda(),
                              batch.target_lengths.cuda(), blank=batch.blank, reduction="mean",
                              max_target_len=batch.max_target_len, logits=True)
    loss.backward()
    ref_loss, ref_grad, _ = _ref(batch, z.detach().cpu())
    assert_loss_close(loss.item(), ref_loss)
    assert_grad_close(z.grad, ref_grad, torch.bfloat16)
