"""GPU parity of the mean_batch and mean_volume reductions against the oracle.

mean_batch is the batch mean of the per-utterance losses and mean_volume
their sum over the sum of the target lengths (after zero_infinity); their
gradients scale every covered row by g / B and g / sum(U).  The batch holds
an unalignable utterance and one without frames, with and without
zero_infinity, in float32 and bfloat16, and one case from logits.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.helpers import assert_grad_close, assert_loss_close, run_gpu

pytestmark = pytest.mark.gpu


def _rows(batch, nll):
    rows = np.ones(batch.log_probs.shape[0], dtype=bool)
    cu, ln = batch.cu_seqlens.numpy(), batch.lengths.numpy()
    for b in range(batch.B):
        if not np.isfinite(nll[b]) and not batch.zero_infinity:
            rows[cu[b]:cu[b] + ln[b]] = False
    return rows


@pytest.mark.parametrize("reduction", ["mean_batch", "mean_volume"])
@pytest.mark.parametrize("zero_infinity", [True, False])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_reduction_matches_the_oracle(cuda_device, reduction, zero_infinity, dtype):
    # utterance 2 cannot align (4 frames, 6 labels); utterance 3 has no frames
    batch = workloads.make_batch([150, 88, 4, 0, 61], [30, 17, 6, 3, 12], 41, dtype=dtype, seed=13,
                                 repeat_prob=0.2, reduction=reduction, zero_infinity=zero_infinity)
    g = torch.tensor([1.7])
    loss, grad, status = run_gpu(batch, grad_loss=g)
    assert status == 0
    ref_loss, ref_grad, nll = oracle.oracle_batch(batch, grad_loss=g.numpy())
    assert_loss_close(loss, ref_loss)
    if zero_infinity:
        assert_grad_close(grad, ref_grad, dtype, rows=_rows(batch, nll))
    else:
        assert np.isinf(loss) and np.isinf(ref_loss)


def test_mean_volume_from_logits(cuda_device):
    batch = workloads.make_batch([120, 77, 40], [25, 14, 9], 65, dtype=torch.float32, seed=31,
                                 reduction="mean_volume")
    z = workloads.unnormalised_logits(batch, seed=3)
    loss, grad, status = run_gpu(batch, grad_loss=torch.tensor([0.6]), log_probs=z.cuda(), logits=True)
    assert status == 0
    ref_loss, ref_grad, _ = oracle.ctc_loss_packed_logits(z, batch.cu_seqlens, batch.lengths, batch.targets,
                                                          batch.target_lengths, batch.blank, False, "mean_volume",
                                                          grad_loss=np.array([0.6]))
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32)
