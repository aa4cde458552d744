"""Parity of the CUDA path with the fp64 oracle, through the C-ABI.

Every named workload is checked element by element (loss and gradient),
the large-vocabulary workload (a 315M-element dense gradient) in the launch
configuration the benchmark times, eight utterances of the oracle at a time,
plus a property every row must satisfy.  Edge cases follow the page's test
file (test_ctc_loss.py of "feat(asr): native CTC loss kernel over
sequence-packed log probabilities").
"""

import math

import numpy as np
import pytest
import torch

import oracle
import packed_sequence_ctc_gb300 as pk
import workloads
from helpers import assert_grad_close, assert_loss_close, run_gpu

pytestmark = pytest.mark.gpu


def _ref(batch, grad_loss=None):
    loss, grad, nll = oracle.oracle_batch(batch, grad_loss=grad_loss)
    return loss, grad, nll


def _defined_rows(batch, nll):
    """Rows whose reference gradient is defined (no infinite loss unless zeroed)."""
    rows = np.zeros(batch.T_total, dtype=bool)
    for b in range(batch.B):
        s = int(batch.cu_seqlens[b])
        e = int(batch.cu_seqlens[b + 1])
        if batch.zero_infinity or np.isfinite(nll[b]):
            rows[s:e] = True
    # rows past cu_seqlens[B] belong to nobody: zero on both sides
    rows[int(batch.cu_seqlens[-1]):] = True
    return rows


@pytest.mark.parametrize("name", ["tiny", "conformer", "longform", "char"])
def test_workload_parity(cuda_device, name):
    batch = workloads.workload(name, device=cuda_device)
    loss, grad, status = run_gpu(batch)
    assert status == 0
    ref_loss, ref_grad, nll = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, batch.log_probs.dtype, rows=_defined_rows(batch, nll))


def test_largevocab_full_parity(cuda_device):
    # the benchmarked workload, in the launch configuration the bench times:
    # every loss and every gradient element of all 64 utterances against the
    # oracle, which runs eight utterances at a time to bound host memory
    batch = workloads.workload("largevocab", device=cuda_device)
    loss, grad, status = run_gpu(batch)
    assert status == 0
    for first in range(0, batch.B, 8):
        sample = list(range(first, min(first + 8, batch.B)))
        sub = workloads.select_utterances(batch, sample)
        ref_loss, ref_grad, _ = _ref(sub)
        assert_loss_close(loss[sample], ref_loss)
        s0, s1 = int(batch.cu_seqlens[sample[0]]), int(batch.cu_seqlens[sample[-1] + 1])
        assert int(sub.T_total) == s1 - s0  # tight layout: the utterances' rows are contiguous
        assert_grad_close(grad[s0:s1], ref_grad, batch.log_probs.dtype)
    # every row: the posteriors of a frame sum to one, so sum_c (exp(lp) - grad) = 1
    lp = batch.log_probs.to(cuda_device).double()
    row_p = (lp.exp() - grad.double()).sum(dim=1).cpu().numpy()
    assert np.all(np.abs(row_p - 1.0) < 1e-2), np.abs(row_p - 1.0).max()


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_page_small_case(cuda_device, reduction, dtype):
    # T=[8,5,2], U=[3,1,0], targets [[1,1,2],[2],[]], D=5 with the blank last
    batch = workloads.make_batch([8, 5, 2], [3, 1, 0], 5, targets=[[1, 1, 2], [2], []], blank=4, seed=7,
                                 sigma=1.0, dtype=dtype, reduction=reduction)
    g = torch.tensor([0.7, -1.3, 2.0]) if reduction == "none" else torch.tensor([1.7])
    loss, grad, status = run_gpu(batch, grad_loss=g)
    ref_loss, ref_grad, _ = _ref(batch, grad_loss=g.double().numpy())
    assert status == 0
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype)


def test_repeated_and_blank_id_labels(cuda_device):
    batch = workloads.make_batch([9, 9, 7], [4, 3, 3], 5, targets=[[1, 1, 2, 2], [4, 4, 1], [2, 4, 2]], blank=4,
                                 seed=3)
    loss, grad, status = run_gpu(batch)
    ref_loss, ref_grad, _ = _ref(batch)
    assert status == 0
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32)


def test_empty_targets(cuda_device):
    batch = workloads.make_batch([6, 3], [0, 0], 3, seed=5, blank=2)
    loss, grad, _ = run_gpu(batch)
    ref_loss, ref_grad, _ = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32)


@pytest.mark.parametrize("zero_infinity", [False, True])
def test_zero_length_utterance(cuda_device, zero_infinity):
    batch = workloads.make_batch([5, 0, 3], [2, 1, 1], 4, targets=[[1, 2], [1], [2]], blank=3, seed=11,
                                 zero_infinity=zero_infinity)
    loss, grad, _ = run_gpu(batch)
    assert loss[1] == (0.0 if zero_infinity else math.inf)
    ref_loss, ref_grad, _ = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32)
    batch = workloads.make_batch([5, 0, 3], [2, 0, 1], 4, targets=[[1, 2], [], [2]], blank=3, seed=11,
                                 zero_infinity=zero_infinity)
    loss, _, _ = run_gpu(batch)
    assert loss[1] == 0.0


@pytest.mark.parametrize("zero_infinity", [False, True])
def test_impossible_alignment(cuda_device, zero_infinity):
    logits = torch.tensor([[1.0, 0.5, -0.5], [0.2, 0.1, 0.0]])
    batch = workloads.make_batch([1, 1], [2, 1], 3, targets=[[0, 0], [1]], blank=2, zero_infinity=zero_infinity)
    batch.log_probs = torch.log_softmax(logits, -1)
    loss, grad, _ = run_gpu(batch)
    if zero_infinity:
        assert loss[0] == 0.0
        assert torch.all(grad[0] == 0)
        assert grad[1].abs().sum() > 0
    else:
        assert math.isinf(loss[0]) and loss[0] > 0
        assert math.isfinite(loss[1])
    ref_loss, _, _ = _ref(batch)
    assert_loss_close(loss, ref_loss)


def test_over_allocated_targets_and_filler_utterances(cuda_device):
    # results must not depend on max_target_len nor on zero-length fillers
    tight = workloads.make_batch([9, 7, 4], [4, 3, 2], 6, seed=17, blank=5, label_low=0, label_high=4)
    l1, g1, _ = run_gpu(tight)
    l2, g2, _ = run_gpu(tight, max_target_len=32)
    assert np.array_equal(l1, l2)
    assert torch.equal(g1, g2)
    wide = workloads.make_batch([9, 7, 4, 0, 0], [4, 3, 2, 0, 0], 6, seed=17, blank=5, label_low=0, label_high=4)
    wide.log_probs = tight.log_probs
    wide.targets = tight.targets
    l3, g3, _ = run_gpu(wide, max_target_len=32)
    assert np.array_equal(l3[:3], l1) and np.all(l3[3:] == 0.0)
    assert torch.equal(g3, g1)


def test_gapped_rows_and_trailing_rows(cuda_device):
    # utterance spans longer than their lengths, and rows after cu_seqlens[B]
    batch = workloads.make_batch([7, 5, 6], [3, 2, 2], 9, seed=21, gaps=[2, 0, 3])
    extra = torch.log_softmax(torch.randn(5, 9), -1)
    batch.log_probs = torch.cat([batch.log_probs, extra])
    loss, grad, _ = run_gpu(batch)
    ref_loss, ref_grad, _ = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32)
    assert torch.all(grad[7:9] == 0) and torch.all(grad[-5 - 3:] == 0)


@pytest.mark.parametrize("D", [1, 2, 3, 29, 31, 1025])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_odd_class_counts(cuda_device, D, dtype):
    U = 0 if D == 1 else 5
    batch = workloads.make_batch([13, 1, 40, 7], [min(U, 4), 0, U, 2 if D > 1 else 0], D, seed=D, dtype=dtype,
                                 label_low=1 if D > 1 else 0, label_high=D - 1, reduction="sum")
    loss, grad, _ = run_gpu(batch)
    ref_loss, ref_grad, nll = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype, rows=_defined_rows(batch, nll))


# a chain warp owns 24 state pairs (8 of its 32 lanes shadow the neighbour):
# targets of 23/24 labels switch from one warp to several, 47/48 from 2 to 3,
# 71/72 from 3 to 4
@pytest.mark.parametrize("U", [22, 23, 24, 25, 26, 27, 28, 29, 30, 31, 32, 33, 46, 47, 48, 49, 55, 56, 57, 63, 64, 65,
                               71, 72, 84, 200, 511, 767, 768, 1000])
def test_state_counts_across_warp_boundaries(cuda_device, U):
    T = 2 * U + 37
    batch = workloads.make_batch([T, T // 2 + 3, 11], [U, min(U, T // 4), 3], 40, seed=U, repeat_prob=0.2,
                                 redraw_infeasible=True, reduction="mean")
    loss, grad, status = run_gpu(batch)
    assert status == 0
    ref_loss, ref_grad, nll = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32, rows=_defined_rows(batch, nll))


def test_two_pairs_per_thread(cuda_device):
    # a target bound above 767 puts two state pairs in each lane
    batch = workloads.make_batch([2600, 300, 50], [1200, 60, 10], 48, seed=5, reduction="sum")
    loss, grad, status = run_gpu(batch, max_target_len=1500)
    assert status == 0
    ref_loss, ref_grad, _ = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32)


def test_four_pairs_per_thread(cuda_device):
    # a target bound above 1919 puts four state pairs in each lane; the
    # targets span several warps (124 pairs each) and some stay in one
    batch = workloads.make_batch([700, 420, 90, 5], [300, 130, 40, 2], 37, seed=9, repeat_prob=0.2,
                                 reduction="none")
    loss, grad, status = run_gpu(batch, max_target_len=2100)
    assert status == 0
    ref_loss, ref_grad, nll = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32, rows=_defined_rows(batch, nll))


@pytest.mark.parametrize("offset", [2, 4, 8])
def test_gradient_buffer_not_congruent_with_log_probs(cuda_device, offset):
    batch = workloads.make_batch([40, 33, 17], [6, 5, 2], 29, seed=9, dtype=torch.bfloat16)
    loss, grad, _ = run_gpu(batch, grad_offset_bytes=offset)
    ref_loss, ref_grad, _ = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.bfloat16)


def test_deterministic(cuda_device):
    batch = workloads.make_batch([300, 280, 90], [60, 70, 20], 50, seed=4, repeat_prob=0.3,
                                 redraw_infeasible=True, label_high=6)
    l1, g1, _ = run_gpu(batch)
    l2, g2, _ = run_gpu(batch)
    assert np.array_equal(l1, l2)
    assert torch.equal(g1, g2)


def test_loss_only_forward(cuda_device):
    batch = workloads.workload("tiny")
    loss, _, status = run_gpu(batch, need_grad=False)
    ref_loss, _, _ = _ref(batch)
    assert status == 0
    assert_loss_close(loss, ref_loss)


def test_empty_batch(cuda_device):
    batch = workloads.make_batch([], [], 7, reduction="sum")
    batch.log_probs = torch.log_softmax(torch.randn(4, 7), -1)  # rows that belong to nobody
    loss, grad, status = run_gpu(batch, grad_loss=torch.tensor([1.0]))
    assert loss == 0.0 and status == 0
    assert torch.all(grad == 0)
    batch.reduction = "mean"
    loss, _, _ = run_gpu(batch, grad_loss=torch.tensor([1.0]))
    assert math.isnan(loss)


@pytest.mark.parametrize("bad,bit", [("negative", 0x1), ("too_long", 0x2), ("label", 0x10), ("length", 0x4)])
def test_device_status_on_malformed_input(cuda_device, bad, bit):
    batch = workloads.make_batch([8, 6], [3, 2], 5, seed=1)
    if bad == "negative":
        batch.target_lengths = torch.tensor([-1, 2], dtype=torch.int32)
        batch.targets = batch.targets[3:]
    elif bad == "too_long":
        batch.max_target_len = 2
    elif bad == "label":
        batch.targets = batch.targets.clone()
        batch.targets[1] = 5
    else:
        batch.lengths = torch.tensor([9, 6], dtype=torch.int32)
    loss, grad, status = run_gpu(batch)
    assert status & bit
    assert math.isnan(loss[0])
    assert math.isfinite(loss[1])
    assert torch.all(grad[:8] == 0)


def test_functional_autograd_matches_oracle(cuda_device):
    batch = workloads.workload("tiny")
    lp = batch.log_probs.to(cuda_device).requires_grad_()
    loss = pk.packed_ctc_loss(lp, batch.cu_seqlens.cuda(), batch.lengths.cuda(), batch.targets.cuda(),
                              batch.target_lengths.cuda(), blank=0, reduction="sum")
    loss.backward()
    batch.reduction = "sum"
    ref_loss, ref_grad, _ = _ref(batch)
    assert_loss_close(loss.item(), ref_loss)
    assert_grad_close(lp.grad, ref_grad, torch.float32)


def test_functional_raises_on_negative_target_length(cuda_device):
    batch = workloads.make_batch([8, 6], [3, 2], 5, seed=1)
    with pytest.raises(ValueError, match="negative"):
        pk.packed_ctc_loss(batch.log_probs.cuda(), batch.cu_seqlens.cuda(), batch.lengths.cuda(),
                           batch.targets.cuda(), torch.tensor([-1, 2], device="cuda"), blank=0, max_target_len=3)
    with pytest.raises(ValueError, match="width"):
        pk.packed_ctc_loss(batch.log_probs.cuda(), batch.cu_seqlens.cuda(), batch.lengths.cuda(),
                           batch.targets.cuda(), batch.target_lengths.cuda(), blank=0, max_target_len=2)
    with pytest.raises(TypeError, match="float64"):  # float64 has a path of its own; integers have none
        pk.packed_ctc_loss(batch.log_probs.to(torch.int32).cuda(), batch.cu_seqlens.cuda(), batch.lengths.cuda(),
                           batch.targets.cuda(), batch.target_lengths.cuda(), blank=0)


def test_maximum_target_length(cuda_device):
    # the longest target the library takes (3839 labels: four state pairs per
    # lane, 31 warps), with a short one beside it
    U = 3839
    batch = workloads.make_batch([U + 240, 30], [U, 6], 64, dtype=torch.float32, seed=31, label_low=1,
                                 label_high=63, redraw_infeasible=True, reduction="none")
    assert batch.max_target_len == U
    loss, grad, status = run_gpu(batch)
    assert status == 0
    ref_loss, ref_grad, nll = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32, rows=_defined_rows(batch, nll))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sixteen_k_vocabulary(cuda_device, dtype):
    # D = 16384: a row of 64 KB (fp32), 33 batches of the row stream
    batch = workloads.make_batch([45, 30, 12], [9, 6, 3], 16384, dtype=dtype, seed=32, label_high=16383,
                                 reduction="mean", gaps=[0, 2, 1])
    loss, grad, status = run_gpu(batch)
    assert status == 0
    ref_loss, ref_grad, _ = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype)


@pytest.mark.parametrize("dtype,stream,offset", [(torch.float32, None, 0), (torch.bfloat16, None, 0),
                                                 (torch.bfloat16, "0", 0), (torch.bfloat16, "0", 2),
                                                 (torch.float32, None, 4)])
def test_vocabulary_wider_than_shared_memory(cuda_device, monkeypatch, dtype, stream, offset):
    # D = 32769, an odd width: an fp32 row (128 KB) is wider than two stream
    # slots and is walked in batches by the row-group stream; a bf16 row fits
    # one team of the bulk-copy stream (stream=None) or takes the row-group
    # stream (stream="0"), with the gradient congruent to the input or not
    if stream is not None:
        monkeypatch.setenv("CTC_PACKED_STREAM", stream)
    D = 32769
    batch = workloads.make_batch([40, 23, 9], [8, 5, 0], D, dtype=dtype, seed=33, label_high=D - 1,
                                 reduction="sum", gaps=[1, 0, 2])
    loss, grad, status = run_gpu(batch, grad_offset_bytes=offset)
    assert status == 0
    ref_loss, ref_grad, _ = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_vocabulary_at_the_limit(cuda_device, dtype):
    # D = 2^20, the widest row the library takes (4 MB in fp32): the row is
    # streamed in 2 KB batches, the class sums bucketed by batch
    D = 1 << 20
    batch = workloads.make_batch([9, 6], [3, 2], D, dtype=dtype, seed=34, label_high=D - 1, reduction="mean",
                                 gaps=[1, 0])
    loss, grad, status = run_gpu(batch)
    assert status == 0
    ref_loss, ref_grad, _ = _ref(batch)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype)
