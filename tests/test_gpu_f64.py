"""GPU parity of the float64 path (ctc_packed_forward_f64 / ctc_packed_backward_f64).

Page "feat(asr): native CTC loss kernel over sequence-packed log
probabilities", test_ctc_loss.py ``test_float64_takes_padded_path``: float64
input is served at float64 precision and compared at atol = rtol = 1e-10.
Every case here compares the loss and every gradient element with the fp64
oracle at that bound, |gpu - oracle| <= 1e-10 + 1e-10 |oracle|: mixed
batches, every reduction with unalignable, empty and gapped utterances,
repeated and blank-valued labels, logits input, the widest rows, every
states-per-thread shape of the recursion CTAs, malformed input, a loss-only
forward followed by a backward, determinism and the autograd wrapper.
"""

import numpy as np
import pytest
import torch

import oracle
import packed_sequence_ctc_gb300 as pk
import workloads
from tests.helpers import to_device

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-10


def _close(gpu, ref, atol=ATOL, rtol=RTOL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    same_inf = np.isinf(gpu) & np.isinf(ref) & (np.sign(gpu) == np.sign(ref))
    both_nan = np.isnan(gpu) & np.isnan(ref)
    with np.errstate(invalid="ignore"):
        ok = same_inf | both_nan | (np.abs(gpu - ref) <= atol + rtol * np.abs(ref))
    return ok


def assert_close64(gpu, ref, what, atol=ATOL, rtol=RTOL, rows=None):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rows is not None:
        gpu, ref = gpu[rows], ref[rows]
    ok = _close(gpu, ref, atol, rtol)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} entries beyond {atol} + {rtol}|ref|; first {bad.tolist()}: "
                             f"gpu {gpu[~ok][:5]} ref {ref[~ok][:5]}")


def run_f64(batch, grad_loss=None, logits=False, log_probs=None, need_grad=True, ws=None):
    d = to_device(batch)
    lp = d["log_probs"] if log_probs is None else log_probs
    assert lp.dtype == torch.float64
    T_total, D = lp.shape
    B = batch.B
    mtl = batch.max_target_len
    ws = pk.Workspace(T_total, B, mtl, D, torch.float64).tensor if ws is None else ws
    red = batch.reduction
    loss = torch.full((B if red == "none" else 1,), float("nan"), dtype=torch.float64, device="cuda")
    flags = (0 if need_grad else pk.FLAG_LOSS_ONLY) | (pk.FLAG_LOGITS if logits else 0)
    pk.ctc_packed_forward(lp, d["cu"], d["lengths"], d["targets"], d["target_lengths"], batch.blank,
                          batch.zero_infinity, red, loss, ws, mtl, flags=flags)
    grad = None
    if need_grad:
        if grad_loss is None:
            grad_loss = torch.ones(B if red == "none" else 1, dtype=torch.float64)
        g_up = torch.as_tensor(grad_loss, dtype=torch.float64).reshape(-1).cuda()
        grad = torch.full_like(lp, float("nan"))
        pk.ctc_packed_backward(lp, d["cu"], d["lengths"], d["targets"], d["target_lengths"], batch.blank,
                               batch.zero_infinity, red, g_up, ws, grad, mtl)
    torch.cuda.synchronize()
    status = pk.ctc_packed_read_status(ws)
    out = loss.cpu().numpy()
    return (out if red == "none" else out[0]), (None if grad is None else grad.cpu().numpy()), status


def _ref(batch, grad_loss=None):
    return oracle.oracle_batch(batch, grad_loss=grad_loss)


def _defined_rows(batch, nll):
    rows = np.ones(batch.T_total, dtype=bool)
    cu, ln = batch.cu_seqlens.numpy(), batch.lengths.numpy()
    for b in range(batch.B):
        if not np.isfinite(nll[b]) and not batch.zero_infinity:
            rows[cu[b]:cu[b] + ln[b]] = False
    return rows


def test_mixed_batch(cuda_device):
    batch = workloads.make_batch([130, 77, 301, 9, 64, 1], [30, 12, 70, 3, 20, 1], 37, dtype=torch.float64,
                                 seed=51, repeat_prob=0.2, redraw_infeasible=True, gaps=[0, 3, 1, 0, 2, 0],
                                 reduction="none")
    gl = np.array([0.5, 1.0, 2.0, -1.0, 0.25, 3.0])
    loss, grad, status = run_f64(batch, grad_loss=gl)
    assert status == 0
    ref_loss, ref_grad, _ = _ref(batch, grad_loss=gl)
    assert_close64(loss, ref_loss, "loss")
    assert_close64(grad, ref_grad, "grad")


@pytest.mark.parametrize("reduction", ["sum", "mean", "mean_batch", "mean_volume"])
@pytest.mark.parametrize("zero_infinity", [False, True])
def test_reductions_with_degenerate_utterances(cuda_device, reduction, zero_infinity):
    # an unalignable utterance (6 frames, 5 labels with 2 repeats), an empty
    # target, an utterance without frames, gaps, a blank of 3 and a label
    # equal to the blank
    batch = workloads.make_batch([40, 6, 25, 0, 33], [9, 5, 0, 2, 7], 11, dtype=torch.float64, seed=52, blank=3,
                                 targets=[[1, 2, 2, 4, 5, 6, 3, 8, 9], [1, 1, 2, 2, 4], [], [5, 6],
                                          [7, 3, 7, 7, 10, 3, 2]],
                                 gaps=[2, 0, 1, 3, 0], zero_infinity=zero_infinity, reduction=reduction)
    loss, grad, status = run_f64(batch, grad_loss=[1.7])
    assert status == 0
    ref_loss, ref_grad, nll = _ref(batch, grad_loss=[1.7])
    assert_close64(loss, ref_loss, "loss")
    assert_close64(grad, ref_grad, "grad", rows=_defined_rows(batch, nll))


def test_logits_input(cuda_device):
    batch = workloads.make_batch([130, 77, 64], [30, 12, 20], 37, dtype=torch.float64, seed=53, repeat_prob=0.2,
                                 redraw_infeasible=True, reduction="mean")
    z = workloads.unnormalised_logits(batch, seed=9).to(torch.float64)
    loss, grad, status = run_f64(batch, logits=True, log_probs=z.cuda())
    assert status == 0
    ref_loss, ref_grad, _ = oracle.ctc_loss_packed_logits(z, batch.cu_seqlens, batch.lengths, batch.targets,
                                                          batch.target_lengths, batch.blank, batch.zero_infinity,
                                                          batch.reduction)
    assert_close64(loss, ref_loss, "loss")
    assert_close64(grad, ref_grad, "grad")


@pytest.mark.parametrize("D", [8193, 32769])
def test_wide_rows(cuda_device, D):
    batch = workloads.make_batch([90, 61, 17], [20, 13, 4], D, dtype=torch.float64, seed=54, sigma=3.0,
                                 reduction="sum", gaps=[1, 0, 2])
    loss, grad, status = run_f64(batch)
    assert status == 0
    ref_loss, ref_grad, _ = _ref(batch)
    assert_close64(loss, ref_loss, "loss")
    assert_close64(grad, ref_grad, "grad")


@pytest.mark.parametrize("U", [600, 1500, 2500])
def test_long_targets(cuda_device, U):
    # 1201, 3001 and 5001 states: one, four and eight states per thread of the
    # recursion CTAs.  The oracle's own log-space rounding grows with the
    # frames times |log alpha| (about T * |lp| * 2^-53 per step), so the bound
    # here is that estimate over the utterance, at least 1e-10.
    T = U + 200
    batch = workloads.make_batch([T, 50], [U, 10], 24, dtype=torch.float64, seed=55 + U, sigma=1.0,
                                 redraw_infeasible=True, reduction="none")
    loss, grad, status = run_f64(batch)
    assert status == 0
    ref_loss, ref_grad, nll = _ref(batch)
    tol = max(ATOL, float(np.nanmax(np.abs(nll))) * T * 2.0 ** -53)
    assert_close64(loss, ref_loss, "loss")
    assert_close64(grad, ref_grad, "grad", atol=tol)


def test_nan_log_probability(cuda_device):
    batch = workloads.make_batch([30, 20], [5, 4], 9, dtype=torch.float64, seed=56, reduction="none")
    lab = int(batch.targets[0])
    batch.log_probs[4, lab] = float("nan")
    loss, grad, status = run_f64(batch)
    assert status == 0
    assert np.isnan(loss[0])
    ref_loss, ref_grad, _ = _ref(batch)
    assert_close64(loss[1:], ref_loss[1:], "loss")
    assert_close64(grad[30:], ref_grad[30:], "grad of the clean utterance")


def test_positive_infinite_log_probability(cuda_device):
    # not a log probability: the utterance's loss is NaN, as with a NaN; the
    # other utterance is unaffected
    batch = workloads.make_batch([30, 20], [5, 4], 9, dtype=torch.float64, seed=58, reduction="none")
    batch.log_probs[7, batch.blank] = float("inf")
    loss, grad, status = run_f64(batch)
    assert status == 0
    assert np.isnan(loss[0])
    ref_loss, ref_grad, _ = _ref(batch)
    assert_close64(loss[1:], ref_loss[1:], "loss")
    assert_close64(grad[30:], ref_grad[30:], "grad of the clean utterance")


def test_label_out_of_range_sets_status(cuda_device):
    batch = workloads.make_batch([30, 20], [3, 2], 9, dtype=torch.float64, seed=57, reduction="none",
                                 targets=[[1, 9, 2], [3, 4]])
    loss, grad, status = run_f64(batch)
    assert status & 0x10
    assert np.isnan(loss[0])
    assert np.all(grad[:30] == 0.0)
    # the well-formed utterance keeps its own loss and rows (the oracle runs
    # on the same rows with an in-range label in the first target)
    clean = workloads.make_batch([30, 20], [3, 2], 9, dtype=torch.float64, seed=57, reduction="none",
                                 targets=[[1, 8, 2], [3, 4]])
    assert torch.equal(clean.log_probs, batch.log_probs)
    ref_loss, ref_grad, _ = _ref(clean)
    assert_close64(loss[1], ref_loss[1], "loss")
    assert_close64(grad[30:], ref_grad[30:], "grad")


def test_backward_after_loss_only_forward(cuda_device):
    batch = workloads.make_batch([30, 20], [5, 4], 9, dtype=torch.float64, seed=58, reduction="sum")
    d = to_device(batch)
    n_lo = pk.ctc_packed_workspace_size_loss_only(batch.T_total, batch.B, batch.max_target_len, 9, torch.float64)
    n = pk.ctc_packed_workspace_size(batch.T_total, batch.B, batch.max_target_len, 9, torch.float64)
    assert 0 < n_lo < n
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    loss, _, status = run_f64(batch, need_grad=False, ws=ws)
    assert status == 0
    ref_loss, _, _ = _ref(batch)
    assert_close64(loss, ref_loss, "loss")
    grad = torch.full_like(d["log_probs"], float("nan"))
    pk.ctc_packed_backward(d["log_probs"], d["cu"], d["lengths"], d["targets"], d["target_lengths"], batch.blank,
                           batch.zero_infinity, "sum", torch.ones(1, dtype=torch.float64, device="cuda"), ws, grad,
                           batch.max_target_len)
    assert pk.ctc_packed_read_status(ws) & 0x40
    assert bool((grad == 0).all())


def test_deterministic(cuda_device):
    batch = workloads.make_batch([230, 177, 301, 64], [50, 40, 70, 20], 129, dtype=torch.float64, seed=59,
                                 repeat_prob=0.3, redraw_infeasible=True, reduction="mean")
    l1, g1, _ = run_f64(batch)
    l2, g2, _ = run_f64(batch)
    assert np.array_equal(np.asarray(l1), np.asarray(l2))
    assert np.array_equal(g1, g2)


def test_autograd_wrapper(cuda_device):
    batch = workloads.make_batch([60, 45], [12, 9], 29, dtype=torch.float64, seed=60, reduction="mean_volume")
    lp = batch.log_probs.cuda().requires_grad_(True)
    loss = pk.packed_ctc_loss(lp, batch.cu_seqlens.cuda(), batch.lengths.cuda(), batch.targets.cuda(),
                              batch.target_lengths.cuda(), blank=batch.blank, reduction="mean_volume")
    assert loss.dtype == torch.float64
    loss.backward()
    ref_loss, ref_grad, _ = _ref(batch)
    assert_close64(loss.item(), ref_loss, "loss")
    assert_close64(lp.grad.cpu().numpy(), ref_grad, "grad")


@pytest.mark.parametrize("reduction,grad_loss", [("sum", 1.0), ("mean", -2.5)])
def test_unnormalised_rows_over_a_wide_range(cuda_device, reduction, grad_loss):
    # raw rows with values in [-720, 5]: the dense exp's table covers
    # |x| < 512 and hands the rest to the library exp, scaled like the table
    # (the upstream factor folded into it); every element is compared with
    # the oracle's
    batch = workloads.make_batch([40, 31], [6, 5], 257, dtype=torch.float64, seed=61, reduction=reduction)
    gen = torch.Generator().manual_seed(62)
    batch.log_probs = torch.rand(batch.log_probs.shape, generator=gen, dtype=torch.float64) * 725.0 - 720.0
    loss, grad, status = run_f64(batch, grad_loss=[grad_loss])
    assert status == 0
    ref_loss, ref_grad, _ = _ref(batch, grad_loss=[grad_loss])
    assert_close64(loss, ref_loss, "loss")
    assert_close64(grad, ref_grad, "grad")
