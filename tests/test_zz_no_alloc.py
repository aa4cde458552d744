"""The loss-only forward that allocates nothing (``ctc_packed_forward_noalloc``).

It serves callers that cannot allocate device memory where they need a loss:
a C host without a device allocator, a process whose memory is held by
another framework's pool, or a scoring loop that must not stall. Its scratch
is one fixed array per device inside the library. So these tests check three
things:
* it gives the losses of the ordinary forward (with a caller-supplied
  workspace) within the loss tolerance, on two calls in a row on one stream
  with different batches, which shows that one call leaves nothing behind
  that changes the next, and the fp64 oracle's losses;
* a batch that nearly fills the array (its loss-only workspace size) still
  runs;
* batches too large for the array are refused before any CUDA call.

The file name puts these tests after all others. They must pass both there
and alone in a fresh process, where the first call also sets up the scratch
address.
"""

import os
import re

import numpy as np
import pytest
import torch

import oracle
import packed_sequence_ctc_gb300 as pk
import workloads
from tests.helpers import assert_loss_close, to_device

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ERR_INVALID, ERR_WORKSPACE, ERR_UNSUPPORTED = 1, 2, 4


@pytest.fixture(scope="module")
def lib():
    from packed_sequence_ctc_gb300 import build as b

    return pk.load_library(b.build())


def _noalloc_raw(lib, T_total, B, mtl, D, dtype=0):
    """Call the entry point with null data pointers: only sizes that the host
    refuses before any CUDA call may be passed here."""
    return lib.ctc_packed_forward_noalloc(None, dtype, T_total, D, None, None, None, None, B, mtl, 0, 0, 0, None,
                                          None)


def test_scratch_size_matches_the_header():
    text = open(os.path.join(ROOT, "include", "ctc_packed.h")).read()
    m = re.search(r"#define CTC_PACKED_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m, "scratch size macro not found"
    assert int(m.group(1)) << int(m.group(2)) == pk.NOALLOC_SCRATCH_BYTES


def test_oversized_batches_are_refused_before_any_cuda_call(lib):
    cap = pk.NOALLOC_SCRATCH_BYTES
    # far beyond the scratch
    assert lib.ctc_packed_workspace_size_loss_only(100_000, 8, 200, 1025, 0) > cap
    assert _noalloc_raw(lib, 100_000, 8, 200, 1025) == ERR_WORKSPACE
    # the smallest frame count that no longer fits is refused too
    T = _largest_fitting_frames(lib, 8, 100, 1025)
    assert lib.ctc_packed_workspace_size_loss_only(T + 1, 8, 100, 1025, 0) > cap
    assert _noalloc_raw(lib, T + 1, 8, 100, 1025) == ERR_WORKSPACE
    # the limit is the loss-only workspace: the full one would be refused
    assert lib.ctc_packed_workspace_size(T, 8, 100, 1025, 0) > cap
    assert pk.ctc_packed_status_string(ERR_WORKSPACE).startswith("workspace")
    # invalid and unsupported sizes keep the ordinary forward's codes
    assert _noalloc_raw(lib, -1, 1, 1, 5) == ERR_INVALID
    assert _noalloc_raw(lib, 10, 1, 1, 0) == ERR_INVALID
    assert _noalloc_raw(lib, 10, 1, 1, (1 << 20) + 1) == ERR_UNSUPPORTED
    assert _noalloc_raw(lib, 10, 1, 1, 5, dtype=7) == ERR_INVALID


def _largest_fitting_frames(lib, B, mtl, D):
    lo, hi = 0, 1 << 24
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if lib.ctc_packed_workspace_size_loss_only(mid, B, mtl, D, 0) <= pk.NOALLOC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    return lo


def _losses(batch, noalloc: bool, stream=None):
    d = to_device(batch)
    T_total, D = d["log_probs"].shape
    red = batch.reduction
    loss = torch.full((batch.B if red == "none" else 1,), float("nan"), dtype=torch.float32, device="cuda")
    args = (d["log_probs"], d["cu"], d["lengths"], d["targets"], d["target_lengths"], batch.blank,
            batch.zero_infinity, red, loss)
    if noalloc:
        pk.ctc_packed_forward_noalloc(*args, batch.max_target_len, stream=stream)
    else:
        ws = pk.Workspace(T_total, batch.B, batch.max_target_len, D, d["log_probs"].dtype).tensor
        pk.ctc_packed_forward(*args, ws, batch.max_target_len, stream=stream)
    return loss, d  # d keeps the inputs alive until the caller synchronises


def _second_batch():
    # conformer-like shapes, an empty utterance and an unalignable one
    return workloads.make_batch([300, 257, 410, 0, 123, 40], [60, 40, 90, 2, 30, 39], 1025,
                                dtype=torch.bfloat16, seed=11, repeat_prob=0.3, reduction="none",
                                redraw_infeasible=False, name="noalloc-second")


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_forward(cuda_device, lib):
    first = workloads.workload("tiny")
    second = _second_batch()
    assert lib.ctc_packed_workspace_size_loss_only(second.log_probs.shape[0], second.B, second.max_target_len, 1025,
                                                   1) <= pk.NOALLOC_SCRATCH_BYTES
    # both calls go onto the same stream back to back, without a host wait
    a, keep_a = _losses(first, noalloc=True)
    b, keep_b = _losses(second, noalloc=True)
    torch.cuda.synchronize()
    ra, _ = _losses(first, noalloc=False)
    rb, _ = _losses(second, noalloc=False)
    torch.cuda.synchronize()
    assert_loss_close(a.double().cpu().numpy(), ra.double().cpu().numpy())
    assert_loss_close(b.double().cpu().numpy(), rb.double().cpu().numpy())
    # the unalignable utterance keeps its +inf
    assert np.isinf(b[-1].item()) and np.isinf(rb[-1].item())
    # and both calls give the fp64 oracle's losses
    ref_a, _, _ = oracle.oracle_batch(first, need_grad=False)
    ref_b, _, _ = oracle.oracle_batch(second, need_grad=False)
    assert_loss_close(a.double().cpu().numpy(), ref_a)
    assert_loss_close(b.double().cpu().numpy(), ref_b)


@pytest.mark.gpu
@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_reductions_match_on_a_second_stream(cuda_device, lib, reduction):
    batch = workloads.make_batch([500, 333, 64], [80, 51, 10], 257, seed=5, reduction=reduction,
                                 zero_infinity=True, name="noalloc-reduced")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a, keep = _losses(batch, noalloc=True, stream=s)
        b, keep2 = _losses(batch, noalloc=True, stream=s)
    s.synchronize()
    ref, _ = _losses(batch, noalloc=False)
    torch.cuda.synchronize()
    assert_loss_close(a.double().cpu().numpy(), ref.double().cpu().numpy())
    assert_loss_close(b.double().cpu().numpy(), ref.double().cpu().numpy())


@pytest.mark.gpu
def test_batch_that_nearly_fills_the_scratch(cuda_device, lib):
    B, mtl, D = 8, 100, 65
    T = _largest_fitting_frames(lib, B, mtl, D)
    assert lib.ctc_packed_workspace_size_loss_only(T, B, mtl, D, 0) > pk.NOALLOC_SCRATCH_BYTES // 2
    per = T // B
    batch = workloads.make_batch([per] * B, [mtl] * (B - 1) + [7], D, seed=3, reduction="none",
                                 max_target_len=mtl, name="noalloc-full")
    assert batch.log_probs.shape[0] <= T
    a, keep = _losses(batch, noalloc=True)
    ref, _ = _losses(batch, noalloc=False)
    torch.cuda.synchronize()
    assert_loss_close(a.double().cpu().numpy(), ref.double().cpu().numpy())
