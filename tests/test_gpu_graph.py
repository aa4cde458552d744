"""Forward + backward captured once in a CUDA graph and replayed with new
contents in the same buffers.  The calls never wait for the host and keep no
state outside the caller's workspace, so a replay must give exactly what eager
calls on the same inputs give (the kernels are deterministic)."""

import pytest
import torch

import packed_sequence_ctc_gb300 as pk
import workloads
from tests.helpers import assert_grad_close, assert_loss_close, to_device
from oracle import oracle_batch

LENGTHS, TARGETS = [300, 200, 57, 1], [40, 25, 9, 0]


def _batch(seed, dtype, reduction):
    return workloads.make_batch(LENGTHS, TARGETS, 1025, dtype=dtype, seed=seed, repeat_prob=0.2,
                                reduction=reduction, max_target_len=48, name=f"graph-{seed}")


def _eager(batch):
    d = to_device(batch)
    T_total, D = d["log_probs"].shape
    ws = pk.Workspace(T_total, batch.B, batch.max_target_len, D, d["log_probs"].dtype).tensor
    n = batch.B if batch.reduction == "none" else 1
    loss = torch.empty(n, device="cuda")
    grad = torch.empty_like(d["log_probs"])
    pk.ctc_packed_forward(d["log_probs"], d["cu"], d["lengths"], d["targets"], d["target_lengths"], batch.blank,
                          batch.zero_infinity, batch.reduction, loss, ws, batch.max_target_len)
    pk.ctc_packed_backward(d["log_probs"], d["cu"], d["lengths"], d["targets"], d["target_lengths"], batch.blank,
                           batch.zero_infinity, batch.reduction, torch.ones(n, device="cuda"), ws, grad,
                           batch.max_target_len)
    torch.cuda.synchronize()
    return loss, grad


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,reduction", [(torch.bfloat16, "mean"), (torch.float32, "none")])
def test_graph_replay_with_new_contents_matches_eager(cuda_device, dtype, reduction):
    first, second = _batch(1, dtype, reduction), _batch(2, dtype, reduction)
    s = to_device(first)  # the static buffers the graph is captured on
    T_total, D = s["log_probs"].shape
    ws = pk.Workspace(T_total, first.B, first.max_target_len, D, dtype).tensor
    n = first.B if reduction == "none" else 1
    loss = torch.empty(n, device="cuda")
    grad = torch.empty_like(s["log_probs"])
    g_up = torch.ones(n, device="cuda")

    def step():
        pk.ctc_packed_forward(s["log_probs"], s["cu"], s["lengths"], s["targets"], s["target_lengths"], first.blank,
                              False, reduction, loss, ws, first.max_target_len)
        pk.ctc_packed_backward(s["log_probs"], s["cu"], s["lengths"], s["targets"], s["target_lengths"],
                               first.blank, False, reduction, g_up, ws, grad, first.max_target_len)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager warm-up on the capture stream's side (launch attributes set up here)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()

    for batch in (first, second, first):
        d = to_device(batch)
        for k in ("log_probs", "targets"):
            s[k].copy_(d[k])
        g.replay()
        torch.cuda.synchronize()
        ref_loss, ref_grad = _eager(batch)
        assert torch.equal(loss, ref_loss)
        assert torch.equal(grad, ref_grad)
    # and the replay of the second batch against the fp64 oracle
    d = to_device(second)
    for k in ("log_probs", "targets"):
        s[k].copy_(d[k])
    g.replay()
    torch.cuda.synchronize()
    o_loss, o_grad, _ = oracle_batch(second)
    out = loss.double().cpu().numpy()
    assert_loss_close(out if reduction == "none" else out[0], o_loss)
    assert_grad_close(grad, o_grad, dtype)
