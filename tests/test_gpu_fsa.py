"""GPU parity of the generic FSA full-sum path (ctc_packed_fsa_forward /
ctc_packed_fsa_backward) against the float64 FSA oracle.

Cases: the CTC lattice written as an FSA (also checked against the CTC
path), seeded random FSAs with weights, several start and final states and
loops, in the three dtypes; a sequence without a path (with and without
zero_infinity), frameless sequences and gap rows; a large vocabulary; and
out-of-range FSA data (and more distinct labels than max_labels), which must
set the status word and a NaN loss; bitwise reproducibility; lattices
of 602 to 2502 states (two to eight states a thread); and sequences with
over a thousand distinct labels (more than two a label thread, with and
without label warps of their own).  The recursions carry
float32 mantissas with integer exponents: losses within 1e-4 relative,
float32 gradients within 2e-5 (on these lengths), half types within one
unit in the last place plus 1e-3.
"""

import numpy as np
import pytest
import torch

import packed_sequence_ctc_gb300 as pk
import workloads
from oracle import fsa_oracle
from tests.helpers import assert_grad_close, assert_loss_close, run_gpu

pytestmark = pytest.mark.gpu


def _run(lp, cu, lengths, fsa, max_states, zero_infinity=False, grad_loss=None, guard=64, max_labels=None):
    dev = "cuda"
    T_total, D = lp.shape
    B = lengths.numel()
    fsa_d = tuple(x.to(dev).contiguous() for x in fsa)
    cu_d, ln_d = cu.to(dev).to(torch.int32), lengths.to(dev).to(torch.int32)
    lp_d = lp.to(dev).contiguous()
    max_labels = _max_labels(fsa) if max_labels is None else max_labels
    n_states, n_edges = int(fsa[1].numel()), int(fsa[4].shape[0])
    ws = torch.empty(pk.ctc_packed_fsa_workspace_size(T_total, B, n_states, n_edges, max_states, max_labels, D),
                     dtype=torch.uint8, device=dev)
    loss = torch.full((B,), float("nan"), device=dev)
    pk.ctc_packed_fsa_forward(lp_d, cu_d, ln_d, fsa_d, max_states, max_labels, zero_infinity, loss, ws)
    g = torch.ones(B) if grad_loss is None else torch.as_tensor(grad_loss, dtype=torch.float32)
    n = T_total * D * lp.element_size()
    raw = torch.full((n + 2 * guard,), 0xA5, dtype=torch.uint8, device=dev)
    grad = raw[guard:guard + n].view(lp.dtype).view(T_total, D)
    pk.ctc_packed_fsa_backward(lp_d, cu_d, ln_d, fsa_d, max_states, max_labels, zero_infinity, g.to(dev), ws, grad)
    torch.cuda.synchronize()
    assert bool((raw[:guard] == 0xA5).all()) and bool((raw[guard + n:] == 0xA5).all()), "write outside the gradient"
    status = pk.ctc_packed_read_status(ws)
    return loss.double().cpu().numpy(), grad.clone(), status, g.numpy()


def _oracle(lp, cu, lengths, fsa, grad_loss, zero_infinity=False):
    so, sw, fw, eo, ed, ew = fsa
    return fsa_oracle.fsa_loss_packed(lp, cu, lengths, so, sw, fw, eo, ed, ew, grad_loss=grad_loss,
                                      zero_infinity=zero_infinity)


def _max_labels(fsa):
    eo, ed = fsa[3], fsa[4]
    return max(1, max(len(set(ed[eo[i]:eo[i + 1], 2].tolist())) for i in range(len(eo) - 1)))


def _max_states(fsa):
    so = fsa[0]
    return int((so[1:] - so[:-1]).max())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ctc_lattice_as_fsa(cuda_device, dtype):
    batch = workloads.make_batch([120, 90, 64, 30], [25, 20, 12, 5], 37, dtype=dtype, seed=17, repeat_prob=0.25,
                                 redraw_infeasible=True, reduction="none")
    offs = np.concatenate([[0], np.cumsum(batch.target_lengths.numpy())])
    tg = batch.targets.numpy()
    fsa = workloads.pack_fsas([workloads.ctc_lattice_fsa(tg[offs[b]:offs[b + 1]], batch.blank)
                               for b in range(batch.B)])
    loss, grad, status, g = _run(batch.log_probs, batch.cu_seqlens, batch.lengths, fsa, _max_states(fsa))
    assert status == 0
    ref_loss, ref_grad = _oracle(batch.log_probs, batch.cu_seqlens, batch.lengths, fsa, g)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype)
    # and the CTC path on the same batch
    ctc_loss, ctc_grad, _ = run_gpu(batch)
    assert_loss_close(loss, ctc_loss)
    assert_grad_close(grad, ctc_grad.double().cpu().numpy(), dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_random_fsas(cuda_device, dtype):
    lengths = [150, 77, 0, 33, 200]
    gaps = [0, 3, 0, 2, 0]
    D = 23
    cu = [0]
    for T, gp in zip(lengths, gaps):
        cu.append(cu[-1] + T + gp)
    gen = torch.Generator().manual_seed(5)
    lp = torch.log_softmax(torch.randn(cu[-1], D, generator=gen) * 2.0, -1).to(dtype)
    fsas = [workloads.random_fsa(S, E, D, seed=100 + i) for i, (S, E) in enumerate([(9, 30), (5, 12), (3, 5),
                                                                                  (40, 150), (17, 60)])]
    fsa = workloads.pack_fsas(fsas)
    cu_t = torch.tensor(cu, dtype=torch.int32)
    ln_t = torch.tensor(lengths, dtype=torch.int32)
    gl = [1.0, -0.5, 2.0, 0.7, 1.3]
    loss, grad, status, g = _run(lp, cu_t, ln_t, fsa, _max_states(fsa), grad_loss=gl)
    assert status == 0
    ref_loss, ref_grad = _oracle(lp, cu_t, ln_t, fsa, g)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype)  # gap rows: 0 on both sides


@pytest.mark.parametrize("zero_infinity", [True, False])
def test_sequence_without_a_path(cuda_device, zero_infinity):
    D = 7
    lp = torch.log_softmax(torch.randn(30, D, generator=torch.Generator().manual_seed(2)), -1)
    inf = float("-inf")
    dead = ([0.0, inf], [inf, 0.0], [(0, 0, 1)], [0.0])  # the final state is never reached
    live = workloads.random_fsa(6, 20, D, seed=9)
    fsa = workloads.pack_fsas([live, dead])
    cu = torch.tensor([0, 18, 30], dtype=torch.int32)
    ln = torch.tensor([18, 12], dtype=torch.int32)
    loss, grad, status, g = _run(lp, cu, ln, fsa, 6, zero_infinity=zero_infinity)
    assert status == 0
    ref_loss, ref_grad = _oracle(lp, cu, ln, fsa, g, zero_infinity=zero_infinity)
    assert_loss_close(loss, ref_loss)
    rows = slice(0, 30) if zero_infinity else slice(0, 18)
    assert_grad_close(grad[rows], ref_grad[rows], torch.float32)


def test_large_vocabulary_ctc_lattices(cuda_device):
    batch = workloads.make_batch([97, 64, 40], [20, 12, 9], 8193, dtype=torch.bfloat16, seed=23, sigma=3.0,
                                 label_high=8192, reduction="none")
    offs = np.concatenate([[0], np.cumsum(batch.target_lengths.numpy())])
    tg = batch.targets.numpy()
    fsa = workloads.pack_fsas([workloads.ctc_lattice_fsa(tg[offs[b]:offs[b + 1]], batch.blank)
                               for b in range(batch.B)])
    loss, grad, status, g = _run(batch.log_probs, batch.cu_seqlens, batch.lengths, fsa, _max_states(fsa))
    assert status == 0
    ref_loss, ref_grad = _oracle(batch.log_probs, batch.cu_seqlens, batch.lengths, fsa, g)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.bfloat16)


def test_out_of_range_fsa_data_sets_the_status(cuda_device):
    D = 5
    lp = torch.log_softmax(torch.randn(20, D, generator=torch.Generator().manual_seed(4)), -1)
    good = workloads.random_fsa(4, 10, D, seed=1)
    bad_state = ([0.0, float("-inf")], [float("-inf"), 0.0], [(0, 7, 1)], [0.0])  # state 7 of 2
    bad_label = ([0.0, float("-inf")], [float("-inf"), 0.0], [(0, 1, 9)], [0.0])  # class 9 of 5
    fsa = workloads.pack_fsas([good, bad_state, bad_label])
    cu = torch.tensor([0, 8, 14, 20], dtype=torch.int32)
    ln = torch.tensor([8, 6, 6], dtype=torch.int32)
    loss, _, status, _ = _run(lp, cu, ln, fsa, 4)
    assert status & 0x80 and status & 0x10
    assert np.isfinite(loss[0]) and np.isnan(loss[1]) and np.isnan(loss[2])


def test_many_edges_per_sequence_and_a_nan(cuda_device):
    # more edges than the threads keep in registers (4 x 256), and a NaN
    # label value in one sequence, which must make only its loss NaN
    D = 19
    lp = torch.log_softmax(torch.randn(130, D, generator=torch.Generator().manual_seed(8)), -1)
    big = workloads.random_fsa(60, 1500, D, seed=77)
    small = workloads.random_fsa(5, 14, D, seed=78)
    fsa = workloads.pack_fsas([big, small, small])
    cu = torch.tensor([0, 70, 100, 130], dtype=torch.int32)
    ln = torch.tensor([70, 30, 30], dtype=torch.int32)
    lp[110, :] = float("nan")  # a row of the third sequence
    loss, grad, status, g = _run(lp, cu, ln, fsa, 60)
    ref_loss, ref_grad = _oracle(lp, cu, ln, fsa, g)
    assert np.isnan(loss[2]) and np.isnan(ref_loss[2])
    assert_loss_close(loss[:2], ref_loss[:2])
    assert_grad_close(grad[:100], ref_grad[:100], torch.float32)


def test_more_labels_than_max_labels_rejects_the_sequence(cuda_device):
    D = 6
    lp = torch.log_softmax(torch.randn(24, D, generator=torch.Generator().manual_seed(5)), -1)
    two = ([0.0, float("-inf")], [float("-inf"), 0.0], [(0, 1, 1), (1, 1, 2), (0, 0, 2)], [0.0, 0.0, 0.0])
    three = ([0.0, float("-inf")], [float("-inf"), 0.0], [(0, 1, 1), (1, 1, 2), (0, 0, 3)], [0.0, 0.0, 0.0])
    fsa = workloads.pack_fsas([two, three])
    cu = torch.tensor([0, 12, 24], dtype=torch.int32)
    ln = torch.tensor([12, 12], dtype=torch.int32)
    loss, grad, status, g = _run(lp, cu, ln, fsa, 2, max_labels=2)
    assert status & 0x80
    assert np.isfinite(loss[0]) and np.isnan(loss[1])
    assert bool((grad[12:] == 0).all())
    ref_loss, ref_grad = _oracle(lp, cu, ln, fsa, g)
    assert_loss_close(loss[:1], ref_loss[:1])
    assert_grad_close(grad[:12], ref_grad[:12], torch.float32)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_deterministic(cuda_device, dtype):
    # every sum runs in a fixed order: two runs agree bit for bit
    D = 23
    lp = torch.log_softmax(torch.randn(420, D, generator=torch.Generator().manual_seed(11)), -1).to(dtype)
    fsa = workloads.pack_fsas([workloads.random_fsa(40, 400, D, seed=31), workloads.random_fsa(25, 900, D, seed=32),
                               workloads.random_fsa(7, 30, D, seed=33)])
    cu = torch.tensor([0, 200, 350, 420], dtype=torch.int32)
    ln = torch.tensor([190, 150, 70], dtype=torch.int32)
    l1, g1, s1, _ = _run(lp, cu, ln, fsa, 40)
    l2, g2, s2, _ = _run(lp, cu, ln, fsa, 40)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(l1, l2)
    assert torch.equal(g1.view(torch.int16) if dtype != torch.float32 else g1.view(torch.int32),
                       g2.view(torch.int16) if dtype != torch.float32 else g2.view(torch.int32))


def test_sequence_beyond_the_shared_memory_lists(cuda_device):
    # one sequence with far more edges than four times the batch's mean keeps
    # its lists in the workspace; the small ones keep theirs in shared memory
    D = 17
    lp = torch.log_softmax(torch.randn(60 + 12 * 20, D, generator=torch.Generator().manual_seed(12)), -1)
    fsas = [workloads.random_fsa(50, 6000, D, seed=90)] + [workloads.random_fsa(4, 10, D, seed=91 + i)
                                                           for i in range(12)]
    fsa = workloads.pack_fsas(fsas)
    cu = torch.tensor([0, 60] + [60 + 20 * (i + 1) for i in range(12)], dtype=torch.int32)
    ln = torch.tensor([60] + [18] * 12, dtype=torch.int32)
    loss, grad, status, g = _run(lp, cu, ln, fsa, 50)
    assert status == 0
    ref_loss, ref_grad = _oracle(lp, cu, ln, fsa, g)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32)


@pytest.mark.parametrize("L", [300, 700, 1250])
def test_many_states_a_thread(cuda_device, L):
    # CTC lattices of 2L + 2 states (the entry state included): 602 (two
    # states a thread), 1402 (four) and 2502 (eight, with the two-frame ring
    # of label words and alpha rows)
    batch = workloads.make_batch([L + 150, 90], [L, 30], 41, seed=29 + L, repeat_prob=0.1, redraw_infeasible=True,
                                 reduction="none")
    offs = np.concatenate([[0], np.cumsum(batch.target_lengths.numpy())])
    tg = batch.targets.numpy()
    fsa = workloads.pack_fsas([workloads.ctc_lattice_fsa(tg[offs[b]:offs[b + 1]], batch.blank)
                               for b in range(batch.B)])
    assert _max_states(fsa) == 2 * L + 2
    loss, grad, status, g = _run(batch.log_probs, batch.cu_seqlens, batch.lengths, fsa, _max_states(fsa))
    assert status == 0
    ref_loss, ref_grad = _oracle(batch.log_probs, batch.cu_seqlens, batch.lengths, fsa, g)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, torch.float32)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("S,E,D", [(40, 3000, 1200), (500, 3000, 2000)])
def test_many_distinct_labels(cuda_device, dtype, S, E, D):
    # about 1 100 (1 550) distinct labels in one sequence: more than two a
    # label thread, whether the labels have warps of their own (40 states:
    # 14 label warps) or the 512 state threads carry them (500 states)
    lp = torch.log_softmax(torch.randn(70, D, generator=torch.Generator().manual_seed(21)) * 2.0, -1).to(dtype)
    fsa = workloads.pack_fsas([workloads.random_fsa(S, E, D, seed=61), workloads.random_fsa(7, 40, D, seed=62)])
    cu = torch.tensor([0, 50, 70], dtype=torch.int32)
    ln = torch.tensor([50, 20], dtype=torch.int32)
    assert _max_labels(fsa) > 1024 if S == 500 else _max_labels(fsa) > 2 * 14 * 32
    loss, grad, status, g = _run(lp, cu, ln, fsa, _max_states(fsa), grad_loss=[0.8, 1.2])
    assert status == 0
    ref_loss, ref_grad = _oracle(lp, cu, ln, fsa, g)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sizes_beyond_the_older_shared_memory_limit(cuda_device, dtype):
    # 2048 states and about 3 100 distinct labels: beyond what the kernels
    # accepted when the backward recursion formed the occupancies itself
    # (CTC_PACKED_ERR_UNSUPPORTED then).  At this size the recursions' edge
    # lists and the row kernel's edge records both stay in the workspace.
    D = 3500
    lp = torch.log_softmax(torch.randn(60, D, generator=torch.Generator().manual_seed(23)) * 2.0, -1).to(dtype)
    fsa = workloads.pack_fsas([workloads.random_fsa(2048, 8000, D, seed=71), workloads.random_fsa(9, 50, D, seed=72)])
    cu = torch.tensor([0, 40, 60], dtype=torch.int32)
    ln = torch.tensor([40, 20], dtype=torch.int32)
    assert _max_states(fsa) == 2048 and _max_labels(fsa) > 3000
    loss, grad, status, g = _run(lp, cu, ln, fsa, _max_states(fsa), grad_loss=[0.9, 1.1])
    assert status == 0
    ref_loss, ref_grad = _oracle(lp, cu, ln, fsa, g)
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
def test_one_and_two_frame_sequences(cuda_device, dtype):
    # a sequence of one frame (its only row is its last frame, where the
    # occupancies take beta_T = exp(final)) and one of two (a 2- and a 3-state
    # chain: both have a path), beside a longer one, with rows between the
    # sequences that no sequence covers
    D = 12
    lp = torch.log_softmax(torch.randn(30, D, generator=torch.Generator().manual_seed(31)), -1).to(dtype)
    fsa = workloads.pack_fsas([workloads.random_fsa(2, 6, D, seed=81), workloads.random_fsa(3, 9, D, seed=82),
                               workloads.random_fsa(6, 18, D, seed=83)])
    cu = torch.tensor([0, 3, 7, 30], dtype=torch.int32)  # spans of 3, 4 and 23 rows
    ln = torch.tensor([1, 2, 20], dtype=torch.int32)
    loss, grad, status, g = _run(lp, cu, ln, fsa, _max_states(fsa), grad_loss=[0.7, 1.3, 0.9])
    assert status == 0
    ref_loss, ref_grad = _oracle(lp, cu, ln, fsa, g)
    assert np.isfinite(ref_loss).all()
    assert_loss_close(loss, ref_loss)
    assert_grad_close(grad, ref_grad, dtype)
