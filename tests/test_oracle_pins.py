"""Pins of the fp64 oracle against things other than itself.

Each check ties the oracle to something fixed by the definition of CTC or by
mathematics, never to a re-typing of its own recursion:

* brute force over every class path of a tiny input (T <= 6, D <= 4), using
  the collapse map of CTC (merge repeats, then drop blanks);
* brute force over every state path of the extended-label lattice, for
  targets that contain the blank id (page "feat(asr): native CTC loss kernel
  over sequence-packed log probabilities", ctc_loss.py ``_alpha_kernel``: a
  target id equal to the blank is a label like any other);
* the closed form for uniform log probabilities, loss = T log D - log C(T+U-R, 2U),
  at the real sizes of the benchmark workloads;
* torch's own CPU ``ctc_loss`` in float64 (the padded kernel the page tests
  against, test_ctc_loss.py ``test_packed_ctc_loss_function``);
* invariants: posteriors of each frame sum to one, so each gradient row of a
  log-softmax input sums to zero, and 0 <= P_t(c) <= 1;
* special cases: no target, a forced unique alignment, infeasible utterances,
  zero-length utterances;
* central finite differences of nll(log_softmax(z)) with respect to z.
"""

import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

RNG = np.random.default_rng(1234)


def log_softmax64(z):
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    return z - m - np.log(np.exp(z - m).sum(axis=-1, keepdims=True))


def collapse(path, blank):
    out, prev = [], None
    for c in path:
        if c != prev and c != blank:
            out.append(c)
        prev = c
    return out


def brute_force_paths(lp, labels, blank):
    """Sum over every class path whose collapse is ``labels``."""
    T, D = lp.shape
    labels = list(labels)
    if T == 0:
        return (0.0 if not labels else math.inf), np.zeros((0, D))
    total = 0.0
    acc = np.zeros((T, D))
    for path in itertools.product(range(D), repeat=T):
        if collapse(path, blank) != labels:
            continue
        p = math.exp(sum(lp[t, c] for t, c in enumerate(path)))
        total += p
        for t, c in enumerate(path):
            acc[t, c] += p
    if total == 0.0:
        return math.inf, None
    return -math.log(total), np.exp(lp) - acc / total


def brute_force_lattice(lp, labels, blank):
    """Sum over every state path of the extended-label lattice."""
    T, D = lp.shape
    ext = [blank]
    for l in labels:
        ext += [l, blank]
    S = len(ext)
    if T == 0:
        return (0.0 if not labels else math.inf), np.zeros((0, D))

    def allowed(s, s2):
        if s2 == s or s2 == s + 1:
            return True
        return s2 == s + 2 and s2 % 2 == 1 and ext[s2] != ext[s]

    total = 0.0
    acc = np.zeros((T, D))
    for states in itertools.product(range(S), repeat=T):
        if states[0] > 1 or states[-1] < S - 2:
            continue
        if not all(allowed(states[i], states[i + 1]) for i in range(T - 1)):
            continue
        p = math.exp(sum(lp[t, ext[s]] for t, s in enumerate(states)))
        total += p
        for t, s in enumerate(states):
            acc[t, ext[s]] += p
    if total == 0.0:
        return math.inf, None
    return -math.log(total), np.exp(lp) - acc / total


def run_one(lp, labels, blank):
    T, D = lp.shape
    nll, grad = oracle.raw_nll_and_grad(lp, [0, T], [T], list(labels), [len(labels)], blank)
    return nll[0], grad


TINY_CASES = [
    # (T, D, labels, blank)
    (1, 2, [], 0),
    (3, 2, [], 1),
    (1, 3, [1], 0),
    (2, 3, [1, 2], 0),
    (3, 3, [1, 1], 0),
    (4, 3, [2, 1, 2], 0),
    (5, 3, [1, 1, 2], 0),
    (6, 3, [2, 2, 2], 0),
    (5, 4, [3, 1], 2),
    (6, 4, [1, 3, 3], 0),
    (6, 4, [0, 2, 1], 3),
    (4, 4, [1, 2, 3], 0),
    (2, 3, [1, 1], 0),  # infeasible: needs 3 frames
    (3, 4, [2, 2, 2], 0),  # infeasible: needs 5 frames
]


@pytest.mark.parametrize("T,D,labels,blank", TINY_CASES)
def test_brute_force_class_paths(T, D, labels, blank):
    lp = log_softmax64(RNG.normal(0, 2, size=(T, D)))
    nll_bf, grad_bf = brute_force_paths(lp, labels, blank)
    nll, grad = run_one(lp, labels, blank)
    if math.isinf(nll_bf):
        assert math.isinf(nll) and nll > 0
        return
    assert abs(nll - nll_bf) <= 1e-10 * max(1.0, abs(nll_bf))
    np.testing.assert_allclose(grad, grad_bf, atol=1e-12, rtol=0)


@pytest.mark.parametrize("T,D,labels,blank", [
    (4, 3, [0, 1], 0),
    (5, 3, [1, 0, 0], 0),
    (5, 4, [2, 3, 2], 2),
    (6, 3, [2, 0, 2], 0),
    (4, 3, [0, 0], 0),
])
def test_brute_force_lattice_blank_id_targets(T, D, labels, blank):
    lp = log_softmax64(RNG.normal(0, 2, size=(T, D)))
    nll_bf, grad_bf = brute_force_lattice(lp, labels, blank)
    nll, grad = run_one(lp, labels, blank)
    if math.isinf(nll_bf):
        assert math.isinf(nll)
        return
    assert abs(nll - nll_bf) <= 1e-10 * max(1.0, abs(nll_bf))
    np.testing.assert_allclose(grad, grad_bf, atol=1e-12, rtol=0)


def test_lattice_brute_force_equals_class_paths_without_blank_labels():
    # the two brute forces agree where both apply, so each pins the other
    for T, D, labels, blank in TINY_CASES[:10]:
        lp = log_softmax64(RNG.normal(0, 1, size=(T, D)))
        a, ga = brute_force_paths(lp, labels, blank)
        b, gb = brute_force_lattice(lp, labels, blank)
        assert (math.isinf(a) and math.isinf(b)) or abs(a - b) < 1e-12 * max(1, abs(a))


def adjacent_repeats(labels):
    return sum(1 for i in range(1, len(labels)) if labels[i] == labels[i - 1])


def closed_form_uniform(T, D, labels):
    U, R = len(labels), adjacent_repeats(labels)
    if T < U + R:
        return math.inf
    n = math.comb(T + U - R, 2 * U)
    return T * math.log(D) - math.log(n)


@pytest.mark.parametrize("T,U,D,repeat", [
    (50, 10, 32, 0.0), (300, 60, 1025, 0.1), (1750, 520, 1025, 0.0), (800, 150, 29, 0.2),
    (600, 140, 8193, 0.0), (7, 3, 5, 0.5), (1, 1, 3, 0.0),
])
def test_closed_form_uniform_at_workload_sizes(T, U, D, repeat):
    rng = np.random.default_rng(T * 7 + U)
    labels = list(rng.integers(1, min(D, 40), size=U))
    for i in range(1, U):
        if rng.random() < repeat:
            labels[i] = labels[i - 1]
    D_small = min(D, 41)  # the loss depends on D only through log D here
    lp = np.full((T, D_small), -math.log(D))
    nll, _ = oracle.raw_nll_and_grad(lp, [0, T], [T], labels, [U], 0, need_grad=False)
    expected = closed_form_uniform(T, D, labels)
    assert abs(nll[0] - expected) <= 1e-9 * max(1.0, abs(expected))


def test_closed_form_infeasible():
    # all-repeat target with more labels than half the frames: T < U + R
    T, U = 8, 5
    labels = [3] * U
    lp = np.full((T, 6), -math.log(6))
    nll, _ = oracle.raw_nll_and_grad(lp, [0, T], [T], labels, [U], 0, need_grad=False)
    assert math.isinf(closed_form_uniform(T, 6, labels)) and np.isposinf(nll[0])
    # one more frame makes it exactly feasible with a single alignment
    T = 2 * U - 1
    lp = log_softmax64(RNG.normal(0, 1, size=(T, 6)))
    nll, _ = oracle.raw_nll_and_grad(lp, [0, T], [T], labels, [U], 0, need_grad=False)
    forced = -sum(lp[t, 3 if t % 2 == 0 else 0] for t in range(T))
    assert abs(nll[0] - forced) < 1e-12 * abs(forced)


def _padded(batch_lp, cu, lengths):
    B = len(lengths)
    T = max(lengths) if B else 0
    D = batch_lp.shape[1]
    pad = torch.zeros(T, B, D, dtype=torch.float64)
    for b in range(B):
        pad[: lengths[b], b] = batch_lp[cu[b]: cu[b] + lengths[b]]
    return pad


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("zero_infinity", [False, True])
def test_against_torch_cpu_ctc_loss(reduction, zero_infinity):
    gen = torch.Generator().manual_seed(5)
    lengths = [23, 9, 17, 1, 30]
    target_lengths = [6, 5, 3, 2, 0]  # utterance 1 and 3 are infeasible (5 labels in 9 frames with repeats / 2 in 1)
    D = 7
    seqs = [[1, 2, 2, 3, 4, 5], [2, 2, 2, 2, 2], [6, 1, 6], [3, 4], []]
    cu = np.cumsum([0] + lengths).tolist()
    lp = torch.log_softmax(torch.randn(cu[-1], D, generator=gen, dtype=torch.float64) * 2, -1)
    flat = [x for s in seqs for x in s]
    loss, grad, nll = oracle.ctc_loss_packed(lp, cu, lengths, flat, target_lengths, 0, zero_infinity, reduction)

    pad = _padded(lp, cu, lengths).requires_grad_()
    tgt = torch.zeros(len(lengths), max(target_lengths), dtype=torch.long)
    for b, s in enumerate(seqs):
        tgt[b, : len(s)] = torch.tensor(s, dtype=torch.long)
    ref = torch.nn.functional.ctc_loss(pad, tgt, torch.tensor(lengths), torch.tensor(target_lengths), blank=0,
                                       reduction=reduction, zero_infinity=zero_infinity)
    np.testing.assert_allclose(np.asarray(loss), ref.detach().numpy(), rtol=1e-10, atol=1e-12)
    if not zero_infinity:
        return  # the gradient of an infinite loss is not defined
    ref.sum().backward()
    ref_grad = np.concatenate([pad.grad[: lengths[b], b].numpy() for b in range(len(lengths))])
    np.testing.assert_allclose(grad, ref_grad, atol=1e-12, rtol=0)


def test_against_torch_cpu_ctc_loss_feasible_gradient():
    gen = torch.Generator().manual_seed(8)
    lengths = [40, 12, 33]
    seqs = [[1, 1, 2, 5, 5, 5, 3], [4, 2], [3, 1, 3, 1, 2, 2]]
    D, blank = 6, 0
    cu = np.cumsum([0] + lengths).tolist()
    lp = torch.log_softmax(torch.randn(cu[-1], D, generator=gen, dtype=torch.float64) * 3, -1)
    flat = [x for s in seqs for x in s]
    tl = [len(s) for s in seqs]
    for reduction in ("none", "sum", "mean"):
        g_up = torch.tensor([0.5, -2.0, 1.5], dtype=torch.float64) if reduction == "none" else torch.tensor(0.7)
        loss, grad, _ = oracle.ctc_loss_packed(lp, cu, lengths, flat, tl, blank, False, reduction,
                                               grad_loss=g_up)
        pad = _padded(lp, cu, lengths).requires_grad_()
        tgt = torch.zeros(3, max(tl), dtype=torch.long)
        for b, s in enumerate(seqs):
            tgt[b, : len(s)] = torch.tensor(s)
        ref = torch.nn.functional.ctc_loss(pad, tgt, torch.tensor(lengths), torch.tensor(tl), blank=blank,
                                           reduction=reduction)
        ref.backward(g_up.to(torch.float64))
        ref_grad = np.concatenate([pad.grad[: lengths[b], b].numpy() for b in range(3)])
        np.testing.assert_allclose(np.asarray(loss), ref.detach().numpy(), rtol=1e-10)
        np.testing.assert_allclose(grad, ref_grad, atol=1e-12, rtol=0)


def test_against_torch_on_tiny_workload():
    batch = workloads.workload("tiny")
    loss, grad, _ = oracle.oracle_batch(batch)
    lengths = batch.lengths.tolist()
    cu = batch.cu_seqlens.tolist()
    pad = _padded(batch.log_probs.double(), cu, lengths).requires_grad_()
    ref = torch.nn.functional.ctc_loss(pad, workloads.padded_targets(batch), torch.tensor(lengths),
                                       batch.target_lengths.long(), blank=0, reduction="none")
    ref.sum().backward()
    np.testing.assert_allclose(loss, ref.detach().numpy(), rtol=1e-11)
    ref_grad = np.concatenate([pad.grad[: lengths[b], b].numpy() for b in range(batch.B)])
    np.testing.assert_allclose(grad, ref_grad, atol=1e-12)


def test_posteriors_sum_to_one_and_rows_sum_to_zero():
    gen = torch.Generator().manual_seed(3)
    lengths = [120, 77, 64]
    D = 11
    seqs = [list(np.random.default_rng(b).integers(1, D, size=u)) for b, u in enumerate([30, 20, 25])]
    cu = np.cumsum([0] + lengths).tolist()
    lp = torch.log_softmax(torch.randn(cu[-1], D, generator=gen, dtype=torch.float64) * 2, -1)
    _, grad = oracle.raw_nll_and_grad(lp, cu, lengths, [x for s in seqs for x in s], [30, 20, 25], 0)
    # rows of exp(lp) sum to 1 and the posteriors of a frame sum to 1
    np.testing.assert_allclose(grad.sum(axis=1), 0.0, atol=1e-12)
    P = np.exp(lp.numpy()) - grad
    assert P.min() > -1e-12 and P.max() < 1 + 1e-12
    # classes outside {blank} and the target carry exp(lp) alone
    for b in range(3):
        rows = slice(cu[b], cu[b] + lengths[b])
        absent = sorted(set(range(D)) - set(seqs[b]) - {0})
        # (numpy's exp and the C library's may differ in the last bit)
        np.testing.assert_allclose(grad[rows][:, absent], np.exp(lp.numpy()[rows][:, absent]), rtol=5e-16, atol=0)


def test_empty_target_is_sum_of_blank_log_probs():
    lp = log_softmax64(RNG.normal(0, 2, size=(37, 9)))
    nll, grad = run_one(lp, [], 4)
    assert abs(nll - (-lp[:, 4].sum())) < 1e-12 * abs(nll)
    # the only path is all-blank: the blank column has posterior 1
    expect = np.exp(lp)
    expect[:, 4] -= 1.0
    np.testing.assert_allclose(grad, expect, atol=1e-13)


def test_zero_length_utterances():
    lp = log_softmax64(RNG.normal(0, 1, size=(5, 4)))
    nll, grad = oracle.raw_nll_and_grad(lp, [0, 5, 5, 5], [5, 0, 0], [1, 2, 1, 3], [2, 2, 0], 0)
    assert np.isfinite(nll[0]) and np.isposinf(nll[1]) and nll[2] == 0.0
    loss, g, _ = oracle.ctc_loss_packed(lp, [0, 5, 5, 5], [5, 0, 0], [1, 2, 1, 3], [2, 2, 0], 0,
                                        zero_infinity=True)
    assert loss[1] == 0.0


def test_gapped_rows_get_zero_gradient():
    lp = log_softmax64(RNG.normal(0, 1, size=(12, 5)))
    # utterance 0 uses 6 of its 8 rows, utterance 1 uses 3 of 4
    _, grad, _ = oracle.ctc_loss_packed(lp, [0, 8, 12], [6, 3], [1, 2, 3], [2, 1], 0)
    assert np.all(grad[6:8] == 0.0) and np.all(grad[11:12] == 0.0)
    assert np.all(grad[:6] != 0.0)


def test_finite_differences_with_respect_to_logits():
    rng = np.random.default_rng(99)
    T, D = 9, 5
    z = rng.normal(0, 1.5, size=(T, D))
    labels = [1, 3, 3, 2]

    def nll_of(zz):
        return run_one(log_softmax64(zz), labels, 0)[0]

    _, grad = run_one(log_softmax64(z), labels, 0)
    h = 1e-6
    fd = np.zeros_like(z)
    for t in range(T):
        for c in range(D):
            zp, zm = z.copy(), z.copy()
            zp[t, c] += h
            zm[t, c] -= h
            fd[t, c] = (nll_of(zp) - nll_of(zm)) / (2 * h)
    np.testing.assert_allclose(grad, fd, atol=1e-7)


def test_reductions_and_scales():
    nll = np.array([2.0, np.inf, 6.0, 0.0])
    tl = np.array([4, 3, 0, 0])
    assert oracle.reduce_losses(nll, tl, "sum", True) == 8.0
    assert abs(oracle.reduce_losses(nll, tl, "mean", True) - (0.5 + 0 + 6.0 + 0) / 4) < 1e-15
    np.testing.assert_array_equal(oracle.utterance_scales(nll, tl, "mean", True), [1 / 16, 0, 1 / 4, 1 / 4])
    np.testing.assert_array_equal(oracle.utterance_scales(nll, tl, "none", False, [1, 2, 3, 4]), [1, 2, 3, 4])
