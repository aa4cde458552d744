"""Pins of the generic FSA full-sum oracle (``oracle.fsa_oracle``).

* The CTC lattice written as an FSA gives the CTC oracle's losses and
  gradients (CTC is the special case the page builds into its recursion).
* On tiny random FSAs, brute force over every edge path gives the loss and
  the per-frame class occupancies.
* Central finite differences of the loss of log_softmax(z) with respect to z.
"""

import itertools

import numpy as np
import pytest

import oracle
from oracle import fsa_oracle as fo

RNG = np.random.default_rng(4242)


def _lsm(z):
    return z - np.log(np.exp(z).sum(axis=1, keepdims=True))


def _pack(fsas):
    """Concatenate per-sequence (start, final, edges, weights)."""
    so, eo = [0], [0]
    sw, fw, ed, ew = [], [], [], []
    for start, final, edges, weights in fsas:
        sw.append(start)
        fw.append(final)
        ed.append(edges.reshape(-1, 3))
        ew.append(weights)
        so.append(so[-1] + len(start))
        eo.append(eo[-1] + len(edges))
    return (np.array(so), np.concatenate(sw), np.concatenate(fw), np.array(eo), np.concatenate(ed),
            np.concatenate(ew))


@pytest.mark.parametrize("zero_infinity", [True, False])
def test_ctc_lattice_as_fsa_gives_the_ctc_oracle(zero_infinity):
    D, blank = 7, 0
    lengths = [12, 9, 0, 3, 10, 0]
    targets = [[1, 2, 2, 3], [4, 0, 4], [2], [5, 5, 5], [], []]  # a blank id as a label, an infeasible one
    cu = np.concatenate([[0], np.cumsum(lengths)])
    lp = _lsm(RNG.normal(0, 1.5, size=(cu[-1], D)))
    fsas = [fo.ctc_topology(t, blank) for t in targets]
    so, sw, fw, eo, ed, ew = _pack(fsas)
    g = np.array([1.0, 0.5, 2.0, 1.5, -1.0, 0.7])
    loss, grad = fo.fsa_loss_packed(lp, cu, lengths, so, sw, fw, eo, ed, ew, grad_loss=g,
                                    zero_infinity=zero_infinity)
    tl = np.array([len(t) for t in targets])
    flat = np.array([c for t in targets for c in t], dtype=np.int64)
    ref_loss, ref_grad, nll = oracle.ctc_loss_packed(lp, cu, lengths, flat, tl, blank, zero_infinity, "none",
                                                     grad_loss=g)
    np.testing.assert_allclose(loss, ref_loss, rtol=1e-12)
    ok = np.isfinite(nll) | zero_infinity
    for b in range(len(lengths)):
        if ok[b]:
            rows = slice(cu[b], cu[b + 1])
            np.testing.assert_allclose(grad[rows], ref_grad[rows], atol=1e-12)


def _random_fsa(S, E, D):
    edges = np.stack([RNG.integers(0, S, E), RNG.integers(0, S, E), RNG.integers(0, D, E)], axis=1)
    weights = RNG.normal(0, 0.5, E)
    start = np.where(RNG.random(S) < 0.5, RNG.normal(0, 0.3, S), -np.inf)
    start[0] = 0.0
    final = np.where(RNG.random(S) < 0.5, RNG.normal(0, 0.3, S), -np.inf)
    final[-1] = 0.0
    return start, final, edges, weights


@pytest.mark.parametrize("T", [0, 1, 3])
def test_brute_force_over_edge_paths(T):
    S, E, D = 3, 6, 3
    start, final, edges, weights = _random_fsa(S, E, D)
    lp = _lsm(RNG.normal(0, 1, size=(T, D)))
    total = 0.0
    occ = np.zeros((T, D))
    if T == 0:
        total = np.sum(np.exp(start + final))
    for path in itertools.product(range(E), repeat=T):
        if T == 0:
            break
        if any(edges[path[i], 1] != edges[path[i + 1], 0] for i in range(T - 1)):
            continue
        sc = start[edges[path[0], 0]] + final[edges[path[-1], 1]]
        sc += sum(weights[e] + lp[t, edges[e, 2]] for t, e in enumerate(path))
        p = np.exp(sc)
        total += p
        for t, e in enumerate(path):
            occ[t, edges[e, 2]] += p
    loss, grad = fo.fsa_sequence(lp, start, final, edges, weights, 1.0, False)
    np.testing.assert_allclose(loss, -np.log(total), rtol=1e-12)
    if T:
        np.testing.assert_allclose(grad, np.exp(lp) - occ / total, atol=1e-12)


def test_gradient_matches_central_differences():
    S, E, D, T = 4, 9, 5, 5
    start, final, edges, weights = _random_fsa(S, E, D)
    z = RNG.normal(0, 1, size=(T, D))
    _, grad = fo.fsa_sequence(_lsm(z), start, final, edges, weights, 1.3, False)
    h = 1e-5
    fd = np.zeros_like(z)
    for t in range(T):
        for c in range(D):
            zp, zm = z.copy(), z.copy()
            zp[t, c] += h
            zm[t, c] -= h
            lp_ = fo.fsa_sequence(_lsm(zp), start, final, edges, weights, 1.0, False)[0]
            lm_ = fo.fsa_sequence(_lsm(zm), start, final, edges, weights, 1.0, False)[0]
            fd[t, c] = 1.3 * (lp_ - lm_) / (2 * h)
    np.testing.assert_allclose(grad, fd, atol=1e-7)


def test_no_path_is_infinite_or_zeroed():
    start = np.array([0.0, -np.inf])
    final = np.array([-np.inf, 0.0])
    edges = np.array([[0, 0, 1]])  # state 1 is never reached
    lp = _lsm(RNG.normal(size=(4, 3)))
    l, g = fo.fsa_sequence(lp, start, final, edges, np.zeros(1), 1.0, False)
    assert np.isposinf(l) and g is None
    l, g = fo.fsa_sequence(lp, start, final, edges, np.zeros(1), 1.0, True)
    assert l == 0.0 and not g.any()
