"""Planted mistakes in the FSA oracle: its pins must catch each one.

Each case copies ``oracle/fsa_oracle.py``, plants one plausible mistake
(edges walked the wrong way, a weight or a final weight dropped, a wrong
occupancy, a wrong sign), loads the copy as a module of its own and checks
that the CTC-lattice pin or the brute-force pin rejects it.  Nothing here
touches a GPU.
"""

import importlib.util
import itertools
import os
import sys

import numpy as np
import pytest

import oracle
from oracle import fsa_oracle

SRC = fsa_oracle.__file__
RNG = np.random.default_rng(9090)

MUTANTS = {
    "forward_edges_reversed": ("np.logaddexp.at(nxt, to, v)", "np.logaddexp.at(nxt, fr, v)"),
    "forward_weight_dropped": ("v = alpha[t][fr] + weights + lp[t, lab]", "v = alpha[t][fr] + lp[t, lab]"),
    "final_weight_dropped": ("Z = _logsumexp(alpha[T] + final)", "Z = _logsumexp(np.where(final > -np.inf, alpha[T], -np.inf))"),
    "loss_sign": ("return -Z, grad", "return Z, grad"),
    "beta_uses_origin": ("v = weights + lp[t, lab] + beta[t + 1][to]", "v = weights + lp[t, lab] + beta[t + 1][fr]"),
    "occupancy_misses_weight": ("occ = np.exp(alpha[t][fr] + weights + lp[t, lab] + beta[t + 1][to] - Z)",
                                "occ = np.exp(alpha[t][fr] + lp[t, lab] + beta[t + 1][to] - Z)"),
    "occupancy_off_by_a_frame": ("occ = np.exp(alpha[t][fr] + weights + lp[t, lab] + beta[t + 1][to] - Z)",
                                 "occ = np.exp(alpha[t + 1][fr] + weights + lp[t, lab] + beta[t + 1][to] - Z)"),
    "grad_without_exp_lp": ("grad[t] = scale * (np.exp(lp[t]) - post)", "grad[t] = scale * (-post)"),
    "ctc_no_skip": ("if s + 2 < S and s % 2 == 1 and ext[s + 2] != ext[s]:", "if False:"),
    "ctc_single_final": ("        final[S - 2] = 0.0\n    # with no frames", "        pass\n    # with no frames"),
}


def _load_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation {name} does not apply"
    path = tmp_path / f"fsa_{name}.py"
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location(f"fsa_mutant_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _lsm(z):
    return z - np.log(np.exp(z).sum(axis=1, keepdims=True))


def _ctc_pin_fails(mod):
    D, blank = 6, 0
    lengths = [9, 7, 5]
    targets = [[1, 2, 2], [3, 1], [4, 4]]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    lp = _lsm(RNG.normal(0, 1.5, size=(cu[-1], D)))
    so, sw, fw, eo, ed, ew = [0], [], [], [0], [], []
    for t in targets:
        st, fi, e, w = mod.ctc_topology(t, blank)
        sw += list(st)
        fw += list(fi)
        ed += [list(x) for x in e]
        ew += list(w)
        so.append(so[-1] + len(st))
        eo.append(eo[-1] + len(e))
    loss, grad = mod.fsa_loss_packed(lp, cu, lengths, np.array(so), np.array(sw), np.array(fw), np.array(eo),
                                     np.array(ed), np.array(ew))
    tl = np.array([len(t) for t in targets])
    flat = np.array([c for t in targets for c in t])
    ref_loss, ref_grad, _ = oracle.ctc_loss_packed(lp, cu, lengths, flat, tl, blank, False, "none")
    return not (np.allclose(loss, ref_loss, rtol=1e-10) and np.allclose(grad, ref_grad, atol=1e-10))


def _brute_force_pin_fails(mod):
    S, E, D, T = 3, 6, 3, 3
    edges = np.stack([RNG.integers(0, S, E), RNG.integers(0, S, E), RNG.integers(0, D, E)], axis=1)
    weights = RNG.normal(0, 0.5, E)
    start = np.array([0.0, -0.3, -np.inf])
    final = np.array([-np.inf, 0.2, 0.0])
    lp = _lsm(RNG.normal(0, 1, size=(T, D)))
    total, occ = 0.0, np.zeros((T, D))
    for path in itertools.product(range(E), repeat=T):
        if any(edges[path[i], 1] != edges[path[i + 1], 0] for i in range(T - 1)):
            continue
        sc = start[edges[path[0], 0]] + final[edges[path[-1], 1]]
        sc += sum(weights[e] + lp[t, edges[e, 2]] for t, e in enumerate(path))
        total += np.exp(sc)
        for t, e in enumerate(path):
            occ[t, edges[e, 2]] += np.exp(sc)
    if total == 0.0:
        return False
    loss, grad = mod.fsa_sequence(lp, start, final, edges, weights, 1.0, False)
    return not (np.isclose(loss, -np.log(total), rtol=1e-10) and grad is not None
                and np.allclose(grad, np.exp(lp) - occ / total, atol=1e-10))


def test_the_unmutated_oracle_passes_both_pins():
    assert not _ctc_pin_fails(fsa_oracle)
    for _ in range(5):
        assert not _brute_force_pin_fails(fsa_oracle)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_each_planted_mistake_is_caught(tmp_path, name):
    mod = _load_mutant(tmp_path, name, *MUTANTS[name])
    caught = _ctc_pin_fails(mod) or any(_brute_force_pin_fails(mod) for _ in range(5))
    assert caught, f"the pins did not catch {name}"
