"""The seeded input generators follow the workload recipe (CPU).

Each named workload: its sizes, length and target-length ranges
(``U ~ U[ceil(T/k), floor(T/m)]``), class ranges, dtypes and reductions;
determinism from its seeds; feasibility where the recipe redraws
infeasible targets, and the long-form workload's one infeasible utterance;
rows of log probabilities that are normalised; and the FSA and logits
generators' structure.
"""

import math

import numpy as np
import pytest
import torch

import workloads

RECIPE = {
    # name: (B, T range, U fraction range (k, m), D, dtype, reduction)
    "conformer": (32, (200, 400), (6, 4), 1025, torch.bfloat16, "mean"),
    "char": (256, (100, 1000), (8, 3), 29, torch.float16, "mean"),
    "largevocab": (64, (400, 800), (8, 4), 8193, torch.bfloat16, "none"),
}


def _repeats(t):
    return sum(1 for i in range(1, len(t)) if t[i] == t[i - 1])


@pytest.mark.parametrize("name", sorted(RECIPE))
def test_named_workload_follows_its_recipe(name):
    B, (tlo, thi), (k, m), D, dtype, red = RECIPE[name]
    w = workloads.workload(name)
    assert w.B == B and w.D == D and w.log_probs.dtype == dtype and w.reduction == red
    Ts, Us = w.lengths.tolist(), w.target_lengths.tolist()
    assert all(tlo <= T <= thi for T in Ts)
    assert all(math.ceil(T / k) <= U <= T // m for T, U in zip(Ts, Us))
    assert w.log_probs.shape == (sum(Ts), D)
    tg = w.targets.tolist()
    assert len(tg) == sum(Us) and all(1 <= c < D for c in tg)  # labels avoid the blank (0)
    off = 0
    for T, U in zip(Ts, Us):
        assert T >= U + _repeats(tg[off:off + U])  # every utterance can align
        off += U
    rows = torch.logsumexp(w.log_probs[:50].float(), dim=1)
    assert torch.allclose(rows, torch.zeros_like(rows), atol=2e-2)  # normalised (up to the cast)


def test_longform_has_one_infeasible_utterance():
    w = workloads.workload("longform")
    assert w.B == 9 and w.zero_infinity and w.reduction == "sum"
    T, U = w.lengths.tolist()[-1], w.target_lengths.tolist()[-1]
    last = w.targets.tolist()[-U:]
    assert len(set(last)) == 1 and T < U + _repeats(last)


def test_generators_are_deterministic():
    a, b = workloads.workload("conformer"), workloads.workload("conformer")
    assert torch.equal(a.log_probs, b.log_probs) and torch.equal(a.targets, b.targets)
    assert torch.equal(workloads.unnormalised_logits(a, seed=3), workloads.unnormalised_logits(b, seed=3))
    assert workloads.random_fsa(7, 20, 5, seed=1) == workloads.random_fsa(7, 20, 5, seed=1)


def test_unnormalised_logits_normalise_back_to_the_batch():
    w = workloads.make_batch([30, 20], [5, 4], 11, dtype=torch.float32, seed=2)
    z = workloads.unnormalised_logits(w, seed=4, offset=20.0)
    assert not torch.allclose(z, w.log_probs)
    assert torch.allclose(torch.log_softmax(z.double(), 1), w.log_probs.double(), atol=1e-5)


def test_fsa_generators():
    start, final, edges, weights = workloads.ctc_lattice_fsa([3, 3, 5], 0)
    S = 2 * 3 + 1
    assert len(start) == S + 1 and start[S] == 0.0 and final[S - 1] == 0.0 and final[S - 2] == 0.0
    assert all(0 <= f < S + 1 and 0 <= t < S for f, t, _ in edges)
    assert (3, 5, 3) not in edges and (1, 3, 3) not in edges  # no skip between the two equal labels
    assert (3, 5, 5) in edges  # the skip from the second 3 over a blank to the 5
    so, sw, fw, eo, ed, ew = workloads.pack_fsas([workloads.random_fsa(4, 9, 6, 1), (start, final, edges, weights)])
    assert so.tolist() == [0, 4, 4 + S + 1] and eo.tolist() == [0, 9, 9 + len(edges)]
    assert ed.shape == (9 + len(edges), 3) and ew.numel() == ed.shape[0] and sw.numel() == fw.numel() == so[-1]
