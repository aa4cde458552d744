"""Planted mistakes: the pins must catch a wrong oracle.

Each case copies the oracle's C source, plants one plausible mistake (a
dropped transition, a wrong index, a sign, a swapped operand), builds the copy
with gcc in a temporary directory and checks that the brute-force and torch
pins reject it.  Nothing here touches a GPU.
"""

import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from oracle import ctc_oracle as driver
from test_oracle_pins import brute_force_lattice, brute_force_paths, log_softmax64

SRC = os.path.join(os.path.dirname(driver.__file__), "ctc_oracle.c")

MUTANTS = {
    "no_skip_transition": ("a = log_add(a, ALPHA(t - 1, s - 2));", "a = a;"),
    "skip_ignores_repeat": ("if (s >= 2 && s % 2 == 1 && ext_label(labels, s, blank) != ext_label(labels, s - 2, blank))",
                            "if (s >= 2 && s % 2 == 1)"),
    "skip_condition_inverted": ("s % 2 == 1 && ext_label(labels, s, blank) != ext_label(labels, s - 2, blank)",
                                "s % 2 == 1 && ext_label(labels, s, blank) == ext_label(labels, s - 2, blank)"),
    "no_advance": ("if (s >= 1) a = log_add(a, ALPHA(t - 1, s - 1));", ""),
    "start_only_blank": ("if (S > 1) ALPHA(0, 1) = LP(0, ext_label(labels, 1, blank));", ""),
    "end_only_last": ("if (S > 1) total = log_add(total, ALPHA(T - 1, S - 2));", ""),
    "nll_sign": ("*nll = -total;", "*nll = total;"),
    "emission_of_blank": ("ALPHA(t, s) = a + LP(t, ext_label(labels, s, blank));", "ALPHA(t, s) = a + LP(t, blank);"),
    "beta_no_skip": ("b = log_add(b, BETA(t + 1, s + 2));", "b = b;"),
    "beta_end_one_state": ("if (S > 1) BETA(T - 1, S - 2) = LP(T - 1, ext_label(labels, S - 2, blank));", ""),
    "posterior_keeps_lp": ("g[c] -= exp(ALPHA(t, s) + BETA(t, s) - LP(t, c) + *nll);",
                           "g[c] -= exp(ALPHA(t, s) + BETA(t, s) + *nll);"),
    "grad_plain_lp": ("for (int64_t c = 0; c < D; ++c) g[c] = exp(LP(t, c));",
                      "for (int64_t c = 0; c < D; ++c) g[c] = 0.0;"),
    "label_index_off_by_one": ("return (s % 2 == 0) ? blank : labels[(s - 1) / 2];",
                               "return (s % 2 == 0) ? blank : labels[s / 2 - (s > 1)];"),
    "zero_length_loss": ("*nll = (U == 0) ? 0.0 : INFINITY;", "*nll = 0.0;"),
}

CASES = [(5, 3, [1, 1, 2], 0), (6, 4, [1, 3, 3], 0), (6, 4, [0, 2, 1], 3), (4, 3, [2, 1, 2], 0),
         (5, 4, [3, 1], 2), (6, 3, [2, 0, 2], 0)]


def _build_mutant(tmp, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation {name} does not apply"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    so = os.path.join(tmp, f"{name}.so")
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", so, path, "-lm"])
    return driver.load_library(so)


def _pins_pass(lib):
    rng = np.random.default_rng(7)
    for T, D, labels, blank in CASES:
        lp = log_softmax64(rng.normal(0, 2, size=(T, D)))
        ref = brute_force_lattice if blank in labels else brute_force_paths
        nll_ref, grad_ref = ref(lp, labels, blank)
        nll, grad = oracle.raw_nll_and_grad(lp, [0, T], [T], labels, [len(labels)], blank, lib=lib)
        if not (abs(nll[0] - nll_ref) <= 1e-10 * max(1, abs(nll_ref))):
            return False
        if not np.allclose(grad, grad_ref, atol=1e-12, rtol=0):
            return False
    # zero-length utterance with a target: the page's loss is inf
    nll, _ = oracle.raw_nll_and_grad(np.zeros((1, 3)), [0, 0, 1], [0, 1], [1], [1, 0], 0, lib=lib)
    return bool(np.isposinf(nll[0]))


def test_unmutated_copy_passes():
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_mutant(tmp, "identity", "log_add", "log_add")
        assert _pins_pass(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    old, new = MUTANTS[name]
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_mutant(tmp, name, old, new)
        assert not _pins_pass(lib), f"planted mistake {name} went unnoticed"
