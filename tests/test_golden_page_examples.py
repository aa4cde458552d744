"""The worked examples of the page's test file, run through the oracle.

The page prints inputs and structural outcomes (an infinite loss, a zeroed
gradient, a zero loss) but no numbers; ``tests/golden/page_examples.json``
records those inputs and outcomes with their citations.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))


def test_impossible_alignment():
    g = GOLDEN["impossible_alignment"]
    lp = torch.log_softmax(torch.tensor(g["logits"], dtype=torch.float64), -1)
    args = (lp, g["cu_seqlens"], g["lengths"], g["targets"], g["target_lengths"], g["blank"])
    loss, _, _ = oracle.ctc_loss_packed(*args, zero_infinity=False, need_grad=False)
    assert np.isposinf(loss[0]) and np.isfinite(loss[1])
    # one frame and one label: the only path emits label 1, so loss = -lp[1, 1]
    logits1 = g["logits"][1]
    assert abs(loss[1] - (math.log(sum(math.exp(x) for x in logits1)) - logits1[1])) < 1e-14
    loss, grad, _ = oracle.ctc_loss_packed(*args, zero_infinity=True)
    assert loss[0] == 0.0
    assert np.all(grad[0] == 0.0)
    assert np.abs(grad[1]).sum() > 0


@pytest.mark.parametrize("zero_infinity", [False, True])
def test_zero_length_utterance(zero_infinity):
    g = GOLDEN["zero_length_utterance"]
    T = sum(g["lengths"])
    lp = torch.log_softmax(torch.randn(T, g["D"], dtype=torch.float64, generator=torch.Generator().manual_seed(11)), -1)
    cu = np.cumsum([0] + g["lengths"]).tolist()
    loss, _, _ = oracle.ctc_loss_packed(lp, cu, g["lengths"], g["targets"], g["target_lengths"], g["blank"],
                                        zero_infinity=zero_infinity, need_grad=False)
    assert loss[1] == (0.0 if zero_infinity else math.inf)
    tl = list(g["target_lengths"])
    tl[1] = 0
    targets = g["targets"][:2] + g["targets"][3:]
    loss, _, _ = oracle.ctc_loss_packed(lp, cu, g["lengths"], targets, tl, g["blank"], zero_infinity=zero_infinity,
                                        need_grad=False)
    assert loss[1] == 0.0
