"""Pins of the oracle's mean_batch and mean_volume reductions.

Read as: mean_batch = (1/B) sum_b loss_b, mean_volume = sum_b loss_b /
sum_b U_b, after zero_infinity.  Pinned against the sum reduction (itself
pinned against torch's CTC loss) and by central finite differences of the
reduced loss, which tie each reduction's gradient scale to its loss.
"""

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(77)


def _batch():
    cu = np.array([0, 9, 15, 15, 22])
    lengths = np.array([9, 6, 0, 7])
    targets = np.array([1, 2, 1, 3, 3, 2, 4, 1])
    target_lengths = np.array([3, 2, 1, 2])  # utterance 2 has no frames: infinite loss
    z = RNG.normal(0, 1.5, size=(22, 5))
    lp = z - np.log(np.exp(z).sum(axis=1, keepdims=True))
    return lp, cu, lengths, targets, target_lengths


@pytest.mark.parametrize("zero_infinity", [True, False])
def test_relations_to_the_sum(zero_infinity):
    lp, cu, ln, tg, tl = _batch()
    total = oracle.ctc_loss_packed(lp, cu, ln, tg, tl, 0, zero_infinity, "sum", need_grad=False)[0]
    mb = oracle.ctc_loss_packed(lp, cu, ln, tg, tl, 0, zero_infinity, "mean_batch", need_grad=False)[0]
    mv = oracle.ctc_loss_packed(lp, cu, ln, tg, tl, 0, zero_infinity, "mean_volume", need_grad=False)[0]
    if zero_infinity:
        assert np.isclose(mb * 4, total, rtol=1e-14) and np.isclose(mv * tl.sum(), total, rtol=1e-14)
    else:
        assert np.isinf(total) and np.isinf(mb) and np.isinf(mv)


@pytest.mark.parametrize("reduction", ["mean_batch", "mean_volume"])
def test_gradient_matches_central_differences(reduction):
    lp, cu, ln, tg, tl = _batch()
    g = 1.7
    _, grad, _ = oracle.ctc_loss_packed(lp, cu, ln, tg, tl, 0, True, reduction, grad_loss=np.array([g]))
    # the loss as a function of free log probabilities (the path's gradient
    # convention is scale * exp(lp) - P, the derivative through log_softmax)
    z0 = lp.copy()

    def loss_of(z):
        lz = z - np.log(np.exp(z).sum(axis=1, keepdims=True))
        return g * oracle.ctc_loss_packed(lz, cu, ln, tg, tl, 0, True, reduction, need_grad=False)[0]

    h = 1e-5
    fd = np.zeros_like(z0)
    for t in range(z0.shape[0]):
        for c in range(z0.shape[1]):
            zp, zm = z0.copy(), z0.copy()
            zp[t, c] += h
            zm[t, c] -= h
            fd[t, c] = (loss_of(zp) - loss_of(zm)) / (2 * h)
    np.testing.assert_allclose(grad, fd, rtol=0, atol=2e-8)


def test_empty_volume_and_empty_batch():
    lp, cu, ln, tg, tl = _batch()
    zero = np.zeros_like(tl)
    v = oracle.ctc_loss_packed(lp, cu, ln, tg[:0], zero, 0, True, "mean_volume", need_grad=False)[0]
    assert np.isposinf(v)  # positive blank-path losses over a zero volume
    e = oracle.ctc_loss_packed(lp[:0], np.array([0]), np.zeros(0, int), tg[:0], np.zeros(0, int), 0, True,
                               "mean_batch", need_grad=False)[0]
    assert np.isnan(e)
