"""Pins of the logits form of the oracle (``oracle.ctc_loss_packed_logits``).

The logits form takes unnormalised scores z, applies log_softmax over each
row and returns the loss with the gradient with respect to z.  It is pinned
by properties that do not come from the oracle itself:
* log_softmax removes any per-row constant, so shifting a row of z changes
  neither the loss nor the gradient;
* central finite differences of the loss with respect to each logit;
* every row of the gradient of a covered frame sums to zero (softmax and the
  frame's posteriors both sum to one), and uncovered frames get zero;
* on already normalised rows the logits form is the log-probability form.
"""

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(20261202)


def _small_batch():
    cu = np.array([0, 7, 7, 12, 16])  # an empty utterance and a 1-row gap at the end
    lengths = np.array([7, 0, 5, 3])
    targets = np.array([1, 2, 2, 3, 1, 4])
    target_lengths = np.array([3, 1, 1, 1])
    return cu, lengths, targets, target_lengths


def test_row_shift_leaves_loss_and_gradient_unchanged():
    cu, ln, tg, tl = _small_batch()
    z = RNG.normal(0, 2, size=(16, 6))
    shift = RNG.uniform(-60, 60, size=(16, 1))
    for red in ("none", "sum", "mean"):
        l0, g0, _ = oracle.ctc_loss_packed_logits(z, cu, ln, tg, tl, 0, reduction=red, zero_infinity=True)
        l1, g1, _ = oracle.ctc_loss_packed_logits(z + shift, cu, ln, tg, tl, 0, reduction=red, zero_infinity=True)
        np.testing.assert_allclose(l1, l0, rtol=1e-12, atol=1e-10)
        np.testing.assert_allclose(g1, g0, rtol=0, atol=1e-12)


def test_gradient_matches_central_differences():
    cu, ln, tg, tl = _small_batch()
    z = RNG.normal(0, 1.5, size=(16, 6))
    gl = np.array([0.7, 1.3, -0.4, 2.0])
    loss, grad, _ = oracle.ctc_loss_packed_logits(z, cu, ln, tg, tl, 0, reduction="none", grad_loss=gl)

    def weighted(zz):
        l, _, _ = oracle.ctc_loss_packed_logits(zz, cu, ln, tg, tl, 0, reduction="none", need_grad=False)
        return float(np.dot(gl, np.where(np.isfinite(l), l, 0.0)))

    h = 1e-5
    fd = np.zeros_like(z)
    for t in range(z.shape[0]):
        for c in range(z.shape[1]):
            zp, zm = z.copy(), z.copy()
            zp[t, c] += h
            zm[t, c] -= h
            fd[t, c] = (weighted(zp) - weighted(zm)) / (2 * h)
    np.testing.assert_allclose(grad, fd, rtol=0, atol=2e-7)


def test_gradient_rows_sum_to_zero_and_uncovered_rows_are_zero():
    cu, ln, tg, tl = _small_batch()
    z = RNG.normal(0, 3, size=(16, 6))
    _, grad, nll = oracle.ctc_loss_packed_logits(z, cu, ln, tg, tl, 0, reduction="sum")
    covered = np.zeros(16, bool)
    for b in range(4):
        covered[cu[b]:cu[b] + ln[b]] = np.isfinite(nll[b])
    np.testing.assert_allclose(grad[covered].sum(axis=1), 0.0, atol=1e-12)
    assert not grad[~covered].any()
    assert covered.sum() == 15 and not covered[15]


def test_normalised_rows_give_the_log_probability_form():
    cu, ln, tg, tl = _small_batch()
    z = RNG.normal(0, 2, size=(16, 6))
    lp = z - np.log(np.exp(z).sum(axis=1, keepdims=True))
    a = oracle.ctc_loss_packed_logits(lp, cu, ln, tg, tl, 0, reduction="mean")
    b = oracle.ctc_loss_packed(lp, cu, ln, tg, tl, 0, reduction="mean")
    np.testing.assert_allclose(a[0], b[0], rtol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


@pytest.mark.parametrize("bad", ["sign", "no_max"])
def test_pins_reject_a_wrong_normalisation(bad):
    # plant a mistake in a copy of the normalisation: the shift pin must fail
    cu, ln, tg, tl = _small_batch()
    z = RNG.normal(0, 2, size=(16, 6))
    shift = RNG.uniform(5, 20, size=(16, 1))

    def wrong(zz):
        if bad == "sign":
            return zz + np.log(np.exp(zz).sum(axis=1, keepdims=True))
        return zz - np.log(np.exp(zz - zz.max()).sum(axis=1, keepdims=True))

    l0 = oracle.ctc_loss_packed(wrong(z), cu, ln, tg, tl, 0, reduction="sum", zero_infinity=True,
                                need_grad=False)[0]
    l1 = oracle.ctc_loss_packed(wrong(z + shift), cu, ln, tg, tl, 0, reduction="sum", zero_infinity=True,
                                need_grad=False)[0]
    assert abs(l1 - l0) > 1e-3
