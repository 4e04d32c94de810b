"""Pins of the float64 cross-entropy oracle (oracle/loss.py) to facts other
than itself: the uniform-logits value log V, a two-word vocabulary worked out
by hand (the logistic loss), invariance of the loss to a shift of all logits,
agreement of the log-sum-exp with scipy, the gradient's zero row sums, and
central finite differences.  CPU only."""
import math

import numpy as np
import scipy.special

import oracle as O


def test_uniform_logits_give_log_v():
    # W = 0: every logit is 0, softmax is uniform, the loss of any target is log V
    rng = np.random.default_rng(0)
    h = rng.standard_normal((5, 8))
    for V in (2, 7, 1000):
        f = O.loss_forward(h, np.zeros((V, 8)), rng.integers(0, V, 5))
        np.testing.assert_allclose(f["loss_rows"], math.log(V), rtol=0, atol=1e-13)


def test_two_word_vocabulary_is_the_logistic_loss():
    # V = 2: l = log(1 + exp(z_other - z_target)) = softplus of the margin
    h = np.array([[1.0, -2.0], [0.5, 0.25]])
    W = np.array([[0.3, 0.7], [-1.1, 0.4]])
    t = np.array([0, 1])
    z = h @ W.T
    want = [math.log1p(math.exp(z[0, 1] - z[0, 0])), math.log1p(math.exp(z[1, 0] - z[1, 1]))]
    np.testing.assert_allclose(O.loss_forward(h, W, t)["loss_rows"], want, rtol=1e-14)


def test_logsumexp_matches_scipy_and_survives_large_logits():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((6, 300)) * 30 + 700      # exp overflows without the shift
    np.testing.assert_allclose(O.logsumexp_rows(z), scipy.special.logsumexp(z, axis=1),
                               rtol=1e-15, atol=1e-12)


def test_gradient_rows_sum_to_zero_and_match_finite_differences():
    rng = np.random.default_rng(2)
    S, H, V = 4, 5, 9
    h = rng.standard_normal((S, H))
    W = rng.standard_normal((V, H))
    t = rng.integers(0, V, S)
    scale = 1.0 / S
    g = O.loss_backward(h, W, t, scale)
    # softmax minus one-hot sums to zero per row, so sum_v dz_iv = 0 and
    # dh_i is orthogonal to sum_v W_v only in that combination: check sum_v dW_v = 0
    np.testing.assert_allclose(g["dW"].sum(axis=0), 0.0, atol=1e-14)
    eps = 1e-6
    for name, base in (("h", h), ("W", W)):
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            saved = base[idx]
            base[idx] = saved + eps
            lp = O.loss_total(h, W, t, scale)
            base[idx] = saved - eps
            lm = O.loss_total(h, W, t, scale)
            base[idx] = saved
            num[idx] = (lp - lm) / (2 * eps)
        an = g["d" + name]
        err = np.max(np.abs(an - num)) / max(1e-12, np.max(np.abs(num)))
        assert err < 1e-7, (name, err)


def test_loss_ignores_a_common_shift_of_the_logits():
    # an extra feature equal to 1 whose weight is the same constant for every
    # word adds that constant to all of a row's logits: the loss must not move
    rng = np.random.default_rng(3)
    h = rng.standard_normal((6, 4))
    W = rng.standard_normal((11, 4))
    t = rng.integers(0, 11, 6)
    base = O.loss_forward(h, W, t)["loss_rows"]
    h1 = np.concatenate([h, np.ones((6, 1))], axis=1)
    W1 = np.concatenate([W, np.full((11, 1), 37.5)], axis=1)
    np.testing.assert_allclose(O.loss_forward(h1, W1, t)["loss_rows"], base, rtol=1e-12, atol=1e-12)
