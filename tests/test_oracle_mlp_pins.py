"""Pins of the float64 MLP oracle (oracle/mlp.py) to facts other than itself:
values of the logistic function and SiLU fixed by their definitions, a
one-unit MLP worked out by hand, the symmetry between the gate and up
projections that SwiGLU does not have, row independence (what makes tiling
exact), and central finite differences for the backward.  CPU only."""
import math

import numpy as np
import pytest

import oracle as O


def test_sigmoid_and_silu_values():
    # sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(-v) = 1 - sigmoid(v),
    # and the tails without overflow
    assert O.sigmoid(0.0) == 0.5
    assert abs(O.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    v = np.linspace(-30, 30, 121)
    np.testing.assert_allclose(O.sigmoid(-v), 1 - O.sigmoid(v), rtol=0, atol=1e-15)
    assert O.sigmoid(-800.0) == 0.0 and O.sigmoid(800.0) == 1.0
    # silu(v) = v sigmoid(v): silu(0) = 0, silu(ln 3) = 0.75 ln 3, silu(v) -> v
    # for large v and -> 0 for large -v
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert O.silu(50.0) == pytest.approx(50.0, abs=1e-15)
    assert abs(O.silu(-50.0)) < 1e-19


def test_silu_grad_matches_finite_differences():
    v = np.linspace(-12, 12, 97)
    h = 1e-6
    num = (O.silu(v + h) - O.silu(v - h)) / (2 * h)
    np.testing.assert_allclose(O.silu_grad(v), num, rtol=0, atol=1e-8)
    # silu'(0) = 1/2 exactly
    assert O.silu_grad(0.0) == 0.5


def test_one_unit_mlp_by_hand():
    # hidden = ffn = 1: y = silu(wg x) (wu x) wd, with distinct gate and up
    # weights so that exchanging the two projections is caught
    x = np.array([[1.5], [-0.5]])
    wg, wu, wd = 0.8, -1.3, 2.1
    f = O.mlp_forward(x, np.array([[wg]]), np.array([[wu]]), np.array([[wd]]))
    for i in range(2):
        gx = wg * x[i, 0]
        want = gx / (1 + math.exp(-gx)) * (wu * x[i, 0]) * wd
        assert abs(f["y"][i, 0] - want) < 1e-15
    swapped = O.mlp_forward(x, np.array([[wu]]), np.array([[wg]]), np.array([[wd]]))
    assert abs(swapped["y"][0, 0] - f["y"][0, 0]) > 0.1


def test_rows_are_independent():
    # each token's output depends on that token alone: computing any subset
    # of rows gives the same values, whatever the tiling (up to the order of
    # the library matmul's float64 additions, which depends on the shape)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((37, 16))
    Wg, Wu = rng.standard_normal((24, 16)) / 4, rng.standard_normal((24, 16)) / 4
    Wd = rng.standard_normal((16, 24)) / 5
    full = O.mlp_forward(x, Wg, Wu, Wd)["y"]
    for lo, hi in [(0, 1), (5, 17), (36, 37), (0, 37)]:
        np.testing.assert_allclose(O.mlp_forward(x[lo:hi], Wg, Wu, Wd)["y"], full[lo:hi],
                                   rtol=0, atol=1e-13)


def test_zero_gate_weights_give_zero_output():
    # silu(0) = 0: with Wg = 0 the MLP outputs zeros and only dWg is non-zero
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 8))
    Wu, Wd = rng.standard_normal((12, 8)), rng.standard_normal((8, 12))
    dy = rng.standard_normal((6, 8))
    gr = O.mlp_backward(x, np.zeros((12, 8)), Wu, Wd, dy)
    assert not gr["y"].any() and not gr["dx"].any() and not gr["dWu"].any()
    assert not gr["dWd"].any()
    # dg = da * u * silu'(0) = (dy Wd) * u / 2
    np.testing.assert_allclose(gr["dWg"], ((dy @ Wd) * (x @ Wu.T) * 0.5).T @ x, rtol=1e-14)


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(11)
    S, hidden, ffn = 5, 6, 7
    args = {"x": rng.standard_normal((S, hidden)),
            "Wg": rng.standard_normal((ffn, hidden)) / 2,
            "Wu": rng.standard_normal((ffn, hidden)) / 2,
            "Wd": rng.standard_normal((hidden, ffn)) / 2}
    dy = rng.standard_normal((S, hidden))
    grads = O.mlp_backward(dy=dy, **args)
    eps = 1e-6
    for name in ("x", "Wg", "Wu", "Wd"):
        base = args[name]
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            saved = base[idx]
            base[idx] = saved + eps
            lp = O.mlp_loss(dy=dy, **args)
            base[idx] = saved - eps
            lm = O.mlp_loss(dy=dy, **args)
            base[idx] = saved
            num[idx] = (lp - lm) / (2 * eps)
        an = grads["d" + name]
        err = np.max(np.abs(an - num)) / max(1e-12, np.max(np.abs(num)))
        assert err < 1e-6, (name, err)
