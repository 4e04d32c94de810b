"""Pins of the float64 oracle against facts that do not come from the oracle
itself: a library attention routine, brute force on tiny inputs, closed forms,
invariants of the method (causality, GQA sharing, head-chunk invariance) and
finite differences for the backward.  CPU only."""
import math
import types

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O


def geom(**kw):
    base = dict(S=None, hidden=16, Hq=4, Hkv=2, d=8, rope_theta=1e4,
                qk_norm=False, norm_eps=1e-6)
    base.update(kw)
    return types.SimpleNamespace(**base)


def rand_layer(rng, g, S, scale_w=None):
    h, d = g.hidden, g.d
    x = rng.standard_normal((S, h))
    Wq = rng.standard_normal((g.Hq * d, h)) / math.sqrt(h)
    Wk = rng.standard_normal((g.Hkv * d, h)) / math.sqrt(h)
    Wv = rng.standard_normal((g.Hkv * d, h)) / math.sqrt(h)
    Wo = rng.standard_normal((h, g.Hq * d)) / math.sqrt(g.Hq * d)
    return x, Wq, Wk, Wv, Wo


# ------------------------------------------------------------- attention --

@pytest.mark.parametrize("n,d", [(1, 4), (37, 8), (130, 64)])
def test_attention_matches_library_sdpa(n, d):
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    o, _ = O.causal_attention(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(t)[None, None] for t in (q, k, v)),
        is_causal=True)[0, 0].numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_attention_brute_force_loops():
    rng = np.random.default_rng(2)
    n, d = 9, 4
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    o, lse = O.causal_attention(q, k, v)
    for i in range(n):
        scores = []
        for j in range(i + 1):
            scores.append(sum(q[i, t] * k[j, t] for t in range(d)) / math.sqrt(d))
        z = sum(math.exp(s) for s in scores)
        assert abs(lse[i] - math.log(z)) < 1e-12
        assert abs(lse[i] - scipy.special.logsumexp(scores)) < 1e-12
        for t in range(d):
            ref = sum(math.exp(scores[j]) / z * v[j, t] for j in range(i + 1))
            assert abs(o[i, t] - ref) < 1e-12


def test_softmax_rows_are_stochastic_and_causal():
    rng = np.random.default_rng(3)
    n, d = 50, 8
    q, k, v = (rng.standard_normal((n, d)) * 3 for _ in range(3))
    _, _, p = O.causal_attention(q, k, v, return_p=True)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(p >= 0)
    assert np.all(p[np.triu_indices(n, 1)] == 0)


def test_identical_keys_give_prefix_mean():
    rng = np.random.default_rng(4)
    n, d = 20, 8
    q, v = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    k = np.tile(rng.standard_normal((1, d)), (n, 1))
    o, lse = O.causal_attention(q, k, v)
    for i in range(n):
        np.testing.assert_allclose(o[i], v[: i + 1].mean(axis=0), atol=1e-12)
        s = q[i] @ k[0] / math.sqrt(d)
        assert abs(lse[i] - (s + math.log(i + 1))) < 1e-12


def test_sampled_rows_equal_full_rows():
    rng = np.random.default_rng(5)
    n, d = 64, 8
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    o, lse = O.causal_attention(q, k, v)
    rows = [0, 5, 31, 63]
    o2, lse2 = O.causal_attention(q[rows], k, v, q_pos=rows)
    np.testing.assert_allclose(o2, o[rows], atol=1e-13)
    np.testing.assert_allclose(lse2, lse[rows], atol=1e-13)


# ------------------------------------------------------------------ RoPE --

def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(6)
    v = rng.standard_normal((1, 64))
    c, s = O.rope_cos_sin(np.array([0]), 64, 5e5)
    np.testing.assert_array_equal(O.apply_rope(v, c, s), v)


def test_rope_matches_complex_rotation():
    # pair (i, i + d/2) as the complex number a + ib, rotated by e^{i pos w_i}
    rng = np.random.default_rng(7)
    d, theta = 16, 1e4
    pos = np.array([0, 1, 7, 1000, 5_242_879])
    v = rng.standard_normal((len(pos), d))
    c, s = O.rope_cos_sin(pos, d, theta)
    r = O.apply_rope(v, c, s)
    w = np.array([theta ** (-(2 * i) / d) for i in range(d // 2)])
    z = (v[:, : d // 2] + 1j * v[:, d // 2:]) * np.exp(1j * np.outer(pos, w))
    np.testing.assert_allclose(r[:, : d // 2], z.real, atol=1e-12)
    np.testing.assert_allclose(r[:, d // 2:], z.imag, atol=1e-12)


def test_rope_preserves_norm_and_transpose_inverts():
    rng = np.random.default_rng(8)
    pos = np.arange(100) * 997
    v = rng.standard_normal((100, 128))
    c, s = O.rope_cos_sin(pos, 128, 5e5)
    r = O.apply_rope(v, c, s)
    np.testing.assert_allclose(np.linalg.norm(r, axis=1),
                               np.linalg.norm(v, axis=1), rtol=1e-13)
    np.testing.assert_allclose(O.apply_rope_transpose(r, c, s), v, atol=1e-12)
    # transpose: <R u, w> == <u, R^T w>
    w = rng.standard_normal((100, 128))
    lhs = np.sum(r * w, axis=1)
    rhs = np.sum(v * O.apply_rope_transpose(w, c, s), axis=1)
    np.testing.assert_allclose(lhs, rhs, atol=1e-11)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(9)
    d = 32
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    base = None
    for shift in [0, 3, 1000, 77777]:
        pi, pj = np.array([10 + shift]), np.array([4 + shift])
        qr = O.apply_rope(q[None], *O.rope_cos_sin(pi, d, 1e4))
        kr = O.apply_rope(k[None], *O.rope_cos_sin(pj, d, 1e4))
        sc = float((qr @ kr.T)[0, 0])
        base = sc if base is None else base
        assert abs(sc - base) < 1e-10


# -------------------------------------------------------------- RMSNorm --

def test_rms_norm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(10)
    a = rng.standard_normal((30, 128)) * 5
    y, r = O.rms_norm(a, None, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-13)
    y2, _ = O.rms_norm(a * 7.5, None, 0.0)
    np.testing.assert_allclose(y2, y, atol=1e-13)
    g = rng.standard_normal(128)
    yg, _ = O.rms_norm(a, g, 0.0)
    np.testing.assert_allclose(yg, y * g, atol=1e-13)


# ----------------------------------------------------------------- layer --

def test_single_token_closed_form():
    # S = 1: softmax weight 1, RoPE identity, so out = sum_h v0(h) Wo_h^T
    rng = np.random.default_rng(11)
    g = geom(Hq=4, Hkv=2, d=8)
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, 1)
    res = O.layer_forward(g, x, Wq, Wk, Wv, Wo)
    expect = np.zeros(g.hidden)
    for h in range(4):
        kv = h // 2
        v0 = Wv[kv * 8:(kv + 1) * 8] @ x[0]
        expect += Wo[:, h * 8:(h + 1) * 8] @ v0
    np.testing.assert_allclose(res["out"][0], expect, atol=1e-12)


def test_causal_prefix_invariance():
    rng = np.random.default_rng(12)
    g = geom(qk_norm=True)
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, 40)
    full = O.layer_forward(g, x, Wq, Wk, Wv, Wo)
    for t in [1, 17, 39]:
        pre = O.layer_forward(g, x[:t], Wq, Wk, Wv, Wo)
        np.testing.assert_allclose(pre["out"], full["out"][:t], atol=1e-12)
        np.testing.assert_allclose(pre["lse"], full["lse"][:, :t], atol=1e-12)


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(13)
    g = geom(Hq=6, Hkv=2, d=8)
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, 25)
    gqa = O.layer_forward(g, x, Wq, Wk, Wv, Wo)
    rep = lambda W: np.concatenate([W[(h // 3) * 8:(h // 3 + 1) * 8]
                                    for h in range(6)])
    mha = O.layer_forward(geom(Hq=6, Hkv=6, d=8), x, Wq, rep(Wk), rep(Wv), Wo)
    np.testing.assert_allclose(gqa["out"], mha["out"], atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv,ch", [(4, 1, 1), (4, 1, 2), (4, 2, 2),
                                       (6, 2, 6), (8, 2, 4), (4, 4, 2)])
def test_head_chunk_invariance(Hq, Hkv, ch):
    """The UPipe loop (chunks of ch heads, each adding its Wo-slice partial
    result) gives the unchunked layer's output."""
    rng = np.random.default_rng(14)
    g = geom(Hq=Hq, Hkv=Hkv, d=8, qk_norm=True)
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, 33)
    full = O.layer_forward(g, x, Wq, Wk, Wv, Wo)
    grp = Hq // Hkv
    acc = np.zeros_like(full["out"])
    for c in range(Hq // ch):
        heads = range(c * ch, (c + 1) * ch)
        kvs = sorted({h // grp for h in heads})
        sub = geom(Hq=ch, Hkv=len(kvs), d=8, qk_norm=True)
        sel = lambda W, idx: np.concatenate([W[i * 8:(i + 1) * 8] for i in idx])
        part = O.layer_forward(sub, x, sel(Wq, heads), sel(Wk, kvs),
                               sel(Wv, kvs), Wo[:, c * ch * 8:(c + 1) * ch * 8])
        np.testing.assert_allclose(part["lse"], full["lse"][list(heads)],
                                   atol=1e-12)
        acc += part["out"]
    np.testing.assert_allclose(acc, full["out"], atol=1e-12)


def test_row_source_callable_matches_array():
    rng = np.random.default_rng(15)
    g = geom(S=50)
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, 50)
    rows = [0, 7, 49]
    a = O.layer_forward(g, x, Wq, Wk, Wv, Wo, rows=rows)
    b = O.layer_forward(g, lambda lo, hi: x[lo:hi], Wq, Wk, Wv, Wo, rows=rows)
    full = O.layer_forward(g, x, Wq, Wk, Wv, Wo)
    np.testing.assert_allclose(a["out"], full["out"][rows], atol=1e-12)
    np.testing.assert_allclose(b["out"], full["out"][rows], atol=1e-12)


def _torch_layer(g, x, Wq, Wk, Wv, Wo, qg, kg):
    """The same layer written independently with torch float64 library ops:
    F.linear projections, F.rms_norm (qk-norm), the rotate-half RoPE in the
    form x cos + rotate_half(x) sin with inverse frequencies 1 / theta^(2i/d),
    repeat_interleave for the GQA groups, causal scaled_dot_product_attention,
    heads concatenated in order and F.linear with Wo."""
    F = torch.nn.functional
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    S, d = x.shape[0], g.d
    X = t(x)
    q = F.linear(X, t(Wq)).view(S, g.Hq, d).transpose(0, 1)       # [Hq, S, d]
    k = F.linear(X, t(Wk)).view(S, g.Hkv, d).transpose(0, 1)
    v = F.linear(X, t(Wv)).view(S, g.Hkv, d).transpose(0, 1)
    if g.qk_norm:
        q = F.rms_norm(q, (d,), None if qg is None else t(qg), g.norm_eps)
        k = F.rms_norm(k, (d,), None if kg is None else t(kg), g.norm_eps)
    inv_freq = 1.0 / (g.rope_theta ** (torch.arange(0, d, 2, dtype=torch.float64) / d))
    ang = torch.outer(torch.arange(S, dtype=torch.float64), inv_freq)
    emb = torch.cat([ang, ang], dim=-1)
    cos, sin = emb.cos(), emb.sin()

    def rotate_half(a):
        return torch.cat([-a[..., d // 2:], a[..., :d // 2]], dim=-1)

    q = q * cos + rotate_half(q) * sin
    k = k * cos + rotate_half(k) * sin
    rep = g.Hq // g.Hkv
    k = k.repeat_interleave(rep, dim=0)
    v = v.repeat_interleave(rep, dim=0)
    o = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True)[0]
    s = (q @ k.transpose(1, 2)) / math.sqrt(d)
    s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    out = F.linear(o.transpose(0, 1).reshape(S, g.Hq * d), t(Wo))
    return out.numpy(), lse.numpy(), o.numpy()


@pytest.mark.parametrize("qk_norm", [False, True])
def test_layer_composition_matches_independent_torch_formulation(qk_norm):
    """Pins the step order and per-tensor placement of ``layer_forward`` at
    S > 1 (where RoPE is not the identity): RoPE on q and k but not v, the
    RMSNorm before RoPE, GQA head h -> kv head h // (Hq/Hkv), and head h's
    output multiplied by Wo's column block h."""
    rng = np.random.default_rng(19)
    g = geom(hidden=32, Hq=6, Hkv=2, d=8, qk_norm=qk_norm, rope_theta=100.0)
    S = 37
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, S)
    qg = 1 + 0.3 * rng.standard_normal(8) if qk_norm else None
    kg = 1 + 0.3 * rng.standard_normal(8) if qk_norm else None
    res = O.layer_forward(g, x, Wq, Wk, Wv, Wo, qg, kg)
    out, lse, o = _torch_layer(g, x, Wq, Wk, Wv, Wo, qg, kg)
    np.testing.assert_allclose(res["out"], out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(res["lse"], lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(res["o"], o, rtol=0, atol=1e-12)


def test_project_kv_blocks_keep_their_positions():
    """K and V projected in blocks of 7 rows (RoPE of each block from its
    own positions) equal the single-block projection, and so does the
    layer computed with that blocking."""
    rng = np.random.default_rng(20)
    g = geom(hidden=16, Hq=4, Hkv=2, d=8, qk_norm=True, rope_theta=50.0)
    S = 40
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, S)
    kg = 1 + 0.3 * rng.standard_normal(8)
    for kvh in range(2):
        K1, V1 = O.project_kv(x, Wk, Wv, g, kvh, S, kg, block=S)
        K7, V7 = O.project_kv(x, Wk, Wv, g, kvh, S, kg, block=7)
        np.testing.assert_allclose(K7, K1, rtol=0, atol=1e-13)
        np.testing.assert_allclose(V7, V1, rtol=0, atol=1e-13)
    a = O.layer_forward(g, x, Wq, Wk, Wv, Wo, None, kg)
    b = O.layer_forward(g, x, Wq, Wk, Wv, Wo, None, kg, rows=[0, 6, 7, 13, 14, 39], kv_block=7)
    np.testing.assert_allclose(b["out"], a["out"][[0, 6, 7, 13, 14, 39]], rtol=0, atol=1e-12)


# -------------------------------------------------------------- backward --

@pytest.mark.parametrize("qk_norm", [False, True])
def test_backward_matches_finite_differences(qk_norm):
    rng = np.random.default_rng(17)
    g = geom(hidden=6, Hq=4, Hkv=2, d=4, qk_norm=qk_norm, norm_eps=1e-6)
    S = 5
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, S)
    dout = rng.standard_normal((S, g.hidden))
    qg = 1 + 0.2 * rng.standard_normal(4) if qk_norm else None
    kg = 1 + 0.2 * rng.standard_normal(4) if qk_norm else None
    args = dict(x=x, Wq=Wq, Wk=Wk, Wv=Wv, Wo=Wo, q_gamma=qg, k_gamma=kg)
    grads = O.layer_backward(g, dout=dout, **args)
    names = {"x": "dx", "Wq": "dWq", "Wk": "dWk", "Wv": "dWv", "Wo": "dWo"}
    if qk_norm:
        names.update(q_gamma="dq_gamma", k_gamma="dk_gamma")
    eps = 1e-6
    for name, gname in names.items():
        base = args[name]
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            saved = base[idx]
            base[idx] = saved + eps
            lp = O.layer_loss(g, dout=dout, **args)
            base[idx] = saved - eps
            lm = O.layer_loss(g, dout=dout, **args)
            base[idx] = saved
            num[idx] = (lp - lm) / (2 * eps)
        an = grads[gname]
        err = np.max(np.abs(an - num)) / max(1e-12, np.max(np.abs(num)))
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("qk_norm", [False, True])
def test_tail_backward_equals_full_backward_rows(qk_norm):
    """The tail-rows dx used at million-token sizes equals the last rows of
    the full chain-rule backward (itself pinned by finite differences)."""
    rng = np.random.default_rng(18)
    g = geom(hidden=24, Hq=4, Hkv=2, d=8, qk_norm=qk_norm)
    S = 40
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, S)
    dout = rng.standard_normal((S, g.hidden))
    qg = 1 + 0.2 * rng.standard_normal(8) if qk_norm else None
    kg = 1 + 0.2 * rng.standard_normal(8) if qk_norm else None
    full = O.layer_backward(g, x, Wq, Wk, Wv, Wo, dout, qg, kg)
    for n in (1, 7, 40):
        tail = O.layer_backward_tail(g, x, Wq, Wk, Wv, Wo, dout[S - n:], n, qg, kg)
        np.testing.assert_allclose(tail, full["dx"][S - n:], atol=1e-12)


@pytest.mark.parametrize("qk_norm", [False, True])
def test_key_rows_backward_equals_full_backward_with_sparse_dout(qk_norm):
    """dx of early key rows from a few gradient-carrying query rows equals the
    full chain-rule backward run with dout zero on every other row."""
    rng = np.random.default_rng(21)
    g = geom(hidden=24, Hq=4, Hkv=2, d=8, qk_norm=qk_norm)
    S = 50
    x, Wq, Wk, Wv, Wo = rand_layer(rng, g, S)
    qg = 1 + 0.2 * rng.standard_normal(8) if qk_norm else None
    kg = 1 + 0.2 * rng.standard_normal(8) if qk_norm else None
    q_rows = [9, 10, 30, 31, 49]
    dout = np.zeros((S, g.hidden))
    dout[q_rows] = rng.standard_normal((len(q_rows), g.hidden))
    full = O.layer_backward(g, x, Wq, Wk, Wv, Wo, dout, qg, kg)
    keys = list(range(9))
    part = O.layer_backward_key_rows(g, x, Wq, Wk, Wv, Wo, q_rows, dout[q_rows], keys, qg, kg)
    np.testing.assert_allclose(part, full["dx"][keys], atol=1e-12)
    assert np.abs(full["dx"][keys]).max() > 1e-3     # the rows do receive gradient
