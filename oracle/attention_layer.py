"""Float64 CPU oracle for the causal GQA attention layer that Untied Ulysses
(UPipe) computes one head chunk at a time.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA path, and the CUDA path never calls it.

What the method computes, and where it is stated
------------------------------------------------
* "Untied Ulysses: Memory-Efficient Context Parallelism via Headwise Chunking"
  (memeeeeeex.com article, section "Untied Ulysses (UPipe)"; talk transcript on
  liquidgold.cc): the heads a GPU owns are split into chunks that are run one
  after another; per chunk the heads are (re)computed, their attention is
  computed over the whole sequence and the partial result is stored, while the
  buffers are reused.  The article's editor's note says the method brings no
  new mathematics: chunking changes memory, not the result.  So the oracle has no
  chunking at all; it computes the layer by its plain definition, head by head,
  and chunk invariance is a property the tests check.
* The Q&A of the talk (aipmzone.com article, Q&A; transcript) names the query,
  key and value matrices and the all-pairs interaction of attention; the
  article's stack section places FlashAttention-style attention over the full
  sequence per head (DeepSpeed Ulysses).
* The layer's geometry (projections, causal mask, GQA grouping, RoPE, Qwen3's
  per-head RMSNorm on q and k, the Wo projection) is not spelled out on the
  pages; it is the standard Llama / Qwen3 attention layer the pages train
  ("Results": Llama3-8B, Qwen3-32B).  Readings where the pages are silent:
    - RoPE is the rotate-half form: pairs (i, i + d/2) rotate by
      pos * theta^(-2i/d), angle computed exactly in float64;
    - RMSNorm: v / sqrt(mean(v^2) + eps) * gamma over the head dimension,
      applied per head to q and per kv head to k, before RoPE;
    - softmax scale 1/sqrt(d), causal mask j <= i, no bias or dropout;
    - query head h reads kv head floor(h / (Hq / Hkv));
    - weights use the nn.Linear layout [out_features, in_features];
    - lse is the natural-log log-sum-exp of the scaled scores, per head/row.

Precision: every step runs in float64 on the exact bf16 input values, with
no intermediate rounding.  The stated tolerances (bf16 inputs, fp32
accumulation) are measured against this plain definition: the oracle does not
model any storage precision of an implementation.
"""
from __future__ import annotations

import math
from typing import Callable, Optional, Sequence, Union

import numpy as np

ArrayOrRows = Union[np.ndarray, Callable[[int, int], np.ndarray]]


# ---------------------------------------------------------------- helpers --

def _rows(x: ArrayOrRows, lo: int, hi: int) -> np.ndarray:
    if callable(x):
        return np.asarray(x(lo, hi), dtype=np.float64)
    return np.asarray(x[lo:hi], dtype=np.float64)


def _nrows(x: ArrayOrRows, S: Optional[int]) -> int:
    if callable(x):
        assert S is not None
        return S
    return x.shape[0]


# ------------------------------------------------------------------- RoPE --

def rope_cos_sin(positions: np.ndarray, d: int, theta: float):
    """cos/sin of the RoPE angles pos * theta^(-2i/d), i = 0 .. d/2-1, in
    float64 (rotate-half RoPE of the Llama/Qwen3 attention layer)."""
    i = np.arange(d // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def apply_rope(v: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate each pair (v[i], v[i + d/2]) by the angle whose cos/sin are given."""
    h = v.shape[-1] // 2
    a, b = v[..., :h], v[..., h:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)


def apply_rope_transpose(g: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """The transpose (= inverse) of ``apply_rope``: rotation by minus the angle.
    This is the backward of RoPE."""
    h = g.shape[-1] // 2
    a, b = g[..., :h], g[..., h:]
    return np.concatenate([a * cos + b * sin, b * cos - a * sin], axis=-1)


# ---------------------------------------------------------------- RMSNorm --

def rms_norm(a: np.ndarray, gamma: Optional[np.ndarray], eps: float):
    """Per-row RMSNorm over the last (head) dimension: a / sqrt(mean(a^2)+eps)
    * gamma.  Returns (y, r) with r the per-row root."""
    r = np.sqrt(np.mean(a * a, axis=-1, keepdims=True) + eps)
    y = a / r
    if gamma is not None:
        y = y * gamma
    return y, r


def rms_norm_backward(dy: np.ndarray, a: np.ndarray, r: np.ndarray,
                      gamma: Optional[np.ndarray]):
    """Gradient of ``rms_norm`` w.r.t. its input and its gain.
    With yhat = a / r: d(yhat_i)/d(a_j) = delta_ij / r - a_i a_j / (n r^3),
    so da = (dyhat - yhat * mean(dyhat * yhat)) / r, dyhat = dy * gamma,
    dgamma = sum over rows of dy * yhat."""
    yhat = a / r
    dyhat = dy * gamma if gamma is not None else dy
    da = (dyhat - yhat * np.mean(dyhat * yhat, axis=-1, keepdims=True)) / r
    dgamma = np.sum(dy * yhat, axis=tuple(range(dy.ndim - 1)))
    return da, dgamma


# --------------------------------------------------------------- attention --

def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     q_pos: Optional[Sequence[int]] = None,
                     return_p: bool = False):
    """Causal softmax attention of one head.

    q: [n, d] queries at positions ``q_pos`` (default 0..n-1);
    k, v: [L, d] keys/values at positions 0..L-1 (L > max(q_pos)).
    s_ij = q_i . k_j / sqrt(d) for j <= pos_i, -inf otherwise;
    lse_i = log sum_j exp(s_ij); p_ij = exp(s_ij - lse_i); o_i = sum_j p_ij v_j.
    """
    n, d = q.shape
    if q_pos is None:
        q_pos = np.arange(n)
    q_pos = np.asarray(q_pos)
    L = int(q_pos.max()) + 1
    s = (q @ k[:L].T) / math.sqrt(d)
    mask = np.arange(L)[None, :] > q_pos[:, None]
    s[mask] = -np.inf
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=1, keepdims=True)
    lse = (np.log(z) + m)[:, 0]
    p = e / z
    o = p @ v[:L]
    if return_p:
        return o, lse, p
    return o, lse


# ------------------------------------------------------------------- layer --

def _head_proj(xr: np.ndarray, W: np.ndarray, head: int, d: int) -> np.ndarray:
    return xr @ np.asarray(W[head * d:(head + 1) * d], dtype=np.float64).T


def _qk_post(a, pos, geom, gamma):
    """RMSNorm (qk-norm layers only), then RoPE."""
    if geom.qk_norm:
        a, _ = rms_norm(a, gamma, geom.norm_eps)
    cos, sin = rope_cos_sin(pos, geom.d, geom.rope_theta)
    return apply_rope(a, cos, sin)


def project_kv(x: ArrayOrRows, Wk, Wv, geom, kv_head: int, upto: int,
               k_gamma=None, block: int = 65536):
    """K (normed, rotated) and V of one kv head for positions 0..upto-1,
    ``block`` rows of x at a time (RoPE takes each block's own positions)."""
    d = geom.d
    K = np.empty((upto, d))
    V = np.empty((upto, d))
    for lo in range(0, upto, block):
        hi = min(upto, lo + block)
        xr = _rows(x, lo, hi)
        K[lo:hi] = _qk_post(_head_proj(xr, Wk, kv_head, d), np.arange(lo, hi),
                            geom, k_gamma)
        V[lo:hi] = _head_proj(xr, Wv, kv_head, d)
    return K, V


def layer_forward(geom, x: ArrayOrRows, Wq, Wk, Wv, Wo, q_gamma=None,
                  k_gamma=None, rows: Optional[Sequence[int]] = None,
                  kv_block: int = 65536):
    """out = sum_h attn_h(x) Wo[:, h*d:(h+1)*d]^T for the query rows ``rows``
    (default: every row).  Returns dict(out [n, hidden], lse [Hq, n],
    o [Hq, n, d])."""
    S = _nrows(x, geom.S)
    rows = np.arange(S) if rows is None else np.asarray(sorted(rows))
    upto = int(rows.max()) + 1
    d, Hq, Hkv = geom.d, geom.Hq, geom.Hkv
    g = Hq // Hkv
    if callable(x):
        xq = np.concatenate([_rows(x, int(r), int(r) + 1) for r in rows])
    else:
        xq = np.asarray(x[rows], dtype=np.float64)
    Wo = np.asarray(Wo, dtype=np.float64)
    out = np.zeros((len(rows), Wo.shape[0]))
    lse = np.empty((Hq, len(rows)))
    o_all = np.empty((Hq, len(rows), d))
    for kvh in range(Hkv):
        K, V = project_kv(x, Wk, Wv, geom, kvh, upto, k_gamma, kv_block)
        for h in range(kvh * g, (kvh + 1) * g):
            q = _qk_post(_head_proj(xq, Wq, h, d), rows, geom, q_gamma)
            o, l = causal_attention(q, K, V, rows)
            lse[h] = l
            o_all[h] = o
            out += o @ Wo[:, h * d:(h + 1) * d].T
    return {"out": out, "lse": lse, "o": o_all}


def layer_backward(geom, x: np.ndarray, Wq, Wk, Wv, Wo, dout: np.ndarray,
                   q_gamma=None, k_gamma=None):
    """Gradients of L = sum(out * dout) w.r.t. x, Wq, Wk, Wv, Wo and the norm
    gains, by the chain rule in float64 over the full sequence (small S).

    Per head h (kv head g):  dWo_h = dout^T o_h;  do = dout Wo_h;
    dv += p^T do;  dp = do v^T;  D = rowsum(do * o);  ds = p * (dp - D);
    dq = ds k / sqrt(d);  dk += ds^T q / sqrt(d);  then RoPE transpose and the
    RMSNorm backward give the gradient of the projection outputs a = x W^T,
    and dW = da^T x, dx += da W.
    """
    x = np.asarray(x, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    Wq, Wk, Wv, Wo = (np.asarray(w, dtype=np.float64) for w in (Wq, Wk, Wv, Wo))
    S, d, Hq, Hkv = x.shape[0], geom.d, geom.Hq, geom.Hkv
    g = Hq // Hkv
    pos = np.arange(S)
    cos, sin = rope_cos_sin(pos, d, geom.rope_theta)
    scale = 1.0 / math.sqrt(d)
    dx = np.zeros_like(x)
    dWq, dWk, dWv, dWo = (np.zeros_like(w) for w in (Wq, Wk, Wv, Wo))
    dgq = np.zeros(d) if geom.qk_norm else None
    dgk = np.zeros(d) if geom.qk_norm else None

    def pre(a, gamma):
        if geom.qk_norm:
            y, r = rms_norm(a, gamma, geom.norm_eps)
        else:
            y, r = a, None
        return apply_rope(y, cos, sin), r

    def post_grad(dqk, a, r, gamma):
        dy = apply_rope_transpose(dqk, cos, sin)
        if geom.qk_norm:
            return rms_norm_backward(dy, a, r, gamma)
        return dy, None

    for kvh in range(Hkv):
        sl = slice(kvh * d, (kvh + 1) * d)
        ak = x @ Wk[sl].T
        v = x @ Wv[sl].T
        k, rk = pre(ak, k_gamma)
        dk = np.zeros((S, d))
        dv = np.zeros((S, d))
        for h in range(kvh * g, (kvh + 1) * g):
            hs = slice(h * d, (h + 1) * d)
            aq = x @ Wq[hs].T
            q, rq = pre(aq, q_gamma)
            o, _, p = causal_attention(q, k, v, return_p=True)
            dWo[:, hs] = dout.T @ o
            do = dout @ Wo[:, hs]
            dv += p.T @ do
            dp = do @ v.T
            D = np.sum(do * o, axis=1, keepdims=True)
            ds = p * (dp - D)
            dq = ds @ k * scale
            dk += ds.T @ q * scale
            daq, dgam = post_grad(dq, aq, rq, q_gamma)
            if dgq is not None:
                dgq += dgam
            dWq[hs] = daq.T @ x
            dx += daq @ Wq[hs]
        dak, dgam = post_grad(dk, ak, rk, k_gamma)
        if dgk is not None:
            dgk += dgam
        dWk[sl] = dak.T @ x
        dWv[sl] = dv.T @ x
        dx += dak @ Wk[sl] + dv @ Wv[sl]
    return {"dx": dx, "dWq": dWq, "dWk": dWk, "dWv": dWv, "dWo": dWo,
            "dq_gamma": dgq, "dk_gamma": dgk}


def layer_backward_tail(geom, x: ArrayOrRows, Wq, Wk, Wv, Wo, dout_tail: np.ndarray,
                        n_tail: int, q_gamma=None, k_gamma=None):
    """dx for the last ``n_tail`` rows of the sequence, exactly (same chain
    rule as ``layer_backward``), without the full-sequence cost.

    Row t >= S - n_tail of dx collects dq_t (which needs P and dP of row t
    against every key j <= t, i.e. the full K and V) and dk_t, dv_t (which
    need only the queries i >= t, all inside the tail).  ``dout_tail`` holds
    rows S - n_tail .. S - 1 of dout.  Returns dx_tail [n_tail, hidden].
    """
    S = _nrows(x, geom.S)
    d, Hq, Hkv = geom.d, geom.Hq, geom.Hkv
    g = Hq // Hkv
    t0 = S - n_tail
    rows = np.arange(t0, S)
    Wq, Wk, Wv, Wo = (np.asarray(w, dtype=np.float64) for w in (Wq, Wk, Wv, Wo))
    dout_tail = np.asarray(dout_tail, dtype=np.float64)
    xt = _rows(x, t0, S)
    cos_t, sin_t = rope_cos_sin(rows, d, geom.rope_theta)
    scale = 1.0 / math.sqrt(d)

    def pre(a, gamma):
        if geom.qk_norm:
            y, r = rms_norm(a, gamma, geom.norm_eps)
        else:
            y, r = a, None
        return apply_rope(y, cos_t, sin_t), r

    def post_grad(dqk, a, r, gamma):
        dy = apply_rope_transpose(dqk, cos_t, sin_t)
        if geom.qk_norm:
            return rms_norm_backward(dy, a, r, gamma)[0]
        return dy

    dx = np.zeros((n_tail, Wq.shape[1]))
    for kvh in range(Hkv):
        sl = slice(kvh * d, (kvh + 1) * d)
        K, V = project_kv(x, Wk, Wv, geom, kvh, S, k_gamma)
        ak_t = xt @ Wk[sl].T
        dk_t = np.zeros((n_tail, d))
        dv_t = np.zeros((n_tail, d))
        for h in range(kvh * g, (kvh + 1) * g):
            hs = slice(h * d, (h + 1) * d)
            aq_t = xt @ Wq[hs].T
            q_t, rq = pre(aq_t, q_gamma)
            o_t, _, p_t = causal_attention(q_t, K, V, rows, return_p=True)   # [n, S]
            do_t = dout_tail @ Wo[:, hs]
            dp_t = do_t @ V.T
            D = np.sum(do_t * o_t, axis=1, keepdims=True)
            ds_t = p_t * (dp_t - D)                                          # [n, S]
            dq_t = ds_t @ K * scale
            # keys in the tail receive only tail queries (causal)
            dk_t += ds_t[:, t0:].T @ q_t * scale
            dv_t += p_t[:, t0:].T @ do_t
            dx += post_grad(dq_t, aq_t, rq, q_gamma) @ Wq[hs]
        _, rk = pre(ak_t, k_gamma)
        dx += post_grad(dk_t, ak_t, rk, k_gamma) @ Wk[sl] + dv_t @ Wv[sl]
    return dx


def layer_backward_key_rows(geom, x: ArrayOrRows, Wq, Wk, Wv, Wo, q_rows: Sequence[int],
                            dout_rows: np.ndarray, key_rows: Sequence[int], q_gamma=None,
                            k_gamma=None):
    """dx of the early rows ``key_rows`` when the upstream gradient is zero
    everywhere except on the query rows ``q_rows`` (``dout_rows`` holds those
    rows of dout), every key row before every query row.  Same chain rule as
    ``layer_backward``.

    A key row j before every gradient-carrying query has dO_j = 0, so its dq
    vanishes and dx_j = dk_j Wk + dv_j Wv with dk_j = sum_i ds_ij q_i / sqrt(d)
    and dv_j = sum_i p_ij do_i over the query rows i only.  Each of those needs
    p_i and o_i over its full causal row (K, V of positions 0..i), but not the
    other queries of the sequence: the longest dk / dv sums of a
    million-token layer (those of its first keys) stay within reach.
    Returns dx_rows [len(key_rows), hidden]."""
    q_rows = np.asarray(sorted(q_rows))
    key_rows = np.asarray(sorted(key_rows))
    assert key_rows.max() < q_rows.min()
    d, Hq, Hkv = geom.d, geom.Hq, geom.Hkv
    g = Hq // Hkv
    Wq, Wk, Wv, Wo = (np.asarray(w, dtype=np.float64) for w in (Wq, Wk, Wv, Wo))
    dout_rows = np.asarray(dout_rows, dtype=np.float64)
    upto = int(q_rows.max()) + 1
    scale = 1.0 / math.sqrt(d)
    xq = np.concatenate([_rows(x, int(r), int(r) + 1) for r in q_rows])
    xk = np.concatenate([_rows(x, int(r), int(r) + 1) for r in key_rows])
    cos_k, sin_k = rope_cos_sin(key_rows, d, geom.rope_theta)
    dx = np.zeros((len(key_rows), Wq.shape[1]))
    for kvh in range(Hkv):
        sl = slice(kvh * d, (kvh + 1) * d)
        K, V = project_kv(x, Wk, Wv, geom, kvh, upto, k_gamma)
        dk = np.zeros((len(key_rows), d))
        dv = np.zeros((len(key_rows), d))
        for h in range(kvh * g, (kvh + 1) * g):
            hs = slice(h * d, (h + 1) * d)
            q = _qk_post(_head_proj(xq, Wq, h, d), q_rows, geom, q_gamma)
            o, _, p = causal_attention(q, K, V, q_rows, return_p=True)    # p [nq, upto]
            do = dout_rows @ Wo[:, hs]
            D = np.sum(do * o, axis=1, keepdims=True)
            pk = p[:, key_rows]
            ds = pk * (do @ V[key_rows].T - D)
            dk += ds.T @ q * scale
            dv += pk.T @ do
        ak = xk @ Wk[sl].T
        if geom.qk_norm:
            _, rk = rms_norm(ak, k_gamma, geom.norm_eps)
            dak = rms_norm_backward(apply_rope_transpose(dk, cos_k, sin_k), ak, rk, k_gamma)[0]
        else:
            dak = apply_rope_transpose(dk, cos_k, sin_k)
        dx += dak @ Wk[sl] + dv @ Wv[sl]
    return dx


def layer_loss(geom, x, Wq, Wk, Wv, Wo, dout, q_gamma=None, k_gamma=None):
    """Scalar L = sum(out * dout); the function whose gradient
    ``layer_backward`` returns (used by the finite-difference pin)."""
    out = layer_forward(geom, x, Wq, Wk, Wv, Wo, q_gamma, k_gamma)["out"]
    return float(np.sum(out * np.asarray(dout, dtype=np.float64)))
