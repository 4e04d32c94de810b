"""GPU parity at the full sizes of the five workloads, in the launch
configurations the benchmark times, against the plain float64 oracle.

A million-token layer is beyond the oracle, so the forward is checked on a
seeded sample of 256 query rows per head (the same rows for every head), and
so is the forward with the fused Wo-slice accumulate in the benchmark's chunk
size (its lse bit-identical to the separate forward's).  The
backward is checked on complete dx rows: with the upstream gradient set to
zero after row T, causality makes dx of the rows up to T depend only on the
prefix [0, T] of the sequence, which the oracle's tail backward covers (the
query rows up to T against the full prefix K and V, and every later query of
that prefix for their dk, dv); the rows after T must come out exactly zero.
T = S - 1 checks the last rows and T = S/2 the middle of the sequence.  The
first rows, whose dk and dv sum over every later query (the backward's
longest accumulations: up to 1M tokens one CTA walks all the queries of a key
tile, 65536 tensor-core accumulation steps at 1M), are checked
with the upstream gradient non-zero on three windows of query rows only: right
after the checked rows, in the middle and at the end.  The weight and gain
gradients are checked in full on the same geometries at 8192 tokens, where
the whole oracle backward is feasible."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import WORKLOADS, make_inputs, sample_rows
from tests._util import f64, assert_close, LSE_ABS, GAIN_MAX_REL, GAIN_MEAN_REL

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_ROWS = 256


def _gpu_fwd(u, w, ch, t):
    sh = u.Shape.of(w, ch)
    out = torch.empty(w.S, w.hidden, device="cuda")
    lse = torch.empty(w.Hq, w.S, device="cuda")
    o = torch.empty(w.S, w.Hq * w.d, device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(u.workspace_bytes(sh, 0), dtype=torch.uint8, device="cuda")
    u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
               t.get("q_gamma"), t.get("k_gamma"), o)
    torch.cuda.synchronize()
    assert u.last_error() == 0
    return out, lse, o


def _gpu_fwd_fused(u, w, ch, t):
    sh = u.Shape.of(w, ch)
    out = torch.empty(w.S, w.hidden, device="cuda")
    lse = torch.empty(w.Hq, w.S, device="cuda")
    ws = torch.empty(u.workspace_bytes(sh, 3), dtype=torch.uint8, device="cuda")
    u.attn_fwd_fused(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
                     t.get("q_gamma"), t.get("k_gamma"))
    torch.cuda.synchronize()
    assert u.last_error() == 0
    return out, lse


@pytest.mark.parametrize("name", ["llama3.2-3b-s65536", "llama3-8b-rank-s1m",
                                  "llama3-8b-rank-s5m", "qwen3-32b-rank-s1m"])
def test_forward_sampled_rows_at_full_size(name):
    import headwise_chunked_attention_gb300 as u
    w = WORKLOADS[name]
    t = make_inputs(w, seed=0, device="cuda", norm_gains="random")
    rows = sample_rows(w.S, N_ROWS)
    got = {}
    for ch in w.chunk_heads:
        out, lse, o = _gpu_fwd(u, w, ch, t)
        got[ch] = (f64(out[rows]), f64(lse[:, rows]),
                   f64(o[rows]).reshape(len(rows), w.Hq, w.d).transpose(1, 0, 2))
        del out, lse, o
        torch.cuda.empty_cache()
    # the fused forward (Wo-slice accumulate inside the attention kernel) in
    # the benchmark's chunk size
    ch0 = w.chunk_heads[0]
    out, lse = _gpu_fwd_fused(u, w, ch0, t)
    fused = (f64(out[rows]), f64(lse[:, rows]))
    del out, lse
    torch.cuda.empty_cache()
    xg = t["x"]
    a = {k: f64(v) for k, v in t.items() if k != "x"}
    ref = O.layer_forward(w, lambda lo, hi: f64(xg[lo:hi]), a["Wq"], a["Wk"], a["Wv"],
                          a["Wo"], a.get("q_gamma"), a.get("k_gamma"), rows=rows)
    for ch, (out, lse, o) in got.items():
        assert_close(out, ref["out"], f"{name} out ch={ch}")
        assert_close(o, ref["o"], f"{name} attention output ch={ch}")
        dl = np.abs(lse - ref["lse"]).max()
        assert dl <= LSE_ABS, f"{name} lse ch={ch}: {dl:.2e}"
    assert_close(fused[0], ref["out"], f"{name} fused out ch={ch0}")
    assert np.array_equal(fused[1], got[ch0][1]), f"{name} fused lse ch={ch0}"
    # the per-head attention output does not depend on the chunk size
    first = got[w.chunk_heads[0]][2]
    for ch in w.chunk_heads[1:]:
        assert np.array_equal(got[ch][2], first), ch


def _gpu_fwd_bwd(u, w, ch, t, dout, saved_o):
    sh = u.Shape.of(w, ch)
    out = torch.empty(w.S, w.hidden, device="cuda")
    lse = torch.empty(w.Hq, w.S, device="cuda")
    ws = torch.empty(u.workspace_bytes(sh, 1), dtype=torch.uint8, device="cuda")
    o = torch.empty(w.S, w.Hq * w.d, device="cuda", dtype=torch.bfloat16) if saved_o else None
    u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
               t.get("q_gamma"), t.get("k_gamma"), o)
    del out
    g = {n: torch.empty(t[s].shape, device="cuda") for n, s in
         [("dx", "x"), ("dWq", "Wq"), ("dWk", "Wk"), ("dWv", "Wv"), ("dWo", "Wo")]}
    dqg = torch.empty(w.d, device="cuda") if w.qk_norm else None
    dkg = torch.empty(w.d, device="cuda") if w.qk_norm else None
    u.attn_bwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], dout, lse, g["dx"],
               g["dWq"], g["dWk"], g["dWv"], g["dWo"], ws, t.get("q_gamma"), t.get("k_gamma"),
               dqg, dkg, attn_o=o)
    torch.cuda.synchronize()
    assert u.last_error() == 0
    g["dq_gamma"], g["dk_gamma"] = dqg, dkg
    return g


@pytest.mark.parametrize("name,saved_o,where", [("llama3-8b-rank-s1m", False, "end"),
                                                ("llama3-8b-rank-s1m", False, "middle"),
                                                ("qwen3-32b-rank-s1m", False, "middle"),
                                                ("llama3-8b-rank-s1m", True, "middle")])
def test_backward_dx_rows_at_full_size(name, saved_o, where):
    # saved_o: the backward takes the forward's attention output
    # (upipe_attn_bwd_saved_o) instead of recomputing it chunk by chunk
    import headwise_chunked_attention_gb300 as u
    w = WORKLOADS[name]
    ch = w.chunk_heads[0]
    t = make_inputs(w, seed=1, device="cuda", with_grad=True, norm_gains="random")
    T = w.S - 1 if where == "end" else w.S // 2 + N_ROWS // 2   # last row with a gradient
    dout = t["dout"].clone()
    dout[T + 1:] = 0
    g = _gpu_fwd_bwd(u, w, ch, t, dout, saved_o)
    for k, v in g.items():
        assert v is None or torch.isfinite(v).all(), k
    # causality: no row after T receives a gradient
    assert torch.count_nonzero(g["dx"][T + 1:]).item() == 0
    n = N_ROWS
    dx_rows = f64(g["dx"][T + 1 - n:T + 1])
    del g
    xg = t["x"]
    a = {k: f64(v) for k, v in t.items() if k not in ("x", "dout")}
    wp = w.with_(S=T + 1)          # the prefix [0, T] of the sequence
    ref = O.layer_backward_tail(wp, lambda lo, hi: f64(xg[lo:hi]), a["Wq"], a["Wk"], a["Wv"],
                                a["Wo"], f64(dout[T + 1 - n:T + 1]), n, a.get("q_gamma"),
                                a.get("k_gamma"))
    assert_close(dx_rows, ref, f"{name} dx rows {T + 1 - n}..{T}")


@pytest.mark.parametrize("name", ["llama3-8b-rank-s1m", "qwen3-32b-rank-s1m"])
def test_backward_weight_gradients_full_geometry(name):
    # every gradient of the layer (dx, dWq, dWk, dWv, dWo and the RMSNorm
    # gains) in full, on the rank geometry at 8192 tokens, every chunk size
    import headwise_chunked_attention_gb300 as u
    w = WORKLOADS[name].with_(S=8192)
    inp = make_inputs(w, seed=2, with_grad=True, norm_gains="random")
    t = {k: v.to("cuda") for k, v in inp.items()}
    a = {k: f64(v) for k, v in inp.items()}
    ref = O.layer_backward(w, a["x"], a["Wq"], a["Wk"], a["Wv"], a["Wo"], a["dout"],
                           a.get("q_gamma"), a.get("k_gamma"))
    for ch in w.chunk_heads:
        g = _gpu_fwd_bwd(u, w, ch, t, t["dout"], False)
        for nm in ("dx", "dWq", "dWk", "dWv", "dWo"):
            assert_close(f64(g[nm]), ref[nm], f"{name} {nm} ch={ch}")
        if w.qk_norm:
            for nm in ("dq_gamma", "dk_gamma"):
                assert_close(f64(g[nm]), ref[nm], f"{name} {nm} ch={ch}",
                             GAIN_MAX_REL, GAIN_MEAN_REL)


@pytest.mark.parametrize("name", ["llama3-8b-rank-s1m", "qwen3-32b-rank-s1m"])
def test_backward_first_rows_at_full_size(name):
    import headwise_chunked_attention_gb300 as u
    w = WORKLOADS[name]
    ch = w.chunk_heads[0]
    t = make_inputs(w, seed=3, device="cuda", with_grad=True, norm_gains="random")
    n = N_ROWS
    q_rows = np.concatenate([np.arange(n, n + 128), np.arange(w.S // 2 - 64, w.S // 2 + 64),
                             np.arange(w.S - 128, w.S)])
    idx = torch.from_numpy(q_rows).to("cuda")
    dout = torch.zeros_like(t["dout"])
    dout[idx] = t["dout"][idx]
    g = _gpu_fwd_bwd(u, w, ch, t, dout, False)
    for k, v in g.items():
        assert v is None or torch.isfinite(v).all(), k
    dx_rows = f64(g["dx"][:n])
    del g
    xg = t["x"]
    a = {k: f64(v) for k, v in t.items() if k not in ("x", "dout")}
    ref = O.layer_backward_key_rows(w, lambda lo, hi: f64(xg[lo:hi]), a["Wq"], a["Wk"],
                                    a["Wv"], a["Wo"], q_rows, f64(dout[idx]), np.arange(n),
                                    a.get("q_gamma"), a.get("k_gamma"))
    assert_close(dx_rows, ref, f"{name} dx rows 0..{n - 1}")


def test_backward_first_rows_at_5m():
    # Past 1M tokens a key tile's query walk is split across CTAs (segments of
    # 8192 sub-tiles, 10 for the first key tiles at 5M), each adding its dK/dV
    # partial: the first rows' dx, whose dk and dv sum over all 5M queries,
    # checked against the oracle with dout non-zero on three windows.  x,
    # dout, dx and out need ~190 GB of the device.
    import gc
    import headwise_chunked_attention_gb300 as u
    # the earlier tests' blocks stay in torch's cache unless released first
    gc.collect()
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < 200e9:
        pytest.skip(f"needs ~190 GB of free device memory, {free / 1e9:.0f} GB free")
    w = WORKLOADS["llama3-8b-rank-s5m"]
    t = make_inputs(w, seed=3, device="cuda")
    n = 192
    q_rows = np.concatenate([np.arange(n, n + 64), np.arange(w.S // 2 - 32, w.S // 2 + 32),
                             np.arange(w.S - 64, w.S)])
    idx = torch.from_numpy(q_rows).to("cuda")
    dout = torch.zeros(w.S, w.hidden, device="cuda", dtype=torch.bfloat16)
    gen = torch.Generator(device="cuda").manual_seed(7)
    dout[idx] = torch.randn(len(q_rows), w.hidden, device="cuda", generator=gen).to(torch.bfloat16)
    sh = u.Shape.of(w, 1)
    ws = torch.empty(u.workspace_bytes(sh, 1), dtype=torch.uint8, device="cuda")
    lse = torch.empty(w.Hq, w.S, device="cuda")
    out = torch.empty(w.S, w.hidden, device="cuda")
    u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws)
    torch.cuda.synchronize()
    del out
    torch.cuda.empty_cache()
    g = {n_: torch.empty(t[s].shape, device="cuda") for n_, s in
         [("dx", "x"), ("dWq", "Wq"), ("dWk", "Wk"), ("dWv", "Wv"), ("dWo", "Wo")]}
    u.attn_bwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], dout, lse, g["dx"], g["dWq"],
               g["dWk"], g["dWv"], g["dWo"], ws)
    torch.cuda.synchronize()
    assert u.last_error() == 0
    for k, v in g.items():           # in blocks: a whole-tensor isfinite needs 80 GB more
        flat = v.view(-1)
        for lo in range(0, flat.numel(), 1 << 28):
            assert torch.isfinite(flat[lo:lo + (1 << 28)]).all().item(), k
    dx_rows = f64(g["dx"][:n])
    del g, ws
    torch.cuda.empty_cache()
    xg = t["x"]
    a = {k: f64(v) for k, v in t.items() if k != "x"}
    ref = O.layer_backward_key_rows(w, lambda lo, hi: f64(xg[lo:hi]), a["Wq"], a["Wk"], a["Wv"],
                                    a["Wo"], q_rows, f64(dout[idx]), np.arange(n))
    assert_close(dx_rows, ref, "5M dx rows 0..191")
