"""GPU parity at the full sizes of the five workloads, in the launch
configurations the benchmark times: the oracle cannot run a whole
million-token layer, so it checks a seeded sample of query rows (the same rows
for every head) exactly, and for the backward the last rows of the sequence,
whose dx needs only tail queries plus the full K and V."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import WORKLOADS, make_inputs, sample_rows
from tests._util import f64, assert_close, LSE_ABS

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_ROWS = 64


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
    xg = t["x"]
    a = {k: f64(v) for k, v in t.items() if k != "x"}
    ref = O.layer_forward(w, lambda lo, hi: f64(xg[lo:hi]), a["Wq"], a["Wk"], a["Wv"],
                          a["Wo"], a.get("q_gamma"), a.get("k_gamma"), rows=rows,
                          store_dtype="bf16")
    for ch, (out, lse, o) in got.items():
        assert_close(out, ref["out"], f"{name} out ch={ch}")
        assert_close(o, ref["o"], f"{name} attention output ch={ch}")
        dl = np.abs(lse - ref["lse"]).max()
        assert dl <= LSE_ABS, f"{name} lse ch={ch}: {dl:.2e}"
    # the per-head attention output does not depend on the chunk size
    first = got[w.chunk_heads[0]][2]
    for ch in w.chunk_heads[1:]:
        assert np.array_equal(got[ch][2], first), ch


@pytest.mark.parametrize("name,saved_o", [("llama3-8b-rank-s1m", False),
                                          ("qwen3-32b-rank-s1m", False),
                                          ("llama3-8b-rank-s1m", True)])
def test_backward_tail_rows_at_full_size(name, saved_o):
    # saved_o: the backward takes the forward's attention output
    # (upipe_attn_bwd_saved_o) instead of recomputing it chunk by chunk
    import headwise_chunked_attention_gb300 as u
    w = WORKLOADS[name]
    ch = w.chunk_heads[0]
    t = make_inputs(w, seed=1, device="cuda", with_grad=True, norm_gains="random")
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
    u.attn_bwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], t["dout"], lse, g["dx"],
               g["dWq"], g["dWk"], g["dWv"], g["dWo"], ws, t.get("q_gamma"), t.get("k_gamma"),
               dqg, dkg, attn_o=o)
    torch.cuda.synchronize()
    assert u.last_error() == 0
    n = N_ROWS
    dx_tail = f64(g["dx"][w.S - n:])
    for k in list(g):
        assert torch.isfinite(g[k]).all(), k
    xg = t["x"]
    a = {k: f64(v) for k, v in t.items() if k not in ("x", "dout")}
    ref = O.layer_backward_tail(w, lambda lo, hi: f64(xg[lo:hi]), a["Wq"], a["Wk"], a["Wv"],
                                a["Wo"], f64(t["dout"][w.S - n:]), n, a.get("q_gamma"),
                                a.get("k_gamma"), store_dtype="bf16")
    assert_close(dx_tail, ref, f"{name} dx tail rows")
