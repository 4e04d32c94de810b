"""GPU parity of the forward whose attention kernel adds each head's partial
result o_h Wo[:, h*d:(h+1)*d]^T into out itself (upipe_attn_fwd_fused,
through the C ABI), against the float64 oracle and against upipe_attn_fwd on
the same seeded inputs.  Both compute the same softmax in the same kernel
code, so lse must be bit-identical; out differs only by the order of its fp32
additions (per head in the fused kernel, per chunk in the separate GEMM)."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import WORKLOADS, Workload, make_inputs
from tests._util import f64, assert_close, LSE_ABS
from tests._guard import guarded

pytestmark = pytest.mark.gpu

# out of the fused forward against out of the separate Wo GEMM: fp32
# summation order only
ORDER_MAX_REL, ORDER_MEAN_REL = 1e-4, 1e-5


def U():
    import headwise_chunked_attention_gb300 as mod
    mod.lib()
    return mod


def run_fused(w, ch, t, expect_error=0):
    # out starts as NaN (the call must overwrite every element); out, lse and
    # the workspace sit inside guard margins that must come back untouched
    u = U()
    shape = u.Shape.of(w, ch)
    g = {"out": guarded((w.S, w.hidden), fill=float("nan")),
         "lse": guarded((w.Hq, w.S), fill=float("nan")),
         "workspace": guarded((u.workspace_bytes(shape, 3),), torch.uint8)}
    out, lse, ws = g["out"].t, g["lse"].t, g["workspace"].t
    u.attn_fwd_fused(shape, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
                     t.get("q_gamma"), t.get("k_gamma"))
    torch.cuda.synchronize()
    rc = u.last_error()
    assert rc == expect_error, f"device error word {rc}, expected {expect_error}"
    for name, b in g.items():
        b.check(name)
    return out, lse


def run_unfused(w, ch, t):
    u = U()
    shape = u.Shape.of(w, ch)
    out = torch.empty(w.S, w.hidden, device="cuda")
    lse = torch.empty(w.Hq, w.S, device="cuda")
    ws = torch.empty(u.workspace_bytes(shape, 0), dtype=torch.uint8, device="cuda")
    u.attn_fwd(shape, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
               t.get("q_gamma"), t.get("k_gamma"))
    torch.cuda.synchronize()
    rc = u.last_error()
    assert rc == 0, f"device error word {rc}"
    return out, lse


def oracle_fwd(w, inp):
    a = {k: f64(v) for k, v in inp.items()}
    return O.layer_forward(w, a["x"], a["Wq"], a["Wk"], a["Wv"], a["Wo"],
                           a.get("q_gamma"), a.get("k_gamma"))


def check(w, ch, inp, ref):
    t = {k: v.cuda() for k, v in inp.items()}
    out, lse = run_fused(w, ch, t)
    assert_close(f64(out), ref["out"], f"{w.name} out ch={ch}")
    dl = np.abs(f64(lse) - ref["lse"]).max()
    assert dl <= LSE_ABS, f"{w.name} lse ch={ch}: {dl:.3e}"
    out_u, lse_u = run_unfused(w, ch, t)
    assert torch.equal(lse, lse_u), f"{w.name} lse ch={ch} differs from upipe_attn_fwd"
    assert_close(f64(out), f64(out_u), f"{w.name} out ch={ch} vs upipe_attn_fwd",
                 ORDER_MAX_REL, ORDER_MEAN_REL)


SMALL = [
    # d = 64, hidden 256: two 128-column blocks of out per CTA
    WORKLOADS["tiny-s2048"],
    # d = 128 GQA with one kv head, ragged S, chunks below and at the group
    # size (g = 4: chunk_heads 1, 2 < g, 4 = g)
    Workload("d128-s1000", S=1000, hidden=256, Hq=4, Hkv=1, d=128,
             chunk_heads=(1, 2, 4), rope_theta=5e5),
    # qk-norm geometry, hidden 384 (three column blocks), chunks spanning
    # several kv groups (g = 2: chunk_heads 4 > g)
    Workload("d128-qknorm-s777", S=777, hidden=384, Hq=4, Hkv=2, d=128,
             chunk_heads=(1, 2, 4), rope_theta=1e6, qk_norm=True),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_fused_forward_matches_oracle(w):
    inp = make_inputs(w, seed=0, norm_gains="random")
    ref = oracle_fwd(w, inp)
    for ch in w.chunk_heads:
        check(w, ch, inp, ref)


@pytest.mark.parametrize("S", [1, 2, 127, 128, 129, 255, 256, 257, 300])
def test_fused_forward_ragged_and_tiny_lengths(S):
    # the last 256-row block is partly (or, for the second 128-row tile, all)
    # past S: the reduce-adds of those rows are dropped at the tensor's edge
    w = Workload("ragged", S=S, hidden=256, Hq=2, Hkv=1, d=128, chunk_heads=(1,),
                 rope_theta=1e4)
    inp = make_inputs(w, seed=S)
    check(w, 1, inp, oracle_fwd(w, inp))


def test_fused_forward_many_heads_and_wide_out():
    # Llama-3.2-3B geometry (24 query heads in 8 groups, hidden 3072: 24
    # column blocks of out per CTA) at 4096 tokens, every chunk size the
    # benchmark sweeps: all heads' CTAs add into the same rows of out
    w = WORKLOADS["llama3.2-3b-s65536"].with_(S=4096)
    inp = make_inputs(w, seed=1)
    t = {k: v.cuda() for k, v in inp.items()}
    for ch in w.chunk_heads:
        out, lse = run_fused(w, ch, t)
        out_u, lse_u = run_unfused(w, ch, t)
        assert torch.equal(lse, lse_u), ch
        assert_close(f64(out), f64(out_u), f"out ch={ch} vs upipe_attn_fwd",
                     ORDER_MAX_REL, ORDER_MEAN_REL)


def test_fused_forward_folds_long_rows():
    # past 65536 keys the attention folds each long row's O out of TMEM into
    # per-SM fp32 rows every 512 KV tiles; the fused tail then takes o from
    # the folded rows plus TMEM, as the separate forward does (d = 64)
    w = Workload("d64-s70000", S=70000, hidden=256, Hq=1, Hkv=1, d=64, chunk_heads=(1,),
                 rope_theta=1e4)
    t = {k: v.cuda() for k, v in make_inputs(w, seed=6).items()}
    out, lse = run_fused(w, 1, t)
    out_u, lse_u = run_unfused(w, 1, t)
    assert torch.equal(lse, lse_u)
    assert_close(f64(out), f64(out_u), "out vs upipe_attn_fwd", ORDER_MAX_REL, ORDER_MEAN_REL)


def test_fused_forward_reports_projection_range_error():
    # a projected value beyond fp16's range is reported, as in upipe_attn_fwd
    w = Workload("range", S=300, hidden=256, Hq=2, Hkv=1, d=64, chunk_heads=(1,),
                 rope_theta=1e4)
    inp = make_inputs(w, seed=4)
    big = dict(inp, x=(inp["x"].float() * 2.0 ** 17).to(torch.bfloat16))
    run_fused(w, 1, {k: v.cuda() for k, v in big.items()}, expect_error=U().ERR_RANGE)
    # the next call starts with a clear error word
    run_fused(w, 1, {k: v.cuda() for k, v in inp.items()})
