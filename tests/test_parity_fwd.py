"""GPU forward parity: the CUDA path (through the C ABI) against the float64
oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import WORKLOADS, Workload, make_inputs, sample_rows
from tests._util import f64, assert_close, LSE_ABS
from tests._guard import guarded

pytestmark = pytest.mark.gpu


def U():
    import headwise_chunked_attention_gb300 as mod
    mod.lib()
    return mod


def run_fwd(w, ch, inp, debug=True, expect_error=0):
    # out, lse, attn_o and the workspace sit inside guard margins that must
    # come back untouched
    u = U()
    dev = "cuda"
    t = {k: v.to(dev) for k, v in inp.items()}
    shape = u.Shape.of(w, ch)
    g = {"out": guarded((w.S, w.hidden)), "lse": guarded((w.Hq, w.S)),
         "workspace": guarded((u.workspace_bytes(shape, 0),), torch.uint8)}
    if debug:
        g["attn_o"] = guarded((w.S, w.Hq * w.d), torch.bfloat16)
    out, lse, ws = g["out"].t, g["lse"].t, g["workspace"].t
    o = g["attn_o"].t if debug else None
    u.attn_fwd(shape, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
               t.get("q_gamma"), t.get("k_gamma"), o)
    torch.cuda.synchronize()
    rc = u.last_error()
    assert rc == expect_error, f"device error word {rc}, expected {expect_error}"
    for name, b in g.items():
        b.check(name)
    return out, lse, o


def oracle_fwd(w, inp, rows=None):
    a = {k: f64(v) for k, v in inp.items()}
    return O.layer_forward(w, a["x"], a["Wq"], a["Wk"], a["Wv"], a["Wo"],
                           a.get("q_gamma"), a.get("k_gamma"), rows=rows)


def check_full(w, ch, inp):
    # against the plain float64 definition: no rounding of any intermediate
    out, lse, o = run_fwd(w, ch, inp)
    ref = oracle_fwd(w, inp)
    assert_close(f64(out), ref["out"], "out")
    o_g = f64(o).reshape(w.S, w.Hq, w.d).transpose(1, 0, 2)
    assert_close(o_g, ref["o"], "attention output")
    dl = np.abs(f64(lse) - ref["lse"]).max()
    assert dl <= LSE_ABS, f"lse max abs err {dl:.3e}"
    return out, lse, o


SMALL = [
    WORKLOADS["tiny-s2048"],
    # d=128 GQA, one kv head, ragged S, several chunk sizes
    Workload("d128-s1000", S=1000, hidden=256, Hq=4, Hkv=1, d=128,
             chunk_heads=(1, 2, 4), rope_theta=5e5),
    Workload("d128-qknorm-s777", S=777, hidden=384, Hq=4, Hkv=2, d=128,
             chunk_heads=(1, 2, 4), rope_theta=1e6, qk_norm=True),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_forward_matches_oracle(w):
    inp = make_inputs(w, seed=0, norm_gains="random")
    for ch in w.chunk_heads:
        check_full(w, ch, inp)


@pytest.mark.parametrize("S", [1, 2, 127, 128, 129, 255, 256, 257, 300])
def test_forward_ragged_and_tiny_lengths(S):
    w = Workload("ragged", S=S, hidden=256, Hq=2, Hkv=1, d=128, chunk_heads=(1,),
                 rope_theta=1e4)
    check_full(w, 1, make_inputs(w, seed=S))


def test_per_head_output_bit_identical_across_chunk_sizes():
    w = Workload("chunks", S=1536, hidden=512, Hq=8, Hkv=2, d=128,
                 chunk_heads=(1, 2, 4, 8), rope_theta=5e5, qk_norm=True)
    inp = make_inputs(w, seed=3, norm_gains="random")
    outs = {}
    for ch in w.chunk_heads:
        _, lse, o = run_fwd(w, ch, inp)
        outs[ch] = (o.cpu(), lse.cpu())
    o1, l1 = outs[1]
    for ch in w.chunk_heads[1:]:
        assert torch.equal(outs[ch][0].view(torch.int16), o1.view(torch.int16)), ch
        assert torch.equal(outs[ch][1], l1), ch


def test_chunked_out_close_to_unchunked():
    w = WORKLOADS["llama3.2-3b-s65536"].with_(S=4096)
    inp = make_inputs(w, seed=1)
    ref, _, _ = run_fwd(w, 24, inp, debug=False)
    for ch in (3, 6):
        out, _, _ = run_fwd(w, ch, inp, debug=False)
        assert_close(f64(out), f64(ref), f"out ch={ch} vs ch=24", 1e-3, 1e-4)


def _late_max_inputs(w, scale):
    inp = make_inputs(w, seed=11)
    x = inp["x"].float()
    x[900:1020] *= scale
    inp["x"] = x.to(torch.bfloat16)
    return inp


LATE = Workload("late-max", S=1500, hidden=256, Hq=2, Hkv=1, d=128, chunk_heads=(1, 2),
                rope_theta=1e4)


def test_forward_row_max_growing_late_in_rows():
    # The hidden rows of keys 900..1019 are scaled by 2, so their scores
    # against every later query are about twice as large: the row max of
    # those queries grows by up to ~8 powers of two inside the eighth KV tile,
    # and the kernel either keeps its running max (growth within the p <= 128
    # allowance) or takes the tile's max and rescales O and l mid-row.  Every
    # row is compared with the plain float64 layer: out and O at the layer's
    # bounds, lse within 1e-3 outside the scaled block.  Inside the block q and
    # k are both doubled, so its scores are 4 times the unit-scale ones and
    # the fp16 rounding of q and k moves them 4 times as far: there the lse
    # bound is 4 x 1e-3 (a fault in the rescale would be off by whole powers
    # of two).
    w = LATE
    inp = _late_max_inputs(w, 2.0)
    out_rows = np.r_[0:900, 1020:w.S]
    blk = np.r_[900:1020]
    ref = oracle_fwd(w, inp)
    for ch in w.chunk_heads:
        out, lse, o = run_fwd(w, ch, inp)
        assert_close(f64(out), ref["out"], f"out ch={ch}")
        o_g = f64(o).reshape(w.S, w.Hq, w.d).transpose(1, 0, 2)
        assert_close(o_g, ref["o"], f"attention output ch={ch}")
        dl = np.abs(f64(lse) - ref["lse"])
        assert dl[:, out_rows].max() <= LSE_ABS, f"lse {dl[:, out_rows].max():.3e} ch={ch}"
        assert dl[:, blk].max() <= 4 * LSE_ABS, f"block lse {dl[:, blk].max():.3e} ch={ch}"


def test_forward_row_max_jump_forces_rescale():
    # Scaled by 6, the block's keys raise every later row's max by 10 to 34
    # powers of two in one tile: each such row must take the new max and
    # rescale mid-row.  The rows after the block are compared with the layer's
    # bounds (their scores against the block are 6 times the unit-scale ones,
    # so lse gets 6 x 1e-3).  The block's own rows (scores 36 times the unit
    # scale, far outside what the unit-scale bounds describe) are checked for
    # the rescale only: finite, and lse within 36 x 1e-3.
    w = LATE
    inp = _late_max_inputs(w, 6.0)
    after = np.r_[1020:w.S]
    blk = np.r_[900:1020]
    ref = oracle_fwd(w, inp)
    for ch in w.chunk_heads:
        out, lse, o = run_fwd(w, ch, inp)
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
        assert_close(f64(out)[after], ref["out"][after], f"out ch={ch}")
        o_g = f64(o).reshape(w.S, w.Hq, w.d).transpose(1, 0, 2)
        assert_close(o_g[:, after], ref["o"][:, after], f"attention output ch={ch}")
        assert_close(f64(out)[:900], ref["out"][:900], f"out before the block ch={ch}")
        dl = np.abs(f64(lse) - ref["lse"])
        assert dl[:, :900].max() <= LSE_ABS
        assert dl[:, after].max() <= 6 * LSE_ABS, f"lse {dl[:, after].max():.3e} ch={ch}"
        assert dl[:, blk].max() <= 36 * LSE_ABS, f"block lse {dl[:, blk].max():.3e} ch={ch}"


def test_forward_reports_values_beyond_fp16_range():
    # q, k, v are kept in fp16: a projection beyond +-65504 does not fit,
    # and the call must report it (UPIPE_ERR_RANGE) instead of returning
    # silently; the next call starts with a clear error word.
    import headwise_chunked_attention_gb300 as u
    w = Workload("range", S=300, hidden=256, Hq=2, Hkv=1, d=128, chunk_heads=(1,),
                 rope_theta=1e4)
    inp = make_inputs(w, seed=5)
    inp["x"] = (inp["x"].float() * 2.0 ** 17).to(torch.bfloat16)
    run_fwd(w, 1, inp, expect_error=u.ERR_RANGE)
    run_fwd(w, 1, make_inputs(w, seed=5))


@pytest.mark.parametrize("w", [
    # 4, 3 and 6 chunks: pairs only, a pair and a single last chunk, pairs
    # across KV groups with the per-head RMSNorm
    Workload("pair4-s1500", S=1500, hidden=256, Hq=4, Hkv=1, d=128, chunk_heads=(1,),
             rope_theta=1e4),
    Workload("pair3-d64-s1000", S=1000, hidden=384, Hq=3, Hkv=1, d=64, chunk_heads=(1,),
             rope_theta=1e4),
    Workload("pair6-qknorm-s777", S=777, hidden=384, Hq=6, Hkv=2, d=128, chunk_heads=(1,),
             rope_theta=1e6, qk_norm=True),
], ids=lambda w: w.name)
def test_paired_accumulates(w):
    # A workspace with the third chunk buffer makes the forward add two
    # chunks' partial results per accumulate: out within the layer's bounds
    # of the oracle and within fp32 summation order of the unpaired forward;
    # lse bit-identical.
    u = U()
    inp = make_inputs(w, seed=0, norm_gains="random")
    t = {k: v.to("cuda") for k, v in inp.items()}
    sh = u.Shape.of(w, 1)
    res = {}
    for mode in (0, 2):
        ws = torch.empty(u.workspace_bytes(sh, mode), device="cuda", dtype=torch.uint8)
        out = torch.empty(w.S, w.hidden, device="cuda")
        lse = torch.empty(w.Hq, w.S, device="cuda")
        u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
                   t.get("q_gamma"), t.get("k_gamma"))
        torch.cuda.synchronize()
        assert u.last_error() == 0
        res[mode] = (f64(out), lse.cpu())
    assert torch.equal(res[0][1], res[2][1])
    scale = np.abs(res[0][0]).max()
    assert np.abs(res[2][0] - res[0][0]).max() / scale < 1e-5
    ref = oracle_fwd(w, inp)
    assert_close(res[2][0], ref["out"], "paired out")
