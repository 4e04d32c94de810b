"""GPU forward parity: the CUDA path (through the C ABI) against the float64
oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import WORKLOADS, Workload, make_inputs, sample_rows
from tests._util import f64, assert_close, LSE_ABS

pytestmark = pytest.mark.gpu


def U():
    import headwise_chunked_attention_gb300 as mod
    mod.lib()
    return mod


def run_fwd(w, ch, inp, debug=True):
    u = U()
    dev = "cuda"
    t = {k: v.to(dev) for k, v in inp.items()}
    shape = u.Shape.of(w, ch)
    out = torch.empty(w.S, w.hidden, device=dev, dtype=torch.float32)
    lse = torch.empty(w.Hq, w.S, device=dev, dtype=torch.float32)
    ws = torch.empty(u.workspace_bytes(shape, 0), device=dev, dtype=torch.uint8)
    o = torch.empty(w.S, w.Hq * w.d, device=dev, dtype=torch.bfloat16) if debug else None
    u.attn_fwd(shape, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
               t.get("q_gamma"), t.get("k_gamma"), o)
    torch.cuda.synchronize()
    assert u.last_error() == 0
    return out, lse, o


def oracle_fwd(w, inp, rows=None, store=None):
    a = {k: f64(v) for k, v in inp.items()}
    return O.layer_forward(w, a["x"], a["Wq"], a["Wk"], a["Wv"], a["Wo"],
                           a.get("q_gamma"), a.get("k_gamma"), rows=rows,
                           store_dtype=store)


def check_full(w, ch, inp):
    out, lse, o = run_fwd(w, ch, inp)
    refb = oracle_fwd(w, inp, store="bf16")
    # q, k, v, P and O are bf16 by design (the workspace precision): the
    # tolerance applies against the oracle that stores q, k, v in bf16
    assert_close(f64(out), refb["out"], "out")
    o_g = f64(o).reshape(w.S, w.Hq, w.d).transpose(1, 0, 2)
    assert_close(o_g, refb["o"], "attention output")
    dl = np.abs(f64(lse) - refb["lse"]).max()
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


def test_forward_row_max_growing_late_in_rows():
    # The hidden rows of keys 900..1019 are scaled by 6, so their scores
    # against every later query are 6 times larger: the row max of each of
    # those queries jumps by 10 to 34 powers of two in the eighth KV tile, and
    # the kernel must take that tile's max and rescale O and l mid-row.
    # The block's own rows are left out of the comparison: their queries are
    # scaled too, so their scores among themselves are 36 times larger, and a
    # one-ulp difference in the bf16 rounding of a projected q or k (float64
    # oracle against the fp32 tensor-core sum) moves such a score by ~1%.
    # Every other row is compared in full, out and O with the layer's bounds.
    # Their scores against the scaled keys are 6 times larger too, and the
    # LSE error (absolute, in the scores' units) grows with them: one ulp of
    # a k element moves such a score 6 times as far, so the LSE bound here is
    # 6 x 1e-3.  A fault in the rescale would be off by whole powers of two.
    w = Workload("late-max", S=1500, hidden=256, Hq=2, Hkv=1, d=128, chunk_heads=(1, 2),
                 rope_theta=1e4)
    inp = make_inputs(w, seed=11)
    x = inp["x"].float()
    x[900:1020] *= 6.0
    inp["x"] = x.to(torch.bfloat16)
    keep = np.r_[0:900, 1020:w.S]
    ref = oracle_fwd(w, inp, store="bf16")
    for ch in w.chunk_heads:
        out, lse, o = run_fwd(w, ch, inp)
        assert_close(f64(out)[keep], ref["out"][keep], f"out ch={ch}")
        o_g = f64(o).reshape(w.S, w.Hq, w.d).transpose(1, 0, 2)
        assert_close(o_g[:, keep], ref["o"][:, keep], f"attention output ch={ch}")
        dl = np.abs(f64(lse)[:, keep] - ref["lse"][:, keep]).max()
        assert dl <= 6 * LSE_ABS, f"lse max abs err {dl:.3e} ch={ch}"


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
    ref = oracle_fwd(w, inp, store="bf16")
    assert_close(res[2][0], ref["out"], "paired out")
