"""GPU backward parity: upipe_attn_bwd (chunked, recomputing Q/K/V and the
attention output per chunk) and upipe_attn_bwd_saved_o (the forward's saved
attention output instead of its recompute) against the float64 chain-rule
oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import WORKLOADS, Workload, make_inputs
from tests._util import f64, assert_close, rel_errs, GAIN_MAX_REL, GAIN_MEAN_REL, MEAN_REL
from tests._guard import guarded

pytestmark = pytest.mark.gpu


def run_fwd_bwd(w, ch, inp, saved_o=False, dout_scale=None):
    import headwise_chunked_attention_gb300 as u
    dev = "cuda"
    t = {k: v.to(dev) for k, v in inp.items()}
    sh = u.Shape.of(w, ch)
    # every buffer the library writes sits inside guard margins that must come
    # back untouched
    gb = {"out": guarded((w.S, w.hidden)), "lse": guarded((w.Hq, w.S)),
          "workspace": guarded((u.workspace_bytes(sh, 1),), torch.uint8)}
    if saved_o:
        gb["attn_o"] = guarded((w.S, w.Hq * w.d), torch.bfloat16)
    out, lse, ws = gb["out"].t, gb["lse"].t, gb["workspace"].t
    o = gb["attn_o"].t if saved_o else None
    u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws,
               t.get("q_gamma"), t.get("k_gamma"), o)
    if saved_o:   # the backward must not depend on what the forward left in ws
        ws.fill_(0xFF)
    dout = t["dout"] if dout_scale is None else (t["dout"].float() * dout_scale).to(torch.bfloat16)
    for n, src in [("dx", "x"), ("dWq", "Wq"), ("dWk", "Wk"), ("dWv", "Wv"), ("dWo", "Wo")]:
        gb[n] = guarded(tuple(t[src].shape), fill=float("nan"))
    if w.qk_norm:
        gb["dq_gamma"] = guarded((w.d,), fill=float("nan"))
        gb["dk_gamma"] = guarded((w.d,), fill=float("nan"))
    g = {n: gb[n].t for n in ("dx", "dWq", "dWk", "dWv", "dWo")}
    dqg = gb["dq_gamma"].t if w.qk_norm else None
    dkg = gb["dk_gamma"].t if w.qk_norm else None
    u.attn_bwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], dout, lse,
               g["dx"], g["dWq"], g["dWk"], g["dWv"], g["dWo"], ws,
               t.get("q_gamma"), t.get("k_gamma"), dqg, dkg, attn_o=o)
    torch.cuda.synchronize()
    rc = u.last_error()
    assert rc == 0, f"device error word {rc}"
    for name, b in gb.items():
        b.check(name)
    g["dq_gamma"], g["dk_gamma"] = dqg, dkg
    return g


def oracle_bwd(w, inp):
    # the plain float64 chain rule: no rounding of any intermediate
    a = {k: f64(v) for k, v in inp.items()}
    return O.layer_backward(w, a["x"], a["Wq"], a["Wk"], a["Wv"], a["Wo"], a["dout"],
                            a.get("q_gamma"), a.get("k_gamma"))


CASES = [
    (WORKLOADS["tiny-s2048"], (2,)),
    (Workload("d128-s1000", S=1000, hidden=256, Hq=4, Hkv=1, d=128,
              chunk_heads=(1, 2, 4), rope_theta=5e5), (1, 2, 4)),
    (Workload("d128-qknorm-s700", S=700, hidden=384, Hq=4, Hkv=2, d=128,
              chunk_heads=(1, 2, 4), rope_theta=1e6, qk_norm=True), (1, 4)),
    (Workload("d64-mha-s333", S=333, hidden=256, Hq=2, Hkv=2, d=64,
              chunk_heads=(1, 2), rope_theta=1e4), (1, 2)),
    # d = 64 with the per-head RMSNorm; chunk_heads 4 spans two KV groups
    (Workload("d64-qknorm-s389", S=389, hidden=256, Hq=4, Hkv=2, d=64,
              chunk_heads=(1, 2, 4), rope_theta=1e6, qk_norm=True), (1, 4)),
]


@pytest.mark.parametrize("w,chs", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_backward_matches_oracle(w, chs):
    inp = make_inputs(w, seed=0, with_grad=True, norm_gains="random")
    ref = oracle_bwd(w, inp)
    for ch in chs:
        g = run_fwd_bwd(w, ch, inp)
        for name in ("dx", "dWq", "dWk", "dWv", "dWo"):
            assert_close(f64(g[name]), ref[name], f"{name} ch={ch}")
        if w.qk_norm:
            for name in ("dq_gamma", "dk_gamma"):
                assert_close(f64(g[name]), ref[name], f"{name} ch={ch}",
                             GAIN_MAX_REL, GAIN_MEAN_REL)


@pytest.mark.parametrize("w,chs", [CASES[1], CASES[2]],
                         ids=lambda c: getattr(c, "name", str(c)))
def test_backward_with_saved_attention_output(w, chs):
    # the saved-O backward computes the same gradients: against the oracle
    # with the same bound, and against the recomputing backward to within the
    # layer's max bound (the recompute forms D = rowsum(dO * o) from the fp32
    # o, the saved-O path from its bf16 copy: the two differ by o's rounding)
    inp = make_inputs(w, seed=0, with_grad=True, norm_gains="random")
    ref = oracle_bwd(w, inp)
    for ch in chs:
        g = run_fwd_bwd(w, ch, inp, saved_o=True)
        r = run_fwd_bwd(w, ch, inp)
        names = ["dx", "dWq", "dWk", "dWv", "dWo"] + (["dq_gamma", "dk_gamma"]
                                                      if w.qk_norm else [])
        for name in names:
            bound = (GAIN_MAX_REL, GAIN_MEAN_REL) if "gamma" in name else ()
            assert_close(f64(g[name]), ref[name], f"saved-O {name} ch={ch}", *bound)
            assert_close(f64(g[name]), f64(r[name]), f"saved-O vs recompute {name} ch={ch}",
                         *bound)


@pytest.mark.parametrize("w,chs", [CASES[1], CASES[4]],
                         ids=lambda c: getattr(c, "name", str(c)))
def test_backward_gradient_magnitude_invariance(w, chs):
    # The backward keeps dO and dS in fp16 with power-of-two factors derived
    # on the device from the norms of dout, Wo, v and dO.  Multiplying dout by
    # a power of two multiplies those factors' inputs by it, so the fp16
    # operands are the same bits and every gradient (the gains' included)
    # scales exactly: tiny (2^-40) and large (2^20) upstream gradients lose no
    # precision.  The fp32 reductions across CTAs (dQ, dK, dV, split-K weight
    # gradients) run in no fixed order, and a one-ulp change of an fp32
    # gradient moves the bf16 low half of its hi/lo split by up to ~2^-18 of
    # the value, so the comparison allows 1e-4 of the tensor's RMS; a lost
    # factor or an fp16 underflow would be off by orders of magnitude more.
    inp = make_inputs(w, seed=0, with_grad=True, norm_gains="random")
    for ch in chs:
        base = {k: f64(v) for k, v in run_fwd_bwd(w, ch, inp).items() if v is not None}
        for e in (-40, 20):
            g = run_fwd_bwd(w, ch, inp, dout_scale=2.0 ** e)
            for name, v in base.items():
                got = f64(g[name]) * 2.0 ** -e
                rms = np.sqrt(np.mean(v * v))
                err = np.max(np.abs(got - v)) / rms
                assert err < 1e-4, f"{name} ch={ch} scale 2^{e}: {err:.2e}"


@pytest.mark.parametrize("walk", [2, 6])
def test_backward_segmented_walks(walk):
    # Past 1M tokens a key tile's walk over the queries is cut into segments
    # run by separate CTAs, each adding its dK / dV partial.  UPIPE_BWD_WALK
    # forces short segments here (2 and 6 sub-tiles of 64 queries), so that
    # small shapes take that path; the environment is read once per process,
    # hence the child process.
    import os
    import subprocess
    import sys
    env = dict(os.environ, UPIPE_BWD_WALK=str(walk))
    child = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_bwd_walk_child.py")
    r = subprocess.run([sys.executable, child], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]


@pytest.mark.parametrize("S", [1, 2, 129])
def test_backward_shortest_and_ragged_lengths(S):
    # one token (every row attends to itself only), two, and one past a tile
    w = Workload("short", S=S, hidden=256, Hq=2, Hkv=1, d=128, chunk_heads=(1, 2),
                 rope_theta=1e4)
    # With one token dq and dk vanish in exact arithmetic (the softmax of one
    # score is constant), so dWq and dWk are exactly zero, and with two tokens
    # they are sums of cancelling terms: their relative error is not
    # meaningful there.  dx (the input gradient) keeps the layer's bounds per
    # token.  A weight-gradient element over one or two tokens is a single
    # product, with nothing to average the 16-bit rounding of its factors
    # (the bf16 attention output in dWo; in dWv the two query heads of the KV
    # group can also cancel, dv = dO_h0 + dO_h1), so for S <= 2 dWv and dWo
    # are held to the mean bound relative to the whole tensor's scale.
    inp = make_inputs(w, seed=S, with_grad=True)
    ref = oracle_bwd(w, inp)
    for ch in w.chunk_heads:
        g = run_fwd_bwd(w, ch, inp)
        assert_close(f64(g["dx"]), ref["dx"], f"S={S} dx ch={ch}")
        if S <= 2:
            for name in ("dWv", "dWo"):
                _, mn = rel_errs(f64(g[name]), ref[name], rowwise=False)
                assert mn <= MEAN_REL, f"S={S} {name} ch={ch}: mean {mn:.2e}"
        else:
            for name in ("dWq", "dWk", "dWv", "dWo"):
                assert_close(f64(g[name]), ref[name], f"S={S} {name} ch={ch}")


def test_backward_of_a_zero_upstream_gradient_is_exactly_zero():
    # dout = 0: the gradient scales' norms are all zero (the scale code's
    # degenerate branch); every gradient must come out exactly 0, not NaN
    w = CASES[2][0]
    inp = make_inputs(w, seed=0, with_grad=True, norm_gains="random")
    for ch in (1, 4):
        g = run_fwd_bwd(w, ch, inp, dout_scale=0.0)
        for name, v in g.items():
            if v is not None:
                assert torch.count_nonzero(v).item() == 0, f"{name} ch={ch}"
