"""GPU checks of the forward's stream contract: with more than one chunk the
forward runs each chunk's Wo-slice accumulate on a library-owned side stream
and joins it back with events, so the caller's stream must see the finished
``out`` (and ``lse``) right after the call, whatever stream the caller uses.
``out`` is bit-reproducible (one store, then one reduce-add per chunk in chunk
order), so every snapshot must equal the reference bit for bit."""
import pytest
import torch

from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

W = Workload("streams-s1000", S=1000, hidden=256, Hq=8, Hkv=2, d=64, chunk_heads=(1,),
             rope_theta=1e4)


def _call(u, sh, t, out, lse, ws, stream=None):
    u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out, lse, ws, stream=stream)


def test_forward_result_is_ordered_on_the_callers_stream():
    import headwise_chunked_attention_gb300 as u
    t = {k: v.cuda() for k, v in make_inputs(W, seed=3).items()}
    sh = u.Shape.of(W, 1)   # 8 chunks: seven accumulates run on the side stream
    ws = torch.empty(u.workspace_bytes(sh, 0), dtype=torch.uint8, device="cuda")
    out = torch.empty(W.S, W.hidden, device="cuda")
    lse = torch.empty(W.Hq, W.S, device="cuda")
    _call(u, sh, t, out, lse, ws)
    torch.cuda.synchronize()
    assert u.last_error() == 0
    out_ref, lse_ref = out.clone(), lse.clone()

    # a caller-created stream: snapshots taken on it right after each call,
    # with the output poisoned in between, must all be the finished result
    s = torch.cuda.Stream()
    snaps = []
    with torch.cuda.stream(s):
        for _ in range(4):
            out.fill_(float("nan"))
            lse.fill_(float("nan"))
            _call(u, sh, t, out, lse, ws)
            snaps.append((out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert u.last_error() == 0
    for o, l in snaps:
        assert torch.equal(o, out_ref)
        assert torch.equal(l, lse_ref)


def test_forward_on_the_legacy_default_stream():
    import headwise_chunked_attention_gb300 as u
    t = {k: v.cuda() for k, v in make_inputs(W, seed=4).items()}
    sh = u.Shape.of(W, 2)
    ws = torch.empty(u.workspace_bytes(sh, 0), dtype=torch.uint8, device="cuda")
    out = torch.empty(W.S, W.hidden, device="cuda")
    lse = torch.empty(W.Hq, W.S, device="cuda")
    _call(u, sh, t, out, lse, ws)
    torch.cuda.synchronize()
    ref = out.clone()
    out.fill_(float("nan"))
    # stream handle 0 is the legacy default stream, which the torch current
    # stream here also is; the clone is ordered after the call on it
    _call(u, sh, t, out, lse, ws, stream=torch.cuda.default_stream())
    got = out.clone()
    torch.cuda.synchronize()
    assert u.last_error() == 0
    assert torch.equal(got, ref)
