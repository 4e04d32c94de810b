"""The forward entry point for callers that cannot allocate device memory.

upipe_attn_fwd_noalloc runs the layer forward on a static device array built
into the library instead of a caller-provided workspace.  This file is named
so that pytest collects it last: if it fails, a run stopped at the first
failure has already run every other test.  It passes alone in a fresh process
and after the other tests, because every call overwrites whatever the shared
array holds before reading it.
"""
import ctypes

import pytest
import torch

from workloads import WORKLOADS, Workload, make_inputs
from tests._guard import guarded

pytestmark = pytest.mark.gpu

UPIPE_ERR_WORKSPACE_TOO_SMALL = 3
STATIC_SCRATCH_BYTES = 64 << 20


def noalloc_fn():
    import headwise_chunked_attention_gb300 as u
    fn = u.lib().upipe_attn_fwd_noalloc
    fn.argtypes = [ctypes.POINTER(u.Shape)] + [ctypes.c_void_p] * 10
    fn.restype = ctypes.c_int
    return fn


def ptr(t):
    return None if t is None else t.data_ptr()


@pytest.mark.parametrize("w,ch", [
    (WORKLOADS["tiny-s2048"], 2),
    (Workload("d128-qknorm-s3000", S=3000, hidden=512, Hq=8, Hkv=2, d=128,
              chunk_heads=(2,), rope_theta=1e6, qk_norm=True), 2),
    # past 65536 tokens the attention folds long rows into per-SM fp32 rows,
    # which then also live in the static array (d = 64: 16 MiB of them)
    (Workload("d64-s70000", S=70000, hidden=256, Hq=1, Hkv=1, d=64,
              chunk_heads=(1,), rope_theta=1e4), 1),
], ids=["tiny", "d128-qknorm", "d64-fold-rows"])
def test_noalloc_forward_matches_allocating_forward(w, ch):
    # The same kernels add the chunks into out in the same order on both
    # paths, so out and lse must be bit-identical to the allocating forward's.
    import headwise_chunked_attention_gb300 as u
    fn = noalloc_fn()
    inp = {k: v.cuda() for k, v in make_inputs(w, seed=5, norm_gains="random").items()}
    shape = u.Shape.of(w, ch)
    assert 0 < u.workspace_bytes(shape, 0) <= STATIC_SCRATCH_BYTES
    # the existing entry point, with a caller-allocated workspace
    out_ref = torch.empty(w.S, w.hidden, device="cuda")
    lse_ref = torch.empty(w.Hq, w.S, device="cuda")
    ws = torch.empty(u.workspace_bytes(shape, 0), dtype=torch.uint8, device="cuda")
    u.attn_fwd(shape, inp["x"], inp["Wq"], inp["Wk"], inp["Wv"], inp["Wo"], out_ref, lse_ref,
               ws, inp.get("q_gamma"), inp.get("k_gamma"))
    torch.cuda.synchronize()
    assert u.last_error() == 0
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):   # two calls in a row share the static scratch
        # out and lse inside guard margins that must come back untouched
        g_out = guarded((w.S, w.hidden), fill=float("nan"))
        g_lse = guarded((w.Hq, w.S), fill=float("nan"))
        out, lse = g_out.t, g_lse.t
        rc = fn(ctypes.byref(shape), ptr(inp["x"]), ptr(inp["Wq"]), ptr(inp["Wk"]),
                ptr(inp["Wv"]), ptr(inp["Wo"]), ptr(inp.get("q_gamma")),
                ptr(inp.get("k_gamma")), ptr(out), ptr(lse), stream)
        assert rc == 0, rc
        torch.cuda.synchronize()
        assert u.last_error() == 0
        g_out.check("out")
        g_lse.check("lse")
        assert torch.equal(out, out_ref), f"out, call {call}"
        assert torch.equal(lse, lse_ref), f"lse, call {call}"


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    import headwise_chunked_attention_gb300 as u
    fn = noalloc_fn()
    w = WORKLOADS["llama3.2-3b-s65536"]
    shape = u.Shape.of(w, 24)
    assert u.workspace_bytes(shape, 0) > STATIC_SCRATCH_BYTES
    fake = [0x100000 + 0x1000 * i for i in range(10)]
    rc = fn(ctypes.byref(shape), *fake[:5], None, None, fake[5], fake[6], None)
    assert rc == UPIPE_ERR_WORKSPACE_TOO_SMALL
