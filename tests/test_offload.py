"""GPU test of the offload of block inputs to host memory and their prefetch
back (upipe_offload / upipe_prefetch / upipe_copy_join, through the C ABI):
a round trip is bit-exact and ordered by the tickets, the copies run beside
a layer forward on the caller's stream without changing its result, and
memory of the wrong kind is refused before anything is enqueued."""
import ctypes

import pytest
import torch

from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def U():
    import headwise_chunked_attention_gb300 as mod
    mod.lib()
    return mod


def test_offload_and_prefetch_round_trip_is_exact():
    u = U()
    g = torch.Generator(device="cuda").manual_seed(1)
    x = torch.randn(3000, 1024, device="cuda", generator=g).to(torch.bfloat16)
    keep = x.clone()
    host = torch.empty(x.shape, dtype=x.dtype).pin_memory()
    t = u.offload(x, host)
    u.copy_join(t)
    x.zero_()                  # ordered after the copy by the join
    t = u.prefetch(host, x)
    u.copy_join(t)
    torch.cuda.synchronize()
    assert torch.equal(x, keep)
    assert torch.equal(host, keep.cpu())


def test_copies_run_beside_a_layer_forward():
    # the block input is offloaded while the layer forward reads it, then
    # overwritten and prefetched back; the forward's output is unchanged and
    # a second forward on the prefetched input gives the same bits
    u = U()
    w = Workload("offload", S=4096, hidden=512, Hq=4, Hkv=2, d=128, chunk_heads=(2,),
                 rope_theta=1e4)
    t = {k: v.cuda() for k, v in make_inputs(w, seed=3).items()}
    sh = u.Shape.of(w, 2)
    ws = torch.empty(u.workspace_bytes(sh, 0), dtype=torch.uint8, device="cuda")
    out0 = torch.empty(w.S, w.hidden, device="cuda")
    lse = torch.empty(w.Hq, w.S, device="cuda")
    u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out0, lse, ws)
    host = torch.empty(t["x"].shape, dtype=torch.bfloat16).pin_memory()
    x_keep = t["x"].clone()
    ticket = u.offload(t["x"], host)
    out1 = torch.empty_like(out0)
    u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out1, lse, ws)
    u.copy_join(ticket)
    t["x"].fill_(7.0)
    ticket = u.prefetch(host, t["x"])
    u.copy_join(ticket)
    out2 = torch.empty_like(out0)
    u.attn_fwd(sh, t["x"], t["Wq"], t["Wk"], t["Wv"], t["Wo"], out2, lse, ws)
    torch.cuda.synchronize()
    assert u.last_error() == 0
    assert torch.equal(t["x"], x_keep)
    assert torch.equal(out1, out0) and torch.equal(out2, out0)


def test_pageable_or_wrong_kind_memory_is_refused():
    u = U()
    L = u.lib()
    x = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    pageable = torch.zeros(1024, dtype=torch.bfloat16)
    pinned = torch.zeros(1024, dtype=torch.bfloat16).pin_memory()
    t = ctypes.c_void_p()
    n = 2048
    # pageable host memory, and both ends on the device
    assert L.upipe_offload(x.data_ptr(), pageable.data_ptr(), n, None, ctypes.byref(t)) == 1
    assert L.upipe_prefetch(x.data_ptr(), x.data_ptr(), n, None, ctypes.byref(t)) == 1
    # host source for an offload (the directions exchanged)
    assert L.upipe_offload(pinned.data_ptr(), x.data_ptr(), n, None, ctypes.byref(t)) == 1
    assert t.value is None
    torch.cuda.synchronize()
    assert u.last_error() == 0
