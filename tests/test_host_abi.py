"""CPU-only checks of the C ABI: the library builds, loads and exports every
function include/upipe.h declares; the workspace planner; host-side argument
validation (no call here reaches the GPU: every case fails validation first)."""
import ctypes
import json
import os
import re

import pytest

from workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def u():
    import headwise_chunked_attention_gb300 as mod
    if not os.path.exists(mod.lib_path()):
        from headwise_chunked_attention_gb300.build import build
        build()
    mod.lib()
    return mod


def declared_functions():
    src = open(os.path.join(ROOT, "include", "upipe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(upipe_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_function(u):
    names = declared_functions()
    assert {"upipe_attn_fwd", "upipe_attn_bwd", "upipe_workspace_bytes"} <= set(names)
    L = u.lib()
    for n in names:
        assert hasattr(L, n), n


def ws(u, w, ch, mode=0, **kw):
    return u.workspace_bytes(u.Shape.of(w.with_(**kw) if kw else w, ch), mode)


def test_workspace_closed_form(u):
    al = lambda b: (b + 255) // 256 * 256
    for w in WORKLOADS.values():
        g = w.Hq // w.Hkv
        for ch in w.chunk_heads:
            kvc = max(1, ch // g)
            S, d = w.S, w.d
            expect = (al(((S >> 10) + 1) * (d // 2) * 8) + 2 * al(1024 * (d // 2) * 8)
                      + 2 * al(S * ch * d * 2) + 2 * al(S * kvc * d * 2))
            if S > 512 * 128:   # per-SM fp32 rows for folding long attention rows
                expect += 256 * 256 * d * 4
            assert ws(u, w, ch) == expect, (w.name, ch)
            # backward: dO (fp16), D, dQ (fp32), dK, dV (fp32) and their bf16
            # low halves, the saved RMSNorm values (qk-norm), and the fp16
            # gradient scales' norm maxima (2 + Hkv + chunks floats)
            bwd = (al(S * ch * d * 2) + al(ch * S * 4) + al(S * ch * d * 4)
                   + 2 * al(S * kvc * d * 4) + 2 * al(S * kvc * d * 2))
            if w.qk_norm:
                bwd += al(S * ch * d * 4) + al(ch * S * 4) + al(S * kvc * d * 4) + al(kvc * S * 4)
            bwd += al((2 + w.Hkv + w.Hq // ch) * 4)
            assert ws(u, w, ch, 1) == expect + bwd, (w.name, ch)
            # mode 2: the forward's third chunk buffer for paired accumulates
            assert ws(u, w, ch, 2) == expect + al(S * ch * d * 2), (w.name, ch)
            # mode 3: the fused forward keeps no attention output, so one
            # chunk buffer (Q) instead of two
            assert ws(u, w, ch, 3) == expect - al(S * ch * d * 2), (w.name, ch)


def test_workspace_affine_in_chunk_heads_and_golden_reduction(u):
    w = WORKLOADS["qwen3-32b-rank-s1m"]
    b = {ch: ws(u, w, ch) for ch in (1, 2, 4, 8)}
    slope = (b[8] - b[1]) / 7
    for ch in (2, 4):
        assert b[ch] == b[1] + slope * (ch - 1)
    qo = lambda ch: slope * ch             # the part that scales with chunk_heads
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "paper_figures.json")))
    want = gold["attention_intermediate_memory_reduction_qwen3_32b"]["value"]
    assert abs((1 - qo(1) / qo(8)) - want) < 1e-12
    # the Q/O part of the forward workspace is 4 GiB at 8 heads, 0.5 GiB at 1
    assert qo(8) == 4 * 2 ** 30 and qo(1) == 2 ** 29


def test_invalid_shapes_give_zero_workspace(u):
    w = WORKLOADS["tiny-s2048"]
    bad = [dict(S=0), dict(Hq=5), dict(Hkv=3), dict(d=96), dict(hidden=200),
           dict(rope_theta=0.0), dict(rope_theta=float("nan"))]
    for kw in bad:
        assert ws(u, w, 2, **kw) == 0, kw
    assert ws(u, w, 3) == 0                   # 3 does not divide Hq = 4
    assert u.workspace_bytes(u.Shape.of(w, 2), 7) == 0
    assert u.workspace_bytes(u.Shape.of(w, 2), 4) == 0


def _fwd(u, shape, ptrs=None, ws_bytes=1 << 40, dbg=None):
    L = u.lib()
    p = ptrs or [0x100000 + 0x1000 * i for i in range(10)]
    return L.upipe_attn_fwd(ctypes.byref(shape) if shape is not None else None,
                            *p[:5], None, None, p[5], p[6], p[7], ws_bytes, dbg, None)


def test_validation_codes_before_any_launch(u):
    w = WORKLOADS["tiny-s2048"]
    sh = u.Shape.of(w, 2)
    assert _fwd(u, None) == 1
    assert _fwd(u, u.Shape.of(w, 3)) == 1
    assert _fwd(u, u.Shape.of(w.with_(d=96), 2)) == 2
    ptrs = [0x100000 + 0x1000 * i for i in range(10)]
    ptrs[0] = 0
    assert _fwd(u, sh, ptrs) == 1                       # NULL x
    ptrs = [0x100000 + 0x1000 * i for i in range(10)]
    ptrs[2] += 8
    assert _fwd(u, sh, ptrs) == 1                       # misaligned Wk
    assert _fwd(u, sh, ws_bytes=1000) == 3              # workspace too small
    L = u.lib()
    for code, text in [(0, b"ok"), (3, b"workspace too small"), (5, b"device wait timed out")]:
        assert L.upipe_strerror(code) == text


def test_binding_marshals_error_codes(u):
    import torch
    w = WORKLOADS["tiny-s2048"]
    x = torch.zeros(4, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        u.attn_fwd(u.Shape.of(w, 2), x, x, x, x, x, x, x, x)   # CPU tensors refused


def test_saved_o_backward_validates_before_any_launch(u):
    # upipe_attn_bwd_saved_o requires the forward's attention output and
    # validates it, like every other argument, before the first launch
    L = u.lib()
    w = WORKLOADS["tiny-s2048"]
    sh = u.Shape.of(w, 2)
    p = [0x100000 + 0x1000 * i for i in range(20)]
    args = lambda o: (ctypes.byref(sh), *p[:5], None, None, p[5], p[6], o,
                      *p[7:12], None, None, p[12], 1 << 40, None)
    assert L.upipe_attn_bwd_saved_o(*args(None)) == 1       # NULL attn_o
    assert L.upipe_attn_bwd_saved_o(*args(p[13] + 8)) == 1  # misaligned attn_o
    bad = u.Shape.of(w, 3)                                   # 3 does not divide Hq
    assert L.upipe_attn_bwd_saved_o(ctypes.byref(bad), *args(p[13])[1:]) == 1


def test_guard_margins_catch_writes_outside_the_buffer():
    # the guard helper itself, on the CPU: writes inside the buffer pass, one
    # byte changed just after its end or just before its start is reported
    import torch
    from tests._guard import guarded
    g = guarded((3, 5), device="cpu")
    g.t.fill_(1.0)
    assert (g.raw.data_ptr() + g.off) % 256 == 0
    g.check("inside only")
    for edge in ("after", "before"):
        h = guarded((3, 5), device="cpu")
        h.raw[h.off + h.nbytes if edge == "after" else h.off - 1] = 0
        with pytest.raises(AssertionError):
            h.check(edge)


def test_fused_forward_validates_before_any_launch(u):
    # upipe_attn_fwd_fused checks the shape, every pointer and the mode-3
    # workspace size on the host and launches nothing when one fails
    L = u.lib()
    w = WORKLOADS["tiny-s2048"]
    sh = u.Shape.of(w, 2)
    need = u.workspace_bytes(sh, 3)
    assert 0 < need < u.workspace_bytes(sh, 0)
    p = [0x100000 + 0x1000 * i for i in range(10)]
    call = lambda shape, ptrs, nbytes: L.upipe_attn_fwd_fused(
        ctypes.byref(shape) if shape is not None else None, *ptrs[:5], None, None,
        ptrs[5], ptrs[6], ptrs[7], nbytes, None)
    assert call(None, p, need) == 1                         # NULL shape
    assert call(u.Shape.of(w, 3), p, need) == 1             # 3 does not divide Hq
    assert call(u.Shape.of(w.with_(d=96), 2), p, need) == 2
    q = list(p)
    q[5] = 0
    assert call(sh, q, need) == 1                           # NULL out
    q = list(p)
    q[6] += 4
    assert call(sh, q, need) == 1                           # misaligned lse
    q = list(p)
    q[7] += 16
    assert call(sh, q, need) == 1                           # workspace not 256-byte aligned
    assert call(sh, p, need - 1) == 3                       # workspace too small


def test_mlp_workspace_and_validation(u):
    # the MLP's workspace is one tile's intermediates: a (bf16) forward, plus
    # dA (fp32), dg and du (bf16) backward, of min(tile_rows, S) rows
    al = lambda b: (b + 255) // 256 * 256
    for S, hidden, ffn, tile in [(300, 256, 384, 128), (77, 128, 128, 256),
                                 (1 << 17, 4096, 14336, 8192)]:
        sh = u.MlpShape(S, hidden, ffn, tile)
        T = min(tile, S)
        assert u.mlp_workspace_bytes(sh, 0) == al(T * ffn * 2)
        assert u.mlp_workspace_bytes(sh, 1) == al(T * ffn * 2) + al(T * ffn * 4) + 2 * al(T * ffn * 2)
    for bad in [u.MlpShape(0, 256, 256, 128), u.MlpShape(100, 200, 256, 128),
                u.MlpShape(100, 256, 200, 128), u.MlpShape(100, 256, 256, 100),
                u.MlpShape(100, 256, 256, 0)]:
        assert u.mlp_workspace_bytes(bad, 0) == 0
    assert u.mlp_workspace_bytes(u.MlpShape(100, 256, 256, 128), 2) == 0
    L = u.lib()
    sh = u.MlpShape(300, 256, 384, 128)
    p = [0x100000 + 0x1000 * i for i in range(12)]
    need0, need1 = u.mlp_workspace_bytes(sh, 0), u.mlp_workspace_bytes(sh, 1)
    fwd = lambda shape, q, n: L.upipe_mlp_fwd(ctypes.byref(shape), *q[:5], q[5], n, None)
    assert fwd(sh, p, need0 - 1) == 3                              # workspace too small
    assert fwd(u.MlpShape(300, 200, 384, 128), p, need0) == 2       # hidden % 128
    q = list(p); q[0] = 0
    assert fwd(sh, q, need0) == 1                                   # NULL x
    q = list(p); q[4] += 8
    assert fwd(sh, q, need0) == 1                                   # misaligned y
    q = list(p); q[5] += 16
    assert fwd(sh, q, need0) == 1                                   # workspace not 256-aligned
    bwd = lambda q, n: L.upipe_mlp_bwd(ctypes.byref(sh), *q[:9], q[9], n, None)
    assert bwd(p, need1 - 1) == 3
    q = list(p); q[8] = 0
    assert bwd(q, need1) == 1                                       # NULL dWd


def test_loss_workspace_and_validation(u):
    # forward: one tile's per-row partials (vocab / 256 or / 128 float2) and
    # target logits; backward: one tile's dz in bf16
    al = lambda b: (b + 255) // 256 * 256
    for S, hidden, vocab, tile in [(300, 256, 1024, 128), (77, 128, 384, 256),
                                   (1 << 17, 4096, 128256, 4096)]:
        sh = u.LossShape(S, hidden, vocab, tile)
        T = min(tile, S)
        bn = 256 if vocab % 256 == 0 else 128
        assert u.loss_workspace_bytes(sh, 0) == al(T * (vocab // bn) * 8) + al(T * 4)
        assert u.loss_workspace_bytes(sh, 1) == al(T * vocab * 2)
    for bad in [u.LossShape(0, 256, 256, 128), u.LossShape(100, 200, 256, 128),
                u.LossShape(100, 256, 200, 128), u.LossShape(100, 256, 256, 64)]:
        assert u.loss_workspace_bytes(bad, 0) == 0
    L = u.lib()
    sh = u.LossShape(300, 256, 1024, 128)
    p = [0x100000 + 0x1000 * i for i in range(12)]
    need0, need1 = u.loss_workspace_bytes(sh, 0), u.loss_workspace_bytes(sh, 1)
    fwd = lambda q, n: L.upipe_loss_fwd(ctypes.byref(sh), *q[:5], q[5], n, None)
    assert fwd(p, need0 - 1) == 3
    q = list(p); q[2] = 0
    assert fwd(q, need0) == 1                                       # NULL targets
    q = list(p); q[3] += 4
    assert fwd(q, need0) == 1                                       # misaligned loss_rows
    bwd = lambda q, n: L.upipe_loss_bwd(ctypes.byref(sh), *q[:4], 1.0, q[4], q[5], q[6], n, None)
    assert bwd(p, need1 - 1) == 3
    q = list(p); q[5] = 0
    assert bwd(q, need1) == 1                                       # NULL dW
    assert L.upipe_strerror(8) == b"loss target outside the vocabulary"


def test_offload_validates_before_enqueueing(u):
    # NULL pointers, zero bytes and a missing ticket are refused on the host
    L = u.lib()
    t = ctypes.c_void_p(1)
    assert L.upipe_offload(0x100000, 0x200000, 64, None, None) == 1
    assert L.upipe_offload(None, 0x200000, 64, None, ctypes.byref(t)) == 1 and t.value is None
    assert L.upipe_prefetch(0x100000, None, 64, None, ctypes.byref(t)) == 1
    assert L.upipe_offload(0x100000, 0x200000, 0, None, ctypes.byref(t)) == 1
    assert L.upipe_copy_join(None, None) == 1
