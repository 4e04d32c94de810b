"""ctypes marshalling for libupipe (include/upipe.h).  No computation here."""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# UPIPE_DEBUG_BOUNDS=1 in the environment loads the debug build (device-side
# bounds checks of every plain global access; build.build(debug=True))
DEBUG_BOUNDS = os.environ.get("UPIPE_DEBUG_BOUNDS", "0") not in ("", "0")
_LIB_PATH = os.path.join(_HERE, "_build_debug" if DEBUG_BOUNDS else "_build", "libupipe.so")
_lib = None

ERR_NAMES = {0: "UPIPE_OK", 1: "UPIPE_ERR_INVALID_ARG", 2: "UPIPE_ERR_UNSUPPORTED",
             3: "UPIPE_ERR_WORKSPACE_TOO_SMALL", 4: "UPIPE_ERR_CUDA",
             5: "UPIPE_ERR_DEVICE_TIMEOUT", 6: "UPIPE_ERR_RANGE", 7: "UPIPE_ERR_BOUNDS",
             8: "UPIPE_ERR_TARGET"}
ERR_DEVICE_TIMEOUT = 5
ERR_RANGE = 6
ERR_BOUNDS = 7
ERR_TARGET = 8


class UpipeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {ERR_NAMES.get(code, code)}")


class Shape(ctypes.Structure):
    """upipe_shape_t."""
    _fields_ = [("S", ctypes.c_int64), ("hidden", ctypes.c_int32),
                ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("chunk_heads", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("qk_norm", ctypes.c_int32),
                ("norm_eps", ctypes.c_float)]

    @classmethod
    def of(cls, w, chunk_heads: Optional[int] = None, S: Optional[int] = None):
        """From any object with S, hidden, Hq, Hkv, d, rope_theta, qk_norm,
        norm_eps (e.g. a workload) and a chunk size."""
        ch = chunk_heads if chunk_heads is not None else w.chunk_heads[0]
        return cls(S if S is not None else w.S, w.hidden, w.Hq, w.Hkv, w.d, ch,
                   float(w.rope_theta), int(bool(w.qk_norm)), float(w.norm_eps))


class MlpShape(ctypes.Structure):
    """upipe_mlp_shape_t: the sequence-tiled MLP's geometry."""
    _fields_ = [("S", ctypes.c_int64), ("hidden", ctypes.c_int32),
                ("ffn", ctypes.c_int32), ("tile_rows", ctypes.c_int32)]


class LossShape(ctypes.Structure):
    """upipe_loss_shape_t: the sequence-tiled loss's geometry."""
    _fields_ = [("S", ctypes.c_int64), ("hidden", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("tile_rows", ctypes.c_int32)]


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load libupipe.so (built by ``build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libupipe.so not built ({_LIB_PATH}); run "
                "headwise_chunked_attention_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        L.upipe_workspace_bytes.argtypes = [ctypes.POINTER(Shape), ctypes.c_int]
        L.upipe_workspace_bytes.restype = ctypes.c_size_t
        L.upipe_attn_fwd.argtypes = [ctypes.POINTER(Shape)] + [P] * 9 + [ctypes.c_size_t, P, P]
        L.upipe_attn_fwd.restype = ctypes.c_int
        L.upipe_attn_fwd_fused.argtypes = ([ctypes.POINTER(Shape)] + [P] * 9 +
                                           [ctypes.c_size_t, P])
        L.upipe_attn_fwd_fused.restype = ctypes.c_int
        L.upipe_attn_bwd.argtypes = ([ctypes.POINTER(Shape)] + [P] * 17 +
                                     [ctypes.c_size_t, P])
        L.upipe_attn_bwd.restype = ctypes.c_int
        L.upipe_attn_bwd_saved_o.argtypes = ([ctypes.POINTER(Shape)] + [P] * 18 +
                                             [ctypes.c_size_t, P])
        L.upipe_attn_bwd_saved_o.restype = ctypes.c_int
        L.upipe_selftest_wait_timeout.argtypes = [ctypes.c_int, P]
        L.upipe_selftest_wait_timeout.restype = ctypes.c_int
        L.upipe_last_error.argtypes = []
        L.upipe_last_error.restype = ctypes.c_int
        L.upipe_profile_attach.argtypes = [ctypes.c_int, P, P, ctypes.c_int]
        L.upipe_profile_attach.restype = None
        L.upipe_profile_count.argtypes = []
        L.upipe_profile_count.restype = ctypes.c_int
        L.upipe_strerror.argtypes = [ctypes.c_int]
        L.upipe_strerror.restype = ctypes.c_char_p
        L.upipe_mlp_workspace_bytes.argtypes = [ctypes.POINTER(MlpShape), ctypes.c_int]
        L.upipe_mlp_workspace_bytes.restype = ctypes.c_size_t
        L.upipe_mlp_fwd.argtypes = [ctypes.POINTER(MlpShape)] + [P] * 6 + [ctypes.c_size_t, P]
        L.upipe_mlp_fwd.restype = ctypes.c_int
        L.upipe_mlp_bwd.argtypes = [ctypes.POINTER(MlpShape)] + [P] * 10 + [ctypes.c_size_t, P]
        L.upipe_mlp_bwd.restype = ctypes.c_int
        L.upipe_loss_workspace_bytes.argtypes = [ctypes.POINTER(LossShape), ctypes.c_int]
        L.upipe_loss_workspace_bytes.restype = ctypes.c_size_t
        L.upipe_loss_fwd.argtypes = [ctypes.POINTER(LossShape)] + [P] * 6 + [ctypes.c_size_t, P]
        L.upipe_loss_fwd.restype = ctypes.c_int
        L.upipe_loss_bwd.argtypes = ([ctypes.POINTER(LossShape)] + [P] * 4 + [ctypes.c_float] +
                                     [P] * 3 + [ctypes.c_size_t, P])
        L.upipe_loss_bwd.restype = ctypes.c_int
        for name in ("upipe_offload", "upipe_prefetch"):
            fn = getattr(L, name)
            fn.argtypes = [P, P, ctypes.c_size_t, P, ctypes.POINTER(ctypes.c_void_p)]
            fn.restype = ctypes.c_int
        L.upipe_copy_join.argtypes = [P, P]
        L.upipe_copy_join.restype = ctypes.c_int
        L.upipe_debug_bounds.argtypes = []
        L.upipe_debug_bounds.restype = ctypes.c_int
        L.upipe_selftest_bounds.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
        L.upipe_selftest_bounds.restype = ctypes.c_int
        L.upipe_gemm_tile_order.argtypes = [ctypes.c_int] * 5 + [
            ctypes.POINTER(ctypes.c_int32), ctypes.c_int64]
        L.upipe_gemm_tile_order.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def workspace_bytes(shape: Shape, mode: int = 0) -> int:
    return int(lib().upipe_workspace_bytes(ctypes.byref(shape), mode))


def _check(rc: int, where: str):
    if rc != 0:
        raise UpipeError(rc, where)


def attn_fwd(shape: Shape, x, Wq, Wk, Wv, Wo, out, lse, workspace,
             q_norm_w=None, k_norm_w=None, attn_o=None, stream=None):
    """upipe_attn_fwd on torch tensors (bf16 inputs, fp32 out/lse, uint8
    workspace); enqueues on ``stream`` (default: current stream).  ``attn_o``
    ([S, Hq*d] bf16 or None) receives every head's attention output."""
    bf = torch.bfloat16
    rc = lib().upipe_attn_fwd(
        ctypes.byref(shape), _ptr(x, bf, "x"), _ptr(Wq, bf, "Wq"), _ptr(Wk, bf, "Wk"),
        _ptr(Wv, bf, "Wv"), _ptr(Wo, bf, "Wo"), _ptr(q_norm_w, torch.float32, "q_norm_w"),
        _ptr(k_norm_w, torch.float32, "k_norm_w"), _ptr(out, torch.float32, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(),
        _ptr(attn_o, bf, "attn_o"), _stream(stream))
    _check(rc, "upipe_attn_fwd")


def attn_fwd_fused(shape: Shape, x, Wq, Wk, Wv, Wo, out, lse, workspace,
                   q_norm_w=None, k_norm_w=None, stream=None):
    """upipe_attn_fwd_fused on torch tensors: the forward with each chunk's
    Wo-slice accumulate done by the attention kernel (workspace of
    ``workspace_bytes(shape, 3)`` bytes)."""
    bf = torch.bfloat16
    rc = lib().upipe_attn_fwd_fused(
        ctypes.byref(shape), _ptr(x, bf, "x"), _ptr(Wq, bf, "Wq"), _ptr(Wk, bf, "Wk"),
        _ptr(Wv, bf, "Wv"), _ptr(Wo, bf, "Wo"), _ptr(q_norm_w, torch.float32, "q_norm_w"),
        _ptr(k_norm_w, torch.float32, "k_norm_w"), _ptr(out, torch.float32, "out"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "upipe_attn_fwd_fused")


def attn_bwd(shape: Shape, x, Wq, Wk, Wv, Wo, dout, lse, dx, dWq, dWk, dWv, dWo,
             workspace, q_norm_w=None, k_norm_w=None, dq_norm_w=None,
             dk_norm_w=None, attn_o=None, stream=None):
    """upipe_attn_bwd on torch tensors; with ``attn_o`` (the forward's
    attention output) upipe_attn_bwd_saved_o, which skips the recompute of
    the attention forward."""
    bf, f = torch.bfloat16, torch.float32
    head = [ctypes.byref(shape), _ptr(x, bf, "x"), _ptr(Wq, bf, "Wq"), _ptr(Wk, bf, "Wk"),
            _ptr(Wv, bf, "Wv"), _ptr(Wo, bf, "Wo"), _ptr(q_norm_w, f, "q_norm_w"),
            _ptr(k_norm_w, f, "k_norm_w"), _ptr(dout, bf, "dout"), _ptr(lse, f, "lse")]
    if attn_o is not None:
        fn, where = lib().upipe_attn_bwd_saved_o, "upipe_attn_bwd_saved_o"
        head.append(_ptr(attn_o, bf, "attn_o"))
    else:
        fn, where = lib().upipe_attn_bwd, "upipe_attn_bwd"
    rc = fn(
        *head,
        _ptr(dx, f, "dx"), _ptr(dWq, f, "dWq"), _ptr(dWk, f, "dWk"), _ptr(dWv, f, "dWv"),
        _ptr(dWo, f, "dWo"), _ptr(dq_norm_w, f, "dq_norm_w"), _ptr(dk_norm_w, f, "dk_norm_w"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(rc, where)


class KernelTimer:
    """Times every launch of one library kernel with CUDA events while the
    context is open: 0 attention forward, 1 attention backward, 2 Wo-slice
    accumulate on all SMs, 3 q/k RoPE/RMSNorm backward, 4 dV hi/lo split,
    5 attention forward with the fused Wo-slice accumulate."""

    def __init__(self, kernel: int, capacity: int):
        self.kernel = kernel
        self.starts = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        self.ends = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        for e in self.starts + self.ends:
            e.record()          # materialise the event handles
        torch.cuda.synchronize()
        arr = ctypes.c_void_p * capacity
        self._s = arr(*[e.cuda_event for e in self.starts])
        self._e = arr(*[e.cuda_event for e in self.ends])
        self.count = 0

    def __enter__(self):
        lib().upipe_profile_attach(self.kernel, self._s, self._e, len(self.starts))
        return self

    def __exit__(self, *exc):
        self.count = int(lib().upipe_profile_count())
        lib().upipe_profile_attach(-1, None, None, 0)

    def durations_ms(self):
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(self.starts[:self.count], self.ends[:self.count])]


def selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test kernel (its waits expire)."""
    _check(lib().upipe_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "upipe_selftest_wait_timeout")


def mlp_workspace_bytes(shape: MlpShape, mode: int = 0) -> int:
    return int(lib().upipe_mlp_workspace_bytes(ctypes.byref(shape), mode))


def mlp_fwd(shape: MlpShape, x, Wg, Wu, Wd, y, workspace, stream=None):
    """upipe_mlp_fwd: y [S, hidden] fp32 = the SwiGLU MLP of x, tile by tile."""
    bf = torch.bfloat16
    rc = lib().upipe_mlp_fwd(
        ctypes.byref(shape), _ptr(x, bf, "x"), _ptr(Wg, bf, "Wg"), _ptr(Wu, bf, "Wu"),
        _ptr(Wd, bf, "Wd"), _ptr(y, torch.float32, "y"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "upipe_mlp_fwd")


def mlp_bwd(shape: MlpShape, x, Wg, Wu, Wd, dy, dx, dWg, dWu, dWd, workspace, stream=None):
    """upipe_mlp_bwd: dx (fp32) and the fp32 weight gradients of sum(y * dy)."""
    bf, f = torch.bfloat16, torch.float32
    rc = lib().upipe_mlp_bwd(
        ctypes.byref(shape), _ptr(x, bf, "x"), _ptr(Wg, bf, "Wg"), _ptr(Wu, bf, "Wu"),
        _ptr(Wd, bf, "Wd"), _ptr(dy, bf, "dy"), _ptr(dx, f, "dx"), _ptr(dWg, f, "dWg"),
        _ptr(dWu, f, "dWu"), _ptr(dWd, f, "dWd"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "upipe_mlp_bwd")


def loss_workspace_bytes(shape: LossShape, mode: int = 0) -> int:
    return int(lib().upipe_loss_workspace_bytes(ctypes.byref(shape), mode))


def loss_fwd(shape: LossShape, h, W, targets, loss_rows, lse, workspace, stream=None):
    """upipe_loss_fwd: per-token losses and log-sum-exps (fp32), tile by tile."""
    bf, f = torch.bfloat16, torch.float32
    rc = lib().upipe_loss_fwd(
        ctypes.byref(shape), _ptr(h, bf, "h"), _ptr(W, bf, "W"), _ptr(targets, torch.int32, "targets"),
        _ptr(loss_rows, f, "loss_rows"), _ptr(lse, f, "lse"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "upipe_loss_fwd")


def loss_bwd(shape: LossShape, h, W, targets, lse, scale, dh, dW, workspace, stream=None):
    """upipe_loss_bwd: dh and dW (fp32) of scale * sum of the token losses."""
    bf, f = torch.bfloat16, torch.float32
    rc = lib().upipe_loss_bwd(
        ctypes.byref(shape), _ptr(h, bf, "h"), _ptr(W, bf, "W"), _ptr(targets, torch.int32, "targets"),
        _ptr(lse, f, "lse"), float(scale), _ptr(dh, f, "dh"), _ptr(dW, f, "dW"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(rc, "upipe_loss_bwd")


def offload(dev_src, host_dst, stream=None):
    """upipe_offload: copy a CUDA tensor into a page-locked CPU tensor of the
    same size on the library's copy stream; returns the ticket to join."""
    if not dev_src.is_cuda or host_dst.is_cuda or not host_dst.is_pinned():
        raise ValueError("offload: a CUDA source and a pinned CPU destination")
    n = dev_src.numel() * dev_src.element_size()
    if host_dst.numel() * host_dst.element_size() != n:
        raise ValueError("offload: sizes differ")
    t = ctypes.c_void_p()
    _check(lib().upipe_offload(dev_src.data_ptr(), host_dst.data_ptr(), n, _stream(stream),
                               ctypes.byref(t)), "upipe_offload")
    return t.value


def prefetch(host_src, dev_dst, stream=None):
    """upipe_prefetch: copy a page-locked CPU tensor into a CUDA tensor of the
    same size on the library's copy stream; returns the ticket to join."""
    if not dev_dst.is_cuda or host_src.is_cuda or not host_src.is_pinned():
        raise ValueError("prefetch: a pinned CPU source and a CUDA destination")
    n = dev_dst.numel() * dev_dst.element_size()
    if host_src.numel() * host_src.element_size() != n:
        raise ValueError("prefetch: sizes differ")
    t = ctypes.c_void_p()
    _check(lib().upipe_prefetch(host_src.data_ptr(), dev_dst.data_ptr(), n, _stream(stream),
                                ctypes.byref(t)), "upipe_prefetch")
    return t.value


def copy_join(ticket, stream=None):
    """upipe_copy_join: the stream (default: current) waits for the copy."""
    _check(lib().upipe_copy_join(ticket, _stream(stream)), "upipe_copy_join")


def debug_bounds() -> bool:
    """True when the loaded library is the bounds-checked debug build."""
    return bool(lib().upipe_debug_bounds())


def selftest_bounds(stream=None) -> bool:
    """Run the bounds-check self-test; True if its write past the declared
    view happened (release build), False if a check refused it (debug build,
    which then reports ERR_BOUNDS through last_error())."""
    written = ctypes.c_int(-1)
    _check(lib().upipe_selftest_bounds(_stream(stream), ctypes.byref(written)),
           "upipe_selftest_bounds")
    return written.value == 1


def gemm_tile_order(num_m: int, num_n: int, kb_total: int, ksplit: int = 1,
                    m_fastest: int = 0) -> list:
    """upipe_gemm_tile_order: the persistent GEMM's tile walk, one
    (row block, column tile, first K block, end K block) tuple per tile index."""
    n = num_m * num_n * ksplit
    out = (ctypes.c_int32 * (4 * n))()
    _check(lib().upipe_gemm_tile_order(num_m, num_n, kb_total, ksplit, m_fastest, out, 4 * n),
           "upipe_gemm_tile_order")
    return [tuple(out[4 * t:4 * t + 4]) for t in range(n)]


def last_error() -> int:
    return int(lib().upipe_last_error())
