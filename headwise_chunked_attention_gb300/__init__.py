"""Headwise-chunked causal GQA attention (Untied Ulysses / UPipe) on GB300.

Thin Python binding of the C ABI in ``include/upipe.h``: argument marshalling
only.  Every step of the layer runs in the CUDA kernels of ``libupipe.so``;
PyTorch only provides device memory and the current stream.  There is no CPU
fallback: without the built library every call raises.
"""
from ._binding import (  # noqa: F401
    UpipeError, Shape, MlpShape, LossShape, KernelTimer, mlp_workspace_bytes, mlp_fwd, mlp_bwd,
    loss_workspace_bytes, loss_fwd, loss_bwd, offload, prefetch, copy_join, attn_bwd, attn_fwd, attn_fwd_fused, last_error, lib, lib_path,
    workspace_bytes, selftest_wait_timeout, selftest_bounds, debug_bounds, gemm_tile_order, ERR_NAMES, ERR_DEVICE_TIMEOUT, ERR_RANGE, ERR_BOUNDS,
    ERR_TARGET, DEBUG_BOUNDS,
)
