"""Shared helpers of the tests: tensor conversion and error metrics."""
import numpy as np
import torch


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a (bf16/fp32) tensor on any device."""
    return t.detach().to("cpu", torch.float64).numpy()


def rel_errs(got, ref, rowwise=True):
    """(max, mean) absolute error relative to outputs of unit scale.

    The tolerance is stated for outputs of unit scale.  A causal attention
    layer's output rows are not of one scale (row i averages ~i values, so
    |out_i| shrinks like 1/sqrt(i)); each row (token, last axis) is therefore
    divided by the reference row's RMS before the error is taken.  With
    ``rowwise=False`` the whole tensor is divided by one RMS."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rowwise and ref.ndim >= 2:
        rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
        rms = np.maximum(rms, 1e-30)
    else:
        rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref) / rms
    return float(err.max()), float(err.mean())


# tolerances of the attention layer (bf16 inputs, fp32 accumulation):
MAX_REL, MEAN_REL, LSE_ABS = 2e-2, 2e-3, 1e-3
# The layer's bounds are stated for its output and its input gradient; the
# weight gradients and the RMSNorm gain gradients are held to the same bounds
# (measured against the float64 layer: gain gradients ~8e-4 mean).
GAIN_MAX_REL, GAIN_MEAN_REL = MAX_REL, MEAN_REL


def assert_close(got, ref, what, max_rel=MAX_REL, mean_rel=MEAN_REL):
    mx, mn = rel_errs(got, ref)
    assert mx <= max_rel and mn <= mean_rel, f"{what}: max {mx:.3e} mean {mn:.3e}"
    return mx, mn
