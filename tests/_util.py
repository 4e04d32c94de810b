"""Shared helpers of the tests: tensor conversion and error metrics."""
import numpy as np
import torch


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a (bf16/fp32) tensor on any device."""
    return t.detach().to("cpu", torch.float64).numpy()


def rel_errs(got, ref):
    """(max, mean) absolute error divided by the RMS of the reference: the
    tolerance is stated for outputs of unit scale."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref)
    return float(err.max()) / rms, float(err.mean()) / rms


# tolerances of the attention layer (bf16 inputs, fp32 accumulation):
MAX_REL, MEAN_REL, LSE_ABS = 2e-2, 2e-3, 1e-3


def assert_close(got, ref, what, max_rel=MAX_REL, mean_rel=MEAN_REL):
    mx, mn = rel_errs(got, ref)
    assert mx <= max_rel and mn <= mean_rel, f"{what}: max {mx:.3e} mean {mn:.3e}"
    return mx, mn
