"""Shared helpers of the parity tests: tolerances and comparisons."""
import numpy as np
import torch

# bf16 inputs, fp32 accumulation: the parity bar of every floating-point output
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def f64(t: torch.Tensor) -> np.ndarray:
    """A tensor (any device, bf16/fp32) as a float64 NumPy array."""
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(got, want, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    mx, mn = float(err.max()), float(err.mean())
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max-abs {mx:.3e} (<= {max_abs}), mean-abs {mn:.3e} (<= {mean_abs})"
    return mx, mn
