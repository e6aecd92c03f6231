"""Shared helpers of the parity tests: tolerances and comparisons."""
import numpy as np
import torch

# bf16 inputs, fp32 accumulation: the parity bar of every floating-point output
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
# Full-size checks must also stay within this fraction of the bars, so that a
# later precision change (the attention's packed bf16 exponentials, for one)
# cannot use up the whole tolerance unnoticed.
MARGIN = 0.25
# (what, max-abs, mean-abs, max bar, mean bar) of every check that asserts the margin;
# tests/conftest.py prints them at the end of the session
RECORD = []


def f64(t: torch.Tensor) -> np.ndarray:
    """A tensor (any device, bf16/fp32) as a float64 NumPy array."""
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(got, want, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what="", margin=False):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    mx, mn = float(err.max()), float(err.mean())
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max-abs {mx:.3e} (<= {max_abs}), mean-abs {mn:.3e} (<= {mean_abs})"
    if margin:
        RECORD.append((what, mx, mn, max_abs, mean_abs))
        print(f"parity {what}: max-abs {mx:.3e} mean-abs {mn:.3e}")
        assert mx <= MARGIN * max_abs and mn <= MARGIN * mean_abs, (
            f"{what}: max-abs {mx:.3e} / mean-abs {mn:.3e} leave less than {1 - MARGIN:.0%} of the bars "
            f"{max_abs} / {mean_abs}")
    return mx, mn
