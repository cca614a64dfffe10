"""Error metric shared by the GPU parity tests.

max |x - ref| / rms(ref), computed separately for each output tensor over all of
its elements (the reference value is unique, so every element is compared).
"""
import numpy as np

TOL_F32 = 1e-4   # float32 inputs
TOL_BF16 = 1e-2  # bf16 inputs, float32 state


def rel_err(x, ref):
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    assert np.all(np.isfinite(x)), "non-finite output"
    rms = np.sqrt(np.mean(ref ** 2))
    if rms == 0.0:
        return float(np.max(np.abs(x)))
    return float(np.max(np.abs(x - ref)) / rms)
