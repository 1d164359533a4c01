"""Helpers shared by the parity tests (comparison only; no attention arithmetic)."""
import numpy as np
import torch

# Tolerances (stated with the workloads): fp32 -> 1e-5 absolute; bf16 -> max abs
# error relative to max |ref| of 2e-2 for O and 5e-2 for dQ/dK/dV; LSE (bf16
# path) 1e-3 absolute.
TOL_F32_ABS = 1e-5
TOL_BF16_O = 2e-2
TOL_BF16_GRAD = 5e-2
TOL_BF16_LSE = 1e-3


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def max_abs(a, b) -> float:
    a, b = to64(a), to64(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    return float(np.abs(a - b).max()) if a.size else 0.0


def rel_max(a, ref) -> float:
    a, ref = to64(a), to64(ref)
    assert a.shape == ref.shape, (a.shape, ref.shape)
    if not a.size:
        return 0.0
    assert np.isfinite(a).all(), "non-finite values in GPU output"
    return float(np.abs(a - ref).max() / max(np.abs(ref).max(), 1e-30))


def grad_within(got, ref, cancel_scale: float) -> bool:
    """bf16 gradient bar: rel_max <= TOL_BF16_GRAD, except where the reference
    is identically zero. A row that sees one key has dQ = 0 exactly (a softmax
    over one element is constant), and the GPU's dS = P (dP - D) there is the
    fp32 rounding residual of two equal sums; the relative bar is undefined, so
    the residual is bounded by fp32 rounding of the cancelling terms instead
    (cancel_scale: a bound on |dP| and |D|, e.g. max|dO| * max|V| * d)."""
    ref64 = to64(ref)
    if ref64.size and np.abs(ref64).max() == 0.0:
        return float(np.abs(to64(got)).max()) <= 1e-6 * max(1.0, cancel_scale)
    return rel_max(got, ref) <= TOL_BF16_GRAD
