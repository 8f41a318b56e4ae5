"""Shared helpers for the parity tests: the pages' error metric and tensor
plumbing.  Holds no attention arithmetic."""

import numpy as np
import torch


def rel_err(got, ref) -> float:
    """max|a - b| / max|b| (the pages' accuracy metric); absolute when max|b| == 0."""
    a = np.asarray(got, dtype=np.float64)
    b = np.asarray(ref, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    den = np.max(np.abs(b)) if b.size else 0.0
    num = np.max(np.abs(a - b)) if b.size else 0.0
    return float(num / den) if den > 0 else float(num)


def lse_check(got, ref, tol):
    """LSE: -inf exactly where the reference is -inf; finite entries within tol
    (relative to max |lse|, floor 1)."""
    a = np.asarray(got, dtype=np.float64)
    b = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), "LSE -inf pattern differs"
    assert np.all(a[~fin] == -np.inf)
    if fin.any():
        err = np.max(np.abs(a[fin] - b[fin])) / max(1.0, np.max(np.abs(b[fin])))
        assert err <= tol, f"LSE error {err:.3e} > {tol:.1e}"


def to_np(t):
    return t.detach().float().cpu().numpy() if t.dtype != torch.float64 else t.detach().cpu().numpy()


def cuda(*ts):
    return tuple(t.cuda() for t in ts)


# bf16 and fp32 targets as stated for the method; fp16 takes the bf16 target's
# multiple of the unit roundoff (1e-2 = 2.56 * 2^-8) at fp16's 2^-11, rounded up
TOL = {"bf16": 1e-2, "fp32": 1e-4, "fp16": 2e-3}
