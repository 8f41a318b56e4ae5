"""Inputs that drive the online softmax through its rescale path: the forward
keeps O unnormalised and rescales it (in TMEM) only when a row's running
maximum grows by more than 2^8, which N(0, 1) inputs at scale 1/sqrt(d)
almost never do.  Here later keys carry larger scores (keys scaled up along
the sequence) and the softmax scale is far from 1/sqrt(d), so rows rescale
at many key tiles; results are checked against the fp64 oracle with the same
scale, for every dtype and head size and both backward variants."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu


def ramped_inputs(p, seed, growth):
    """q, k, v, do as the workloads draw them, with key j scaled by
    1 + growth * j / Lkv (later keys score higher), rounded to the dtype."""
    q, k, v, do = W.make_inputs(p, seed)
    ramp = 1.0 + growth * torch.arange(p.Lkv, dtype=torch.float64) / p.Lkv
    k = (k.double() * ramp[None, :, None, None]).to(k.dtype)
    return q, k, v, do


def run_case(p, scale, growth, deterministic, seed=0):
    import exact_attention_34_gb300 as ea

    q, k, v, do = ramped_inputs(p, seed, growth)
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, scale=scale, causal=p.causal)
    grads = ea.backward(qd, kd, vd, o, lse, dod, scale=scale, causal=p.causal, deterministic=deterministic)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    tol = TOL[p.dtype]
    o_ref, lse_ref = oracle.forward(q, k, v, scale=scale, causal=p.causal)
    assert rel_err(to_np(o), o_ref) <= tol
    lse_check(to_np(lse), lse_ref, tol)
    ref = oracle.backward(q, k, v, do, scale=scale, causal=p.causal)
    gmax = max(float(np.max(np.abs(r))) for r in ref) or 1.0
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        g = to_np(g)
        assert np.all(np.isfinite(g)), name
        err = float(np.max(np.abs(g - r))) / max(float(np.max(np.abs(r))), 0.1 * gmax)
        assert err <= tol, f"{name} rel err {err:.3e}"


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_growing_scores(causal, d, dtype, deterministic):
    p = W.Problem(2, 700, 700, 4, 2, d, dtype, causal, None, "ramp")
    run_case(p, scale=2.0 / np.sqrt(d), growth=3.0, deterministic=deterministic)


@pytest.mark.parametrize("scale", [0.02, 0.5])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_scale_far_from_default(scale, dtype):
    p = W.Problem(2, 600, 900, 4, 4, 128, dtype, False, None, "scale")
    run_case(p, scale=scale, growth=1.0, deterministic=True)


@pytest.mark.parametrize("deterministic", [True, False])
def test_growing_scores_head_dim_256(deterministic):
    p = W.Problem(2, 520, 700, 4, 2, 256, "bf16", True, None, "ramp256")
    run_case(p, scale=2.0 / 16.0, growth=3.0, deterministic=deterministic)


# Key ramps for the window cases: 3x and 4x along the sequence.  A window's dQ
# is a strongly cancelling sum (each row of dS sums to zero over few keys), so
# the 16-bit operands show through: P and dS enter the MMAs rounded to the
# format, and delta = rowsum(dO * O) is taken from the stored 16-bit O.  With
# bf16's 8-bit mantissa that costs up to ~6e-3 at 3x and ~1.2e-2 at 4x (dQ,
# seed 3, window (100, 50)); fp16 (three more bits) stays below 1e-3.  The
# pages' 1e-2 target is stated for their N(0, 1) workloads; the 4x bf16 case is
# held to 2e-2, every other case to the target.
WINDOW_GROWTHS = (2.0, 3.0)
BF16_STEEP_RAMP_TOL = 2e-2


@pytest.mark.parametrize("growth", WINDOW_GROWTHS)
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("window", [(200, 0), (100, 50)])
def test_growing_scores_with_window(window, dtype, growth):
    """The left-bounded kernel builds (a window) through the rescale path:
    rows rescale hundreds of times while keys grow 3x or 4x along the
    sequence."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 700, 700, 4, 2, 128, dtype, False, None, "rampwin")
    q, k, v, do = ramped_inputs(p, 3, growth)
    scale = 2.0 / np.sqrt(128)
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, scale=scale, window=window)
    grads = ea.backward(qd, kd, vd, o, lse, dod, scale=scale, window=window)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    o_ref, lse_ref = oracle.forward(q, k, v, scale=scale, window=window)
    assert rel_err(to_np(o), o_ref) <= TOL[dtype]
    lse_check(to_np(lse), lse_ref, TOL[dtype])
    tol = BF16_STEEP_RAMP_TOL if (dtype == "bf16" and growth >= 3.0) else TOL[dtype]
    for name, g, r in zip(("dQ", "dK", "dV"), grads, oracle.backward(q, k, v, do, scale=scale, window=window)):
        assert rel_err(to_np(g), r) <= tol, name
