"""Local-window (sliding) masks on the GPU against the fp64 oracle: windows on
one or both sides of the bottom-right aligned diagonal, narrower and wider than
a tile, with KV lengths, GQA, Lq != Lkv, both backward variants, bf16 and fp32,
and the special cases that reduce to causal, to no mask and to one key per row."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu


def kvt(kv_lens):
    return None if kv_lens is None else torch.tensor(kv_lens, dtype=torch.int32).cuda()


def run_window(p, window, deterministic=True, check_bwd=True, seed=0):
    import exact_attention_34_gb300 as ea

    q, k, v, do = W.make_inputs(p, seed)
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, kv_lens=kvt(p.kv_lens), window=window)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.forward(q, k, v, kv_lens=p.kv_lens, window=window)
    tol = TOL[p.dtype]
    assert rel_err(to_np(o), o_ref) <= tol
    lse_check(to_np(lse), lse_ref, tol)
    if check_bwd:
        grads = ea.backward(qd, kd, vd, o, lse, dod, kv_lens=kvt(p.kv_lens), window=window,
                            deterministic=deterministic)
        torch.cuda.synchronize()
        ref = oracle.backward(q, k, v, do, kv_lens=p.kv_lens, window=window)
        for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
            e = rel_err(to_np(g), r)
            assert e <= tol, f"{name} rel err {e:.3e}"
    assert ea.attn_device_status()[1] == 0
    return o, lse


CASES = [
    # B, Lq, Lkv, Hq, Hkv, d, kv_lens, window
    (2, 600, 600, 4, 2, 128, None, (256, 0)),       # causal sliding window over several tiles
    (2, 1000, 1000, 2, 2, 64, None, (100, 50)),     # two-sided, narrower than a tile
    (2, 300, 1000, 4, 2, 128, None, (-1, 200)),     # right side bounded only, Lq < Lkv
    (2, 1000, 300, 4, 1, 128, None, (64, -1)),      # left side bounded only, Lq > Lkv
    (3, 512, 700, 4, 4, 128, (700, 200, 0), (130, 130)),  # with KV lengths and an empty batch
    (1, 385, 385, 2, 2, 64, None, (0, 3)),          # ragged, one key back and three ahead
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("case", CASES)
def test_window_fwd_bwd(case, dtype):
    B, Lq, Lkv, Hq, Hkv, d, kl, win = case
    run_window(W.Problem(B, Lq, Lkv, Hq, Hkv, d, dtype, False, kl, "window"), win)


@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[4]])
def test_window_single_pass_backward(case):
    B, Lq, Lkv, Hq, Hkv, d, kl, win = case
    run_window(W.Problem(B, Lq, Lkv, Hq, Hkv, d, "bf16", False, kl, "window_atomic"), win, deterministic=False)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_zero_width_window_is_one_key_per_row(dtype):
    """window (0, 0), Lq == Lkv: row i sees key i only, so O = V exactly and
    the exact dQ and dK are 0 (kernel rounding noise only)."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 300, 300, 2, 2, 128, dtype, False, None, "w00")
    q, k, v, do = (t.cuda() for t in W.make_inputs(p))
    o, lse = ea.forward(q, k, v, window=(0, 0))
    dq, dk, dv = ea.backward(q, k, v, o, lse, do, window=(0, 0))
    torch.cuda.synchronize()
    # The forward's P of the one key is exactly 1, so O = V to within an ulp
    # of the output type.  The backward's P = 2^(s sl2 - lse2) recomputes s: in
    # bf16 to within its rounding; in float32 the forward's scores come from
    # split bf16 tensor-core products (about 2^-16 of relative error each)
    # while the backward's may be summed differently, so dV = P dO is held to
    # the float32 target (1e-4) rather than to an ulp
    rt = 2.0 ** -7 if dtype == "bf16" else 1e-6
    assert torch.allclose(o.float(), v.float(), rtol=rt, atol=0)
    rt_bwd = 2.0 ** -7 if dtype == "bf16" else 1e-4
    assert torch.allclose(dv.float(), do.float(), rtol=rt_bwd, atol=1e-30)
    assert dq.abs().max() <= 1e-2 * do.abs().max() and dk.abs().max() <= 1e-2 * do.abs().max()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_window_special_cases_match_causal_and_unmasked_bitwise(dtype):
    """(-1, 0) is the causal path and windows at least as long as the
    sequences are no mask: the same kernels, so the results are identical."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 700, 900, 4, 2, 128, dtype, False, (900, 450), "wspecial")
    q, k, v, do = (t.cuda() for t in W.make_inputs(p))
    kl = kvt(p.kv_lens)
    for window, causal in (((-1, 0), True), ((-1, -1), False), ((5000, 5000), False)):
        a = ea.forward(q, k, v, kv_lens=kl, window=window)
        b = ea.forward(q, k, v, kv_lens=kl, causal=causal)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        ga = ea.backward(q, k, v, a[0], a[1], do, kv_lens=kl, window=window)
        gb = ea.backward(q, k, v, b[0], b[1], do, kv_lens=kl, causal=causal)
        for x, y in zip(ga, gb):
            assert torch.equal(x, y)


def test_window_full_size_headline_shapes():
    """bf16 B4 H8 T8192 d128 with a 1024-key causal sliding window (the
    headline shapes); the oracle checks batch 3, head 2: O/LSE on sampled rows
    and all of dQ, dK, dV for that head."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(4, 8192, 8192, 8, 8, 128, "bf16", False, None, "window_full")
    win = (1024, 0)
    q, k, v, do = W.make_inputs(p)
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, window=win)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, window=win)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    b, h = 3, 2
    sl = lambda t: t[b:b + 1, :, h:h + 1]  # noqa: E731
    rows = np.array([0, 1, 1023, 1024, 1025, 5000, 8191])
    o_ref, lse_ref = oracle.forward(sl(q), sl(k), sl(v), window=win, rows=rows)
    assert rel_err(to_np(sl(o))[:, rows], o_ref) <= TOL["bf16"]
    lse_check(to_np(lse[b:b + 1, h:h + 1])[:, :, rows], lse_ref, TOL["bf16"])
    ref = oracle.backward(sl(q), sl(k), sl(v), sl(do), window=win)
    for g, r in zip((dq, dk, dv), ref):
        assert rel_err(to_np(sl(g)), r) <= TOL["bf16"]
