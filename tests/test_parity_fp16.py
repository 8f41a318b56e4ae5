"""fp16 inputs on the tensor-core path (the same kernels as bf16 with fp16
operands, fp32 accumulation) against the fp64 oracle: forward, both backward
variants, KV lengths + GQA + Lq != Lkv, a local window, the preprocess and the
split-KV decode with its combine."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu
TOL16 = TOL["fp16"]


def kvt(kl):
    return None if kl is None else torch.tensor(kl, dtype=torch.int32).cuda()


CASES = [
    # B, Lq, Lkv, Hq, Hkv, d, causal, kv_lens
    (2, 600, 600, 4, 2, 128, True, None),
    (2, 600, 600, 2, 2, 64, False, None),
    (2, 300, 1000, 4, 2, 128, True, None),
    (4, 256, 1500, 8, 2, 128, False, (1500, 700, 1, 0)),
    (1, 1, 700, 4, 1, 128, True, None),
]


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("case", CASES)
def test_fp16_fwd_bwd(case, deterministic):
    import exact_attention_34_gb300 as ea

    B, Lq, Lkv, Hq, Hkv, d, causal, kl = case
    p = W.Problem(B, Lq, Lkv, Hq, Hkv, d, "fp16", causal, kl, "fp16")
    q, k, v, do = W.make_inputs(p)
    assert q.dtype == torch.float16
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, causal=causal, kv_lens=kvt(kl))
    assert o.dtype == torch.float16
    o_ref, lse_ref = oracle.forward(q, k, v, causal=causal, kv_lens=kl)
    assert rel_err(to_np(o), o_ref) <= TOL16
    lse_check(to_np(lse), lse_ref, TOL16)
    grads = ea.backward(qd, kd, vd, o, lse, dod, causal=causal, kv_lens=kvt(kl), deterministic=deterministic)
    torch.cuda.synchronize()
    ref = oracle.backward(q, k, v, do, causal=causal, kv_lens=kl)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        assert g.dtype == torch.float16
        e = rel_err(to_np(g), r)
        assert e <= TOL16, f"{name} rel err {e:.3e}"
    assert ea.attn_device_status()[1] == 0


def test_fp16_is_more_accurate_than_bf16():
    """The same problem in fp16 and bf16: fp16's 3 extra mantissa bits show up
    as a smaller error against the oracle (a check that fp16 really runs as
    fp16 operands, not through a bf16 conversion)."""
    import exact_attention_34_gb300 as ea

    errs = {}
    for dt in ("fp16", "bf16"):
        p = W.Problem(2, 512, 512, 4, 4, 128, dt, True, None, "cmp")
        q, k, v, do = W.make_inputs(p)
        o, lse = ea.forward(*cuda(q, k, v), causal=True)
        errs[dt] = rel_err(to_np(o), oracle.forward(q, k, v, causal=True)[0])
    assert errs["fp16"] < errs["bf16"] / 3


def test_fp16_window():
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 700, 700, 4, 2, 128, "fp16", False, None, "fp16win")
    q, k, v, do = W.make_inputs(p)
    qd, kd, vd, dod = cuda(q, k, v, do)
    win = (200, 10)
    o, lse = ea.forward(qd, kd, vd, window=win)
    grads = ea.backward(qd, kd, vd, o, lse, dod, window=win)
    torch.cuda.synchronize()
    assert rel_err(to_np(o), oracle.forward(q, k, v, window=win)[0]) <= TOL16
    for g, r in zip(grads, oracle.backward(q, k, v, do, window=win)):
        assert rel_err(to_np(g), r) <= TOL16


def test_fp16_preprocess():
    import exact_attention_34_gb300 as ea

    p = W.Problem(3, 333, 333, 4, 4, 128, "fp16", False, None, "pre16")
    o, _, _, do = W.make_inputs(p, seed=5)
    delta = torch.empty(p.B, p.Hq, p.Lq, device="cuda", dtype=torch.float32)
    ea.attn_bwd_preprocess(o.cuda(), do.cuda(), delta)
    torch.cuda.synchronize()
    assert rel_err(to_np(delta), oracle.backward_preprocess(o, do)) <= 1e-5


@pytest.mark.parametrize("Lq,causal", [(1, False), (16, True)])
def test_fp16_decode(Lq, causal):
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, Lq, 5000, 8, 2, 128, "fp16", causal, (5000, 1200), "dec16")
    q, k, v, _ = W.make_inputs(p)
    o, lse = ea.decode(*cuda(q, k, v), causal=causal, kv_lens=kvt(p.kv_lens), num_splits=6)
    torch.cuda.synchronize()
    assert o.dtype == torch.float16
    o_ref, lse_ref = oracle.forward(q, k, v, causal=causal, kv_lens=p.kv_lens)
    assert rel_err(to_np(o), o_ref) <= TOL16
    lse_check(to_np(lse), lse_ref, TOL16)
