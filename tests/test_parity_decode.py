"""GPU split-KV decode parity: per-split partials against the oracle's
partials (same documented partition), the combined output against the exact
forward, and the combine step alone on seeded random partials."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu


def run_decode(p, num_splits, check_partials=True, seed=0):
    import exact_attention_34_gb300 as ea

    q, k, v = W.make_inputs(p, seed, with_do=False)
    kl = torch.tensor(p.kv_lens, dtype=torch.int32).cuda()
    o, lse, op, lp = ea.decode(*cuda(q, k, v), causal=p.causal, kv_lens=kl, num_splits=num_splits,
                               return_partials=True)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    tol = TOL[p.dtype]
    o_ref, lse_ref = oracle.forward(q, k, v, causal=p.causal, kv_lens=p.kv_lens)
    assert rel_err(to_np(o), o_ref) <= tol
    lse_check(to_np(lse), lse_ref, tol)
    if check_partials:
        op_ref, lp_ref = oracle.splitkv_partials(q, k, v, op.shape[2], causal=p.causal, kv_lens=p.kv_lens)
        assert rel_err(to_np(op), op_ref) <= tol
        lse_check(to_np(lp), lp_ref, tol)
    return o, lse


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("Lq,causal", [(1, False), (16, True), (3, True), (1, True)])
def test_small_decode(dtype, Lq, causal):
    p = W.Problem(3, Lq, 3000, 8, 2, 128, dtype, causal, (3000, 1000, 5), "decode_small")
    run_decode(p, num_splits=5)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_decode_mha_and_d64(dtype):
    p = W.Problem(2, 2, 1024, 4, 4, 64, dtype, False, (1024, 130), "decode_mha")
    run_decode(p, num_splits=3)


def test_decode_auto_splits():
    p = W.Problem(2, 1, 4096, 32, 8, 128, "bf16", False, (4096, 2000), "decode_auto")
    run_decode(p, num_splits=0, check_partials=False)


@pytest.mark.parametrize("Lq,causal", [(1, False), (16, True)])
def test_decode_full_size_sampled(Lq, causal):
    """B8 Hq32 Hkv8 over a 131072-key cache; the oracle checks batches 0 and 5."""
    import exact_attention_34_gb300 as ea

    p = W.decode(Lq, causal)
    q, k, v = W.make_inputs(p, 0, with_do=False)
    kl = torch.tensor(p.kv_lens, dtype=torch.int32).cuda()
    o, lse = ea.decode(*cuda(q, k, v), causal=causal, kv_lens=kl)
    torch.cuda.synchronize()
    G = p.Hq // p.Hkv
    for b in (0, 5):
        for hk in (0, 7):
            n = p.kv_lens[b]
            qs = q[b:b + 1, :, hk * G:(hk + 1) * G]
            o_ref, lse_ref = oracle.forward(qs, k[b:b + 1, :n, hk:hk + 1], v[b:b + 1, :n, hk:hk + 1],
                                            causal=causal)
            got = to_np(o[b:b + 1, :, hk * G:(hk + 1) * G])
            assert rel_err(got, o_ref) <= TOL["bf16"]
            lse_check(to_np(lse[b:b + 1, hk * G:(hk + 1) * G]), lse_ref, TOL["bf16"])


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_combine_alone(dtype):
    import exact_attention_34_gb300 as ea

    g = torch.Generator().manual_seed(3)
    B, Hq, S, Lq, d = 2, 3, 7, 4, 128
    op = torch.randn(B, Hq, S, Lq, d, generator=g)
    lp = torch.randn(B, Hq, S, Lq, generator=g) * 3
    lp[0, 1, 2:] = -float("inf")      # empty splits
    lp[1, 2, :, 1] = -float("inf")    # a row with every split empty
    op[1, 2, :, 1] = 0
    o = torch.empty(B, Lq, Hq, d, device="cuda", dtype=W.DTYPES[dtype])
    lse = torch.empty(B, Hq, Lq, device="cuda")
    ea.attn_decode_combine(op.cuda(), lp.cuda(), o, lse)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.combine(op, lp)
    assert rel_err(to_np(o), o_ref) <= TOL[dtype]
    lse_check(to_np(lse), lse_ref, 1e-6)
    assert np.all(to_np(o)[1, 1, 2] == 0)
