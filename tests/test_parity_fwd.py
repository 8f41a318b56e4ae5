"""GPU forward parity: the CUDA library through its C ABI against the fp64
oracle on the same seeded inputs, max|a-b|/max|b| per output tensor."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu


def kv_tensor(p):
    return None if p.kv_lens is None else torch.tensor(p.kv_lens, dtype=torch.int32).cuda()


def run_fwd(p, rows=None, heads=None, seed=0):
    import exact_attention_34_gb300 as ea

    q, k, v = W.make_inputs(p, seed, with_do=False)
    o, lse = ea.forward(*cuda(q, k, v), causal=p.causal, kv_lens=kv_tensor(p))
    torch.cuda.synchronize()
    st, code, _ = ea.attn_device_status()
    assert code == 0
    o_ref, lse_ref = oracle.forward(q, k, v, causal=p.causal, kv_lens=p.kv_lens, rows=rows, heads=heads)
    o_np, lse_np = to_np(o), to_np(lse)
    if rows is not None:
        o_np, lse_np = o_np[:, rows], lse_np[:, :, rows]
    if heads is not None:
        o_np, o_ref = o_np[:, :, heads], o_ref[:, :, heads]
        lse_np, lse_ref = lse_np[:, heads], lse_ref[:, heads]
    tol = TOL[p.dtype]
    e = rel_err(o_np, o_ref)
    assert e <= tol, f"{p.name}: O rel err {e:.3e} > {tol:.0e}"
    lse_check(lse_np, lse_ref, tol)
    return q, k, v, o, lse


def test_tiny_fp32_exact_check():
    run_fwd(W.tiny())


SMALL = [(T, d, c) for T in (128, 600, 1000) for d in (64, 128) for c in (False, True)]


@pytest.mark.parametrize("T,d,causal", SMALL)
def test_bf16_small_grid(T, d, causal):
    run_fwd(W.Problem(2, T, T, 2, 2, d, "bf16", causal, None, f"small_T{T}_d{d}_c{int(causal)}"))


@pytest.mark.parametrize("T,d,causal", [(600, 64, True), (300, 128, False), (1000, 128, True)])
def test_fp32_small_grid(T, d, causal):
    run_fwd(W.Problem(2, T, T, 2, 2, d, "fp32", causal, None, "fp32_small"))


@pytest.mark.parametrize("Lq,Lkv,causal", [(300, 1000, True), (1000, 300, True), (257, 1500, False),
                                           (130, 129, True)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_lq_ne_lkv(Lq, Lkv, causal, dtype):
    run_fwd(W.Problem(2, Lq, Lkv, 4, 2, 128, dtype, causal, None, "lq_ne_lkv"))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("fp32", 128)])
def test_kvlens_gqa_small(causal, dtype, d):
    p = W.Problem(4, 256, 2048, 8, 2, d, dtype, causal, (1900, 700, 1, 0), "kvlen_small")
    q, k, v, o, lse = run_fwd(p)
    o_np, lse_np = to_np(o), to_np(lse)
    # batch 3 has no key: zeros and -inf; batch 2 has one key: exactly v_0 (non-causal)
    assert np.all(o_np[3] == 0) and np.all(lse_np[3] == -np.inf)
    if not causal:
        vk = to_np(v)[2, 0]  # [Hkv, d]
        G = p.Hq // p.Hkv
        for h in range(p.Hq):
            assert np.array_equal(o_np[2, :, h], np.broadcast_to(vk[h // G], o_np[2, :, h].shape))


def test_headline_sampled():
    """bf16 causal B4 H8 T8192 d128 at full size, sampled rows of two heads."""
    p = W.headline()
    rows = np.unique(np.concatenate([np.arange(0, 8192, 509), [0, 1, 127, 128, 255, 256, 4095, 8190, 8191]]))
    run_fwd(p, rows=rows, heads=[0, 5])


def test_kvlen_gqa_full_sampled():
    """KVLenMask + GQA + Lq != Lkv at full size (B4 Hq8 Hkv2 Lq2048 Lkv16384)."""
    p = W.kvlen_gqa()
    rows = np.unique(np.concatenate([np.arange(0, 2048, 97), [2047]]))
    run_fwd(p, rows=rows, heads=[0, 3, 6])


@pytest.mark.parametrize("T", W.RAGGED_T)
def test_ragged_full_sampled(T):
    p = W.grid(T, 128, True)
    rows = np.unique(np.concatenate([np.arange(0, T, 37), [T - 1]]))
    run_fwd(p, rows=rows, heads=[1, 7])
