"""GPU backward parity (dQ, dK, dV and the delta preprocess) against the fp64
oracle, plus bitwise reproducibility of the two-pass backward."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, rel_err, to_np

pytestmark = pytest.mark.gpu


def kv_tensor(p):
    return None if p.kv_lens is None else torch.tensor(p.kv_lens, dtype=torch.int32).cuda()


def gpu_fwd_bwd(p, deterministic=True, seed=0):
    import exact_attention_34_gb300 as ea

    q, k, v, do = W.make_inputs(p, seed)
    qd, kd, vd, dod = cuda(q, k, v, do)
    kl = kv_tensor(p)
    o, lse = ea.forward(qd, kd, vd, causal=p.causal, kv_lens=kl)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, causal=p.causal, kv_lens=kl, deterministic=deterministic)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    return (q, k, v, do), (o, lse), (dq, dk, dv)


def check_grads(p, got, ref, tol=None):
    tol = TOL[p.dtype] if tol is None else tol
    for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
        e = rel_err(a, b)
        assert e <= tol, f"{p.name}: {name} rel err {e:.3e} > {tol:.0e}"


def run_bwd(p, deterministic=True):
    (q, k, v, do), _, (dq, dk, dv) = gpu_fwd_bwd(p, deterministic)
    ref = oracle.backward(q, k, v, do, causal=p.causal, kv_lens=p.kv_lens)
    check_grads(p, (to_np(dq), to_np(dk), to_np(dv)), ref)
    return dq, dk, dv


@pytest.mark.parametrize("deterministic", [True, False])
def test_tiny_fp32_exact_check(deterministic):
    run_bwd(W.tiny(), deterministic)


CASES = [(T, d, c) for T in (128, 600) for d in (64, 128) for c in (False, True)]


@pytest.mark.parametrize("T,d,causal", CASES)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_small_grid(T, d, causal, dtype):
    run_bwd(W.Problem(2, T, T, 2, 2, d, dtype, causal, None, f"bwd_T{T}_d{d}_c{int(causal)}_{dtype}"))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_atomic_variant(dtype):
    run_bwd(W.Problem(2, 600, 600, 4, 2, 128, dtype, True, None, "bwd_atomic"), deterministic=False)


@pytest.mark.parametrize("T,d,causal", CASES)
def test_atomic_small_grid(T, d, causal):
    run_bwd(W.Problem(2, T, T, 2, 2, d, "bf16", causal, None, f"atomic_T{T}_d{d}_c{int(causal)}"), False)


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("Lq,Lkv,causal", [(300, 1000, True), (1000, 300, True), (257, 700, False)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_lq_ne_lkv(Lq, Lkv, causal, dtype, deterministic):
    run_bwd(W.Problem(2, Lq, Lkv, 4, 2, 128, dtype, causal, None, "bwd_lq_ne_lkv"), deterministic)


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_kvlens_gqa_single_key_and_empty(deterministic, dtype):
    p = W.Problem(4, 256, 1500, 8, 2, 128, dtype, False, (1500, 700, 1, 0), "bwd_kvlen")
    dq, dk, dv = run_bwd(p, deterministic)
    dq, dk, dv = to_np(dq), to_np(dk), to_np(dv)
    # empty batch: all gradients zero; keys past the length: dK = dV = 0
    assert np.all(dq[3] == 0) and np.all(dk[3] == 0) and np.all(dv[3] == 0)
    assert np.all(dk[1, 700:] == 0) and np.all(dv[1, 700:] == 0)
    assert np.all(dk[2, 1:] == 0) and np.all(dv[2, 1:] == 0)
    # single valid key: exact dQ = dK = 0, kernel rounding noise only
    assert np.max(np.abs(dq[2])) <= 1e-2 * np.max(np.abs(dq))
    assert np.max(np.abs(dk[2])) <= 1e-2 * np.max(np.abs(dk))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_two_pass_is_bitwise_reproducible(dtype):
    p = W.Problem(2, 700, 700, 4, 2, 128, dtype, True, None, "bwd_repeat")
    _, _, g1 = gpu_fwd_bwd(p, True)
    _, _, g2 = gpu_fwd_bwd(p, True)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("fp32", 128)])
def test_preprocess(dtype, d):
    import exact_attention_34_gb300 as ea

    p = W.Problem(3, 333, 333, 4, 4, d, dtype, False, None, "pre")
    o, _, _, do = W.make_inputs(p, seed=5)  # any tensors: delta = rowsum(o * do)
    delta = torch.empty(p.B, p.Hq, p.Lq, device="cuda", dtype=torch.float32)
    ea.attn_bwd_preprocess(o.cuda(), do.cuda(), delta)
    torch.cuda.synchronize()
    ref = oracle.backward_preprocess(o, do)
    assert rel_err(to_np(delta), ref) <= 1e-5


@pytest.mark.parametrize("deterministic", [True, False])
def test_headline_full_size_one_head(deterministic):
    """bf16 causal B4 H8 T8192 d128, full-size run; the oracle checks batch 1, head 6."""
    p = W.headline()
    (q, k, v, do), _, (dq, dk, dv) = gpu_fwd_bwd(p, deterministic)
    b, h = 1, 6
    sl = lambda t: t[b:b + 1, :, h:h + 1]  # noqa: E731
    ref = oracle.backward(sl(q), sl(k), sl(v), sl(do), causal=True)
    check_grads(p, (to_np(sl(dq)), to_np(sl(dk)), to_np(sl(dv))), ref)


def test_kvlen_gqa_full_size_one_group():
    """KVLenMask + GQA config at full size; the oracle checks batch 0 and batch 2
    (single key), KV head 1 with its 4 query heads."""
    p = W.kvlen_gqa()
    (q, k, v, do), _, (dq, dk, dv) = gpu_fwd_bwd(p, True)
    G = p.Hq // p.Hkv
    for b in (0, 2):
        hk = 1
        sq = lambda t: t[b:b + 1, :, hk * G:(hk + 1) * G]  # noqa: E731
        sk = lambda t: t[b:b + 1, :, hk:hk + 1]  # noqa: E731
        ref = oracle.backward(sq(q), sk(k), sk(v), sq(do), kv_lens=[p.kv_lens[b]])
        got = (to_np(sq(dq)), to_np(sk(dk)), to_np(sk(dv)))
        if b == 2:  # exact gradients are dQ = dK = 0: absolute noise bound
            assert np.max(np.abs(got[0])) < 1e-2 and np.max(np.abs(got[1])) < 1e-2
            assert rel_err(got[2], ref[2]) <= TOL["bf16"]
        else:
            check_grads(p, got, ref)


def check_one_slice(p, inputs, grads, b, h):
    q, k, v, do = inputs
    sl = lambda t: t[b:b + 1, :, h:h + 1]  # noqa: E731
    ref = oracle.backward(sl(q), sl(k), sl(v), sl(do), causal=p.causal)
    check_grads(p, tuple(to_np(sl(g)) for g in grads), ref)


# The attention grid's largest cells and the ragged lengths at their full size
# (B4 H8), run through the same launch configuration the bench times (grouped
# launch order over all 32 (batch, head) pairs, the head_dim 64 K/V ring); the
# oracle checks two (batch, head) slices of each.
FULL = [(8192, 64, False, "bf16"), (8192, 64, True, "bf16"), (3000, 64, True, "bf16"), (3000, 128, True, "bf16"),
        (1500, 128, False, "bf16"), (2048, 128, True, "fp32")]


@pytest.mark.slow
@pytest.mark.parametrize("T,d,causal,dtype", FULL)
def test_grid_full_size_two_slices(T, d, causal, dtype):
    p = W.grid(T, d, causal, dtype)
    inputs, _, grads = gpu_fwd_bwd(p, True)
    for b, h in ((0, 3), (3, 7)):
        check_one_slice(p, inputs, grads, b, h)


@pytest.mark.slow
@pytest.mark.parametrize("T,d", [(8192, 64), (3000, 128)])
def test_grid_full_size_atomic(T, d):
    p = W.grid(T, d, True)
    inputs, _, grads = gpu_fwd_bwd(p, False)
    check_one_slice(p, inputs, grads, 2, 5)
