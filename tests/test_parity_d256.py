"""head_dim 256 against the fp64 oracle: its own tensor-core kernels (one
query tile per forward CTA, 64-key steps), bf16 and fp16, with every mask
kind, KV lengths, GQA, Lq != Lkv and ragged tails."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu


def kvt(kl):
    return None if kl is None else torch.tensor(kl, dtype=torch.int32).cuda()


CASES = [
    # B, Lq, Lkv, Hq, Hkv, causal, kv_lens, window
    (2, 600, 600, 4, 2, True, None, None),
    (2, 300, 900, 4, 4, False, None, None),
    (2, 900, 300, 2, 2, True, None, None),
    (3, 256, 700, 8, 2, False, (700, 129, 0), None),
    (2, 500, 500, 2, 1, False, None, (64, 0)),
    (1, 64, 64, 1, 1, False, None, None),
    (1, 1, 5, 2, 1, False, None, None),
]


def segments_of(B, L, seed):
    rng = np.random.default_rng(seed)
    out = np.zeros((B, L), dtype=np.int32)
    for b in range(B):
        i, doc = 0, 0
        while i < L:
            n = int(rng.integers(1, 300))
            out[b, i:i + n] = doc
            i, doc = i + n, doc + 1
    return out


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("case", CASES)
def test_d256_forward(case, dtype):
    import exact_attention_34_gb300 as ea

    B, Lq, Lkv, Hq, Hkv, causal, kl, win = case
    p = W.Problem(B, Lq, Lkv, Hq, Hkv, 256, dtype, causal, kl, "d256")
    q, k, v, _ = W.make_inputs(p)
    o, lse = ea.forward(*cuda(q, k, v), causal=causal, kv_lens=kvt(kl), window=win)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    o_ref, lse_ref = oracle.forward(q, k, v, causal=causal, kv_lens=kl, window=win)
    assert rel_err(to_np(o), o_ref) <= TOL[dtype]
    lse_check(to_np(lse), lse_ref, TOL[dtype])


@pytest.mark.parametrize("use_info", [True, False])
def test_d256_forward_segments(use_info):
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 700, 700, 4, 2, 256, "bf16", True, None, "d256seg")
    q, k, v, _ = W.make_inputs(p)
    ids = segments_of(2, 700, 3)
    segs = (torch.tensor(ids).cuda(), torch.tensor(ids).cuda())
    if not use_info:
        segs = segs + (None,)
    o, lse = ea.forward(*cuda(q, k, v), causal=True, segments=segs)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    o_ref, lse_ref = oracle.forward(q, k, v, causal=True, segments=(ids, ids))
    assert rel_err(to_np(o), o_ref) <= TOL["bf16"]
    lse_check(to_np(lse), lse_ref, TOL["bf16"])


def test_d256_forward_full_size_sampled():
    """bf16 causal B2 H4 T8192 d256; the oracle checks one (batch, head)."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 8192, 8192, 4, 4, 256, "bf16", True, None, "d256big")
    q, k, v, _ = W.make_inputs(p)
    o, lse = ea.forward(*cuda(q, k, v), causal=True)
    torch.cuda.synchronize()
    b, h = 1, 2
    sl = lambda t: t[b:b + 1, :, h:h + 1]  # noqa: E731
    o_ref, lse_ref = oracle.forward(sl(q), sl(k), sl(v), causal=True)
    assert rel_err(to_np(sl(o)), o_ref) <= TOL["bf16"]
    lse_check(to_np(lse[b:b + 1, h:h + 1]), lse_ref, TOL["bf16"])


def check_bwd(p, window=None, segments=None, deterministic=True, seed=0):
    import exact_attention_34_gb300 as ea

    q, k, v, do = W.make_inputs(p, seed)
    qd, kd, vd, dod = cuda(q, k, v, do)
    kl = kvt(p.kv_lens)
    segs = None if segments is None else (torch.tensor(segments[0]).cuda(), torch.tensor(segments[1]).cuda())
    o, lse = ea.forward(qd, kd, vd, causal=p.causal, kv_lens=kl, window=window, segments=segs)
    grads = ea.backward(qd, kd, vd, o, lse, dod, causal=p.causal, kv_lens=kl, window=window, segments=segs,
                        deterministic=deterministic)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    ref = oracle.backward(q, k, v, do, causal=p.causal, kv_lens=p.kv_lens, window=window, segments=segments)
    gmax = max(float(np.max(np.abs(r))) for r in ref) or 1.0
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        g = to_np(g)
        assert np.all(np.isfinite(g)), name
        scale = max(float(np.max(np.abs(r))), 0.1 * gmax)  # single-key rows: exact zeros, bound the noise
        err = float(np.max(np.abs(g - r))) / scale
        assert err <= TOL[p.dtype], f"{name} rel err {err:.3e}"
    return grads


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("case", CASES)
def test_d256_backward(case, dtype, deterministic):
    B, Lq, Lkv, Hq, Hkv, causal, kl, win = case
    check_bwd(W.Problem(B, Lq, Lkv, Hq, Hkv, 256, dtype, causal, kl, "d256bwd"), window=win,
              deterministic=deterministic)


@pytest.mark.parametrize("use_causal", [False, True])
def test_d256_backward_segments(use_causal):
    p = W.Problem(2, 700, 700, 4, 2, 256, "bf16", use_causal, None, "d256segbwd")
    ids = segments_of(2, 700, 5)
    check_bwd(p, segments=(ids, ids))


def test_d256_backward_is_bitwise_reproducible():
    p = W.Problem(2, 700, 700, 4, 2, 256, "bf16", True, None, "d256rep")
    g1 = check_bwd(p)
    g2 = check_bwd(p)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_d256_backward_full_size_sampled():
    """bf16 causal B2 Hq8 Hkv2 T4096 d256; the oracle checks one KV group of batch 1."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 4096, 4096, 8, 2, 256, "bf16", True, None, "d256bwdbig")
    q, k, v, do = W.make_inputs(p)
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, causal=True)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    b, hk, G = 1, 1, 4
    sq = lambda t: t[b:b + 1, :, hk * G:(hk + 1) * G]  # noqa: E731
    sk = lambda t: t[b:b + 1, :, hk:hk + 1]  # noqa: E731
    ref = oracle.backward(sq(q), sk(k), sk(v), sq(do), causal=True)
    for name, g, r in zip(("dQ", "dK", "dV"), (sq(dq), sk(dk), sk(dv)), ref):
        e = rel_err(to_np(g), r)
        assert e <= TOL["bf16"], f"{name} rel err {e:.3e}"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("Lq,causal", [(1, False), (16, True)])
def test_d256_decode(Lq, causal, dtype):
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, Lq, 3000, 8, 2, 256, dtype, causal, (3000, 900), "dec256")
    q, k, v, _ = W.make_inputs(p)
    o, lse = ea.decode(*cuda(q, k, v), causal=causal, kv_lens=kvt(p.kv_lens), num_splits=4)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    o_ref, lse_ref = oracle.forward(q, k, v, causal=causal, kv_lens=p.kv_lens)
    assert rel_err(to_np(o), o_ref) <= TOL[dtype]
    lse_check(to_np(lse), lse_ref, TOL[dtype])
