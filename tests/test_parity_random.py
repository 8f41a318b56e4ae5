"""Seeded random configurations against the fp64 oracle: dtype, head_dim,
lengths (tile multiples, ragged, one), GQA group, KV lengths (incl. 0, 1 and
past Lkv), causal or a window, and the backward variant are drawn together, so
combinations no hand-written case lists are exercised too."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    dtype = ["bf16", "fp16", "fp32"][rng.integers(3)]
    d = int(rng.choice([32, 64, 128]))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 4))
    lens = [1, 17, 64, 127, 128, 129, 300, 511, 700]
    Lq, Lkv = int(rng.choice(lens)), int(rng.choice(lens))
    mask = rng.integers(3)  # 0 none, 1 causal, 2 window
    window = None
    causal = mask == 1
    if mask == 2:
        window = (int(rng.choice([-1, 0, 5, 100, 400])), int(rng.choice([-1, 0, 3, 64])))
    kv_lens = None
    if rng.random() < 0.5:
        kv_lens = [int(rng.choice([0, 1, Lkv // 2, Lkv, Lkv + 7])) for _ in range(B)]
    deterministic = bool(rng.random() < 0.6)
    return W.Problem(B, Lq, Lkv, Hkv * G, Hkv, d, dtype, causal, kv_lens, f"rand{seed}"), window, deterministic


@pytest.mark.parametrize("seed", range(40))
def test_random_configuration(seed):
    import exact_attention_34_gb300 as ea

    p, window, deterministic = draw(seed)
    q, k, v, do = W.make_inputs(p, seed)
    qd, kd, vd, dod = cuda(q, k, v, do)
    kl = None if p.kv_lens is None else torch.tensor(p.kv_lens, dtype=torch.int32).cuda()
    o, lse = ea.forward(qd, kd, vd, causal=p.causal, kv_lens=kl, window=window)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, causal=p.causal, kv_lens=kl, window=window,
                             deterministic=deterministic)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    tol = TOL[p.dtype]
    o_ref, lse_ref = oracle.forward(q, k, v, causal=p.causal, kv_lens=p.kv_lens, window=window)
    assert rel_err(to_np(o), o_ref) <= tol, ("O", p, window)
    lse_check(to_np(lse), lse_ref, tol)
    ref = oracle.backward(q, k, v, do, causal=p.causal, kv_lens=p.kv_lens, window=window)
    # a tensor whose exact gradient is (nearly) all zero -- e.g. dQ and dK when
    # every valid row has a single key -- only carries rounding noise; bound it
    # against the largest reference gradient instead of its own zero scale
    gmax = max(float(np.max(np.abs(r))) if r.size else 0.0 for r in ref) or 1.0
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        g = to_np(g)
        assert np.all(np.isfinite(g)), (name, p, window)
        scale = max(float(np.max(np.abs(r))) if r.size else 0.0, 0.1 * gmax)
        err = float(np.max(np.abs(g - r))) / scale if r.size else 0.0
        assert err <= tol, (name, err, p, window, deterministic)


def draw_ext(seed):
    """Also head_dim 256 (16-bit only) and segment ids (packed runs or i.i.d.
    ids from a small range, with or without the block summary)."""
    rng = np.random.default_rng(5000 + seed)
    dtype = ["bf16", "fp16", "fp32"][rng.integers(3)]
    d = int(rng.choice([32, 64, 128, 256] if dtype != "fp32" else [32, 64, 128]))
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 4))
    lens = [1, 64, 129, 255, 300, 511, 700]
    Lq, Lkv = int(rng.choice(lens)), int(rng.choice(lens))
    mask = rng.integers(3)  # 0 none, 1 causal, 2 window
    window = None
    causal = mask == 1
    if mask == 2:
        window = (int(rng.choice([-1, 0, 5, 100, 400])), int(rng.choice([-1, 0, 3, 64])))
    kv_lens = None
    if rng.random() < 0.4:
        kv_lens = [int(rng.choice([0, 1, Lkv // 2, Lkv])) for _ in range(B)]
    segments = None
    if rng.random() < 0.5:
        def ids(L):
            if rng.random() < 0.5:  # packed runs
                out = np.zeros((B, L), dtype=np.int32)
                for b in range(B):
                    i, doc = 0, 0
                    while i < L:
                        n = int(rng.integers(1, 200))
                        out[b, i:i + n] = doc
                        i, doc = i + n, doc + 1
                return out
            return rng.integers(0, 4, size=(B, L)).astype(np.int32)
        segments = (ids(Lq), ids(Lkv), bool(rng.random() < 0.7))
    deterministic = bool(rng.random() < 0.6)
    p = W.Problem(B, Lq, Lkv, Hkv * G, Hkv, d, dtype, causal, kv_lens, f"randx{seed}")
    return p, window, segments, deterministic


@pytest.mark.parametrize("seed", range(40))
def test_random_configuration_with_segments_and_d256(seed):
    import exact_attention_34_gb300 as ea

    p, window, segments, deterministic = draw_ext(seed)
    q, k, v, do = W.make_inputs(p, seed)
    qd, kd, vd, dod = cuda(q, k, v, do)
    kl = None if p.kv_lens is None else torch.tensor(p.kv_lens, dtype=torch.int32).cuda()
    segs, seg_np = None, None
    if segments is not None:
        seg_np = (segments[0], segments[1])
        segs = (torch.tensor(segments[0]).cuda(), torch.tensor(segments[1]).cuda())
        if not segments[2]:
            segs = segs + (None,)
    o, lse = ea.forward(qd, kd, vd, causal=p.causal, kv_lens=kl, window=window, segments=segs)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, causal=p.causal, kv_lens=kl, window=window, segments=segs,
                             deterministic=deterministic)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    tol = TOL[p.dtype]
    ctx = (p, window, segments is not None, deterministic)
    o_ref, lse_ref = oracle.forward(q, k, v, causal=p.causal, kv_lens=p.kv_lens, window=window, segments=seg_np)
    assert rel_err(to_np(o), o_ref) <= tol, ("O", ctx)
    lse_check(to_np(lse), lse_ref, tol)
    ref = oracle.backward(q, k, v, do, causal=p.causal, kv_lens=p.kv_lens, window=window, segments=seg_np)
    gmax = max(float(np.max(np.abs(r))) if r.size else 0.0 for r in ref) or 1.0
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        g = to_np(g)
        assert np.all(np.isfinite(g)), (name, ctx)
        scale = max(float(np.max(np.abs(r))) if r.size else 0.0, 0.1 * gmax)
        err = float(np.max(np.abs(g - r))) / scale if r.size else 0.0
        assert err <= tol, (name, err, ctx)
