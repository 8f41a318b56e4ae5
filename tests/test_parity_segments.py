"""Segment (document) masks on the GPU against the fp64 oracle: packed
documents (sorted ids) and arbitrary unsorted ids, with causal and window
masks, KV lengths, GQA, Lq != Lkv, all dtypes and both backward variants."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu


def doc_ids(B, L, seed, mean_len):
    """Packed documents: ids 0, 1, 2, ... in runs of random length."""
    rng = np.random.default_rng(seed)
    out = np.zeros((B, L), dtype=np.int32)
    for b in range(B):
        i, doc = 0, 0
        while i < L:
            n = int(rng.integers(1, 2 * mean_len))
            out[b, i:i + n] = doc
            i, doc = i + n, doc + 1
    return out


def check(p, qs, ks, window=None, deterministic=True, seed=0):
    import exact_attention_34_gb300 as ea

    q, k, v, do = W.make_inputs(p, seed)
    qd, kd, vd, dod = cuda(q, k, v, do)
    segs = (torch.tensor(qs).cuda(), torch.tensor(ks).cuda())
    kl = None if p.kv_lens is None else torch.tensor(p.kv_lens, dtype=torch.int32).cuda()
    o, lse = ea.forward(qd, kd, vd, causal=p.causal, kv_lens=kl, window=window, segments=segs)
    grads = ea.backward(qd, kd, vd, o, lse, dod, causal=p.causal, kv_lens=kl, window=window, segments=segs,
                        deterministic=deterministic)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    tol = TOL[p.dtype]
    win = window if window is not None else None
    o_ref, lse_ref = oracle.forward(q, k, v, causal=p.causal, kv_lens=p.kv_lens, window=win, segments=(qs, ks))
    assert rel_err(to_np(o), o_ref) <= tol
    lse_check(to_np(lse), lse_ref, tol)
    ref = oracle.backward(q, k, v, do, causal=p.causal, kv_lens=p.kv_lens, window=win, segments=(qs, ks))
    gmax = max(float(np.max(np.abs(r))) for r in ref) or 1.0
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        g = to_np(g)
        assert np.all(np.isfinite(g)), name
        scale = max(float(np.max(np.abs(r))), 0.1 * gmax)  # single-key rows: exact zeros, bound the noise
        assert float(np.max(np.abs(g - r))) / scale <= tol, name
    return o, lse


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_documents(causal, dtype, deterministic):
    p = W.Problem(2, 700, 700, 4, 2, 128, dtype, causal, None, "docs")
    ids = doc_ids(2, 700, 1, 150)
    check(p, ids, ids, deterministic=deterministic)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d", [32, 64])
def test_unsorted_ids_lq_ne_lkv_kvlens(dtype, d):
    rng = np.random.default_rng(7)
    p = W.Problem(3, 300, 520, 8, 2, d, dtype, False, (520, 200, 1), "unsorted")
    qs = rng.integers(0, 3, size=(3, 300)).astype(np.int32)
    ks = rng.integers(0, 3, size=(3, 520)).astype(np.int32)
    check(p, qs, ks)


@pytest.mark.parametrize("deterministic", [True, False])
def test_segments_with_window(deterministic):
    p = W.Problem(2, 600, 600, 4, 4, 128, "bf16", False, None, "segwin")
    ids = doc_ids(2, 600, 2, 200)
    check(p, ids, ids, window=(100, 0), deterministic=deterministic)


def test_rows_without_a_matching_key():
    """Query ids that no key carries give o = 0 and lse = -inf."""
    p = W.Problem(1, 256, 256, 2, 2, 128, "bf16", False, None, "nomatch")
    qs = np.zeros((1, 256), dtype=np.int32)
    qs[0, 100:140] = 7  # no key has id 7
    ks = np.zeros((1, 256), dtype=np.int32)
    o, lse = check(p, qs, ks)
    assert torch.all(o[0, 100:140] == 0)
    assert torch.all(lse[0, :, 100:140] == -float("inf"))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_one_shared_id_equals_no_mask(dtype):
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 400, 400, 4, 2, 64, dtype, True, None, "sameid")
    q, k, v, do = (t.cuda() for t in W.make_inputs(p))
    z = torch.zeros(2, 400, dtype=torch.int32, device="cuda")
    a = ea.forward(q, k, v, causal=True, segments=(z, z))
    b = ea.forward(q, k, v, causal=True)
    tol = TOL[dtype] / 10
    assert rel_err(to_np(a[0]), to_np(b[0])) <= tol
    ga = ea.backward(q, k, v, a[0], a[1], do, causal=True, segments=(z, z))
    gb = ea.backward(q, k, v, b[0], b[1], do, causal=True)
    for x, y in zip(ga, gb):
        assert rel_err(to_np(x), to_np(y)) <= tol
