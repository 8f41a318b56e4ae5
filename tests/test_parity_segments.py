"""Segment (document) masks on the GPU against the fp64 oracle: packed
documents (sorted ids) and arbitrary unsorted ids, with causal and window
masks, KV lengths, GQA, Lq != Lkv, all dtypes and both backward variants;
with the block summary (tile skipping, single-id tiles unmasked) and without
it; and the block summary itself against a brute-force count."""

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


def check(p, qs, ks, window=None, deterministic=True, seed=0, use_info=True):
    import exact_attention_34_gb300 as ea

    q, k, v, do = W.make_inputs(p, seed)
    qd, kd, vd, dod = cuda(q, k, v, do)
    segs = (torch.tensor(qs).cuda(), torch.tensor(ks).cuda())
    if not use_info:
        segs = segs + (None,)
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


@pytest.mark.parametrize("use_info", [True, False])
@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_documents(causal, dtype, deterministic, use_info):
    p = W.Problem(2, 700, 700, 4, 2, 128, dtype, causal, None, "docs")
    ids = doc_ids(2, 700, 1, 150)
    check(p, ids, ids, deterministic=deterministic, use_info=use_info)


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_block_aligned_documents(d, deterministic):
    """Documents of 256 and 384 tokens: every tile inside a document holds one
    id on both sides (the unmasked path), tiles across documents are dropped."""
    p = W.Problem(2, 1664, 1664, 4, 2, d, "bf16", True, None, "aligned_docs")
    lens = [256, 384, 256, 384, 384]
    ids = np.repeat(np.arange(len(lens), dtype=np.int32), lens)[None].repeat(2, 0)
    check(p, ids, ids, deterministic=deterministic)


def block_shuffled_ids(B, L, seed, nblk_ids):
    """Ids constant over 128-blocks in a shuffled order, with some blocks split
    in two at a ragged offset: query tiles of one CTA see disjoint key ranges."""
    rng = np.random.default_rng(seed)
    nb = (L + 127) // 128
    out = np.zeros((B, L), dtype=np.int32)
    for b in range(B):
        ids = rng.permutation(nblk_ids)[:nb] if nb <= nblk_ids else rng.integers(0, nblk_ids, nb)
        for i in range(nb):
            out[b, 128 * i:128 * (i + 1)] = ids[i]
            if rng.random() < 0.3:
                cut = 128 * i + int(rng.integers(1, 127))
                out[b, cut:128 * (i + 1)] = rng.integers(0, nblk_ids)
    return out


@pytest.mark.parametrize("use_info", [True, False])
@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("causal", [False, True])
def test_block_shuffled_ids(causal, deterministic, use_info):
    p = W.Problem(2, 1100, 900, 4, 2, 128, "bf16", causal, None, "shuffled")
    qs = block_shuffled_ids(2, 1100, 3, 12)
    ks = block_shuffled_ids(2, 900, 4, 12)
    check(p, qs, ks, deterministic=deterministic, use_info=use_info)


def summary_brute_force(qs, ks):
    """Expected block summary: per 128-block (min id, max id, other-side span)."""
    def blocks(ids):
        return [ids[i:i + 128] for i in range(0, len(ids), 128)]

    B, Lq = qs.shape
    Lkv = ks.shape[1]
    qrec, krec = [], []
    for b in range(B):
        qb, kb = blocks(qs[b]), blocks(ks[b])
        qmm = [(int(x.min()), int(x.max())) for x in qb]
        kmm = [(int(x.min()), int(x.max())) for x in kb]
        for mine, other, L_other, out in ((qmm, kmm, Lkv, qrec), (kmm, qmm, Lq, krec)):
            for lo, hi in mine:
                hit = [c for c, (olo, ohi) in enumerate(other) if olo <= hi and ohi >= lo]
                span = (128 * hit[0], min(L_other, 128 * (hit[-1] + 1))) if hit else (0, 0)
                out.append((lo, hi) + span)
    return np.array(qrec + krec, dtype=np.int32)


@pytest.mark.parametrize("B,Lq,Lkv,kind", [(3, 700, 300, "random"), (2, 1100, 900, "shuffled"),
                                           (1, 5000, 5000, "docs"), (2, 1, 129, "random"),
                                           (1, 40000, 300, "shuffled")])
def test_segment_info_matches_brute_force(B, Lq, Lkv, kind):
    import exact_attention_34_gb300 as ea

    rng = np.random.default_rng(B * 7 + Lq)
    if kind == "random":
        qs = rng.integers(-5, 5, size=(B, Lq)).astype(np.int32)
        ks = rng.integers(-5, 5, size=(B, Lkv)).astype(np.int32)
    elif kind == "shuffled":
        qs, ks = block_shuffled_ids(B, Lq, 1, 400), block_shuffled_ids(B, Lkv, 2, 400)
    else:
        qs = doc_ids(B, Lq, 5, 300)
        ks = qs.copy()
    info = ea.segment_info(torch.tensor(qs).cuda(), torch.tensor(ks).cuda())
    torch.cuda.synchronize()
    got = info.cpu().view(torch.int32).numpy().reshape(-1, 4)
    np.testing.assert_array_equal(got, summary_brute_force(qs, ks))


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
