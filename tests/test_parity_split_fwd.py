"""GPU parity of the split forward (attn_fwd_split): each pair of query tiles
cuts its key range into pieces that write float32 partials, and the
log-sum-exp combine merges them.  Checked against the fp64 oracle over the
masks it takes (KV lengths with empty and one-key batch elements, causal,
windows, GQA, ragged lengths, head_dim 32/64/128, bf16/fp16), at piece counts
from 2 to more pieces than tiles, at the full KVLenMask + GQA workload
(sampled rows), for a backward fed by its o and lse, and run to run."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu


def kv_tensor(p):
    return None if p.kv_lens is None else torch.tensor(p.kv_lens, dtype=torch.int32).cuda()


def check(p, num_splits, window=None, seed=0, rows=None, heads=None):
    import exact_attention_34_gb300 as ea

    q, k, v = W.make_inputs(p, seed, with_do=False)
    causal = p.causal if window is None else False
    o, lse = ea.forward(*cuda(q, k, v), causal=causal, kv_lens=kv_tensor(p), window=window, num_splits=num_splits)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    o_ref, lse_ref = oracle.forward(q, k, v, causal=causal, kv_lens=p.kv_lens, window=window, rows=rows, heads=heads)
    o_np, lse_np = to_np(o), to_np(lse)
    if rows is not None:
        o_np, lse_np = o_np[:, rows], lse_np[:, :, rows]
    if heads is not None:
        o_np, o_ref = o_np[:, :, heads], o_ref[:, :, heads]
        lse_np, lse_ref = lse_np[:, heads], lse_ref[:, heads]
    tol = TOL[p.dtype]
    e = rel_err(o_np, o_ref)
    assert e <= tol, f"{p.name} splits={num_splits}: O rel err {e:.3e}"
    lse_check(lse_np, lse_ref, tol)
    return q, k, v, o, lse


@pytest.mark.parametrize("num_splits", [0, 2, 3, 8, 64])
def test_kv_lengths_gqa(num_splits):
    """Most keys in one batch element, one with a single key, one with none;
    64 pieces is more pieces than the 40 key tiles (one tile a piece)."""
    p = W.Problem(4, 300, 5000, 8, 2, 128, "bf16", False, (4700, 236, 1, 0), "split_kvlen")
    check(p, num_splits)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_causal_ragged(d, dtype):
    p = W.Problem(1, 1500, 1500, 2, 1, d, dtype, True, None, "split_causal")
    check(p, 4)


@pytest.mark.parametrize("window", [(700, 30), (-1, 0), (200, -1), (0, 0)])
def test_windows_with_kv_lengths(window):
    p = W.Problem(2, 900, 3000, 4, 2, 64, "bf16", False, (2900, 1300), "split_window")
    check(p, 5, window=window)


def test_offset_causal_lq_below_lkv():
    """Bottom-right aligned causal with Lq < Lkv: a row's keys end at its
    diagonal; pieces of the upper pair hold fewer tiles than the lower."""
    p = W.Problem(2, 333, 4100, 4, 4, 128, "bf16", True, (4100, 2000), "split_offset")
    check(p, 3)


def test_all_empty():
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 200, 2048, 2, 2, 64, "bf16", False, (0, 0), "split_empty")
    q, k, v = (t.cuda() for t in W.make_inputs(p, 0, with_do=False))
    o, lse = ea.forward(q, k, v, kv_lens=kv_tensor(p), num_splits=4)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_matches_unsplit_and_is_reproducible():
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 512, 8192, 8, 2, 128, "bf16", True, (8192, 3000), "split_repro")
    q, k, v = (t.cuda() for t in W.make_inputs(p, 1, with_do=False))
    kl = kv_tensor(p)
    o1, l1 = ea.forward(q, k, v, causal=True, kv_lens=kl)
    o2, l2 = ea.forward(q, k, v, causal=True, kv_lens=kl, num_splits=6)
    o3, l3 = ea.forward(q, k, v, causal=True, kv_lens=kl, num_splits=6)
    torch.cuda.synchronize()
    assert torch.equal(o2, o3) and torch.equal(l2, l3)
    assert rel_err(to_np(o2), to_np(o1)) <= 1e-2
    assert float((l2 - l1).abs().max()) <= 1e-4 * max(1.0, float(l1.abs().max()))


@pytest.mark.parametrize("d,dtype", [(256, "bf16"), (128, "fp32")])
def test_unsplit_builds_ignore_num_splits(d, dtype):
    """head_dim 256 and float32 run the plain forward: the same bits."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(1, 300, 2000, 2, 1, d, dtype, True, None, "split_ignored")
    q, k, v = (t.cuda() for t in W.make_inputs(p, 0, with_do=False))
    o1, l1 = ea.forward(q, k, v, causal=True)
    o2, l2 = ea.forward(q, k, v, causal=True, num_splits=4)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_backward_from_split_forward():
    """The backward takes the combined o and lse as its residuals."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 400, 2600, 4, 2, 64, "bf16", False, (2600, 900), "split_bwd")
    q, k, v, do = W.make_inputs(p, 2)
    qd, kd, vd, dod = cuda(q, k, v, do)
    kl = kv_tensor(p)
    o, lse = ea.forward(qd, kd, vd, kv_lens=kl, num_splits=4)
    grads = ea.backward(qd, kd, vd, o, lse, dod, kv_lens=kl)
    torch.cuda.synchronize()
    for name, g, r in zip(("dQ", "dK", "dV"), grads, oracle.backward(q, k, v, do, kv_lens=p.kv_lens)):
        assert rel_err(to_np(g), r) <= TOL["bf16"], name


def test_kvlen_gqa_full_sampled():
    """The full KVLenMask + GQA workload (B4 Hq8 Hkv2 Lq2048 Lkv16384) with the
    library's piece count, sampled rows of three heads."""
    p = W.kvlen_gqa()
    rows = np.unique(np.concatenate([np.arange(0, 2048, 97), [0, 255, 256, 2047]]))
    check(p, 0, rows=rows, heads=[0, 3, 6])
