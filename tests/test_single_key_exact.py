"""A row whose softmax runs over a single key has probability exactly 1, so
its output is that key's value row, bit for bit, whatever the dtype, and its
log-sum-exp is the scaled score.  This pins the kernels' running row maximum
exactly: a maximum taken over anything but the row's valid scores (a stale
column, a read past the tile) leaves P below 1 and moves O by an ulp, which
the relative tolerances of the other parity tests cannot see.  Covers the
head_dim 64/128/256 forwards (bf16, fp16), the split forward, segment masks
and the split-KV decode."""

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(B, Lq, Lkv, Hq, Hkv, d, dtype, seed=0):
    p = W.Problem(B, Lq, Lkv, Hq, Hkv, d, dtype, False, None, "single_key")
    q, k, v = (t.cuda() for t in W.make_inputs(p, seed, with_do=False))
    return q, k, v


def _expect_v0(o, v, rows_mask=None):
    """o[b, i, h] == v[b, 0, h // G] for every (b, i, h) the mask selects."""
    B, Lq, Hq, d = o.shape
    G = Hq // v.shape[2]
    v0 = v[:, 0].repeat_interleave(G, dim=1)[:, None].expand(B, Lq, Hq, d)
    same = (o == v0).all(dim=-1)
    if rows_mask is not None:
        same = same | ~rows_mask
    bad = (~same).nonzero()
    assert bad.numel() == 0, f"{bad.shape[0]} rows differ from v0, first {bad[:4].tolist()}"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_kv_length_one(d, dtype):
    import exact_attention_34_gb300 as ea

    q, k, v = _inputs(3, 300, 520, 8, 2, d, dtype)
    kl = torch.ones(3, dtype=torch.int32, device="cuda")
    o, lse = ea.forward(q, k, v, kv_lens=kl)
    torch.cuda.synchronize()
    _expect_v0(o, v)
    # lse = scale * <q, k0>, computed here in float64 from the same rounded inputs
    G = 4
    k0 = k[:, 0].double().repeat_interleave(G, dim=1)  # [B, Hq, d]
    ref = (q.double() * k0[:, None]).sum(-1).permute(0, 2, 1) / np.sqrt(d)
    assert float((lse.double() - ref).abs().max()) <= 1e-5 * max(1.0, float(ref.abs().max()))


@pytest.mark.parametrize("d", [32, 64, 128])
def test_kv_length_one_fp32(d):
    """float32: head_dim 64/128 run on the tensor cores with split operands
    (V in three exact bf16 parts, P = 1 exact), 32 on the CUDA cores."""
    import exact_attention_34_gb300 as ea

    q, k, v = _inputs(3, 300, 520, 8, 2, d, "fp32")
    kl = torch.ones(3, dtype=torch.int32, device="cuda")
    o, _ = ea.forward(q, k, v, kv_lens=kl)
    torch.cuda.synchronize()
    _expect_v0(o, v)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_causal_first_row(d):
    """Equal lengths, causal: row 0 sees key 0 only."""
    import exact_attention_34_gb300 as ea

    q, k, v = _inputs(2, 384, 384, 4, 4, d, "bf16", seed=3)
    o, _ = ea.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o[:, 0], v[:, 0])


def test_segments_single_matching_key():
    """kv length 1 under a segment mask: rows whose id matches key 0's id see
    exactly that key; the others see none (o = 0)."""
    import exact_attention_34_gb300 as ea

    rng = np.random.default_rng(7)
    for d in (32, 64, 128):
        q, k, v = _inputs(3, 300, 520, 8, 2, d, "bf16")
        qs = rng.integers(0, 3, size=(3, 300)).astype(np.int32)
        ks = rng.integers(0, 3, size=(3, 520)).astype(np.int32)
        kl = torch.tensor([520, 200, 1], dtype=torch.int32, device="cuda")
        o, lse = ea.forward(q, k, v, kv_lens=kl, segments=(torch.tensor(qs).cuda(), torch.tensor(ks).cuda()))
        torch.cuda.synchronize()
        match = torch.tensor(qs[2] == ks[2, 0], device="cuda")[:, None].expand(300, 8)
        _expect_v0(o[2:3], v[2:3], match[None])
        assert torch.all(o[2][~match] == 0) and torch.all(torch.isneginf(lse[2].T[~match]))


def test_split_forward_and_decode():
    import exact_attention_34_gb300 as ea

    q, k, v = _inputs(2, 512, 8192, 8, 2, 128, "bf16", seed=5)
    kl = torch.ones(2, dtype=torch.int32, device="cuda")
    o, _ = ea.forward(q, k, v, kv_lens=kl, num_splits=4)
    torch.cuda.synchronize()
    _expect_v0(o, v)
    qd = q[:, :1].contiguous()
    od, _ = ea.decode(qd, k, v, kv_lens=kl, num_splits=3)
    torch.cuda.synchronize()
    _expect_v0(od, v)
