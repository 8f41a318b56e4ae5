"""The single-pass backward with dQ added in key-tile order (deterministic = 2)
against the fp64 oracle, and its bitwise reproducibility.

Each 128-row query tile's dQ is a sum over the key tiles that see it, taken
in increasing key-tile order through a turn counter per query tile; the CTAs
take their key tiles from a ticket counter.  These tests cover the masks
(none, causal, windows, KV lengths with empty and single-key batches,
segments with and without the block summary), GQA, Lq != Lkv, ragged tails,
head_dim 32/64/128 and both 16-bit formats; repeat runs must agree bit for
bit, on small problems and at the full headline size, where 152 CTAs at a
time claim 2048 key tiles and wait on one another's turns."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, rel_err, to_np

pytestmark = pytest.mark.gpu

ORDERED = 2


def run(p, window=None, segments=None, seed=0):
    import exact_attention_34_gb300 as ea

    q, k, v, do = W.make_inputs(p, seed)
    qd, kd, vd, dod = cuda(q, k, v, do)
    kl = None if p.kv_lens is None else torch.tensor(p.kv_lens, dtype=torch.int32).cuda()
    segs = None
    if segments is not None:
        segs = (torch.tensor(segments[0]).cuda(), torch.tensor(segments[1]).cuda())
        if not segments[2]:
            segs = segs + (None,)
    o, lse = ea.forward(qd, kd, vd, causal=p.causal, kv_lens=kl, window=window, segments=segs)
    grads = ea.backward(qd, kd, vd, o, lse, dod, causal=p.causal, kv_lens=kl, window=window, segments=segs,
                        deterministic=ORDERED)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    return (q, k, v, do), grads


def check(p, window=None, segments=None, seed=0):
    (q, k, v, do), grads = run(p, window, segments, seed)
    seg_np = None if segments is None else (segments[0], segments[1])
    ref = oracle.backward(q, k, v, do, causal=p.causal, kv_lens=p.kv_lens, window=window, segments=seg_np)
    tol = TOL[p.dtype]
    gmax = max(float(np.max(np.abs(r))) if r.size else 0.0 for r in ref) or 1.0
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        g = to_np(g)
        assert np.all(np.isfinite(g)), name
        # single-key rows have exact zero dQ/dK: bound their noise by the largest gradient
        scale = max(float(np.max(np.abs(r))) if r.size else 0.0, 0.1 * gmax)
        err = float(np.max(np.abs(g - r))) / scale if r.size else 0.0
        assert err <= tol, (name, err, p.name, window)
    return grads


CASES = [(T, d, c) for T in (128, 600, 1100) for d in (64, 128) for c in (False, True)]


@pytest.mark.parametrize("T,d,causal", CASES)
def test_small_grid(T, d, causal):
    check(W.Problem(2, T, T, 2, 2, d, "bf16", causal, None, f"ordered_T{T}_d{d}_c{int(causal)}"))


@pytest.mark.parametrize("Lq,Lkv,causal", [(300, 1000, True), (1000, 300, True), (257, 700, False), (1, 900, True)])
def test_lq_ne_lkv(Lq, Lkv, causal):
    check(W.Problem(2, Lq, Lkv, 4, 2, 128, "bf16", causal, None, "ordered_lq_ne_lkv"))


@pytest.mark.parametrize("causal", [False, True])
def test_kvlens_gqa_single_key_and_empty(causal):
    p = W.Problem(4, 256, 1500, 8, 2, 128, "bf16", causal, (1500, 700, 1, 0), "ordered_kvlen")
    dq, dk, dv = (to_np(g) for g in check(p))
    assert np.all(dq[3] == 0) and np.all(dk[3] == 0) and np.all(dv[3] == 0)
    assert np.all(dk[1, 700:] == 0) and np.all(dv[1, 700:] == 0)


@pytest.mark.parametrize("window", [(100, 50), (0, 0), (300, -1), (-1, 200)])
def test_windows(window):
    check(W.Problem(2, 900, 1000, 4, 2, 128, "bf16", False, (1000, 640), "ordered_window"), window=window)


@pytest.mark.parametrize("use_info", [True, False])
def test_segments(use_info):
    rng = np.random.default_rng(3)
    B, L = 2, 700

    def docs():
        out = np.zeros((B, L), dtype=np.int32)
        for b in range(B):
            i, doc = 0, 0
            while i < L:
                n = int(rng.integers(1, 300))
                out[b, i:i + n] = doc
                i, doc = i + n, doc + 1
        return out

    ids = docs()
    check(W.Problem(B, L, L, 4, 4, 64, "bf16", True, None, "ordered_segments"), segments=(ids, ids, use_info))


@pytest.mark.parametrize("d", [32, 64, 128])
def test_fp16_and_head_dims(d):
    check(W.Problem(2, 517, 517, 4, 2, d, "fp16", True, None, f"ordered_fp16_d{d}"))


def test_bitwise_repeat_gqa():
    p = W.Problem(2, 2048, 2048, 8, 2, 128, "bf16", True, None, "ordered_repeat")
    _, g1 = run(p)
    _, g2 = run(p)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


@pytest.mark.slow
def test_headline_full_size_bitwise_and_one_slice():
    """bf16 causal B4 H8 T8192 d128: two runs agree bit for bit; the oracle
    checks batch 2, head 1."""
    p = W.headline()
    (q, k, v, do), g1 = run(p)
    _, g2 = run(p)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    b, h = 2, 1
    sl = lambda t: t[b:b + 1, :, h:h + 1]  # noqa: E731
    ref = oracle.backward(sl(q), sl(k), sl(v), sl(do), causal=True)
    for name, g, r in zip(("dQ", "dK", "dV"), g1, ref):
        assert rel_err(to_np(sl(g)), r) <= TOL["bf16"], name


def test_unsupported_combinations_are_refused():
    import exact_attention_34_gb300 as ea

    for p in (W.Problem(1, 128, 128, 2, 2, 64, "fp32", False, None, "f32"),
              W.Problem(1, 128, 128, 2, 2, 256, "bf16", False, None, "d256")):
        q, k, v, do = cuda(*W.make_inputs(p, 0))
        o, lse = ea.forward(q, k, v)
        with pytest.raises(ea.AttnError) as e:
            ea.backward(q, k, v, o, lse, do, deterministic=ORDERED)
        assert e.value.status == ea.ATTN_ERR_UNSUPPORTED


def draw(seed):
    """A seeded configuration: format, head_dim, GQA group, lengths (tile
    multiples, ragged, one), KV lengths (0, 1, partial, past Lkv), causal or a
    window."""
    rng = np.random.default_rng(7000 + seed)
    dtype = ["bf16", "fp16"][rng.integers(2)]
    d = int(rng.choice([32, 64, 128]))
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 4))
    lens = [1, 64, 127, 128, 129, 300, 511, 700, 1030]
    Lq, Lkv = int(rng.choice(lens)), int(rng.choice(lens))
    mask = rng.integers(3)
    window = None
    causal = mask == 1
    if mask == 2:
        window = (int(rng.choice([-1, 0, 5, 100, 400])), int(rng.choice([-1, 0, 3, 64])))
    kv_lens = None
    if rng.random() < 0.5:
        kv_lens = tuple(int(rng.choice([0, 1, Lkv // 2, Lkv, Lkv + 7])) for _ in range(B))
    return W.Problem(B, Lq, Lkv, Hkv * G, Hkv, d, dtype, causal, kv_lens, f"ordered_rand{seed}"), window


@pytest.mark.parametrize("seed", range(24))
def test_random_configuration(seed):
    p, window = draw(seed)
    check(p, window=window, seed=seed)
