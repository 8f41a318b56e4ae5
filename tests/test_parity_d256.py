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
