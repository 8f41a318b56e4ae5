"""head_dim 32 against the fp64 oracle: the tensor-core kernels run it as 64
with zero-filled columns (bf16 and fp16, both backward variants, masks,
split-KV decode) and the fp32 kernels natively."""

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
    (3, 256, 700, 8, 2, False, (700, 129, 0), None),
    (2, 500, 500, 2, 1, False, None, (64, 0)),
]


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("case", CASES)
def test_d32_fwd_bwd(case, dtype, deterministic):
    import exact_attention_34_gb300 as ea

    B, Lq, Lkv, Hq, Hkv, causal, kl, win = case
    p = W.Problem(B, Lq, Lkv, Hq, Hkv, 32, dtype, causal, kl, "d32")
    q, k, v, do = W.make_inputs(p)
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, causal=causal, kv_lens=kvt(kl), window=win)
    grads = ea.backward(qd, kd, vd, o, lse, dod, causal=causal, kv_lens=kvt(kl), window=win,
                        deterministic=deterministic)
    torch.cuda.synchronize()
    tol = TOL[dtype]
    o_ref, lse_ref = oracle.forward(q, k, v, causal=causal, kv_lens=kl, window=win)
    assert rel_err(to_np(o), o_ref) <= tol
    lse_check(to_np(lse), lse_ref, tol)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, oracle.backward(q, k, v, do, causal=causal, kv_lens=kl,
                                                                    window=win)):
        e = rel_err(to_np(g), r)
        assert e <= tol, f"{name} rel err {e:.3e}"
    assert ea.attn_device_status()[1] == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("Lq,causal", [(1, False), (16, True)])
def test_d32_decode(Lq, causal, dtype):
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, Lq, 3000, 8, 2, 32, dtype, causal, (3000, 900), "dec32")
    q, k, v, _ = W.make_inputs(p)
    o, lse = ea.decode(*cuda(q, k, v), causal=causal, kv_lens=kvt(p.kv_lens), num_splits=4)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.forward(q, k, v, causal=causal, kv_lens=p.kv_lens)
    assert rel_err(to_np(o), o_ref) <= TOL[dtype]
    lse_check(to_np(lse), lse_ref, TOL[dtype])


def test_d32_outputs_touch_only_their_columns():
    """The padded columns never reach memory: a guard band after each output
    tensor stays untouched (outputs are views into larger buffers)."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 300, 300, 4, 2, 32, "bf16", True, None, "d32guard")
    q, k, v, do = (t.cuda() for t in W.make_inputs(p))
    n = q.numel()
    buf = torch.full((n + 4096,), 7.0, device="cuda", dtype=torch.bfloat16)
    o = buf[:n].view_as(q)
    lse = torch.empty(p.B, p.Hq, p.Lq, device="cuda")
    ea.attn_fwd(q, k, v, o, lse, causal=True)
    torch.cuda.synchronize()
    assert torch.all(buf[n:] == 7.0)
