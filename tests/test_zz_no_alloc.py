"""The allocation-free backward entry point (attn_bwd_static_scratch), called
through the C ABI, against the regular attn_bwd with a caller workspace and
against the fp64 oracle.

Callers that cannot allocate device memory where they run the backward
(hosts whose device memory belongs to a fixed pool or another runtime,
latency-critical loops that must not hit cudaMalloc's implicit device
synchronisation, embeddings that only hand over existing tensors) use this
entry point; its scratch is a static array inside the library shared by every
call on a device.  Both entry points run the same deterministic kernels, so
their results must agree bit for bit.  This file is collected last so a run
that stops at the first failure has already run every other test."""

import ctypes

import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, rel_err, to_np

pytestmark = pytest.mark.gpu


def _static_bwd(ea, q, k, v, o, lse, do, causal, kv):
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    B, Lq, Hq, d = q.shape
    Lkv, Hkv = k.shape[1], k.shape[2]
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    st = ea.lib().attn_bwd_static_scratch(P(q), P(k), P(v), P(o), P(lse), P(do), P(dq), P(dk), P(dv), B, Lq, Lkv,
                                          Hq, Hkv, d, 1.0 / d ** 0.5, int(causal), P(kv),
                                          ea.ATTN_BF16 if q.dtype == torch.bfloat16 else ea.ATTN_FP32,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, ea.lib().attn_last_error().decode()
    return dq, dk, dv


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_static_scratch_backward_matches_workspace_backward(dtype):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 700, 900, 4, 2, 128, dtype, True, (900, 333), "no_alloc")
    q_h, k_h, v_h, do_h = W.make_inputs(p, seed=7)
    q, k, v, do = (t.cuda() for t in (q_h, k_h, v_h, do_h))
    kv = torch.tensor(p.kv_lens, dtype=torch.int32, device="cuda")
    o, lse = ea.forward(q, k, v, causal=True, kv_lens=kv)
    ref = ea.backward(q, k, v, o, lse, do, causal=True, kv_lens=kv, deterministic=True)
    for _ in range(2):  # two calls in a row share (and reuse) the static scratch
        got = _static_bwd(ea, q, k, v, o, lse, do, True, kv)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
    # and the result itself against the fp64 oracle
    exact = oracle.backward(q_h, k_h, v_h, do_h, causal=True, kv_lens=p.kv_lens)
    for a, b in zip(got, exact):
        assert rel_err(to_np(a), b) <= TOL[dtype]


def test_static_scratch_rejects_oversized_problem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_34_gb300 as ea

    # B*Hq*roundup(Lq,128) = 8*32*4096 > 524288: rejected before any launch
    fake = ctypes.c_void_p(0x10000)
    st = ea.lib().attn_bwd_static_scratch(*([fake] * 9), 8, 4096, 4096, 32, 8, 128, 0.1, 0, None, ea.ATTN_BF16, None)
    assert st == ea.ATTN_ERR_WORKSPACE
    assert "static scratch" in ea.lib().attn_last_error().decode()
