"""Edge cases of the method on the GPU, against the fp64 oracle: one query, one
key, tails one row past a tile, wide GQA groups, every batch empty, the longest
sequence the pages ran (fwd+bwd at T = 65,536, memory linear in T), and the
library's calls captured into and replayed from a CUDA graph."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, lse_check, rel_err, to_np

pytestmark = pytest.mark.gpu


def kvt(p):
    return None if p.kv_lens is None else torch.tensor(p.kv_lens, dtype=torch.int32).cuda()


def fwd_bwd_check(p, check_bwd=True, seed=0):
    import exact_attention_34_gb300 as ea

    q, k, v, do = W.make_inputs(p, seed)
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, causal=p.causal, kv_lens=kvt(p))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.forward(q, k, v, causal=p.causal, kv_lens=p.kv_lens)
    tol = TOL[p.dtype]
    assert rel_err(to_np(o), o_ref) <= tol
    lse_check(to_np(lse), lse_ref, tol)
    if check_bwd:
        grads = ea.backward(qd, kd, vd, o, lse, dod, causal=p.causal, kv_lens=kvt(p))
        torch.cuda.synchronize()
        ref = oracle.backward(q, k, v, do, causal=p.causal, kv_lens=p.kv_lens)
        for g, r in zip(grads, ref):
            assert rel_err(to_np(g), r) <= tol
    assert ea.attn_device_status()[1] == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("Lq,Lkv,causal", [(1, 1, False), (1, 1, True), (1, 700, False), (1, 700, True),
                                           (700, 1, False), (700, 1, True), (129, 129, True), (257, 255, False),
                                           (383, 385, True)])
def test_degenerate_lengths(dtype, Lq, Lkv, causal):
    fwd_bwd_check(W.Problem(2, Lq, Lkv, 4, 2, 128, dtype, causal, None, "edge"))


@pytest.mark.parametrize("d", [64, 128])
def test_wide_gqa_group(d):
    fwd_bwd_check(W.Problem(2, 300, 520, 16, 2, d, "bf16", True, None, "gqa8"))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_every_batch_empty(dtype):
    import exact_attention_34_gb300 as ea

    p = W.Problem(3, 200, 300, 4, 4, 64, dtype, False, (0, 0, 0), "all_empty")
    q, k, v, do = (t.cuda() for t in W.make_inputs(p))
    o, lse = ea.forward(q, k, v, kv_lens=kvt(p))
    dq, dk, dv = ea.backward(q, k, v, o, lse, do, kv_lens=kvt(p))
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(lse == -float("inf"))
    assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_d64_kvlens_and_lengths_past_lkv(causal):
    # a length above Lkv is clamped; a length of 1 gives the single-key case
    fwd_bwd_check(W.Problem(3, 256, 400, 4, 1, 64, "bf16", causal, (400, 9999, 1), "d64_kv"))


def test_atomic_backward_d64_gqa():
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 300, 333, 8, 2, 64, "bf16", True, None, "atomic_d64")
    q, k, v, do = W.make_inputs(p)
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, causal=True)
    grads = ea.backward(qd, kd, vd, o, lse, dod, causal=True, deterministic=False)
    torch.cuda.synchronize()
    for g, r in zip(grads, oracle.backward(q, k, v, do, causal=True)):
        assert rel_err(to_np(g), r) <= TOL["bf16"]


def test_longest_sequence_fwd_bwd():
    """fwd+bwd at T = 65,536, B4 H8 d128 causal (the longest length the pages
    ran); memory stays linear in T.  The oracle checks sampled query rows of one
    head: O and LSE, and dQ (which only needs its own rows)."""
    import exact_attention_34_gb300 as ea

    T = 65536
    p = W.Problem(4, T, T, 8, 8, 128, "bf16", True, None, "T64k")
    q, k, v, do = W.make_inputs(p)
    qd, kd, vd, dod = cuda(q, k, v, do)
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    o, lse = ea.forward(qd, kd, vd, causal=True)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    # outputs + residuals + workspace only: no T x T buffer anywhere
    extra = torch.cuda.max_memory_allocated() - base
    assert extra < 6 * qd.numel() * qd.element_size()
    b, h = 2, 5
    rows = np.array([0, 1, 4095, 30000, 65534, 65535])
    sl = lambda t: t[b:b + 1, :, h:h + 1]  # noqa: E731
    o_ref, lse_ref = oracle.forward(sl(q), sl(k), sl(v), causal=True, rows=rows)
    assert rel_err(to_np(sl(o))[:, rows], o_ref) <= TOL["bf16"]
    lse_check(to_np(lse[b:b + 1, h:h + 1])[:, :, rows], lse_ref, TOL["bf16"])
    dq_ref, _, _ = oracle.backward(sl(q), sl(k), sl(v), sl(do), causal=True, rows=rows)
    assert rel_err(to_np(sl(dq))[:, rows], dq_ref[:, rows]) <= TOL["bf16"]


def test_cuda_graph_capture_and_replay():
    """The C calls only launch kernels on the given stream (no allocation or
    synchronisation), so a whole fwd+bwd step can be captured once and replayed."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 640, 640, 4, 2, 128, "bf16", True, None, "graph")
    q, k, v, do = (t.cuda() for t in W.make_inputs(p))
    o, lse = torch.empty_like(q), torch.empty(p.B, p.Hq, p.Lq, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(ea.attn_bwd_workspace_size(p.B, p.Lq, p.Hq, p.d, True, q.dtype), device="cuda",
                     dtype=torch.uint8)
    s = torch.cuda.Stream()

    def step():
        ea.attn_fwd(q, k, v, o, lse, causal=True, stream=s)
        ea.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, causal=True, stream=s)

    with torch.cuda.stream(s):
        step()  # first call sets per-device kernel attributes outside the capture
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for t in (o, dq, dk, dv):
        t.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip((o, dq, dk, dv), ref):
        assert torch.equal(a, b)  # deterministic path: replay is bitwise identical
