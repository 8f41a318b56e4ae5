"""Guard bands around every output and workspace buffer.

Each output tensor (and each caller workspace) is a view into a larger device
buffer whose leading and trailing bands hold a canary value.  After the call
the bands must be untouched, so no kernel writes before or past its buffer,
including on ragged lengths, KV lengths of 0 and 1, GQA and Lq != Lkv.  The
values written must also equal those of the same call into plain tensors:
bitwise for the deterministic paths, within the parity tolerance for the
atomic-dQ backward.  compute-sanitizer is closed on this machine; these bands are
the out-of-bounds-write check in its place."""

import pytest
import torch

import workloads as W
from tests._helpers import TOL, rel_err, to_np

pytestmark = pytest.mark.gpu

BAND = 4096  # canary elements on each side (keeps the view 16-byte aligned)
CANARY = {torch.bfloat16: 7.0, torch.float16: 7.0, torch.float32: -12345.0, torch.uint8: 0xA5}


class Guarded:
    """A contiguous view of `shape` inside a buffer with canary bands."""

    def __init__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        self.n, self.fill = n, CANARY[dtype]
        self.buf = torch.full((n + 2 * BAND,), self.fill, device="cuda", dtype=dtype)
        self.t = self.buf[BAND:BAND + n].view(*shape)

    def check(self, what):
        lead, tail = self.buf[:BAND], self.buf[BAND + self.n:]
        assert torch.all(lead == self.fill), f"{what}: written before the buffer"
        assert torch.all(tail == self.fill), f"{what}: written past the buffer"


def _inputs(p, seed=0):
    q, k, v, do = (t.cuda() for t in W.make_inputs(p, seed))
    kl = torch.tensor(p.kv_lens, dtype=torch.int32, device="cuda") if p.kv_lens is not None else None
    return q, k, v, do, kl


CASES = [
    W.Problem(2, 300, 555, 4, 2, 128, "bf16", False, (555, 1), "ragged_kvl1"),
    W.Problem(2, 333, 333, 4, 4, 64, "bf16", True, None, "ragged_causal"),
    W.Problem(2, 200, 700, 4, 1, 128, "fp16", True, (700, 0), "offset_causal_kvl0"),
    W.Problem(2, 190, 260, 2, 2, 64, "fp32", True, (260, 77), "fp32"),
    W.Problem(1, 300, 300, 2, 1, 256, "bf16", True, None, "d256"),
]


@pytest.mark.parametrize("p", CASES, ids=lambda p: p.name)
def test_forward_and_backward_stay_inside_their_buffers(p):
    import exact_attention_34_gb300 as ea

    q, k, v, do, kl = _inputs(p)
    dt = q.dtype
    o = Guarded(q.shape, dt)
    lse = Guarded((p.B, p.Hq, p.Lq), torch.float32)
    ea.attn_fwd(q, k, v, o.t, lse.t, causal=p.causal, kv_lens=kl)
    o_ref, lse_ref = ea.forward(q, k, v, causal=p.causal, kv_lens=kl)
    torch.cuda.synchronize()
    o.check("o")
    lse.check("lse")
    assert torch.equal(o.t, o_ref) and torch.equal(lse.t, lse_ref)

    variants = (True,) if p.d == 256 else (True, False) if p.dtype == "fp32" else (True, False, 2)
    for det in variants:
        dq, dk, dv = Guarded(q.shape, dt), Guarded(k.shape, dt), Guarded(v.shape, dt)
        ws = Guarded((ea.attn_bwd_workspace_size(p.B, p.Lq, p.Hq, p.d, det, dt),), torch.uint8)
        ea.attn_bwd(q, k, v, o_ref, lse_ref, do, dq.t, dk.t, dv.t, ws.t, causal=p.causal, kv_lens=kl,
                    deterministic=det)
        ref = ea.backward(q, k, v, o_ref, lse_ref, do, causal=p.causal, kv_lens=kl, deterministic=det)
        torch.cuda.synchronize()
        assert ea.attn_device_status()[1] == 0
        for g, name in ((dq, "dq"), (dk, "dk"), (dv, "dv"), (ws, "workspace")):
            g.check(f"{name} (deterministic={det})")
        for got, want in zip((dq.t, dk.t, dv.t), ref):
            if det:
                assert torch.equal(got, want)
            else:
                assert rel_err(to_np(got), to_np(want)) <= TOL[p.dtype]


@pytest.mark.parametrize("Lq,causal", [(1, False), (16, True)])
def test_decode_and_combine_stay_inside_their_buffers(Lq, causal):
    import exact_attention_34_gb300 as ea

    p = W.Problem(3, Lq, 1000, 8, 2, 128, "bf16", causal, (1000, 17, 0), "decode_guard")
    q, k, v, _, kl = _inputs(p)
    S = 3
    op = Guarded((p.B, p.Hq, S, p.Lq, p.d), torch.float32)
    lp = Guarded((p.B, p.Hq, S, p.Lq), torch.float32)
    ea.attn_decode_splitkv(q, k, v, op.t, lp.t, S, causal=causal, kv_lens=kl)
    o, lse = Guarded(q.shape, q.dtype), Guarded((p.B, p.Hq, p.Lq), torch.float32)
    ea.attn_decode_combine(op.t, lp.t, o.t, lse.t)
    ref = ea.decode(q, k, v, causal=causal, kv_lens=kl, num_splits=S, return_partials=True)
    torch.cuda.synchronize()
    for g, name in ((op, "o_part"), (lp, "lse_part"), (o, "o"), (lse, "lse")):
        g.check(name)
    assert torch.equal(o.t, ref[0]) and torch.equal(lse.t, ref[1])
    assert torch.equal(op.t, ref[2]) and torch.equal(lp.t, ref[3])


def test_split_forward_stays_inside_its_buffers():
    import exact_attention_34_gb300 as ea

    p = W.Problem(3, 384, 3000, 4, 2, 128, "bf16", False, (3000, 129, 0), "split_guard")
    q, k, v, _, kl = _inputs(p)
    S = 3
    o, lse = Guarded(q.shape, q.dtype), Guarded((p.B, p.Hq, p.Lq), torch.float32)
    ws = Guarded((ea.attn_fwd_split_workspace_size(p.B, p.Lq, p.Hq, p.d, S),), torch.uint8)
    ea.attn_fwd_split(q, k, v, o.t, lse.t, ws.t, S, kv_lens=kl)
    o_ref, lse_ref = ea.forward(q, k, v, kv_lens=kl, num_splits=S)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    for g, name in ((o, "o"), (lse, "lse"), (ws, "workspace")):
        g.check(name)
    assert torch.equal(o.t, o_ref) and torch.equal(lse.t, lse_ref)


def test_window_and_segment_calls_stay_inside_their_buffers():
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 450, 450, 4, 2, 64, "bf16", True, None, "mask_guard")
    q, k, v, do, _ = _inputs(p)
    dt = q.dtype

    def outputs():
        return (Guarded(q.shape, dt), Guarded((p.B, p.Hq, p.Lq), torch.float32), Guarded(q.shape, dt),
                Guarded(k.shape, dt), Guarded(v.shape, dt),
                Guarded((ea.attn_bwd_workspace_size(p.B, p.Lq, p.Hq, p.d, True, dt),), torch.uint8))

    # local window: 64 keys back, 16 ahead
    win = (64, 16)
    o, lse, dq, dk, dv, ws = outputs()
    ea.attn_fwd_window(q, k, v, o.t, lse.t, win)
    ea.attn_bwd_window(q, k, v, o.t, lse.t, do, dq.t, dk.t, dv.t, ws.t, win)
    o_ref, lse_ref = ea.forward(q, k, v, window=win)
    ref = ea.backward(q, k, v, o_ref, lse_ref, do, window=win)
    torch.cuda.synchronize()
    for g, name in zip((o, lse, dq, dk, dv, ws), ("o", "lse", "dq", "dk", "dv", "workspace")):
        g.check(f"window {name}")
    for got, want in zip((o.t, lse.t, dq.t, dk.t, dv.t), (o_ref, lse_ref) + tuple(ref)):
        assert torch.equal(got, want)

    # segments: documents of 100, 250 and 100 tokens, causal within each
    ids = torch.tensor([0] * 100 + [1] * 250 + [2] * 100, dtype=torch.int32, device="cuda").repeat(p.B, 1)
    info = Guarded((ea.attn_segment_info_size(p.B, p.Lq, p.Lq),), torch.uint8)
    ea.attn_segment_info(ids, ids, info.t)
    o, lse, dq, dk, dv, ws = outputs()
    ea.attn_fwd_segments(q, k, v, o.t, lse.t, ids, ids, window=(-1, 0), segment_info=info.t)
    ea.attn_bwd_segments(q, k, v, o.t, lse.t, do, dq.t, dk.t, dv.t, ws.t, ids, ids, window=(-1, 0),
                         segment_info=info.t)
    segs = (ids, ids, ea.segment_info(ids, ids))
    o_ref, lse_ref = ea.forward(q, k, v, causal=True, segments=segs)
    ref = ea.backward(q, k, v, o_ref, lse_ref, do, causal=True, segments=segs)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    info.check("segment info")
    assert torch.equal(info.t, segs[2])
    for g, name in zip((o, lse, dq, dk, dv, ws), ("o", "lse", "dq", "dk", "dv", "workspace")):
        g.check(f"segments {name}")
    for got, want in zip((o.t, lse.t, dq.t, dk.t, dv.t), (o_ref, lse_ref) + tuple(ref)):
        assert torch.equal(got, want)
