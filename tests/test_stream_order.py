"""Stream order under overlapped launches.

The library's kernels start while the kernel before them in the stream is
still draining (programmatic dependent launch): each one waits for its
predecessor before it reads what that kernel writes, the dQ pass runs beside
the dK/dV pass, and the last CTA of every such grid waits before it exits.
These tests check what that must preserve: an operation queued right after a
call (no synchronisation in between) sees the call's complete outputs, and
back-to-back calls that reuse one set of buffers and one workspace give the
results of the same calls run one at a time."""

import numpy as np
import pytest
import torch

import workloads as W
from tests._helpers import cuda

pytestmark = pytest.mark.gpu


def inputs(p, seed):
    return cuda(*W.make_inputs(p, seed))


CASES = [
    (W.Problem(2, 700, 900, 4, 2, 128, "bf16", True, None, "so_d128"), True),
    (W.Problem(2, 700, 900, 4, 2, 64, "fp16", False, None, "so_d64"), True),
    (W.Problem(1, 600, 600, 2, 2, 256, "bf16", True, None, "so_d256"), True),
    (W.Problem(2, 300, 500, 2, 2, 128, "fp32", True, None, "so_f32"), True),
    (W.Problem(2, 700, 900, 4, 2, 128, "bf16", True, None, "so_atomic"), False),
    (W.Problem(2, 700, 900, 4, 2, 128, "bf16", True, None, "so_ordered"), 2),
]


@pytest.mark.parametrize("p,det", CASES, ids=[c[0].name for c in CASES])
def test_outputs_complete_for_the_next_operation(p, det):
    """Copies queued right after forward and backward equal the outputs read
    after a synchronisation."""
    import exact_attention_34_gb300 as ea

    q, k, v, do = inputs(p, 1)
    o, lse = ea.forward(q, k, v, causal=p.causal)
    o_copy, lse_copy = o.clone(), lse.clone()
    grads = ea.backward(q, k, v, o, lse, do, causal=p.causal, deterministic=det)
    copies = [g.clone() for g in grads]
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    assert torch.equal(o_copy, o) and torch.equal(lse_copy, lse)
    for c, g in zip(copies, grads):
        assert torch.equal(c, g)


@pytest.mark.parametrize("p,det", CASES[:4], ids=[c[0].name for c in CASES[:4]])
def test_back_to_back_calls_reusing_buffers(p, det):
    """Three fwd+bwd steps on different inputs into one set of buffers and one
    workspace, queued without synchronisation, each result copied right after
    its call: every copy equals the same step run alone."""
    import exact_attention_34_gb300 as ea

    steps = [inputs(p, s) for s in (2, 3, 4)]
    B, Lq, Hq, d = p.B, p.Lq, p.Hq, p.d
    q0, k0, v0, _ = steps[0]
    o, lse = torch.empty_like(q0), torch.empty((B, Hq, Lq), dtype=torch.float32, device=q0.device)
    dq, dk, dv = torch.empty_like(q0), torch.empty_like(k0), torch.empty_like(v0)
    ws = torch.empty(max(ea.attn_bwd_workspace_size(B, Lq, Hq, d, det, q0.dtype), 256), dtype=torch.uint8,
                     device=q0.device)
    queued = []
    for q, k, v, do in steps:
        ea.attn_fwd(q, k, v, o, lse, causal=p.causal)
        ea.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, causal=p.causal, deterministic=det)
        queued.append(tuple(t.clone() for t in (o, lse, dq, dk, dv)))
    torch.cuda.synchronize()
    for (q, k, v, do), got in zip(steps, queued):
        o1, lse1 = ea.forward(q, k, v, causal=p.causal)
        torch.cuda.synchronize()
        g1 = ea.backward(q, k, v, o1, lse1, do, causal=p.causal, deterministic=det)
        torch.cuda.synchronize()
        for a, b in zip(got, (o1, lse1) + tuple(g1)):
            assert torch.equal(a, b)
    assert ea.attn_device_status()[1] == 0


def test_backward_twice_on_one_workspace():
    """Two backward calls in a row on one workspace (the second's preprocess
    rewrites delta while nothing of the first may still read it)."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 1030, 1030, 8, 2, 128, "bf16", True, None, "so_twice")
    q, k, v, do = inputs(p, 5)
    do2 = torch.randn_like(do)
    o, lse = ea.forward(q, k, v, causal=True)
    ws = torch.empty(ea.attn_bwd_workspace_size(p.B, p.Lq, p.Hq, p.d, True, q.dtype), dtype=torch.uint8,
                     device=q.device)
    out = []
    for g in (do, do2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ea.attn_bwd(q, k, v, o, lse, g, dq, dk, dv, ws, causal=True)
        out.append((dq, dk, dv))
    torch.cuda.synchronize()
    for g, got in zip((do, do2), out):
        ref = ea.backward(q, k, v, o, lse, g, causal=True)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_decode_then_copy():
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 1, 5000, 8, 2, 128, "bf16", False, (5000, 1777), "so_decode")
    q, k, v, _ = inputs(p, 6)
    kl = torch.tensor(p.kv_lens, dtype=torch.int32, device=q.device)
    o, lse = ea.decode(q, k, v, kv_lens=kl)
    o_copy, lse_copy = o.clone(), lse.clone()
    torch.cuda.synchronize()
    assert torch.equal(o_copy, o) and torch.equal(lse_copy, lse)


def test_plain_stream_order_gives_identical_results(tmp_path):
    """The same fwd+bwd with the overlapped launches turned off
    (EXACT_ATTN_NO_PDL=1, in a fresh process) gives the same bits."""
    import os
    import subprocess
    import sys

    import exact_attention_34_gb300 as ea

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = (
        "import sys, torch; sys.path.insert(0, %r)\n"
        "import exact_attention_34_gb300 as ea, workloads as W\n"
        "from tests._helpers import cuda\n"
        "p = W.Problem(2, 900, 1100, 8, 2, 128, 'bf16', True, None, 'so_nopdl')\n"
        "q, k, v, do = cuda(*W.make_inputs(p, 7))\n"
        "o, lse = ea.forward(q, k, v, causal=True)\n"
        "g = ea.backward(q, k, v, o, lse, do, causal=True)\n"
        "torch.save([t.cpu() for t in (o, lse) + tuple(g)], %r)\n"
    ) % (root, str(tmp_path / "plain.pt"))
    env = dict(os.environ, EXACT_ATTN_NO_PDL="1")
    subprocess.run([sys.executable, "-c", script], check=True, env=env, cwd=root, timeout=600)
    plain = torch.load(tmp_path / "plain.pt")
    p = W.Problem(2, 900, 1100, 8, 2, 128, "bf16", True, None, "so_nopdl")
    q, k, v, do = inputs(p, 7)
    o, lse = ea.forward(q, k, v, causal=True)
    g = ea.backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    for a, b in zip((o, lse) + tuple(g), plain):
        assert torch.equal(a.cpu(), b)


def _random_call(rng, ea, dev):
    """One seeded library call and a function that runs it (returning its
    outputs, freshly allocated)."""
    kind = rng.choice(["fwd_bwd", "fwd_bwd", "window", "segments", "split", "decode", "d256", "fp32"])
    B = int(rng.integers(1, 3))
    Hkv = int(rng.choice([1, 2]))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    d = 64 if kind == "d256" else int(rng.choice([64, 128]))
    d = 256 if kind == "d256" else d
    dtype = "fp32" if kind == "fp32" else str(rng.choice(["bf16", "fp16"]))
    Lq = 1 if kind == "decode" else int(rng.choice([129, 300, 640]))
    Lkv = int(rng.choice([129, 300, 640, 1500]))
    if kind in ("window", "segments"):
        Lkv = Lq
    causal = bool(rng.integers(2)) and kind in ("fwd_bwd", "d256", "fp32")
    p = W.Problem(B, Lq, Lkv, Hq, Hkv, d, dtype, causal, None, f"mix_{kind}")
    q, k, v, do = inputs(p, int(rng.integers(1 << 30)))
    det = int(rng.choice([1, 2])) if (kind == "fwd_bwd" and dtype != "fp32" and d <= 128) else 1
    window = (int(rng.integers(0, 200)), int(rng.integers(0, 50))) if kind == "window" else None
    segs = None
    if kind == "segments":
        ids = torch.tensor(np.sort(rng.integers(0, 4, size=(B, Lq)), axis=1).astype(np.int32), device=dev)
        segs = (ids, ids)
    kl = None
    if kind in ("split", "decode"):
        kl = torch.tensor([int(rng.integers(0, Lkv + 1)) for _ in range(B)], dtype=torch.int32, device=dev)

    def run():
        if kind == "decode":
            return ea.decode(q, k, v, kv_lens=kl)
        if kind == "split":
            return ea.forward(q, k, v, kv_lens=kl, num_splits=2)
        o, lse = ea.forward(q, k, v, causal=causal, window=window, segments=segs)
        return (o, lse) + tuple(ea.backward(q, k, v, o, lse, do, causal=causal, window=window, segments=segs,
                                            deterministic=det))

    return run


@pytest.mark.parametrize("seed", range(3))
def test_random_mixed_calls_queued_back_to_back(seed):
    """Twenty seeded calls of every kind (masks, backward variants, head_dim
    256, fp32, split forward, decode) queued on one stream without
    synchronisation, each output copied right after its call: every copy
    equals the same call run alone."""
    import exact_attention_34_gb300 as ea

    rng = np.random.default_rng(900 + seed)
    dev = torch.device("cuda")
    calls = [_random_call(rng, ea, dev) for _ in range(20)]
    queued = [[t.clone() for t in run()] for run in calls]
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    for run, got in zip(calls, queued):
        ref = run()
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
