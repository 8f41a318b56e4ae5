"""Calls from several host threads at once, each on its own stream (ctypes
releases the GIL, so the library's host code runs concurrently): every
result must equal, bitwise, the same call made alone (deterministic paths),
so no call shares mutable state with another."""

import threading

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

CASES = [
    W.Problem(2, 700, 900, 4, 2, 128, "bf16", True, (900, 333), "c0"),
    W.Problem(1, 1000, 1000, 8, 8, 64, "fp16", False, None, "c1"),
    W.Problem(2, 512, 512, 4, 1, 256, "bf16", True, None, "c2"),
    W.Problem(2, 300, 300, 2, 2, 128, "fp32", True, None, "c3"),
]


def _run(ea, tensors, p, stream):
    q, k, v, do, kl = tensors
    with torch.cuda.stream(stream):
        o, lse = ea.forward(q, k, v, causal=p.causal, kv_lens=kl)
        dq, dk, dv = ea.backward(q, k, v, o, lse, do, causal=p.causal, kv_lens=kl)
        dec = ea.decode(q[:, :1].contiguous(), k, v, kv_lens=kl, num_splits=3)
    return o, lse, dq, dk, dv, dec[0], dec[1]


def test_threads_on_separate_streams_match_serial_calls():
    import exact_attention_34_gb300 as ea

    inputs = []
    for i, p in enumerate(CASES):
        q, k, v, do = (t.cuda() for t in W.make_inputs(p, seed=i))
        kl = None if p.kv_lens is None else torch.tensor(p.kv_lens, dtype=torch.int32, device="cuda")
        inputs.append((q, k, v, do, kl))
    serial = []
    for p, t in zip(CASES, inputs):
        serial.append(_run(ea, t, p, torch.cuda.current_stream()))
    torch.cuda.synchronize()

    results = [None] * len(CASES)
    errors = []
    streams = [torch.cuda.Stream() for _ in CASES]

    def worker(i):
        try:
            for _ in range(3):
                results[i] = _run(ea, inputs[i], CASES[i], streams[i])
        except Exception as exc:  # reported below
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(CASES))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert ea.attn_device_status()[1] == 0
    for i, (a, b) in enumerate(zip(serial, results)):
        for x, y in zip(a, b):
            assert torch.equal(x, y), CASES[i].name
