"""Failure detection on the GPU without a fault: the kernels' bounded wait is
run out on purpose (a barrier phase nothing completes), the device status word
reports it with the waiting site, and the context stays usable -- the next
calls compute correct results."""

import time

import pytest
import torch

import oracle
import workloads as W
from tests._helpers import TOL, cuda, rel_err, to_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_and_the_device_stays_usable():
    import exact_attention_34_gb300 as ea

    torch.cuda.synchronize()
    ea.attn_device_status(reset=True)
    t0 = time.perf_counter()
    ea.attn_selftest_wait_timeout(4242)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    st, code, site = ea.attn_device_status(reset=True)
    assert (st, code, site) == (ea.ATTN_ERR_DEVICE, 1, 4242)
    assert 1.5 <= waited <= 30.0, waited  # the 2 s limit of the global timer
    assert ea.attn_device_status(reset=True)[1] == 0  # the reset took
    # the same context still runs the real kernels correctly
    p = W.Problem(1, 300, 300, 2, 2, 128, "bf16", True, None, "after_timeout")
    q, k, v, do = W.make_inputs(p)
    qd, kd, vd, dod = cuda(q, k, v, do)
    o, lse = ea.forward(qd, kd, vd, causal=True)
    grads = ea.backward(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    o_ref, _ = oracle.forward(q, k, v, causal=True)
    assert rel_err(to_np(o), o_ref) <= TOL["bf16"]
    for g, r in zip(grads, oracle.backward(q, k, v, do, causal=True)):
        assert rel_err(to_np(g), r) <= TOL["bf16"]
