"""The inputs of test_parity_rescale.py do drive the forward through its
lazy rescale: replaying the kernel's rule on the exact scores (128-key tiles in
key order; a row's O is rescaled when a tile's maximum, in log2 units, exceeds
the running maximum by more than 8) gives many rescale events, while the plain
workload inputs give almost none.  No GPU."""

import numpy as np

import workloads as W
from tests.test_parity_rescale import WINDOW_GROWTHS, ramped_inputs

THRESHOLD = 8.0  # log2 units, as in the forward kernel


def rescale_events(q, k, scale, causal, window=None):
    q = q.double().numpy()
    k = k.double().numpy()
    B, Lq, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    Lkv = k.shape[1]
    events = 0
    for b in range(B):
        for h in range(Hq):
            s = q[b, :, h] @ k[b, :, h // G].T * scale * np.log2(np.e)
            if causal:
                s = np.where(np.arange(Lkv)[None, :] <= np.arange(Lq)[:, None] + Lkv - Lq, s, -np.inf)
            if window is not None:
                i, j = np.arange(Lq)[:, None] + Lkv - Lq, np.arange(Lkv)[None, :]
                s = np.where((j >= i - window[0]) & (j <= i + window[1]), s, -np.inf)
            m_used = np.full(Lq, -np.inf)
            for j0 in range(0, Lkv, 128):
                m_tile = s[:, j0:j0 + 128].max(axis=1)
                grow = (m_tile > m_used + THRESHOLD) & np.isfinite(m_used)
                events += int(grow.sum())
                m_used = np.where(m_tile > m_used + THRESHOLD, m_tile, m_used)
    return events


def test_ramped_inputs_rescale_often():
    p = W.Problem(2, 700, 700, 4, 2, 128, "bf16", False, None, "ramp")
    q, k, _, _ = ramped_inputs(p, 0, 3.0)
    assert rescale_events(q, k, 2.0 / np.sqrt(128), False) >= 500


def test_plain_inputs_rarely_rescale():
    p = W.Problem(2, 700, 700, 4, 2, 128, "bf16", False, None, "plain")
    q, k, _, _ = W.make_inputs(p, 0)
    assert rescale_events(q, k, 1.0 / np.sqrt(128), False) <= 5


def test_window_inputs_rescale():
    p = W.Problem(2, 700, 700, 4, 2, 128, "bf16", False, None, "rampwin")
    for growth in WINDOW_GROWTHS:
        q, k, _, _ = ramped_inputs(p, 3, growth)
        for window in ((200, 0), (100, 50)):
            assert rescale_events(q, k, 2.0 / np.sqrt(128), False, window) >= 300
