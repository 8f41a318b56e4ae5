"""Pins for the fp64 oracle: every check here is independent of the oracle's own
formulas -- a hand-worked closed form, central finite differences, a library
routine (torch float64 SDPA with autograd, scipy logsumexp), invariants the
mathematics fixes, and a pure-Python brute force on tiny inputs.

CPU only; runs in seconds.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------
# closed form worked by hand (tests/golden/two_keys_closed_form.json)
# --------------------------------------------------------------------------

def _golden():
    with open(os.path.join(HERE, "golden", "two_keys_closed_form.json")) as f:
        return json.load(f)


def test_closed_form_two_keys():
    g = _golden()
    q, k, v, do = (np.array(g[n]) for n in ("q", "k", "v", "do"))
    o, lse = oracle.forward(q, k, v, scale=g["scale"])
    dq, dk, dv = oracle.backward(q, k, v, do, scale=g["scale"])
    exp = g["full"]
    np.testing.assert_allclose(o, exp["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, exp["lse"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dq, exp["dq"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, exp["dk"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, exp["dv"], rtol=0, atol=1e-14)


def test_closed_form_kv_len_one_and_zero():
    g = _golden()
    q, k, v, do = (np.array(g[n]) for n in ("q", "k", "v", "do"))
    o, lse = oracle.forward(q, k, v, scale=g["scale"], kv_lens=[1])
    dq, dk, dv = oracle.backward(q, k, v, do, scale=g["scale"], kv_lens=[1])
    exp = g["kv_len_1"]
    for got, name in ((o, "o"), (lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        assert np.array_equal(got, np.array(exp[name])), name  # exact, no rounding
    o, lse = oracle.forward(q, k, v, scale=g["scale"], kv_lens=[0])
    dq, dk, dv = oracle.backward(q, k, v, do, scale=g["scale"], kv_lens=[0])
    assert np.all(o == 0) and np.all(lse == -np.inf)
    assert np.all(dq == 0) and np.all(dk == 0) and np.all(dv == 0)


# --------------------------------------------------------------------------
# pure-Python brute force (no numpy in the arithmetic)
# --------------------------------------------------------------------------

def brute_force(q, k, v, scale, causal, kv_lens):
    B, Lq, Hq, d = q.shape
    Lkv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    o = [[[[0.0] * d for _ in range(Hq)] for _ in range(Lq)] for _ in range(B)]
    lse = [[[0.0] * Lq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        kvl = Lkv if kv_lens is None else max(0, min(Lkv, int(kv_lens[b])))
        for h in range(Hq):
            hk = h // G
            for i in range(Lq):
                keys = [j for j in range(Lkv)
                        if j < kvl and (not causal or j <= i + kvl - Lq)]
                if not keys:
                    lse[b][h][i] = -math.inf
                    continue
                sc = {}
                for j in keys:
                    s = 0.0
                    for c in range(d):
                        s += float(q[b, i, h, c]) * float(k[b, j, hk, c])
                    sc[j] = s * scale
                mx = max(sc.values())
                z = sum(math.exp(sc[j] - mx) for j in keys)
                for j in keys:
                    p = math.exp(sc[j] - mx) / z
                    for c in range(d):
                        o[b][i][h][c] += p * float(v[b, j, hk, c])
                lse[b][h][i] = mx + math.log(z)
    return np.array(o), np.array(lse)


CASES = [
    # B, Lq, Lkv, Hq, Hkv, d, causal, kv_lens
    (1, 4, 4, 2, 2, 3, False, None),
    (2, 5, 5, 2, 1, 4, True, None),
    (2, 3, 6, 4, 2, 3, True, None),       # Lq < Lkv, bottom-right causal
    (2, 6, 3, 2, 2, 3, True, None),       # Lq > Lkv: the first rows see no key
    (3, 4, 6, 2, 1, 3, False, [6, 1, 0]),  # KV lengths incl. single key and empty
    (3, 4, 6, 4, 2, 2, True, [5, 9, 2]),   # lengths + causal offset, one clamped
]


@pytest.mark.parametrize("case", CASES)
def test_forward_matches_brute_force(case):
    B, Lq, Lkv, Hq, Hkv, d, causal, kl = case
    q = rnd((B, Lq, Hq, d), 1)
    k = rnd((B, Lkv, Hkv, d), 2)
    v = rnd((B, Lkv, Hkv, d), 3)
    o, lse = oracle.forward(q, k, v, scale=0.7, causal=causal, kv_lens=kl)
    ob, lb = brute_force(q, k, v, 0.7, causal, kl)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(lb)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# gradient: central finite differences in fp64
# --------------------------------------------------------------------------

def _loss(q, k, v, do, scale, causal, kl):
    o, _ = oracle.forward(q, k, v, scale=scale, causal=causal, kv_lens=kl)
    return float(np.sum(o * do))


@pytest.mark.parametrize("case", CASES)
def test_backward_matches_finite_differences(case):
    B, Lq, Lkv, Hq, Hkv, d, causal, kl = case
    q = rnd((B, Lq, Hq, d), 11)
    k = rnd((B, Lkv, Hkv, d), 12)
    v = rnd((B, Lkv, Hkv, d), 13)
    do = rnd((B, Lq, Hq, d), 14)
    scale = 0.7
    dq, dk, dv = oracle.backward(q, k, v, do, scale=scale, causal=causal, kv_lens=kl)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            fp = _loss(q, k, v, do, scale, causal, kl)
            x[idx] = old - h
            fm = _loss(q, k, v, do, scale, causal, kl)
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        denom = max(1.0, np.max(np.abs(num)))
        assert np.max(np.abs(num - g)) / denom < 1e-6


# --------------------------------------------------------------------------
# library cross-check: torch float64 SDPA (math path on CPU) + autograd
# --------------------------------------------------------------------------

def _torch_ref(q, k, v, do, scale, mask=None, gqa=False):
    tq, tk, tv = (torch.tensor(x).permute(0, 2, 1, 3).contiguous().requires_grad_(True)
                  for x in (q, k, v))
    o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale, enable_gqa=gqa)
    (o * torch.tensor(do).permute(0, 2, 1, 3)).sum().backward()
    t = lambda x: x.detach().permute(0, 2, 1, 3).numpy()  # noqa: E731
    return t(o), t(tq.grad), t(tk.grad), t(tv.grad)


@pytest.mark.parametrize("Lq,Lkv,causal,Hq,Hkv", [
    (7, 7, False, 2, 2), (7, 7, True, 2, 2), (5, 9, True, 4, 2), (9, 9, False, 4, 1),
])
def test_against_torch_sdpa_float64(Lq, Lkv, causal, Hq, Hkv):
    from torch.nn.attention.bias import causal_lower_right

    B, d, scale = 2, 8, 0.37
    q, k, v, do = rnd((B, Lq, Hq, d), 21), rnd((B, Lkv, Hkv, d), 22), \
        rnd((B, Lkv, Hkv, d), 23), rnd((B, Lq, Hq, d), 24)
    mask = causal_lower_right(Lq, Lkv) if causal else None
    o_t, dq_t, dk_t, dv_t = _torch_ref(q, k, v, do, scale, mask, gqa=Hq != Hkv)
    o, lse = oracle.forward(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = oracle.backward(q, k, v, do, scale=scale, causal=causal)
    for a, b in ((o, o_t), (dq, dq_t), (dk, dk_t), (dv, dv_t)):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_kv_lens_against_torch_boolean_mask():
    B, Lq, Lkv, H, d, scale = 3, 5, 8, 2, 4, 0.5
    kl = [8, 3, 1]
    q, k, v, do = rnd((B, Lq, H, d), 31), rnd((B, Lkv, H, d), 32), \
        rnd((B, Lkv, H, d), 33), rnd((B, Lq, H, d), 34)
    mask = torch.zeros(B, 1, Lq, Lkv, dtype=torch.bool)
    for b in range(B):
        mask[b, :, :, :kl[b]] = True
    o_t, dq_t, dk_t, dv_t = _torch_ref(q, k, v, do, scale, mask)
    o, _ = oracle.forward(q, k, v, scale=scale, kv_lens=kl)
    dq, dk, dv = oracle.backward(q, k, v, do, scale=scale, kv_lens=kl)
    for a, b in ((o, o_t), (dq, dq_t), (dk, dk_t), (dv, dv_t)):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_lse_against_scipy_logsumexp():
    B, L, H, d = 2, 6, 2, 5
    q, k, v = rnd((B, L, H, d), 41), rnd((B, L, H, d), 42), rnd((B, L, H, d), 43)
    _, lse = oracle.forward(q, k, v, scale=0.9, causal=True)
    for b in range(B):
        for h in range(H):
            s = 0.9 * q[b, :, h, :] @ k[b, :, h, :].T
            for i in range(L):
                assert abs(lse[b, h, i] - logsumexp(s[i, :i + 1])) < 1e-12


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_probability_rows_sum_to_one_and_respect_mask():
    q, k = rnd((2, 6, 4, 3), 51), rnd((2, 9, 2, 3), 52)
    p = oracle.probabilities(q, k, causal=True, kv_lens=[9, 4])
    s = p.sum(axis=-1)
    # every row that has a valid key sums to one; rows without sum to zero
    has = np.zeros_like(s, dtype=bool)
    for b, kvl in enumerate([9, 4]):
        for i in range(6):
            has[b, :, i] = min(kvl, i + kvl - 6 + 1) > 0
    np.testing.assert_allclose(s[has], 1.0, rtol=0, atol=1e-14)
    assert np.all(s[~has] == 0)
    assert np.all(p >= 0)


def test_constant_v_gives_v():
    q, k = rnd((2, 5, 2, 4), 61), rnd((2, 7, 1, 4), 62)
    v = np.broadcast_to(rnd((1, 1, 1, 4), 63), (2, 7, 1, 4)).copy()
    o, _ = oracle.forward(q, k, v, causal=True)
    np.testing.assert_allclose(o, np.broadcast_to(v[:, :1], o.shape), rtol=0, atol=1e-14)


def test_single_valid_key_exact_zero_gradients():
    q, k, v, do = rnd((1, 4, 2, 3), 71), rnd((1, 5, 2, 3), 72), rnd((1, 5, 2, 3), 73), \
        rnd((1, 4, 2, 3), 74)
    o, lse = oracle.forward(q, k, v, kv_lens=[1])
    assert np.array_equal(o, np.broadcast_to(v[:, :1], o.shape))
    np.testing.assert_allclose(lse, np.einsum("bihc,bhc->bhi", q, k[:, 0]) / math.sqrt(3),
                               rtol=1e-14)
    dq, dk, dv = oracle.backward(q, k, v, do, kv_lens=[1])
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv[:, 0], do.sum(axis=1), rtol=1e-14)
    assert np.all(dv[:, 1:] == 0)


def test_empty_rows_give_zeros():
    q, k, v, do = rnd((2, 3, 2, 4), 81), rnd((2, 4, 2, 4), 82), rnd((2, 4, 2, 4), 83), \
        rnd((2, 3, 2, 4), 84)
    o, lse = oracle.forward(q, k, v, kv_lens=[0, 4])
    assert np.all(o[0] == 0) and np.all(lse[0] == -np.inf)
    dq, dk, dv = oracle.backward(q, k, v, do, kv_lens=[0, 4])
    assert np.all(dq[0] == 0) and np.all(dk[0] == 0) and np.all(dv[0] == 0)
    # causal with Lq > Lkv: rows 0 .. Lq-Lkv-1 have no key
    o, lse = oracle.forward(rnd((1, 5, 1, 4), 85), k[:1, :2, :1], v[:1, :2, :1], causal=True)
    assert np.all(o[0, :3] == 0) and np.all(lse[0, :, :3] == -np.inf)
    assert np.all(np.isfinite(lse[0, :, 3:]))


def test_causal_length_one_gives_v():
    q, k, v = rnd((3, 1, 2, 4), 91), rnd((3, 1, 2, 4), 92), rnd((3, 1, 2, 4), 93)
    o, _ = oracle.forward(q, k, v, causal=True)
    assert np.array_equal(o, v)


def test_gqa_equals_repeated_kv():
    B, L, Hq, Hkv, d = 2, 6, 6, 2, 3
    q, k, v, do = rnd((B, L, Hq, d), 101), rnd((B, L, Hkv, d), 102), rnd((B, L, Hkv, d), 103), \
        rnd((B, L, Hq, d), 104)
    kr, vr = np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2)
    o, lse = oracle.forward(q, k, v, causal=True, kv_lens=[6, 3])
    o2, lse2 = oracle.forward(q, kr, vr, causal=True, kv_lens=[6, 3])
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-15)
    dq, dk, dv = oracle.backward(q, k, v, do, causal=True, kv_lens=[6, 3])
    dq2, dk2, dv2 = oracle.backward(q, kr, vr, do, causal=True, kv_lens=[6, 3])
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-14)
    # the gradient of a repeated K/V is the sum over the copies of the group
    G = Hq // Hkv
    np.testing.assert_allclose(dk, dk2.reshape(B, L, Hkv, G, d).sum(3), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, dv2.reshape(B, L, Hkv, G, d).sum(3), rtol=0, atol=1e-14)


def test_preprocess_equals_sum_p_dp():
    q, k, v, do = rnd((2, 5, 2, 3), 111), rnd((2, 7, 2, 3), 112), rnd((2, 7, 2, 3), 113), \
        rnd((2, 5, 2, 3), 114)
    o, _ = oracle.forward(q, k, v, causal=True, kv_lens=[7, 2])
    D = oracle.backward_preprocess(o, do)
    p = oracle.probabilities(q, k, causal=True, kv_lens=[7, 2])
    dp = np.einsum("bihc,bjhc->bhij", do, v)
    np.testing.assert_allclose(D, np.sum(p * dp, axis=-1), rtol=1e-13, atol=1e-14)


def test_sampled_rows_and_heads_match_full():
    q, k, v = rnd((2, 9, 4, 3), 121), rnd((2, 11, 2, 3), 122), rnd((2, 11, 2, 3), 123)
    o, lse = oracle.forward(q, k, v, causal=True, kv_lens=[11, 6])
    rows = [0, 4, 8]
    os_, ls_ = oracle.forward(q, k, v, causal=True, kv_lens=[11, 6], rows=rows, heads=[1, 3],
                              row_block=2)
    np.testing.assert_allclose(os_[:, :, [1, 3]], o[:, rows][:, :, [1, 3]], rtol=0, atol=1e-14)
    np.testing.assert_allclose(ls_[:, [1, 3]], lse[:, [1, 3]][:, :, rows], rtol=0, atol=1e-14)


def test_kv_lens_clamped():
    q, k, v = rnd((2, 3, 1, 2), 131), rnd((2, 4, 1, 2), 132), rnd((2, 4, 1, 2), 133)
    o1, _ = oracle.forward(q, k, v, kv_lens=[-5, 99])
    o2, _ = oracle.forward(q, k, v, kv_lens=[0, 4])
    assert np.array_equal(o1, o2)


# --------------------------------------------------------------------------
# split-KV partials and their log-sum-exp combine
# --------------------------------------------------------------------------

def test_split_bounds_partition_the_valid_keys():
    for Lkv, S, kvl in ((1000, 3, 1000), (1000, 3, 500), (131072, 32, 4096), (300, 8, 7)):
        bounds = oracle.split_bounds(kvl, Lkv, S, tile=128)
        covered = []
        for lo, hi in bounds:
            assert lo % 128 == 0 and hi >= lo
            covered.extend(range(lo, hi))
        assert covered == list(range(kvl))


@pytest.mark.parametrize("Lq,causal,kl", [(1, False, [700, 129, 0]), (3, True, [700, 129, 2])])
def test_splitkv_combine_equals_forward(Lq, causal, kl):
    B, Lkv, Hq, Hkv, d = 3, 700, 4, 2, 3
    q, k, v = rnd((B, Lq, Hq, d), 141), rnd((B, Lkv, Hkv, d), 142), rnd((B, Lkv, Hkv, d), 143)
    op, lp = oracle.splitkv_partials(q, k, v, num_splits=4, causal=causal, kv_lens=kl)
    o, lse = oracle.combine(op, lp)
    o_ref, lse_ref = oracle.forward(q, k, v, causal=causal, kv_lens=kl)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=1e-12, atol=1e-13)
    # an empty split carries O = 0 and LSE = -inf
    assert np.all(lp[2, :, 1:] == -np.inf) and np.all(op[2, :, 1:] == 0)


def test_combine_closed_form():
    # two splits with LSE ln 1 and ln 3 -> weights 1/4, 3/4; a third split empty
    op = np.zeros((1, 1, 3, 1, 2))
    op[0, 0, 0, 0] = [1.0, 2.0]
    op[0, 0, 1, 0] = [5.0, -2.0]
    lp = np.array([[[[0.0], [math.log(3.0)], [-np.inf]]]])
    o, lse = oracle.combine(op, lp)
    np.testing.assert_allclose(o[0, 0, 0], [4.0, -1.0], rtol=0, atol=1e-14)
    assert abs(lse[0, 0, 0] - math.log(4.0)) < 1e-15
    o, lse = oracle.combine(np.zeros((1, 1, 2, 1, 2)), np.full((1, 1, 2, 1), -np.inf))
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_backward_row_partition_adds_up():
    q, k, v, do = rnd((2, 7, 4, 3), 151), rnd((2, 9, 2, 3), 152), rnd((2, 9, 2, 3), 153), \
        rnd((2, 7, 4, 3), 154)
    full = oracle.backward(q, k, v, do, causal=True, kv_lens=[9, 5])
    a = oracle.backward(q, k, v, do, causal=True, kv_lens=[9, 5], rows=[0, 2, 3], row_block=2)
    b = oracle.backward(q, k, v, do, causal=True, kv_lens=[9, 5], rows=[1, 4, 5, 6])
    np.testing.assert_allclose(a[1] + b[1], full[1], rtol=0, atol=1e-14)
    np.testing.assert_allclose(a[2] + b[2], full[2], rtol=0, atol=1e-14)
    np.testing.assert_allclose(a[0][:, [0, 2, 3]], full[0][:, [0, 2, 3]], rtol=0, atol=1e-15)
    assert np.all(np.isnan(a[0][:, [1, 4, 5, 6]]))


# --------------------------------------------------------------------------
# local-window masks ("Attention performance", section "Short sequences and
# the default dispatch": position-only masks include window masks)
# --------------------------------------------------------------------------

def brute_force_window(q, k, v, scale, kv_lens, left, right):
    """Pure-Python loops with the window written per (i, j): key j is kept for
    row i iff it lies within `left` keys before and `right` keys after the
    row's diagonal position i + kvl - Lq (negative = unbounded)."""
    B, Lq, Hq, d = q.shape
    Lkv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    o = np.zeros((B, Lq, Hq, d))
    lse = np.full((B, Hq, Lq), -math.inf)
    for b in range(B):
        kvl = Lkv if kv_lens is None else max(0, min(Lkv, int(kv_lens[b])))
        for h in range(Hq):
            for i in range(Lq):
                centre = i + kvl - Lq
                keys = []
                for j in range(kvl):
                    before = centre - j  # > 0: j lies before the diagonal
                    if left >= 0 and before > left:
                        continue
                    if right >= 0 and -before > right:
                        continue
                    keys.append(j)
                if not keys:
                    continue
                sc = {j: scale * sum(float(q[b, i, h, c]) * float(k[b, j, h // G, c]) for c in range(d))
                      for j in keys}
                mx = max(sc.values())
                z = sum(math.exp(sc[j] - mx) for j in keys)
                for j in keys:
                    w = math.exp(sc[j] - mx) / z
                    for c in range(d):
                        o[b, i, h, c] += w * float(v[b, j, h // G, c])
                lse[b, h, i] = mx + math.log(z)
    return o, lse


WINDOW_CASES = [
    # B, Lq, Lkv, Hq, Hkv, d, kv_lens, (left, right)
    (1, 6, 6, 2, 2, 3, None, (2, 0)),        # causal sliding window
    (1, 6, 6, 2, 1, 3, None, (1, 2)),        # two-sided
    (2, 4, 7, 2, 2, 2, None, (-1, 1)),       # right-bounded only, Lq < Lkv
    (2, 7, 4, 2, 1, 3, None, (0, -1)),       # left-bounded only, Lq > Lkv
    (3, 5, 6, 2, 2, 2, [6, 2, 0], (1, 1)),   # with KV lengths, one empty batch
    (1, 5, 5, 2, 2, 3, None, (0, 0)),        # one key per row
]


@pytest.mark.parametrize("case", WINDOW_CASES)
def test_window_forward_matches_brute_force(case):
    B, Lq, Lkv, Hq, Hkv, d, kl, win = case
    q, k, v = rnd((B, Lq, Hq, d), 41), rnd((B, Lkv, Hkv, d), 42), rnd((B, Lkv, Hkv, d), 43)
    o, lse = oracle.forward(q, k, v, scale=0.6, kv_lens=kl, window=win)
    ob, lb = brute_force_window(q, k, v, 0.6, kl, *win)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(lb)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", WINDOW_CASES[:5])
def test_window_backward_matches_finite_differences(case):
    B, Lq, Lkv, Hq, Hkv, d, kl, win = case
    q, k, v, do = rnd((B, Lq, Hq, d), 51), rnd((B, Lkv, Hkv, d), 52), rnd((B, Lkv, Hkv, d), 53), \
        rnd((B, Lq, Hq, d), 54)
    dq, dk, dv = oracle.backward(q, k, v, do, scale=0.6, kv_lens=kl, window=win)

    def loss():
        o, _ = oracle.forward(q, k, v, scale=0.6, kv_lens=kl, window=win)
        return float(np.sum(o * do))

    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            fp = loss()
            x[idx] = old - h
            fm = loss()
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        assert np.max(np.abs(num - g)) / max(1.0, np.max(np.abs(num))) < 1e-6


@pytest.mark.parametrize("Lq,Lkv,left,right", [(9, 9, 3, 0), (9, 9, 2, 3), (6, 11, 4, 1), (11, 6, -1, 5)])
def test_window_against_torch_band_mask(Lq, Lkv, left, right):
    """torch float64 SDPA with a band mask built by tril/triu (a library
    construction independent of the oracle's index arithmetic)."""
    B, H, d, scale = 2, 2, 5, 0.45
    q, k, v, do = rnd((B, Lq, H, d), 61), rnd((B, Lkv, H, d), 62), rnd((B, Lkv, H, d), 63), rnd((B, Lq, H, d), 64)
    ones = torch.ones(Lq, Lkv, dtype=torch.bool)
    off = Lkv - Lq
    band = torch.tril(ones, diagonal=off + right) if right >= 0 else ones
    if left >= 0:
        band = band & torch.triu(ones, diagonal=off - left)
    assert band.any(dim=1).all()  # torch's SDPA returns NaN on empty rows; keep every row non-empty here
    o_t, dq_t, dk_t, dv_t = _torch_ref(q, k, v, do, scale, band)
    o, _ = oracle.forward(q, k, v, scale=scale, window=(left, right))
    dq, dk, dv = oracle.backward(q, k, v, do, scale=scale, window=(left, right))
    for a, b in ((o, o_t), (dq, dq_t), (dk, dk_t), (dv, dv_t)):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_window_special_cases_reduce_to_causal_and_unmasked():
    B, Lq, Lkv, H, d = 2, 7, 9, 2, 3
    q, k, v, do = rnd((B, Lq, H, d), 71), rnd((B, Lkv, H, d), 72), rnd((B, Lkv, H, d), 73), rnd((B, Lq, H, d), 74)
    kl = [9, 5]
    for win, causal in (((-1, 0), True), ((-1, -1), False), ((None, None), False)):
        a = oracle.forward(q, k, v, kv_lens=kl, window=win)
        b = oracle.forward(q, k, v, kv_lens=kl, causal=causal)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        ga = oracle.backward(q, k, v, do, kv_lens=kl, window=win)
        gb = oracle.backward(q, k, v, do, kv_lens=kl, causal=causal)
        for x, y in zip(ga, gb):
            assert np.array_equal(x, y)


def test_window_zero_width_gives_the_diagonal_value():
    """window (0, 0) with Lq == Lkv: row i sees only key i, so O[i] = V[i]
    exactly and dQ = dK = 0 exactly (a single valid key)."""
    B, L, H, d = 2, 6, 2, 4
    q, k, v, do = rnd((B, L, H, d), 81), rnd((B, L, H, d), 82), rnd((B, L, H, d), 83), rnd((B, L, H, d), 84)
    o, lse = oracle.forward(q, k, v, window=(0, 0))
    np.testing.assert_array_equal(o, v)
    dq, dk, dv = oracle.backward(q, k, v, do, window=(0, 0))
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv, do, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# segment (document) masks: ids per token, a key is kept only for rows with
# the same id ("Attention performance", section "H100 (Hopper)" / "Mosaic
# GPU" list segments among the masks; flex-attention style document masks)
# --------------------------------------------------------------------------

def brute_force_segments(q, k, v, scale, qseg, kseg, causal):
    B, Lq, Hq, d = q.shape
    Lkv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    o = np.zeros((B, Lq, Hq, d))
    for b in range(B):
        for h in range(Hq):
            for i in range(Lq):
                keys = [j for j in range(Lkv) if qseg[b][i] == kseg[b][j] and (not causal or j <= i + Lkv - Lq)]
                if not keys:
                    continue
                sc = [scale * sum(float(q[b, i, h, c]) * float(k[b, j, h // G, c]) for c in range(d)) for j in keys]
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                z = sum(w)
                for wj, j in zip(w, keys):
                    for c in range(d):
                        o[b, i, h, c] += wj / z * float(v[b, j, h // G, c])
    return o


SEG_CASES = [
    # B, Lq, Lkv, H, d, causal, q segment ids, kv segment ids
    (1, 6, 6, 2, 3, False, [[0, 0, 1, 1, 1, 2]], [[0, 0, 1, 1, 1, 2]]),
    (1, 6, 6, 2, 3, True, [[0, 0, 1, 1, 1, 2]], [[0, 0, 1, 1, 1, 2]]),
    (2, 4, 7, 2, 2, False, [[3, 1, 1, 9], [0, 0, 0, 0]], [[1, 3, 3, 1, 7, 7, 1], [0, 1, 0, 1, 0, 1, 0]]),
]


@pytest.mark.parametrize("case", SEG_CASES)
def test_segments_forward_matches_brute_force(case):
    B, Lq, Lkv, H, d, causal, qs, ks = case
    q, k, v = rnd((B, Lq, H, d), 91), rnd((B, Lkv, H, d), 92), rnd((B, Lkv, H, d), 93)
    o, _ = oracle.forward(q, k, v, scale=0.8, causal=causal, segments=(qs, ks))
    np.testing.assert_allclose(o, brute_force_segments(q, k, v, 0.8, qs, ks, causal), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", SEG_CASES)
def test_segments_backward_matches_finite_differences(case):
    B, Lq, Lkv, H, d, causal, qs, ks = case
    q, k, v, do = rnd((B, Lq, H, d), 94), rnd((B, Lkv, H, d), 95), rnd((B, Lkv, H, d), 96), rnd((B, Lq, H, d), 97)
    dq, dk, dv = oracle.backward(q, k, v, do, scale=0.8, causal=causal, segments=(qs, ks))

    def loss():
        o, _ = oracle.forward(q, k, v, scale=0.8, causal=causal, segments=(qs, ks))
        return float(np.sum(o * do))

    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            fp = loss()
            x[idx] = old - h
            fm = loss()
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        assert np.max(np.abs(num - g)) / max(1.0, np.max(np.abs(num))) < 1e-6


def test_segments_against_torch_boolean_mask():
    """torch float64 SDPA with the mask built by comparing the id tensors."""
    B, Lq, Lkv, H, d, scale = 2, 9, 9, 2, 4, 0.5
    rng = np.random.default_rng(3)
    qs = np.sort(rng.integers(0, 3, size=(B, Lq)), axis=1)
    ks = qs.copy()
    q, k, v, do = rnd((B, Lq, H, d), 101), rnd((B, Lkv, H, d), 102), rnd((B, Lkv, H, d), 103), rnd((B, Lq, H, d), 104)
    mask = torch.tensor(qs)[:, None, :, None] == torch.tensor(ks)[:, None, None, :]
    o_t, dq_t, dk_t, dv_t = _torch_ref(q, k, v, do, scale, mask)
    o, _ = oracle.forward(q, k, v, scale=scale, segments=(qs, ks))
    dq, dk, dv = oracle.backward(q, k, v, do, scale=scale, segments=(qs, ks))
    for a, b in ((o, o_t), (dq, dq_t), (dk, dk_t), (dv, dv_t)):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_segments_special_cases():
    """one shared id is no mask; per-token unique ids with Lq == Lkv leave each
    row its own key (O = V exactly, dQ = dK = 0)."""
    B, L, H, d = 2, 7, 2, 3
    q, k, v, do = rnd((B, L, H, d), 111), rnd((B, L, H, d), 112), rnd((B, L, H, d), 113), rnd((B, L, H, d), 114)
    same = np.zeros((B, L), dtype=np.int64)
    a, b_ = oracle.forward(q, k, v, segments=(same, same)), oracle.forward(q, k, v)
    assert np.array_equal(a[0], b_[0]) and np.array_equal(a[1], b_[1])
    uniq = np.tile(np.arange(L), (B, 1))
    o, _ = oracle.forward(q, k, v, segments=(uniq, uniq))
    np.testing.assert_array_equal(o, v)
    dq, dk, dv = oracle.backward(q, k, v, do, segments=(uniq, uniq))
    assert np.all(dq == 0) and np.all(dk == 0)
