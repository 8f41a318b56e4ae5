"""Maximum sizes: a KV sequence whose K and V tensors hold more than 2^31
elements (4.3 GB each in bf16), so every offset past 2^31 must be computed in
64 bits.  The outputs are checked through properties that hold at any size:
with K = 0 every score is 0, so each row's softmax is uniform over the N keys:
  O_i = mean_j V_j,  LSE_i = ln N,  dQ = 0,  dV_j = (1/N) sum_{h,i} dO_hi,
  dK_j = (s/N) sum_{h,i} (dO_hi . (V_j - mean V)) q_hi.
V is zero except in two 256-key regions, one at the start and one past element
2^31, so the results depend on the far keys."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

N = (1 << 24) + 384  # keys: N * 128 > 2^31 elements per K/V tensor
D = 128
HQ, HKV, LQ = 4, 1, 128
REGIONS = (slice(0, 256), slice(N - 256, N))


def _inputs():
    g = torch.Generator(device="cuda").manual_seed(3)
    q = torch.randn(1, LQ, HQ, D, device="cuda", generator=g).to(torch.bfloat16)
    do = torch.randn(1, LQ, HQ, D, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.zeros(1, N, HKV, D, device="cuda", dtype=torch.bfloat16)
    v = torch.zeros(1, N, HKV, D, device="cuda", dtype=torch.bfloat16)
    for r in REGIONS:
        v[0, r] = torch.randn(256, HKV, D, device="cuda", generator=g).to(torch.bfloat16)
    return q, k, v, do


def _v_mean(v):
    tot = np.zeros(D)
    for r in REGIONS:
        tot += v[0, r, 0].double().cpu().numpy().sum(axis=0)
    return tot / N


def test_forward_backward_over_a_2_31_element_cache():
    import exact_attention_34_gb300 as ea

    q, k, v, do = _inputs()
    assert k.numel() > (1 << 31)
    o, lse = ea.forward(q, k, v)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    vbar = _v_mean(v)
    o_np = o.double().cpu().numpy()[0]  # [LQ, HQ, D]
    assert np.max(np.abs(o_np - vbar)) <= 1e-2 * np.max(np.abs(vbar))
    np.testing.assert_allclose(lse.cpu().numpy(), np.log(N), rtol=1e-5)

    dq, dk, dv = ea.backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    assert torch.count_nonzero(dq).item() == 0
    dos = do.double().cpu().numpy()[0]  # [LQ, HQ, D]
    qs = q.double().cpu().numpy()[0]
    dv_ref = dos.sum(axis=(0, 1)) / N
    s = 1.0 / np.sqrt(D)
    # sample keys at the start, in the middle, in both V regions and past 2^31 elements
    for j in (0, 100, 255, 256, 1 << 20, (1 << 24) - 1, 1 << 24, N - 257, N - 200, N - 1):
        dv_j = dv[0, j, 0].double().cpu().numpy()
        assert np.max(np.abs(dv_j - dv_ref)) <= 1e-2 * np.max(np.abs(dv_ref)), j
        vj = v[0, j, 0].double().cpu().numpy()
        coef = np.einsum("ihd,d->ih", dos, vj - vbar)  # dO_hi . (V_j - mean V)
        dk_ref = (s / N) * np.einsum("ih,ihd->d", coef, qs)
        dk_j = dk[0, j, 0].double().cpu().numpy()
        assert np.max(np.abs(dk_j - dk_ref)) <= 1e-2 * np.max(np.abs(dk_ref)), j


def test_decode_over_a_2_31_element_cache():
    import exact_attention_34_gb300 as ea

    _, k, v, _ = _inputs()
    g = torch.Generator(device="cuda").manual_seed(4)
    q1 = torch.randn(1, 1, HQ, D, device="cuda", generator=g).to(torch.bfloat16)
    o, lse = ea.decode(q1, k, v)
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    vbar = _v_mean(v)
    assert np.max(np.abs(o.double().cpu().numpy()[0, 0] - vbar)) <= 1e-2 * np.max(np.abs(vbar))
    np.testing.assert_allclose(lse.cpu().numpy(), np.log(N), rtol=1e-5)
