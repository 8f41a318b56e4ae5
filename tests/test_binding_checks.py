"""The Python binding refuses tensors the library would misread -- on the
CPU, non-contiguous views, mixed dtypes, mismatched shapes -- before any call
reaches the C ABI (no GPU needed: the checks run first)."""

import pytest
import torch

import exact_attention_34_gb300 as ea


def qkv(B=1, L=128, H=2, d=64, dtype=torch.bfloat16):
    q = torch.zeros(B, L, H, d, dtype=dtype)
    return q, q.clone(), q.clone()


def test_cpu_tensors_are_refused():
    q, k, v = qkv()
    with pytest.raises(ValueError, match="CUDA"):
        ea.attn_fwd(q, k, v, q.clone(), torch.zeros(1, 2, 128))


def test_shape_and_dtype_mismatches_are_refused():
    q, k, v = qkv()
    with pytest.raises(ValueError, match="batch or head_dim"):
        ea._dims(q, torch.zeros(1, 128, 2, 32, dtype=q.dtype))
    with pytest.raises(ValueError, match="k's shape"):
        ea._dims(q, k, torch.zeros(1, 100, 2, 64, dtype=q.dtype))
    with pytest.raises(TypeError, match="one dtype"):
        ea._dims(q, k.float(), v)
    with pytest.raises(TypeError, match="one dtype"):
        ea._dims(q, k, v.float())
    with pytest.raises(ValueError, match="multiple of KV heads"):
        ea._dims(torch.zeros(1, 128, 3, 64), torch.zeros(1, 128, 2, 64))
    with pytest.raises(ValueError, match="head_dim"):
        ea._dims(torch.zeros(128, 64), k)


def test_non_contiguous_views_are_refused():
    q = torch.zeros(1, 2, 128, 64).transpose(1, 2)  # [1, 128, 2, 64] view, not contiguous
    assert not q.is_contiguous()
    with pytest.raises(ValueError, match="contiguous"):
        ea._ptr(q)
