"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only draws random tensors and
per-batch KV lengths, so both the fp64 oracle and the CUDA library can be fed
the very same rounded inputs.

Recipe (the pages benchmark random inputs, no dataset):

* ``torch.Generator().manual_seed(seed)`` (seed 0 unless stated), then
  ``torch.randn`` in float32 in the order q, k, v, dO, each cast to the
  working dtype (round to nearest even for bf16);
* KV lengths from a second generator seeded with 1: uniform integers in the
  configuration's range, with fixed overrides for the single-key / empty rows.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32, "fp16": torch.float16}


@dataclass(frozen=True)
class Problem:
    """Shape of one attention call."""

    B: int
    Lq: int
    Lkv: int
    Hq: int
    Hkv: int
    d: int
    dtype: str = "bf16"
    causal: bool = False
    kv_lens: tuple | None = None  # per-batch KV lengths, or None for all Lkv
    name: str = ""
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


def make_inputs(p: Problem, seed: int = 0, with_do: bool = True):
    """q, k, v (and dO) as CPU tensors of ``p.dtype``, drawn in that order."""
    g = torch.Generator().manual_seed(seed)
    dt = DTYPES[p.dtype]
    q = torch.randn(p.B, p.Lq, p.Hq, p.d, generator=g, dtype=torch.float32).to(dt)
    k = torch.randn(p.B, p.Lkv, p.Hkv, p.d, generator=g, dtype=torch.float32).to(dt)
    v = torch.randn(p.B, p.Lkv, p.Hkv, p.d, generator=g, dtype=torch.float32).to(dt)
    out = [q, k, v]
    if with_do:
        out.append(torch.randn(p.B, p.Lq, p.Hq, p.d, generator=g, dtype=torch.float32).to(dt))
    return tuple(out)


def uniform_kv_lens(B: int, lo: int, hi: int, seed: int = 1, overrides: dict | None = None):
    """Per-batch KV lengths uniform in [lo, hi], then ``overrides`` {b: len}."""
    g = torch.Generator().manual_seed(seed)
    kl = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    for b, val in (overrides or {}).items():
        kl[b] = val
    return tuple(int(x) for x in kl)


# --- the five workloads -----------------------------------------------------

def tiny() -> Problem:
    """Exact check: fp32, B1 Hq=Hkv=2, L=128, d=64, non-causal, no mask."""
    return Problem(1, 128, 128, 2, 2, 64, "fp32", False, None, "tiny")


def grid(T: int, d: int, causal: bool, dtype: str = "bf16") -> Problem:
    """Attention grid / ragged lengths: B4 H8, Lq = Lkv = T."""
    return Problem(4, T, T, 8, 8, d, dtype, causal, None, f"grid_T{T}_d{d}_c{int(causal)}_{dtype}")


GRID_T = (128, 512, 1024, 2048, 4096, 8192)
RAGGED_T = (600, 1500, 3000)


def kvlen_gqa() -> Problem:
    """KVLenMask + GQA + Lq != Lkv: B4 Hq8 Hkv2 Lq2048 Lkv16384 d128 bf16,
    lengths uniform in [1, 16384] with batch 2 at 1 key and batch 3 at 0."""
    kl = uniform_kv_lens(4, 1, 16384, seed=1, overrides={2: 1, 3: 0})
    return Problem(4, 2048, 16384, 8, 2, 128, "bf16", False, kl, "kvlen_gqa")


def decode(Lq: int = 1, causal: bool = False, Lkv: int = 131072, B: int = 8) -> Problem:
    """Split-KV decode: B8 Hq32 Hkv8 d128 bf16 over a 128k-key cache, lengths
    uniform in [4096, 131072]; Lq=16 runs with the causal offset."""
    kl = uniform_kv_lens(B, 4096, Lkv, seed=1)
    return Problem(B, Lq, Lkv, 32, 8, 128, "bf16", causal, kl, f"decode_Lq{Lq}_c{int(causal)}")


def headline() -> Problem:
    """bf16 causal fwd+bwd at B4 H8 T8192 d128."""
    return grid(8192, 128, True, "bf16")


def fwd_flops(p: Problem) -> float:
    """Counted forward FLOPs: 4 * B * Hq * Lq * Lkv * d, exactly halved when
    causal with Lq == Lkv and no lengths; with KV lengths (or a causal decode
    offset) counted over valid keys only."""
    if p.kv_lens is None and not p.causal:
        return 4.0 * p.B * p.Hq * p.Lq * p.Lkv * p.d
    if p.kv_lens is None and p.causal and p.Lq == p.Lkv:
        return 2.0 * p.B * p.Hq * p.Lq * p.Lkv * p.d
    kl = p.kv_lens if p.kv_lens is not None else (p.Lkv,) * p.B
    n = 0
    for kvl in kl:
        kvl = max(0, min(int(kvl), p.Lkv))
        if not p.causal:
            n += p.Lq * kvl
        else:
            for i in range(p.Lq):
                n += max(0, min(kvl, i + kvl - p.Lq + 1))
    return 4.0 * p.Hq * p.d * n
