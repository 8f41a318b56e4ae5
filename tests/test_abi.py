"""Host-side checks of the C-ABI library: it builds, loads, exports every
symbol include/attn.h declares, and rejects bad arguments with the documented
status before launching anything.  No GPU needed."""

import ctypes
import os
import re

import pytest

import exact_attention_34_gb300 as ea
from exact_attention_34_gb300 import build as eb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    eb.build()
    return ea.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = header_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(ea.EXPORTED)


def test_status_strings(L):
    for code, name in [(0, "ATTN_OK"), (1, "ATTN_ERR_INVALID_ARG"), (2, "ATTN_ERR_UNSUPPORTED"),
                       (3, "ATTN_ERR_WORKSPACE"), (4, "ATTN_ERR_CUDA"), (5, "ATTN_ERR_DEVICE")]:
        assert ea.status_string(code) == name
    assert ea.status_string(99) == "ATTN_ERR_UNKNOWN"


FAKE = 0x10000  # 16-byte aligned fake device address; never dereferenced (validation fails first)


def fwd(L, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Lq=128, Lkv=128, Hq=2, Hkv=2, d=64, scale=0.125,
        causal=0, kv=None, dt=0):
    return L.attn_fwd(q, k, v, o, lse, B, Lq, Lkv, Hq, Hkv, d, scale, causal, kv, dt, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(Lq=-1), 1), (dict(Lkv=0), 1), (dict(Hq=3, Hkv=2), 1), (dict(d=96), 2),
    (dict(d=48), 2), (dict(d=256, dt=1), 2), (dict(d=512), 2), (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(scale=-1.0), 1),
    (dict(causal=2), 1), (dict(dt=7), 1), (dict(q=None), 1), (dict(lse=None), 1), (dict(k=FAKE + 8), 1),
    (dict(kv=FAKE + 2), 1),
])
def test_fwd_rejects_bad_arguments(L, kw, code):
    assert fwd(L, **kw) == code
    assert len(L.attn_last_error()) > 0


def test_bwd_workspace_rules(L):
    B, Lq, Hq, d = 2, 300, 4, 128
    det = L.attn_bwd_workspace_size(B, Lq, Hq, d, 1, 0)
    atom = L.attn_bwd_workspace_size(B, Lq, Hq, d, 0, 0)
    assert det >= B * Hq * Lq * 4 and det % 256 == 0
    assert atom >= det + B * Lq * Hq * d * 4
    args = [FAKE] * 9 + [B, Lq, Lq, Hq, Hq, d, 0.1, 0, None, 0, 1]
    assert L.attn_bwd(*args, None, det, None) == 3          # no workspace
    assert L.attn_bwd(*args, FAKE, det - 1, None) == 3      # too small
    assert L.attn_bwd(*args, FAKE + 16, det, None) == 1     # misaligned workspace
    args_atomic = [FAKE] * 9 + [B, Lq, Lq, Hq, Hq, d, 0.1, 0, None, 0, 0]
    assert L.attn_bwd(*args_atomic, FAKE, det, None) == 3   # atomic needs the dQ buffer too
    bad_det = [FAKE] * 9 + [B, Lq, Lq, Hq, Hq, d, 0.1, 0, None, 0, 3]
    assert L.attn_bwd(*bad_det, FAKE, atom, None) == 1


def test_bwd_ordered_single_pass_rules(L):
    """deterministic = 2: the dQ buffer plus one turn counter per (batch, head,
    query tile) and a ticket; 16-bit types at head_dim <= 128 only."""
    B, Lq, Hq, d = 2, 300, 4, 128
    atom = L.attn_bwd_workspace_size(B, Lq, Hq, d, 0, 0)
    ordered = L.attn_bwd_workspace_size(B, Lq, Hq, d, 2, 0)
    assert ordered >= atom + (B * Hq * 3 + 1) * 4 and ordered % 256 == 0
    args = [FAKE] * 9 + [B, Lq, Lq, Hq, Hq, d, 0.1, 0, None, 0, 2]
    assert L.attn_bwd(*args, FAKE, atom, None) == 3          # the counters do not fit
    f32 = [FAKE] * 9 + [B, Lq, Lq, Hq, Hq, d, 0.1, 0, None, 1, 2]
    assert L.attn_bwd(*f32, FAKE, 1 << 30, None) == 2        # float32: unsupported
    assert "deterministic = 1" in L.attn_last_error().decode()
    d256 = [FAKE] * 9 + [B, Lq, Lq, Hq, Hq, 256, 0.1, 0, None, 0, 2]
    assert L.attn_bwd(*d256, FAKE, 1 << 30, None) == 2       # head_dim 256: unsupported


def test_decode_rules(L):
    s = L.attn_decode_num_splits(8, 1, 131072, 32, 8, 128)
    assert 1 <= s <= 1024
    assert L.attn_decode_num_splits(1, 1, 100, 1, 1, 64) == 1
    # G * Lq must fit one 128-row tile
    args = [FAKE] * 5 + [1, 64, 4096, 8, 2, 128, 0.1, 0, None, 4, 0, None]
    assert L.attn_decode_splitkv(*args) == 2
    assert L.attn_decode_splitkv(*([FAKE] * 5 + [1, 16, 4096, 32, 8, 128, 0.1, 1, None, -1, 0, None])) == 1
    assert L.attn_decode_combine(FAKE, FAKE, FAKE, FAKE, 1, 1, 4, 128, 0, 0, None) == 1
    assert L.attn_decode_workspace_size(8, 1, 32, 128, 16) >= 8 * 32 * 16 * 128 * 4 + 8 * 32 * 16 * 4


def test_preprocess_rejects_bad_arguments(L):
    assert L.attn_bwd_preprocess(FAKE, FAKE, None, 1, 128, 2, 64, 0, None) == 1
    assert L.attn_bwd_preprocess(FAKE, FAKE, FAKE, 1, 128, 2, 80, 0, None) == 2


def test_segment_info_rules(L):
    # one int4 record per 128-position block of each side, per batch element
    assert L.attn_segment_info_size(2, 300, 129) == 2 * (3 + 2) * 16
    assert L.attn_segment_info_size(1, 1, 1) == 32
    assert L.attn_segment_info_size(0, 128, 128) == 0
    need = L.attn_segment_info_size(2, 300, 129)
    assert L.attn_segment_info(FAKE, FAKE, 2, 300, 129, FAKE, need - 1, None) == 3  # too small
    assert L.attn_segment_info(FAKE, FAKE, 2, 300, 129, None, need, None) == 1
    assert L.attn_segment_info(FAKE, FAKE, 2, 300, 129, FAKE + 4, need, None) == 1
    assert L.attn_segment_info(None, FAKE, 2, 300, 129, FAKE, need, None) == 1
    assert L.attn_segment_info(FAKE, FAKE, 0, 300, 129, FAKE, need, None) == 1


def test_segment_entry_points_reject_bad_arguments(L):
    base = [FAKE] * 5 + [1, 128, 128, 2, 2, 64, 0.125, -1, 0]
    # q_segment, kv_segment, segment_info, kv_lens, dtype, stream
    assert L.attn_fwd_segments(*base, None, FAKE, None, None, 0, None) == 1
    assert L.attn_fwd_segments(*base, FAKE, FAKE + 4, None, None, 0, None) == 1
    assert L.attn_fwd_segments(*base, FAKE, FAKE, FAKE + 8, None, 0, None) == 1  # misaligned info
    assert L.attn_fwd_segments(*([FAKE] * 5 + [1, 128, 128, 2, 2, 80, 0.125, -1, 0]), FAKE, FAKE, None, None, 0,
                               None) == 2
    bbase = [FAKE] * 9 + [1, 128, 128, 2, 2, 64, 0.125, -1, 0]
    assert L.attn_bwd_segments(*bbase, FAKE, None, None, None, 0, 1, FAKE, 1 << 20, None) == 1
    assert L.attn_bwd_segments(*bbase, FAKE, FAKE, FAKE + 8, None, 0, 1, FAKE, 1 << 20, None) == 1


def test_split_forward_rules(L):
    # the library's choice: one batch element may hold every key when KV lengths
    # are given (B=4 H8 Lq 2048 Lkv 16384: 64 busy pairs, two pieces fill one
    # wave); a full grid is not split; one pair alone is cut in four (rounds of
    # 1/s plus 5 % a piece); head_dim 256 and float32 are never split
    assert L.attn_fwd_num_splits(4, 2048, 16384, 8, 128, 1, 0) == 2
    assert L.attn_fwd_num_splits(4, 8192, 8192, 8, 128, 0, 0) == 1
    assert L.attn_fwd_num_splits(1, 256, 65536, 1, 64, 0, 2) == 4
    assert L.attn_fwd_num_splits(1, 256, 65536, 1, 256, 0, 0) == 1
    assert L.attn_fwd_num_splits(1, 256, 65536, 1, 128, 0, 1) == 1
    assert L.attn_fwd_num_splits(1, 256, 1000, 1, 128, 0, 0) == 1  # under 8 tiles a piece
    assert L.attn_fwd_num_splits(0, 256, 65536, 1, 128, 0, 0) == 1
    # partial outputs, log-sum-exps and one counter per query-tile pair, each
    # 256-byte aligned; nothing for one piece or d = 256
    rows = 2 * 4 * 3 * 300
    pairs = 2 * 4 * 2
    assert L.attn_fwd_split_workspace_size(2, 300, 4, 64, 3) == (-(-rows * 64 * 4 // 256) * 256 + -(-rows * 4 // 256) * 256
                                                                 + -(-pairs * 4 // 256) * 256)
    assert L.attn_fwd_split_workspace_size(2, 300, 4, 64, 1) == 0
    assert L.attn_fwd_split_workspace_size(2, 300, 4, 256, 3) == 0
    base = [FAKE] * 5 + [2, 300, 4096, 4, 2, 64, 0.125, -1, 0, None]
    need = L.attn_fwd_split_workspace_size(2, 300, 4, 64, 3)
    assert L.attn_fwd_split(*base, -1, FAKE, need, 0, None) == 1
    assert L.attn_fwd_split(*base, 2000, FAKE, 1 << 40, 0, None) == 1
    assert L.attn_fwd_split(*base, 3, None, need, 0, None) == 3
    assert L.attn_fwd_split(*base, 3, FAKE, need - 1, 0, None) == 3
    assert L.attn_fwd_split(*base, 3, FAKE + 16, need, 0, None) == 1  # workspace not 256-byte aligned
    assert L.attn_fwd_split(*([FAKE] * 5 + [2, 300, 4096, 4, 2, 96, 0.125, -1, 0, None]), 3, FAKE, need, 0,
                            None) == 2
    assert L.attn_fwd_split(*([FAKE] * 4 + [None] + [2, 300, 4096, 4, 2, 64, 0.125, -1, 0, None]), 3, FAKE, need, 0,
                            None) == 1
