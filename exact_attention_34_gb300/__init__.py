"""Python binding of the GB300 exact-attention C-ABI library (``libattn.so``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind ``include/attn.h``.  PyTorch supplies device memory and streams.
The functions named like the C entry points (``attn_fwd``, ``attn_bwd``, ...)
take torch tensors, read the sizes off their shapes and raise ``AttnError`` on
any status other than ``ATTN_OK``.  ``forward`` / ``backward`` / ``decode``
are conveniences that allocate the outputs with torch first.

There is no fallback: if ``libattn.so`` is missing or fails to load, importing
the functions raises.  Build it with ``exact_attention_34_gb300.build.build()``
(or ``__graft_entry__.build()``).
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

from .build import LIB as _LIB_PATH

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_WORKSPACE = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_DEVICE = 5

ATTN_BF16 = 0
ATTN_FP32 = 1
ATTN_FP16 = 2

_DT = {torch.bfloat16: ATTN_BF16, torch.float32: ATTN_FP32, torch.float16: ATTN_FP16}


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}: {detail}")


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libattn.so once (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is not built; run exact_attention_34_gb300.build.build()")
    L = ctypes.CDLL(_LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "attn_status_string": (ctypes.c_char_p, [I]),
        "attn_last_error": (ctypes.c_char_p, []),
        "attn_fwd": (I, [P, P, P, P, P, I, I, I, I, I, I, F, I, P, I, P]),
        "attn_bwd_preprocess": (I, [P, P, P, I, I, I, I, I, P]),
        "attn_bwd_workspace_size": (S, [I, I, I, I, I, I]),
        "attn_bwd": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, I, I, P, S, P]),
        "attn_decode_num_splits": (I, [I, I, I, I, I, I]),
        "attn_decode_splitkv": (I, [P, P, P, P, P, I, I, I, I, I, I, F, I, P, I, I, P]),
        "attn_decode_combine": (I, [P, P, P, P, I, I, I, I, I, I, P]),
        "attn_decode_workspace_size": (S, [I, I, I, I, I]),
        "attn_device_status": (I, [ctypes.POINTER(I), ctypes.POINTER(I), I]),
        "attn_timing_enable": (I, [I]),
        "attn_timing_query": (I, [ctypes.c_char_p, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I)]),
        "attn_bwd_static_scratch": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, I, P]),
        "attn_fwd_window": (I, [P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, I, P]),
        "attn_bwd_window": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, I, I, P, S, P]),
        "attn_fwd_segments": (I, [P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, P, P, P, I, P]),
        "attn_bwd_segments": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, P, P, P, I, I, P, S, P]),
        "attn_segment_info_size": (S, [I, I, I]),
        "attn_segment_info": (I, [P, P, I, I, I, P, S, P]),
        "attn_selftest_wait_timeout": (I, [I, P]),
        "attn_fwd_num_splits": (I, [I, I, I, I, I, I, I]),
        "attn_fwd_split_workspace_size": (S, [I, I, I, I, I]),
        "attn_fwd_split": (I, [P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, I, P, S, I, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


EXPORTED = (
    "attn_status_string", "attn_last_error", "attn_fwd", "attn_bwd_preprocess", "attn_bwd_workspace_size",
    "attn_bwd", "attn_decode_num_splits", "attn_decode_splitkv", "attn_decode_combine",
    "attn_decode_workspace_size", "attn_device_status", "attn_timing_enable", "attn_timing_query",
    "attn_bwd_static_scratch", "attn_fwd_window", "attn_bwd_window", "attn_fwd_segments", "attn_bwd_segments",
    "attn_segment_info_size", "attn_segment_info", "attn_selftest_wait_timeout", "attn_fwd_num_splits",
    "attn_fwd_split_workspace_size", "attn_fwd_split",
)


def status_string(s: int) -> str:
    return lib().attn_status_string(int(s)).decode()


def _check(status: int, where: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, where, lib().attn_last_error().decode())


def _ptr(t):
    """Device address of a tensor the library reads or writes.  The library
    indexes dense row-major memory on the GPU, so anything else is refused
    here rather than read with the wrong strides."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor (shape {tuple(t.shape)}, strides {t.stride()}); "
                         "call .contiguous() first")
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    return t.data_ptr()  # a plain int: ctypes converts it for the void* argument


# torch's current stream as a raw handle, without building a Stream object
# (a few microseconds per call, which short calls notice)
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, like=None):
    """The stream handle to pass: `stream`, else torch's current stream on the
    device of tensor `like` (or the current device)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_current_stream is not None:
        return _raw_current_stream(like.get_device() if like is not None else torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _dtype(t) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def _dims(q, k, v=None):
    """(B, Lq, Lkv, Hq, Hkv, d) of q [B, Lq, Hq, d] and k (and v) [B, Lkv, Hkv, d]."""
    qs, ks = q.shape, k.shape
    if len(qs) != 4 or len(ks) != 4:
        raise ValueError("q and k must be [batch, seq, heads, head_dim]")
    B, Lq, Hq, d = qs
    kB, Lkv, Hkv, kd = ks
    if kB != B or kd != d:
        raise ValueError(f"k {tuple(ks)} does not match q {tuple(qs)} in batch or head_dim")
    dt = q.dtype
    if v is not None and v.shape != ks:
        raise ValueError(f"v {tuple(v.shape)} must have k's shape {tuple(ks)}")
    if k.dtype != dt or (v is not None and v.dtype != dt):
        raise TypeError("q, k and v must share one dtype")
    if Hkv == 0 or Hq % Hkv != 0:
        raise ValueError(f"query heads {Hq} must be a multiple of KV heads {Hkv}")
    return B, Lq, Lkv, Hq, Hkv, d


_default_scales = {}


def _scale(scale, d):
    if scale is not None:
        return float(scale)
    s = _default_scales.get(d)
    if s is None:
        s = _default_scales[d] = 1.0 / math.sqrt(d)
    return s


# ---- entry points with the C names -------------------------------------------

def attn_fwd(q, k, v, o, lse, scale=None, causal=False, kv_lens=None, stream=None):
    _attn_fwd(_dims(q, k, v), q, k, v, o, lse, scale, causal, kv_lens, stream)


def _attn_fwd(dims, q, k, v, o, lse, scale, causal, kv_lens, stream):
    B, Lq, Lkv, Hq, Hkv, d = dims
    st = (_lib or lib()).attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Lq, Lkv, Hq, Hkv, d,
                                  _scale(scale, d), 1 if causal else 0, _ptr(kv_lens), _dtype(q), _stream(stream, q))
    if st:
        _check(st, "attn_fwd")


def _window(window):
    """(left, right) with None or a negative value meaning unbounded."""
    left, right = window
    return (-1 if left is None else int(left)), (-1 if right is None else int(right))


def attn_fwd_window(q, k, v, o, lse, window, scale=None, kv_lens=None, stream=None):
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k, v)
    wl, wr = _window(window)
    _check(lib().attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Lq, Lkv, Hq, Hkv, d,
                                 _scale(scale, d), wl, wr, _ptr(kv_lens), _dtype(q), _stream(stream, q)),
           "attn_fwd_window")


def attn_fwd_num_splits(B, Lq, Lkv, Hq, d, has_kv_lens, dtype) -> int:
    return int(lib().attn_fwd_num_splits(B, Lq, Lkv, Hq, d, int(bool(has_kv_lens)), _DT[dtype]))


def attn_fwd_split_workspace_size(B, Lq, Hq, d, num_splits) -> int:
    return int(lib().attn_fwd_split_workspace_size(B, Lq, Hq, d, num_splits))


def attn_fwd_split(q, k, v, o, lse, workspace, num_splits, window=(-1, -1), scale=None, kv_lens=None, stream=None):
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k, v)
    wl, wr = _window(window)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().attn_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Lq, Lkv, Hq, Hkv, d,
                                _scale(scale, d), wl, wr, _ptr(kv_lens), int(num_splits), _ptr(workspace), nbytes,
                                _dtype(q), _stream(stream, q)),
           "attn_fwd_split")


def attn_segment_info_size(B, Lq, Lkv) -> int:
    return int(lib().attn_segment_info_size(B, Lq, Lkv))


def attn_segment_info(q_segment, kv_segment, info, stream=None):
    B, Lq = q_segment.shape
    Lkv = kv_segment.shape[1]
    _check(lib().attn_segment_info(_ptr(q_segment), _ptr(kv_segment), B, Lq, Lkv, _ptr(info),
                                   info.numel() * info.element_size(), _stream(stream, info)),
           "attn_segment_info")


def segment_info(q_segment, kv_segment, stream=None):
    """Block summary of the segment ids (a uint8 device tensor) for the
    segment entry points; recompute it whenever the ids change."""
    B, Lq = q_segment.shape
    info = torch.empty(attn_segment_info_size(B, Lq, kv_segment.shape[1]), device=q_segment.device,
                       dtype=torch.uint8)
    attn_segment_info(q_segment, kv_segment, info, stream)
    return info


def attn_fwd_segments(q, k, v, o, lse, q_segment, kv_segment, window=(-1, -1), scale=None, kv_lens=None,
                      stream=None, segment_info=None):
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k, v)
    wl, wr = _window(window)
    _check(lib().attn_fwd_segments(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Lq, Lkv, Hq, Hkv, d,
                                   _scale(scale, d), wl, wr, _ptr(q_segment), _ptr(kv_segment), _ptr(segment_info),
                                   _ptr(kv_lens), _dtype(q), _stream(stream, q)),
           "attn_fwd_segments")


def attn_bwd_preprocess(o, dout, delta, stream=None):
    B, Lq, Hq, d = o.shape
    _check(lib().attn_bwd_preprocess(_ptr(o), _ptr(dout), _ptr(delta), B, Lq, Hq, d, _dtype(o), _stream(stream, o)),
           "attn_bwd_preprocess")


def _det(deterministic) -> int:
    """The C ABI's backward variant: True/1 two-pass, False/0 single pass with
    atomic dQ, 2 single pass with dQ added in key-tile order."""
    return int(deterministic)


_ws_sizes = {}


def attn_bwd_workspace_size(B, Lq, Hq, d, deterministic=True, dtype=torch.bfloat16) -> int:
    key = (B, Lq, Hq, d, _det(deterministic), dtype)
    n = _ws_sizes.get(key)
    if n is None:  # a pure function of its arguments: asked once per shape
        n = _ws_sizes[key] = int(lib().attn_bwd_workspace_size(B, Lq, Hq, d, key[4], _DT[dtype]))
    return n


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, scale=None, causal=False, kv_lens=None,
             deterministic=True, stream=None):
    _attn_bwd(_dims(q, k, v), q, k, v, o, lse, dout, dq, dk, dv, workspace, scale, causal, kv_lens, deterministic,
              stream)


def _attn_bwd(dims, q, k, v, o, lse, dout, dq, dk, dv, workspace, scale, causal, kv_lens, deterministic, stream):
    B, Lq, Lkv, Hq, Hkv, d = dims
    ws_bytes = workspace.numel() * workspace.element_size()
    st = (_lib or lib()).attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                  _ptr(dv), B, Lq, Lkv, Hq, Hkv, d, _scale(scale, d), 1 if causal else 0,
                                  _ptr(kv_lens), _dtype(q), _det(deterministic), _ptr(workspace), ws_bytes,
                                  _stream(stream, q))
    if st:
        _check(st, "attn_bwd")


def attn_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, workspace, window, scale=None, kv_lens=None,
                    deterministic=True, stream=None):
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k, v)
    wl, wr = _window(window)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, Lq, Lkv, Hq, Hkv, d, _scale(scale, d), wl, wr, _ptr(kv_lens),
                                 _dtype(q), _det(deterministic), _ptr(workspace), ws_bytes, _stream(stream, q)),
           "attn_bwd_window")


def attn_bwd_segments(q, k, v, o, lse, dout, dq, dk, dv, workspace, q_segment, kv_segment, window=(-1, -1),
                      scale=None, kv_lens=None, deterministic=True, stream=None, segment_info=None):
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k, v)
    wl, wr = _window(window)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().attn_bwd_segments(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                   _ptr(dv), B, Lq, Lkv, Hq, Hkv, d, _scale(scale, d), wl, wr, _ptr(q_segment),
                                   _ptr(kv_segment), _ptr(segment_info), _ptr(kv_lens), _dtype(q),
                                   _det(deterministic),
                                   _ptr(workspace), ws_bytes, _stream(stream, q)),
           "attn_bwd_segments")


def attn_decode_num_splits(B, Lq, Lkv, Hq, Hkv, d) -> int:
    return int(lib().attn_decode_num_splits(B, Lq, Lkv, Hq, Hkv, d))


def attn_decode_splitkv(q, k_cache, v_cache, o_part, lse_part, num_splits, scale=None, causal=False,
                        kv_lens=None, stream=None):
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k_cache, v_cache)
    _check(lib().attn_decode_splitkv(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o_part), _ptr(lse_part), B, Lq,
                                     Lkv, Hq, Hkv, d, _scale(scale, d), int(bool(causal)), _ptr(kv_lens),
                                     int(num_splits), _dtype(q), _stream(stream, q)),
           "attn_decode_splitkv")


def attn_decode_combine(o_part, lse_part, o, lse, stream=None):
    B, Hq, S, Lq, d = o_part.shape
    _check(lib().attn_decode_combine(_ptr(o_part), _ptr(lse_part), _ptr(o), _ptr(lse), B, Lq, Hq, d, S, _dtype(o),
                                     _stream(stream, o)),
           "attn_decode_combine")


def attn_decode_workspace_size(B, Lq, Hq, d, num_splits) -> int:
    return int(lib().attn_decode_workspace_size(B, Lq, Hq, d, num_splits))


def attn_device_status(reset=True):
    code, site = ctypes.c_int(0), ctypes.c_int(0)
    st = lib().attn_device_status(ctypes.byref(code), ctypes.byref(site), int(bool(reset)))
    return st, code.value, site.value


def attn_selftest_wait_timeout(site, stream=None):
    """Run the kernels' bounded-wait failure path once (about 2 s); the
    outcome is read with attn_device_status()."""
    _check(lib().attn_selftest_wait_timeout(int(site), _stream(stream)), "attn_selftest_wait_timeout")


def attn_bwd_static_scratch(q, k, v, o, lse, dout, dq, dk, dv, scale=None, causal=False, kv_lens=None,
                            stream=None):
    """Deterministic backward with the library's own static scratch: no
    workspace argument and no device allocation, for callers that cannot
    allocate device memory where they run the backward (fixed memory pools or
    another runtime's allocator, loops that must not take cudaMalloc's
    implicit synchronisation, embeddings that only pass existing tensors).
    The first call on each device looks up the scratch's device address, so
    make it before any stream capture.  Calls on one device must not overlap
    on the GPU."""
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k, v)
    _check(lib().attn_bwd_static_scratch(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                         _ptr(dk), _ptr(dv), B, Lq, Lkv, Hq, Hkv, d, _scale(scale, d),
                                         int(bool(causal)), _ptr(kv_lens), _dtype(q), _stream(stream, q)),
           "attn_bwd_static_scratch")


def attn_timing_enable(on=True):
    _check(lib().attn_timing_enable(int(bool(on))), "attn_timing_enable")


def attn_timing_query(kernel: str):
    """(total milliseconds, launches) recorded for one kernel name."""
    ms, n = ctypes.c_double(0.0), ctypes.c_int(0)
    _check(lib().attn_timing_query(kernel.encode(), ctypes.byref(ms), ctypes.byref(n)), "attn_timing_query")
    return ms.value, n.value


# ---- conveniences that allocate outputs with torch ------------------------------

def _mask_window(causal, window):
    if window is not None and causal:
        raise ValueError("pass either causal or window (causal is window (-1, 0))")
    return window if window is not None else ((-1, 0) if causal else (-1, -1))


def _segment_info_of(segments, stream):
    if len(segments) > 2:
        return segments[2]
    return segment_info(segments[0], segments[1], stream)


def forward(q, k, v, scale=None, causal=False, kv_lens=None, stream=None, window=None, segments=None,
            num_splits=1):
    """(o, lse) for q [B,Lq,Hq,d], k/v [B,Lkv,Hkv,d] on the GPU.  window =
    (left, right) selects the local-window mask (causal must then be False);
    segments = (q_segment [B,Lq], kv_segment [B,Lkv]) int32 adds a segment mask;
    a third element, the segment_info() of those ids, saves recomputing it
    (None there: no tile skipping, ids compared on every tile).  num_splits
    other than 1 splits each query tile pair's key range over up to that many
    programs (0: the library's choice), through a float32 workspace and a
    log-sum-exp combine (not with segments)."""
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k, v)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)  # (new_empty costs twice as much)
    if num_splits != 1:
        if segments is not None:
            raise ValueError("num_splits applies to the causal, window and KV-length masks, not to segments")
        S = num_splits if num_splits > 0 else attn_fwd_num_splits(B, Lq, Lkv, Hq, d, kv_lens is not None, q.dtype)
        nbytes = attn_fwd_split_workspace_size(B, Lq, Hq, d, S)
        ws = torch.empty(nbytes, device=q.device, dtype=torch.uint8) if nbytes > 0 else None
        attn_fwd_split(q, k, v, o, lse, ws, S, _mask_window(causal, window), scale, kv_lens, stream)
        return o, lse
    if segments is not None:
        attn_fwd_segments(q, k, v, o, lse, segments[0], segments[1], _mask_window(causal, window), scale, kv_lens,
                          stream, _segment_info_of(segments, stream))
    elif window is not None:
        if causal:
            raise ValueError("pass either causal or window (causal is window (-1, 0))")
        attn_fwd_window(q, k, v, o, lse, window, scale, kv_lens, stream)
    else:
        _attn_fwd((B, Lq, Lkv, Hq, Hkv, d), q, k, v, o, lse, scale, causal, kv_lens, stream)
    return o, lse


def backward(q, k, v, o, lse, dout, scale=None, causal=False, kv_lens=None, deterministic=True, stream=None,
             window=None, segments=None):
    """(dq, dk, dv) given the forward's o and lse (same mask arguments as
    forward).  deterministic: True (two-pass), False (single pass, atomic dQ)
    or 2 (single pass, dQ added in key-tile order; reproducible)."""
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k, v)
    nbytes = attn_bwd_workspace_size(B, Lq, Hq, d, deterministic, q.dtype)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if segments is not None:
        attn_bwd_segments(q, k, v, o, lse, dout, dq, dk, dv, ws, segments[0], segments[1],
                          _mask_window(causal, window), scale, kv_lens, deterministic, stream,
                          _segment_info_of(segments, stream))
    elif window is not None:
        if causal:
            raise ValueError("pass either causal or window (causal is window (-1, 0))")
        attn_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, ws, window, scale, kv_lens, deterministic, stream)
    else:
        _attn_bwd((B, Lq, Lkv, Hq, Hkv, d), q, k, v, o, lse, dout, dq, dk, dv, ws, scale, causal, kv_lens,
                  deterministic, stream)
    return dq, dk, dv


def decode(q, k_cache, v_cache, scale=None, causal=False, kv_lens=None, num_splits=0, stream=None,
           return_partials=False):
    """Split-KV decode + log-sum-exp combine: (o, lse) [and the partials]."""
    B, Lq, Lkv, Hq, Hkv, d = _dims(q, k_cache, v_cache)
    S = num_splits if num_splits > 0 else attn_decode_num_splits(B, Lq, Lkv, Hq, Hkv, d)
    o_part = torch.empty(B, Hq, S, Lq, d, device=q.device, dtype=torch.float32)
    lse_part = torch.empty(B, Hq, S, Lq, device=q.device, dtype=torch.float32)
    attn_decode_splitkv(q, k_cache, v_cache, o_part, lse_part, S, scale, causal, kv_lens, stream)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    attn_decode_combine(o_part, lse_part, o, lse, stream)
    if return_partials:
        return o, lse, o_part, lse_part
    return o, lse
