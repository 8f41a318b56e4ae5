"""Plain fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check of ``__graft_entry__`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code with the CUDA library (no headers, helpers, tables or constants).

What it computes is the textbook definition of exact softmax attention, written
out densely (the full row of scores is materialised; there is no online softmax,
no tiling of the key axis and no exp2 rewriting), so a reader can check it by eye
against the pages:

* layout ``[batch, seq, heads, head_dim]`` for q, k, v, o and every gradient --
  probjax "Attention performance", section "Attention performance" (inputs are
  [batch, seq, heads, head_dim]);
* the residuals kept for the backward are the output and the log-sum-exp, and
  the backward recomputes the probabilities from the log-sum-exp -- same page,
  sections "Memory" and "CPU";
* per-batch KV lengths (KVLenMask): keys at or past a batch element's length
  are invalid, rows without a valid key return zeros, dK/dV of padded keys are
  zero -- probjax "H100 (Hopper)", section "Mosaic GPU";
* equal-length causal masking and local-window masks -- "Attention
  performance", section "Short sequences and the default dispatch"
  (position-only masks: causal, length or window);
* GQA: query head h reads KV head h // G, K/V are never repeated -- same page,
  section "Grouped-query attention and decoding";
* split-KV decoding combines per-split partial results by their log-sum-exp --
  same section.

Readings where the pages are silent (each listed in the design notes):

* causal with Lq != Lkv (and with KV lengths) is aligned to the bottom right of
  the batch element's valid keys: key j is valid for query row i of batch b iff
  ``j < kvl[b]`` and ``j <= i + kvl[b] - Lq``; for Lq == Lkv with no KV lengths
  this is the usual ``j <= i``;
* the log-sum-exp is the natural logarithm, ``lse[b, h, i]``, and ``-inf`` on a
  row with no valid key (whose output is 0);
* segment (document) masks compare per-token ids: key j is valid for row i
  of batch b only if ``q_segment[b, i] == kv_segment[b, j]`` (on top of the
  position masks);
* a local window ``(left, right)`` is taken around the same bottom-right
  aligned diagonal: key j is valid for row i iff
  ``i + kvl[b] - Lq - left <= j <= i + kvl[b] - Lq + right`` (and ``j < kvl[b]``);
  a negative or missing bound is unbounded, so ``(-1, 0)`` is causal and
  ``(-1, -1)`` is no mask; combined with ``causal=True`` both conditions hold;
* KV lengths outside [0, Lkv] are clamped into it;
* the default scale is 1/sqrt(head_dim).

All arithmetic is float64.  Inputs of any dtype are upcast exactly (bf16 and
fp32 values are exactly representable in fp64), so the oracle sees the same
rounded tensors the GPU sees.

Parity status: every public function here is pinned by tests in
``tests/test_oracle.py`` (finite differences, closed forms, invariants, a
library cross-check and a brute-force loop); none is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Exact upcast to float64 (accepts numpy arrays and CPU torch tensors)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # local: only needed when a tensor is passed

        x = x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def effective_kv_lens(B: int, Lkv: int, kv_lens) -> np.ndarray:
    """Per-batch KV length ``kvl[b]``: Lkv when no lengths are given, else the
    given length clamped into [0, Lkv] (a reading: the pages never pass an
    out-of-range length)."""
    if kv_lens is None:
        return np.full(B, Lkv, dtype=np.int64)
    kl = np.asarray(kv_lens if not hasattr(kv_lens, "numpy") else kv_lens.cpu().numpy())
    kl = kl.astype(np.int64).reshape(-1)
    if kl.shape[0] != B:
        raise ValueError("kv_lens must have one entry per batch element")
    return np.clip(kl, 0, Lkv)


def valid_keys(rows: np.ndarray, Lq: int, Lkv: int, kvl_b: int, causal: bool, window=None, q_seg_b=None,
               kv_seg_b=None) -> np.ndarray:
    """Boolean matrix ``[len(rows), Lkv]``: is key j valid for query row i.

    KVLenMask: ``j < kvl_b``.  Causal (bottom-right reading for Lq != Lkv):
    ``j <= i + kvl_b - Lq``.  Local window ``(left, right)`` around the same
    diagonal: ``j >= i + kvl_b - Lq - left`` when left >= 0 and
    ``j <= i + kvl_b - Lq + right`` when right >= 0.
    """
    j = np.arange(Lkv)[None, :]
    i = np.asarray(rows, dtype=np.int64)[:, None]
    diag = i + kvl_b - Lq
    ok = j < kvl_b
    if causal:
        ok = ok & (j <= diag)
    if window is not None:
        left, right = window
        if left is not None and left >= 0:
            ok = ok & (j >= diag - left)
        if right is not None and right >= 0:
            ok = ok & (j <= diag + right)
    if q_seg_b is not None:
        qs = np.asarray(q_seg_b)[np.asarray(rows, dtype=np.int64)][:, None]
        ok = ok & (qs == np.asarray(kv_seg_b)[None, :])
    return np.broadcast_to(ok, (len(rows), Lkv)).copy()


def _segments_of(segments, b):
    """(q_segment[b], kv_segment[b]) as int64 arrays, or (None, None)."""
    if segments is None:
        return None, None
    qs, ks = segments
    qs = np.asarray(qs if not hasattr(qs, "numpy") else qs.cpu().numpy()).astype(np.int64)
    ks = np.asarray(ks if not hasattr(ks, "numpy") else ks.cpu().numpy()).astype(np.int64)
    return qs[b], ks[b]


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [batch, seq, heads, head_dim]")
    B, Lq, Hq, d = q.shape
    Bk, Lkv, Hkv, dk = k.shape
    if v.shape != k.shape or Bk != B or dk != d:
        raise ValueError("k and v must be [B, Lkv, Hkv, d] matching q")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv (GQA)")
    return B, Lq, Lkv, Hq, Hkv, d


def _head_probs(qh, kh, scale, mask):
    """Softmax probabilities of one (batch, head) slice, dense.

    ``qh [n, d]``, ``kh [Lkv, d]``, ``mask [n, Lkv]`` -> ``P [n, Lkv]`` and the
    natural-log log-sum-exp ``[n]`` (``-inf`` and a zero row of P where the row
    has no valid key).
    """
    s = scale * (qh @ kh.T)
    s = np.where(mask, s, NEG_INF)
    has = mask.any(axis=1)
    m = np.where(has, np.max(np.where(mask, s, -np.finfo(np.float64).max), axis=1), 0.0)
    e = np.where(mask, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    p = np.where(has[:, None], e / np.where(has, l, 1.0)[:, None], 0.0)
    lse = np.where(has, m + np.log(np.where(has, l, 1.0)), NEG_INF)
    return p, lse


def forward(q, k, v, scale=None, causal=False, kv_lens=None, rows=None, heads=None, window=None, segments=None,
            row_block: int = 1024):
    """Exact attention forward: ``O = softmax(scale * Q K^T) V`` and ``LSE``.

    Returns ``(o [B, len(rows), Hq, d], lse [B, Hq, len(rows)])`` in float64.
    ``rows`` (absolute query-row indices, default all) and ``heads`` (query
    heads, default all; other heads are left as NaN) let a test check sampled
    outputs of a large problem one by one.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Lq, Lkv, Hq, Hkv, d = _check_shapes(q, k, v)
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kvl = effective_kv_lens(B, Lkv, kv_lens)
    rows = np.arange(Lq) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = range(Hq) if heads is None else heads
    o = np.full((B, len(rows), Hq, d), np.nan)
    lse = np.full((B, Hq, len(rows)), np.nan)
    for b in range(B):
        for hq in heads:
            hk = hq // G
            for r0 in range(0, len(rows), row_block):
                rr = rows[r0:r0 + row_block]
                mask = valid_keys(rr, Lq, Lkv, int(kvl[b]), causal, window, *_segments_of(segments, b))
                p, l_ = _head_probs(q[b, rr, hq, :], k[b, :, hk, :], scale, mask)
                o[b, r0:r0 + len(rr), hq, :] = p @ v[b, :, hk, :]
                lse[b, hq, r0:r0 + len(rr)] = l_
    return o, lse


def probabilities(q, k, scale=None, causal=False, kv_lens=None, window=None, segments=None):
    """The full probability tensor ``P [B, Hq, Lq, Lkv]`` (tiny inputs only)."""
    q, k = _f64(q), _f64(k)
    B, Lq, Hq, d = q.shape
    Lkv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kvl = effective_kv_lens(B, Lkv, kv_lens)
    out = np.zeros((B, Hq, Lq, Lkv))
    rows = np.arange(Lq)
    for b in range(B):
        for hq in range(Hq):
            mask = valid_keys(rows, Lq, Lkv, int(kvl[b]), causal, window, *_segments_of(segments, b))
            out[b, hq], _ = _head_probs(q[b, :, hq, :], k[b, :, hq // G, :], scale, mask)
    return out


def backward(q, k, v, do, scale=None, causal=False, kv_lens=None, kv_heads=None, window=None, segments=None,
             row_block: int = 1024, rows=None):
    """Analytic gradient of ``sum(O * dO)`` with respect to q, k and v.

    With ``P`` the probabilities (recomputed, as the pages' kernels do from the
    residual log-sum-exp):

    * ``dV_j = sum over the G heads of the group and over rows i of P_ij dO_i``
    * ``dP_ij = <dO_i, v_j>``, ``D_i = sum_j P_ij dP_ij``, ``dS = P * (dP - D)``
    * ``dQ_i = scale * sum_j dS_ij k_j``, ``dK_j = scale * sum_{g,i} dS_ij q_i``

    Keys past a batch element's KV length get dK = dV = 0; rows without a valid
    key get dQ = 0.  ``kv_heads`` restricts the work to some KV heads (with all
    their query heads); other entries are left as NaN.  ``rows`` restricts the
    sums to some query rows: dQ of those rows, and dK / dV summed over those
    rows only (a bounded sample of the work; the sums over a partition of the
    rows add up to the full gradient).

    Returns ``(dq, dk, dv)`` in float64 with the shapes of q, k, v.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Lq, Lkv, Hq, Hkv, d = _check_shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError("do must have the shape of q")
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kvl = effective_kv_lens(B, Lkv, kv_lens)
    kv_heads = range(Hkv) if kv_heads is None else kv_heads
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    all_rows = np.arange(Lq) if rows is None else np.asarray(rows, dtype=np.int64)
    for b in range(B):
        for hk in kv_heads:
            kh, vh = k[b, :, hk, :], v[b, :, hk, :]
            acc_dk = np.zeros((Lkv, d))
            acc_dv = np.zeros((Lkv, d))
            for hq in range(hk * G, (hk + 1) * G):
                for r0 in range(0, len(all_rows), row_block):
                    rr = all_rows[r0:r0 + row_block]
                    mask = valid_keys(rr, Lq, Lkv, int(kvl[b]), causal, window, *_segments_of(segments, b))
                    p, _ = _head_probs(q[b, rr, hq, :], kh, scale, mask)
                    doh = do[b, rr, hq, :]
                    acc_dv += p.T @ doh
                    dp = doh @ vh.T
                    D = np.sum(p * dp, axis=1)
                    ds = p * (dp - D[:, None])
                    dq[b, rr, hq, :] = scale * (ds @ kh)
                    acc_dk += scale * (ds.T @ q[b, rr, hq, :])
            dk[b, :, hk, :] = acc_dk
            dv[b, :, hk, :] = acc_dv
    return dq, dk, dv


def backward_preprocess(o, do):
    """``D[b, h, i] = sum_c dO[b, i, h, c] * O[b, i, h, c]`` (float64).

    This equals ``sum_j P_ij dP_ij`` of the backward above because
    ``O_i = sum_j P_ij v_j``; the GPU backward computes D this way from the
    stored output.  Returns ``[B, Hq, Lq]``.
    """
    o, do = _f64(o), _f64(do)
    return np.einsum("bihc,bihc->bhi", do, o)


def split_bounds(kvl_b: int, Lkv: int, num_splits: int, tile: int = 128):
    """Key range ``[lo, hi)`` of every split of one batch element.

    The split-KV decode divides the key axis into ``num_splits`` equal chunks
    of ``C = tile * ceil(ceil(Lkv / num_splits) / tile)`` keys; split s covers
    ``[s*C, min((s+1)*C, kvl[b]))`` and is empty when ``s*C >= kvl[b]``.  This
    is the library's documented partition (the pages only say the keys are
    split across programs); it is restated here, not imported.
    """
    per = -(-Lkv // num_splits)
    C = tile * (-(-per // tile))
    out = []
    for s in range(num_splits):
        lo = s * C
        hi = min((s + 1) * C, kvl_b)
        out.append((lo, max(lo, hi)))
    return out


def splitkv_partials(q, k, v, num_splits, scale=None, causal=False, kv_lens=None, tile=128):
    """Per-split partial results of the split-KV decode.

    For every split s (key range from :func:`split_bounds`) this is the exact
    attention of each query row over the valid keys inside the split:
    ``O_s`` normalised within the split and ``LSE_s`` its natural log-sum-exp
    (``O_s = 0``, ``LSE_s = -inf`` where the row has no valid key in it).

    Returns ``(o_part [B, Hq, S, Lq, d], lse_part [B, Hq, S, Lq])`` float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Lq, Lkv, Hq, Hkv, d = _check_shapes(q, k, v)
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kvl = effective_kv_lens(B, Lkv, kv_lens)
    S = int(num_splits)
    o_part = np.zeros((B, Hq, S, Lq, d))
    lse_part = np.full((B, Hq, S, Lq), NEG_INF)
    rows = np.arange(Lq)
    for b in range(B):
        base = valid_keys(rows, Lq, Lkv, int(kvl[b]), causal)
        for s, (lo, hi) in enumerate(split_bounds(int(kvl[b]), Lkv, S, tile)):
            if hi <= lo:
                continue
            mask = base.copy()
            mask[:, :lo] = False
            mask[:, hi:] = False
            for hq in range(Hq):
                p, l_ = _head_probs(q[b, :, hq, :], k[b, :, hq // G, :], scale, mask)
                o_part[b, hq, s] = p @ v[b, :, hq // G, :]
                lse_part[b, hq, s] = l_
    return o_part, lse_part


def combine(o_part, lse_part):
    """Log-sum-exp combine of split partials.

    ``LSE = log sum_s exp(LSE_s)`` and ``O = sum_s exp(LSE_s - LSE) O_s``;
    splits with ``LSE_s = -inf`` contribute nothing, and a row whose splits are
    all empty gets ``O = 0``, ``LSE = -inf``.

    ``o_part [B, Hq, S, Lq, d]``, ``lse_part [B, Hq, S, Lq]`` ->
    ``(o [B, Lq, Hq, d], lse [B, Hq, Lq])``.
    """
    o_part, lse_part = _f64(o_part), _f64(lse_part)
    finite = np.isfinite(lse_part)
    any_f = finite.any(axis=2)
    m = np.where(any_f, np.max(np.where(finite, lse_part, -np.finfo(np.float64).max), axis=2), 0.0)
    w = np.where(finite, np.exp(np.where(finite, lse_part, 0.0) - m[:, :, None, :]), 0.0)
    tot = w.sum(axis=2)
    lse = np.where(any_f, m + np.log(np.where(any_f, tot, 1.0)), NEG_INF)
    wn = np.where(any_f[:, :, None, :], w / np.where(any_f, tot, 1.0)[:, :, None, :], 0.0)
    o = np.einsum("bhsi,bhsic->bihc", wn, o_part)
    return o, lse
