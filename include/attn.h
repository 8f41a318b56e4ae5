/*
 * attn.h -- C ABI of a GB300 (sm_103a) exact scaled-dot-product attention
 * library: forward, backward (dQ, dK, dV) and split-KV decode.
 *
 * What it computes (probjax benchmark pages, "Attention performance"):
 *   O = softmax(scale * Q K^T) V over the valid keys of each query row, and
 *   the per-row natural log-sum-exp LSE that the backward recomputes from
 *   (sections "Attention performance" and "Memory": the kernels keep the
 *   output and the log-sum-exp as residuals).
 *
 * Tensor layout (section "Attention performance": inputs are
 * [batch, seq, heads, head_dim]):
 *   q, o, dout, dq   [B, Lq,  Hq,  d]   dense, d innermost
 *   k, v, dk, dv     [B, Lkv, Hkv, d]   dense, d innermost
 *   lse, delta       [B, Hq, Lq]        float32
 * GQA ("Grouped-query attention and decoding"): Hq = G * Hkv and query head h
 * reads KV head h / G directly; K and V are never repeated.
 *
 * Valid keys.  With kvl[b] = kv_lens[b] clamped into [0, Lkv] (Lkv when
 * kv_lens is NULL), key j is valid for query row i of batch b iff
 *   j < kvl[b]                          (KVLenMask, "H100 (Hopper)",
 *                                         section "Mosaic GPU")
 *   and, when causal, j <= i + kvl[b] - Lq   (causal aligned to the bottom
 *                                         right; equal-length causal j <= i)
 * A row without a valid key has O = 0, LSE = -inf and dQ = 0; keys at or past
 * kvl[b] get dK = dV = 0 (same section).
 *
 * Conventions for every call:
 *   - The caller allocates every buffer and owns the stream; the library never
 *     allocates, frees or synchronises.  Calls are asynchronous on `stream`
 *     (NULL = the legacy default stream).  Pointers named here are device
 *     pointers unless stated otherwise.
 *   - Stream order holds: every output of a call is complete for the next
 *     operation queued on its stream, and the call reads its inputs only
 *     after the operations queued before it have completed.  Internally the
 *     kernels are launched with programmatic stream serialization, so that
 *     each one starts while the kernel before it drains and waits on the GPU
 *     before it reads what that kernel writes; setting the environment
 *     variable EXACT_ATTN_NO_PDL=1 before the first call turns this off.
 *   - Every tensor pointer must be 16-byte aligned and, for bf16, every row
 *     stride (Hq*d, Hkv*d elements) is then a multiple of 16 bytes.
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns an error code and launches nothing.  Values that live
 *     on the device (kv_lens) cannot be checked there and are clamped into
 *     [0, Lkv] by the kernels.
 *   - dtype ATTN_BF16 / ATTN_FP16: q/k/v/o/dout/dq/dk/dv are bf16 / fp16;
 *     ATTN_FP32: all float32.  lse, delta, partials and workspaces are always
 *     float32.
 *   - head_dim d must be 32, 64, 128 or 256 (32 runs through the 64-wide
 *     kernels with zero-filled columns, as the pages' kernels pad it; 256 has
 *     its own 16-bit kernels and is ATTN_ERR_UNSUPPORTED with ATTN_FP32).
 *     At d = 256 the backward is deterministic for either value of
 *     `deterministic`.
 *   - Calls are thread-safe: no mutable global state is shared between calls
 *     (tensor-map descriptors are passed by value; the small cache that saves
 *     re-encoding them is per host thread).
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without pulling in CUDA headers. */
typedef struct CUstream_st* attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* bad size, NULL or misaligned pointer, Hq % Hkv != 0 */
  ATTN_ERR_UNSUPPORTED = 2, /* valid call this build cannot compute exactly (e.g. d) */
  ATTN_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the size query says */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call or kernel launch failed */
  ATTN_ERR_DEVICE = 5       /* a kernel reported a device-side fault (see attn_device_status) */
} attn_status;

/* Element type of q, k, v, o, dout, dq, dk, dv (lse, delta and the decode
 * partials are always float32).  bf16 and fp16 run on the tensor cores with
 * fp32 accumulation.  fp32 at head_dim 64 and 128 (forward, and the two-pass
 * backward) also runs on the tensor cores: every float32 operand is split
 * into bf16 parts (two, or three exact ones where a difference cancels) and
 * each product taken as the few bf16 MMAs that keep its error near float32
 * rounding (within 1e-4 of the exact result); softmax and statistics stay in
 * float32.  Head_dim 32, segment ids, the atomic backward and the decode run
 * fp32 on the CUDA cores. */
typedef enum { ATTN_BF16 = 0, ATTN_FP32 = 1, ATTN_FP16 = 2 } attn_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* attn_status_string(attn_status s);

/* Detail message of the last error returned on the calling thread ("" if none). */
const char* attn_last_error(void);

/*
 * Forward.  Writes o [B,Lq,Hq,d] (dtype) and lse [B,Hq,Lq] (float32, natural
 * log, -inf on rows without a valid key).  scale is the softmax scale (pass
 * 1/sqrt(d) for the standard one; it must be finite and > 0).  kv_lens is
 * a device int32 [B] or NULL.  causal is 0 or 1.
 * Fused, memory-linear tiled kernel with online softmax ("Attention
 * performance", section "When to use which": memory grows linearly in T).
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Lq, int Lkv,
                     int Hq, int Hkv, int d, float scale, int causal, const int32_t* kv_lens, attn_dtype dtype,
                     attn_stream_t stream);

/*
 * Backward preprocess: delta[b,h,i] = sum_c dout[b,i,h,c] * o[b,i,h,c] in
 * float32 ([B,Hq,Lq]).  attn_bwd runs it itself; it is exported so the step
 * can be checked and timed on its own.
 */
attn_status attn_bwd_preprocess(const void* o, const void* dout, float* delta, int B, int Lq, int Hq, int d,
                                attn_dtype dtype, attn_stream_t stream);

/*
 * Bytes of device workspace attn_bwd needs ("Attention performance", section
 * "When to use which", backward pass: one pass with atomic dQ, or the split
 * into a dK/dV pass and a dQ pass).  `deterministic` picks the variant:
 *   1: the two-pass backward (a dK/dV kernel per KV block, then a separate
 *      dQ kernel; bitwise reproducible), workspace = delta and lse*log2(e)
 *      per padded query row;
 *   0: the single-pass backward with dQ accumulated by float32 atomic adds
 *      (summation order not reproducible), workspace = the above + a float32
 *      dQ buffer [B,Lq,Hq,d];
 *   2: the single-pass backward with each query tile's dQ parts added in
 *      key-tile order (a turn counter per query tile; bitwise reproducible),
 *      workspace = the above + one int32 per (batch, query head, 128-row
 *      query tile) + 4 bytes.  16-bit types at head_dim <= 128 only
 *      (ATTN_ERR_UNSUPPORTED otherwise).
 */
size_t attn_bwd_workspace_size(int B, int Lq, int Hq, int d, int deterministic, attn_dtype dtype);

/*
 * Backward: given the forward's o and lse and the output gradient dout,
 * writes dq [B,Lq,Hq,d], dk and dv [B,Lkv,Hkv,d] (dtype).  For GQA, dk/dv sum
 * over the G query heads of each KV head.  workspace must be 256-byte aligned
 * and at least attn_bwd_workspace_size(...) bytes; its contents on entry do
 * not matter.
 */
attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, int B, int Lq, int Lkv, int Hq, int Hkv, int d, float scale,
                     int causal, const int32_t* kv_lens, attn_dtype dtype, int deterministic, void* workspace,
                     size_t workspace_bytes, attn_stream_t stream);

/*
 * Local-window (sliding) attention, forward and backward ("Attention
 * performance", section "Short sequences and the default dispatch": window
 * masks are among the position-only masks the fused kernel computes).  Same
 * arguments, outputs, workspace and errors as attn_fwd / attn_bwd, with the
 * causal flag replaced by a window around each row's diagonal: key j is valid
 * for query row i of batch b iff j < kvl[b] and
 *     i + kvl[b] - Lq - window_left  <=  j  <=  i + kvl[b] - Lq + window_right
 * (kvl[b] = Lkv without kv_lens; the diagonal is aligned to the bottom right,
 * as for causal).  A negative bound is unbounded on that side, so (-1, 0) is
 * causal and (-1, -1) is no mask.  Key tiles outside every row's window are
 * neither loaded nor computed; rows whose window holds no valid key get o = 0,
 * lse = -inf and dq = 0.
 */
attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Lq, int Lkv,
                            int Hq, int Hkv, int d, float scale, int window_left, int window_right,
                            const int32_t* kv_lens, attn_dtype dtype, attn_stream_t stream);
attn_status attn_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int B, int Lq, int Lkv, int Hq, int Hkv,
                            int d, float scale, int window_left, int window_right, const int32_t* kv_lens,
                            attn_dtype dtype, int deterministic, void* workspace, size_t workspace_bytes,
                            attn_stream_t stream);

/*
 * Segment (document) masks on top of the window masks above ("H100 (Hopper)",
 * section "Mosaic GPU", lists segments beside KV lengths, causal and local
 * windows): key j is valid for query row i of batch b only if, in addition,
 * q_segment[b][i] == kv_segment[b][j].  q_segment is a device int32 [B, Lq],
 * kv_segment a device int32 [B, Lkv], both 16-byte aligned and required; ids
 * are arbitrary int32 values and need not be sorted.  Rows with no valid key
 * get o = 0, lse = -inf and dq = 0.  Otherwise as attn_fwd_window /
 * attn_bwd_window.
 *
 * segment_info (optional, device, 16-byte aligned) is the block summary that
 * attn_segment_info writes for the same q_segment, kv_segment, B, Lq and Lkv.
 * With it the 16-bit kernels drop the tiles whose query and key blocks share no
 * id and skip the per-element id compare on tiles where both blocks hold one
 * and the same id (packed documents run at the speed of their own causal
 * blocks).  The library does not check that it matches the ids: after the ids
 * change, recompute it.  NULL: every tile inside the position masks is
 * computed and its ids compared per element (same results, slower).
 */
attn_status attn_fwd_segments(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Lq,
                              int Lkv, int Hq, int Hkv, int d, float scale, int window_left, int window_right,
                              const int32_t* q_segment, const int32_t* kv_segment, const void* segment_info,
                              const int32_t* kv_lens, attn_dtype dtype, attn_stream_t stream);
attn_status attn_bwd_segments(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int Lq, int Lkv, int Hq,
                              int Hkv, int d, float scale, int window_left, int window_right,
                              const int32_t* q_segment, const int32_t* kv_segment, const void* segment_info,
                              const int32_t* kv_lens, attn_dtype dtype, int deterministic, void* workspace,
                              size_t workspace_bytes, attn_stream_t stream);

/*
 * Block summary of segment ids for attn_fwd_segments / attn_bwd_segments.
 * For every 128-position block of q_segment ([B, Lq]) and of kv_segment
 * ([B, Lkv]) it records the smallest and largest id and the range of the other
 * side's positions whose blocks' id ranges meet it: B*ceil(Lq/128) query
 * records then B*ceil(Lkv/128) key records of four int32 each, which is
 * attn_segment_info_size(B, Lq, Lkv) bytes (0 for non-positive sizes).  info
 * is caller-owned device memory, 16-byte aligned; it is written by two small
 * kernels on `stream`.  Positions past a batch element's KV length still enter
 * the summary (they only widen it).  Returns ATTN_ERR_WORKSPACE when
 * info_bytes is too small.
 */
size_t attn_segment_info_size(int B, int Lq, int Lkv);
attn_status attn_segment_info(const int32_t* q_segment, const int32_t* kv_segment, int B, int Lq, int Lkv,
                              void* info, size_t info_bytes, attn_stream_t stream);

/*
 * Forward with each query tile's key range split across programs: the
 * split-KV scheme of the decode ("Attention performance", section
 * "Grouped-query attention and decoding") applied to the whole forward, for
 * KV-length masks that put most keys in a few batch elements and for grids
 * too small to fill the GPU.  Arguments, outputs, masks and errors as
 * attn_fwd_window, plus:
 *   num_splits  the most pieces one pair of 128-row query tiles cuts its key
 *               range into; 0 picks attn_fwd_num_splits(...).  A pair whose
 *               masks and KV length leave n KV tiles of 128 keys cuts them into
 *               min(num_splits, ceil(n / C)) near-equal pieces,
 *               C = ceil(ceil(Lkv / 128) / num_splits), so short ranges stay
 *               whole and a batch element's pieces follow its own length.
 *   workspace   device memory, 256-byte aligned, at least
 *               attn_fwd_split_workspace_size(B, Lq, Hq, d, num_splits) bytes;
 *               its contents on entry do not matter.  It receives each piece's
 *               float32 output (normalised within the piece) and log-sum-exp,
 *               and one ticket counter per pair (zeroed by the call with a
 *               memset on `stream`).  The piece of a pair that finishes last
 *               (by an atomic ticket; no program waits on another) merges the
 *               pieces by their log-sum-exps, as attn_decode_combine does, and
 *               writes o and lse; a pair left whole writes them directly.
 * attn_fwd_num_splits is the library's choice: with kv_lens (has_kv_lens != 0)
 * it assumes every key may sit in one batch element, so only that element's
 * ceil(Lq/256)*Hq tile pairs are busy (all B elements' pairs otherwise); it
 * cuts only while the busy pairs are fewer than the SMs, weighs the rounds
 * of programs saved against a fixed cost per piece, and keeps each piece at 8
 * KV tiles or more and the count at most 8 and at most Lkv / 4096.
 * num_splits = 1, head_dim 256 and float32 run attn_fwd_window as is and use
 * no workspace (workspace may then be NULL).  Results equal attn_fwd_window's
 * up to rounding (pieces are normalised and combined in float32), and are the
 * same on every run: the merge adds the pieces in a fixed order, whichever
 * piece performs it.
 */
int attn_fwd_num_splits(int B, int Lq, int Lkv, int Hq, int d, int has_kv_lens, attn_dtype dtype);
size_t attn_fwd_split_workspace_size(int B, int Lq, int Hq, int d, int num_splits);
attn_status attn_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Lq, int Lkv,
                           int Hq, int Hkv, int d, float scale, int window_left, int window_right,
                           const int32_t* kv_lens, int num_splits, void* workspace, size_t workspace_bytes,
                           attn_dtype dtype, attn_stream_t stream);

/*
 * Split-KV decode for few queries over a long KV cache ("Attention
 * performance", section "Grouped-query attention and decoding"): the keys are
 * split across programs, the G query heads of a KV head (times the Lq rows)
 * are packed into one tile, and the partial results are combined by their
 * log-sum-exp.
 *
 * Partition: with C = 128 * ceil(ceil(Lkv / num_splits) / 128), split s of
 * batch b covers keys [s*C, min((s+1)*C, kvl[b])) and is empty when
 * s*C >= kvl[b].  Supported for Lq * (Hq / Hkv) <= 128.
 *
 * attn_decode_splitkv writes, per split, the attention over the split's valid
 * keys, normalised within the split:
 *   o_part   float32 [B, Hq, num_splits, Lq, d]
 *   lse_part float32 [B, Hq, num_splits, Lq]   (-inf, with o_part = 0, where
 *                                               the row has no valid key in it)
 * num_splits = 0 picks attn_decode_num_splits(...).  The same num_splits must
 * be passed to attn_decode_combine.
 */
int attn_decode_num_splits(int B, int Lq, int Lkv, int Hq, int Hkv, int d);
attn_status attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, float* o_part,
                                float* lse_part, int B, int Lq, int Lkv, int Hq, int Hkv, int d, float scale,
                                int causal, const int32_t* kv_lens, int num_splits, attn_dtype dtype,
                                attn_stream_t stream);

/*
 * Log-sum-exp combine: lse = log sum_s exp(lse_part_s) and
 * o = sum_s exp(lse_part_s - lse) o_part_s, cast to dtype; rows whose splits
 * are all empty get o = 0 and lse = -inf.  o [B,Lq,Hq,d], lse [B,Hq,Lq].
 */
attn_status attn_decode_combine(const float* o_part, const float* lse_part, void* o, float* lse, int B, int Lq,
                                int Hq, int d, int num_splits, attn_dtype dtype, attn_stream_t stream);

/* Bytes of o_part plus lse_part for a decode call (num_splits > 0). */
size_t attn_decode_workspace_size(int B, int Lq, int Hq, int d, int num_splits);

/*
 * Device-side status of the current device: kernels never trap; a pipeline
 * wait that runs out of time (2 s) records code 1 and a site here and the
 * kernel ends early; a kernel that finds its shared-memory window misaligned
 * records code 2 and does nothing.  Synchronises the device.  Writes code/site (host
 * pointers, nullable) and clears the status when reset != 0.  Returns
 * ATTN_ERR_DEVICE when a code was set, ATTN_OK otherwise.
 */
attn_status attn_device_status(int* code, int* site, int reset);

/*
 * Diagnostic: runs the bounded-wait failure path of the kernels on purpose.
 * One CTA waits for an mbarrier phase that nothing completes; after the wait
 * limit (2 s of the GPU's global timer) it records code 1 at `site` in the
 * device status word, stops its other waiting warp, frees its TMEM and exits.
 * The device stays usable.  Asynchronous on `stream`; read the outcome with
 * attn_device_status.  Returns ATTN_ERR_CUDA if the launch fails.
 */
attn_status attn_selftest_wait_timeout(int site, attn_stream_t stream);

/*
 * Per-kernel timing for benchmarks (the pages time each case between device
 * synchronisations, "GPU and CPU performance", section "Methodology"; this is
 * the library-side counterpart).  attn_timing_enable(1) clears old records and
 * brackets every kernel launched from then on with CUDA events on its stream
 * (events are created by the library and reused; no device memory is
 * allocated).  attn_timing_enable(0) stops recording.  attn_timing_query waits
 * for the recorded launches of one kernel ("fwd", "bwd_preprocess",
 * "bwd_dkdv", "bwd_dkdv_atomic", "bwd_dkdv_ordered", "bwd_dq", "dq_convert",
 * "decode", "combine", the float32 tensor-core kernels "fwd_split_f32",
 * "bwd_dkdv_split_f32", "bwd_dq_split_f32", or the float32 CUDA-core kernels
 * "fwd_f32", "decode_f32", "bwd_dkdv_f32", "bwd_dq_f32", "dq_convert_f32")
 * and returns their summed milliseconds and
 * count (host pointers).  Process-wide; meant for single-threaded benchmarks.
 */
attn_status attn_timing_enable(int on);
attn_status attn_timing_query(const char* kernel, double* total_ms, int* launches);

/*
 * Deterministic backward that needs no workspace from the caller (the paper
 * has no counterpart; this is a convenience of this library).  Same arguments
 * and results as attn_bwd with deterministic = 1, minus the workspace.
 *
 * For callers that cannot allocate device memory where they run the backward:
 * hosts whose device memory belongs to a fixed pool or another runtime's
 * allocator, latency-critical loops that must not take cudaMalloc's implicit
 * device synchronisation, or embeddings that only hand over existing tensors.
 * The scratch (two floats per padded query row) lives in a 4 MiB device array
 * inside the library, held by every GPU that loads it until the process
 * exits.  Limit: B * Hq * roundup(Lq, 128) <= 524288 (e.g. B4 H8
 * Lq16384); larger problems return ATTN_ERR_WORKSPACE with a message.
 *
 * The first call on each device looks up the array's device address with that
 * device current; make that first call before any stream capture.  Allocates
 * nothing (no cudaMalloc/cudaFree, no library allocator).  All calls on a
 * device share the one array: calls that overlap on the GPU (different
 * streams, or host threads racing) corrupt each other's scratch -- serialise
 * them.  No scratch content needs clearing between calls.
 */
attn_status attn_bwd_static_scratch(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk, void* dv, int B, int Lq, int Lkv, int Hq,
                                    int Hkv, int d, float scale, int causal, const int32_t* kv_lens,
                                    attn_dtype dtype, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
