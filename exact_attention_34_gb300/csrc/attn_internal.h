// Internal interface between the C-ABI layer (attn_api.cu) and the kernel
// translation units.  Not installed; the public ABI is include/attn.h.
#pragma once

#include <atomic>
#include <cstdlib>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103_ptx.cuh"

namespace attn {

// Problem description shared by every kernel family.  All pointers are device
// pointers; sizes are validated by the ABI layer before a launch.
// Position masks.  Key j is valid for query row i of a batch element with kvl
// valid keys iff lo <= j < hi, where with the row's diagonal position
// diag = i + kvl - Lq:  lo = max(0, diag - wl),  hi = min(kvl, diag + wr + 1).
// kWinInf marks an unbounded side: no mask is (kWinInf, kWinInf), causal is
// (kWinInf, 0), a local window (left, right) bounds both sides.
constexpr int kWinInf = 1 << 30;

struct Span {
  int lo, hi;  // [lo, hi); empty when hi <= lo
};

// Valid keys of query row i.
__host__ __device__ __forceinline__ Span key_span(int i, int Lq, int kvl, int wl, int wr) {
  const int diag = i + kvl - Lq;
  Span s;
  s.lo = wl >= kWinInf ? 0 : max(0, diag - wl);
  s.hi = wr >= kWinInf ? kvl : min(kvl, diag + wr + 1);
  return s;
}

// Query rows that see key j (j < kvl): i >= j - (kvl - Lq) - wr and
// i <= j - (kvl - Lq) + wl.
__host__ __device__ __forceinline__ Span query_span(int j, int Lq, int kvl, int wl, int wr) {
  const int off = kvl - Lq;
  Span s;
  s.lo = wr >= kWinInf ? 0 : max(0, j - off - wr);
  s.hi = wl >= kWinInf ? Lq : min(Lq, j - off + wl + 1);
  return s;
}

// Element formats of the tensors a call reads and writes.
enum Elem : int { kElemF32 = 0, kElemBF16 = 1, kElemF16 = 2 };

struct Problem {
  int B, Lq, Lkv, Hq, Hkv, d, G;
  int f16;                 // 16-bit kernels: 1 = fp16 tensors, 0 = bf16
  int causal;              // launch-order hint: later query rows see more keys
  int wl, wr;              // position mask (see key_span)
  float scale;             // softmax scale (> 0)
  const int32_t* kv_lens;  // [B] or nullptr
  const int32_t* q_seg;    // [B, Lq] segment ids or nullptr (then kv_seg is nullptr too)
  const int32_t* kv_seg;   // [B, Lkv]
  const int4* seg_qblk;    // [B, ceil(Lq/128)] SegBlock records or nullptr (no tile skipping)
  const int4* seg_kblk;    // [B, ceil(Lkv/128)]
};

// Segment summary of one 128-position block of a sequence, as an int4:
//   x, y  the smallest and largest segment id in the block;
//   z, w  the positions [z, w) of the other side (keys for a query block,
//         queries for a key block) that may share an id with the block: the
//         span from the first to the last other-side block whose id range
//         meets [x, y] (empty when z == w).
// Every pair (query, key) with equal ids lies inside both blocks' spans, so a
// kernel may drop the tiles outside them; a query block and a key block that
// both hold the single id u (x == y == u) match on every pair, so the id
// compare can be skipped for that tile.
constexpr int kSegBlock = 128;
__device__ __forceinline__ int4 seg_block(const int4* tab, int b, int nblk, int blk) {
  return __ldg(tab + static_cast<size_t>(b) * nblk + blk);
}
__device__ __forceinline__ bool seg_same_single_id(int4 a, int4 c) {
  return a.x == a.y && c.x == c.y && a.x == c.x;
}

// Segment ids of 4 consecutive positions col.. of one sequence (ids past n,
// the sequence's valid length, are never read and come back as 0: those
// positions are masked by their span).  vec: the sequence's ids start
// 16-byte aligned, so a full group is one vector load.
__device__ __forceinline__ int4 load_ids4(const int32_t* __restrict__ ids, int col, int n, bool vec) {
  if (vec && col + 3 < n) return __ldg(reinterpret_cast<const int4*>(ids + col));
  int4 r;
  r.x = col < n ? __ldg(ids + col) : 0;
  r.y = col + 1 < n ? __ldg(ids + col + 1) : 0;
  r.z = col + 2 < n ? __ldg(ids + col + 2) : 0;
  r.w = col + 3 < n ? __ldg(ids + col + 3) : 0;
  return r;
}

// ---- forward ---------------------------------------------------------------
struct FwdArgs {
  Problem pb;
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  // split key ranges (16-bit, head_dim <= 128): pieces write fp32 partials
  // and the last piece of each pair merges them into o and lse; n_split = 1
  // writes them directly
  int n_split = 1;
  int split_chunk = 0;      // KV tiles per piece before a stream is cut further
  float* o_part = nullptr;  // [B, Hq, n_split, Lq, d]
  float* lse_part = nullptr;  // [B, Hq, n_split, Lq]
  int* counters = nullptr;    // one ticket counter per query-tile pair, zeroed before the launch
};
cudaError_t launch_fwd_16(const FwdArgs& a, DeviceStatus* st, cudaStream_t s);  // bf16 or fp16
cudaError_t launch_fwd_f32(const FwdArgs& a, DeviceStatus* st, cudaStream_t s);
cudaError_t launch_fwd_d256(const FwdArgs& a, DeviceStatus* st, cudaStream_t s);  // 16-bit, d = 256
// float32 on the bf16 tensor cores by splitting each operand into bf16 hi + lo
// (head_dim 64 and 128, no segment ids); the CUDA-core kernels take the rest
bool split_f32_applies(const Problem& pb);
cudaError_t launch_fwd_split_f32(const FwdArgs& a, DeviceStatus* st, cudaStream_t s);

// ---- backward --------------------------------------------------------------
struct BwdArgs {
  Problem pb;
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  float* delta;   // workspace [B, Hq, Lq_pad]
  float* lse2;    // workspace [B, Hq, Lq_pad]: lse * log2(e), +inf on empty and pad rows
  float* dq_acc;  // workspace [B, Lq, Hq, d] (single-pass variants)
  int* dq_turn;   // workspace: [B, Hq, ceil(Lq/128)] turn counters, then the ticket (ordered single pass)
  size_t turn_bytes;
  int Lq_pad;     // Lq rounded up to a multiple of 128
  int deterministic;  // 0 single pass (atomic dQ), 1 two-pass, 2 single pass with ordered dQ adds
  int* ticket;
};

// delta = rowsum(dO * O) in the padded [B, Hq, Lq_pad] layout; optional lse2,
// pad-row fill and dQ-accumulator zeroing (see small_kernels.cu).
struct PreprocessArgs {
  const void* o;
  const void* dout;
  const float* lse;  // needed when lse2 != nullptr
  float* delta;
  float* lse2;       // nullable
  float* dq_acc;     // nullable
  int B, Lq, Lq_pad, Hq, d;
  int elem;  // Elem of o and dout
};
cudaError_t launch_bwd_preprocess(const PreprocessArgs& a, cudaStream_t s);
cudaError_t launch_bwd_16(const BwdArgs& a, DeviceStatus* st, cudaStream_t s);
cudaError_t launch_bwd_f32(const BwdArgs& a, DeviceStatus* st, cudaStream_t s);
cudaError_t launch_bwd_d256(const BwdArgs& a, DeviceStatus* st, cudaStream_t s);  // 16-bit, d = 256
// float32 deterministic backward on the bf16 tensor cores (split operands;
// where split_f32_applies)
cudaError_t launch_bwd_split_f32(const BwdArgs& a, DeviceStatus* st, cudaStream_t s);

// ---- segment summary ----------------------------------------------------------
// Writes the SegBlock records of q_seg ([B, Lq]) and kv_seg ([B, Lkv]) into
// info: B * ceil(Lq/128) query records, then B * ceil(Lkv/128) key records.
cudaError_t launch_segment_info(const int32_t* q_seg, const int32_t* kv_seg, int B, int Lq, int Lkv, int4* info,
                                cudaStream_t s);

// ---- split-KV decode ---------------------------------------------------------
struct DecodeArgs {
  Problem pb;
  const void* q;
  const void* k;
  const void* v;
  float* o_part;
  float* lse_part;
  int num_splits;
  int chunk;  // keys per split, a multiple of 128
};
cudaError_t launch_decode_16(const DecodeArgs& a, DeviceStatus* st, cudaStream_t s);
cudaError_t launch_decode_f32(const DecodeArgs& a, DeviceStatus* st, cudaStream_t s);
cudaError_t launch_decode_combine(const float* o_part, const float* lse_part, void* o, float* lse, int B, int Lq,
                                  int Hq, int d, int num_splits, int elem, cudaStream_t s);

// ---- host helpers (attn_api.cu) ---------------------------------------------
// Tiled TMA descriptor over a [B, L, H, d] tensor: dims (d, L, H, B), box
// (box_inner, box_rows, 1, 1), 128-byte swizzle, zero fill out of bounds.
bool make_bshd_tmap(CUtensorMap* map, const void* base, int elem, int B, int L, int H, int d, int box_inner,
                    int box_rows);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Opt kernel K into `bytes` of dynamic shared memory, once per device (the
// attribute call is slow compared with a launch of a small problem).  Setting
// it twice from racing threads is harmless.
template <auto K>
cudaError_t ensure_dynamic_smem(int bytes) {
  // per device: the size already set (callers on several host threads may
  // both set it once; the attribute call is idempotent)
  static std::atomic<int> done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_relaxed) == bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(bytes, std::memory_order_relaxed);
  return e;
}

// Launch k so that it may overlap the kernel before it in the stream
// (programmatic stream serialization): its CTAs start once every CTA of that
// kernel has run griddepcontrol.launch_dependents (or exited).  k must run
// griddepcontrol.wait before it reads anything that kernel may still be
// writing, and at least one of its CTAs must run it before exiting, so that k
// still completes after its predecessor and the stream's next operation
// follows both.  Forwards, the decode, the combine and the preprocess wait
// before their first global read; a first backward pass after the
// preprocess waits after its prologue and only then triggers; a pass that
// reads nothing its predecessor writes (dQ after dK/dV, dK after dV at
// head_dim 256) does not wait at its start, since everything it reads was
// complete before its predecessor's CTAs triggered, and its last CTA waits
// before exiting.  The environment variable EXACT_ATTN_NO_PDL=1 turns the
// overlap off (plain stream order).
bool overlap_launch_enabled();
template <typename... P, typename... A>
cudaError_t launch_overlapping(void (*k)(P...), dim3 grid, int block, int smem, cudaStream_t s, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = overlap_launch_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, std::forward<A>(args)...);
}

// Opt-in per-kernel timing (attn_timing_enable): while enabled, a KernelTimer
// around a launch records CUDA events before and after it on its stream.
class KernelTimer {
 public:
  KernelTimer(const char* name, cudaStream_t s);
  ~KernelTimer();
  KernelTimer(const KernelTimer&) = delete;
  KernelTimer& operator=(const KernelTimer&) = delete;

 private:
  int slot_;
  cudaStream_t stream_;
};

// Launch order of the tiled kernels: a 1-D grid over (batch, head) pairs x
// tiles.  Pairs go in groups of `group`, so that the tensors a pair's CTAs
// share (K/V for query tiles, Q/dO for key tiles) stay in L2 while the group
// runs; inside a group the tile rank is the slower index (rank 0 = most work
// under causal masking starts first) and the pair the faster one.
struct TileCoord {
  int pair, rank;
};

__device__ __forceinline__ TileCoord grouped_tile(int linear, int n_pairs, int n_tiles, int group) {
  const int per_group = group * n_tiles;
  const int g = linear / per_group;
  const int first = g * group;
  const int in_group = min(group, n_pairs - first);
  const int l = linear - g * per_group;
  return {first + l % in_group, l / in_group};
}

#ifndef ATTN_L2_GROUP_BYTES
#define ATTN_L2_GROUP_BYTES (32l << 20)
#endif

// Pairs per group: as many as keep `group` x bytes_per_pair within the L2
// budget above, a multiple of `align` (the G query heads of one KV head share
// its K/V), at least `align`, at most n_pairs.
inline int l2_pair_group(long bytes_per_pair, int n_pairs, int align) {
  long g = bytes_per_pair > 0 ? ATTN_L2_GROUP_BYTES / bytes_per_pair : n_pairs;
  g = (g / align) * align;
  if (g < align) g = align;
  if (g > n_pairs) g = n_pairs;
  return static_cast<int>(g);
}

}  // namespace attn
