// Pieces shared by the backward kernels (two-pass dK/dV, dQ, single pass):
// kernel parameters, the TMEM -> bf16 row store and the probability half of
// the dK/dV softmax.
#pragma once
#include "attn_internal.h"

namespace attn {
namespace bwd {

constexpr float kLog2e = 1.4426950408889634f;

struct BwdKParams {
  const float* lse2;   // [B, Hq, Lq_pad], log2 domain, +inf on empty/pad rows
  const float* delta;  // [B, Hq, Lq_pad]
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;       // single-pass variants: [B, Lq, Hq, dh] fp32, zeroed by the preprocess (waited for before the first add)
  int* dq_turn;        // ordered single pass: [B, Hq, nq] turn counters, zeroed before the launch
  int* ticket;         // ordered single pass: work-item ticket, zeroed before the launch
  int nq;              // 128-row query tiles per sequence
  int rev;             // ordered single pass: turns go from the last key tile down (causal-like masks)
  const int32_t* kv_lens;
  int Lq, Lkv, Hq, Hkv, G, causal, wl, wr, Lq_pad, n_tiles, n_pairs, pair_group;
  int dh;  // stored head_dim (32 runs as D = 64 with zero-filled columns)
  const int32_t* q_seg;   // [B, Lq] segment ids (kSeg builds)
  const int32_t* kv_seg;  // [B, Lkv]
  const int4* seg_qblk;   // segment block summary (kSeg builds; nullptr: none)
  const int4* seg_kblk;
  int nqb, nkb;           // 128-position blocks per sequence: ceil(Lq/128), ceil(Lkv/128)
  float scale, scale_log2;
  DeviceStatus* status;
};

// Store the first ncols (a multiple of 32, <= D) of one row of fp32 values
// from TMEM in the 16-bit format (fp16 when kF16, else bf16), times `mul`.
template <int D, bool kF16>
__device__ __forceinline__ void store_row16(uint32_t taddr, uint16_t* dst, float mul, bool do_store, bool zero,
                                            int ncols) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    if (c * 32 >= ncols) break;
    uint32_t r[32];
    if (!zero) {
      tmem_ld32(taddr + c * 32, r);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = 0u;
    }
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack2<kF16>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
    if (do_store) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
  }
}

// P^T for the warpgroup's 64 queries [c0, c0 + 64): probabilities kept in
// `pr` (fp32) and written packed over columns [c0, c0 + 32) of S^T.  With
// MASK, query q_lo + c0 + c keeps its probability only if the key is valid and
// the query lies in [q_min, q_max) (the rows that see this key).
template <bool MASK, bool kUpper, bool kF16, bool kSeg = false>
__device__ __forceinline__ void dkdv_probs(uint32_t s_col, int c0, const float* lse2, float sl2, bool key_ok,
                                           int q_lo, int q_min, int q_max, float (&pr)[64],
                                           uint32_t seg_lo = 0u, uint32_t seg_hi = 0u) {
  uint32_t sa[32], sb[32];
  tmem_ld32_pair(s_col + c0, s_col + c0 + 32, sa, sb);
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c0 + 4 * i);
    float t[4];  // s sl2 - lse2, two columns per paired FMA
    f2_unpack(f2_fma(f2_pack(__uint_as_float(i < 8 ? sa[4 * i] : sb[4 * i - 32]),
                             __uint_as_float(i < 8 ? sa[4 * i + 1] : sb[4 * i + 1 - 32])),
                     sl2x2, f2_pack(-l4.x, -l4.y)),
              t[0], t[1]);
    f2_unpack(f2_fma(f2_pack(__uint_as_float(i < 8 ? sa[4 * i + 2] : sb[4 * i + 2 - 32]),
                             __uint_as_float(i < 8 ? sa[4 * i + 3] : sb[4 * i + 3 - 32])),
                     sl2x2, f2_pack(-l4.z, -l4.w)),
              t[2], t[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = 4 * i + e;
      float pv = ex2_approx(t[e]);
      if (MASK) pv = (key_ok && q_lo + c0 + c >= q_min && (!kUpper || q_lo + c0 + c < q_max)) ? pv : 0.f;
      if (kSeg) pv = (((c < 32 ? seg_lo >> c : seg_hi >> (c - 32)) & 1u) != 0u) ? pv : 0.f;
      pr[c] = pv;
    }
  }
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) pk[i] = pack2<kF16>(pr[2 * i], pr[2 * i + 1]);
  tmem_st32(s_col + c0, pk);
}

// Bit c (c < 32) of the result: id[col + c] == mine, for the ids of one
// sequence with n valid positions (positions past n never match).
__device__ __forceinline__ uint32_t segment_bits32(const int32_t* ids, int col, int n, bool vec, int mine) {
  uint32_t bits = 0u;
#pragma unroll 2
  for (int i = 0; i < 32; i += 4) {
    const int4 id = load_ids4(ids, col + i, n, vec);
    bits |= (static_cast<uint32_t>(id.x == mine && col + i < n) | (static_cast<uint32_t>(id.y == mine && col + i + 1 < n) << 1) |
             (static_cast<uint32_t>(id.z == mine && col + i + 2 < n) << 2) |
             (static_cast<uint32_t>(id.w == mine && col + i + 3 < n) << 3))
            << i;
  }
  return bits;
}

// Single-pass backward after the preprocess: the dK/dV kernel that also
// sums dQ into kp.dq_acc (grid = KV heads x batch x key tiles), then the dQ
// convert over n_dq values.  ordered: the sums of each query tile run in
// key-tile order (bitwise reproducible); otherwise as the adds arrive.  All
// six tensor maps (inputs, and dK/dV for the epilogue's stores) use boxes of
// 64 columns x 128 rows.
template <int D>
cudaError_t launch_single_pass(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                               const BwdKParams& kp, dim3 grid, long n_dq, bool f16, bool ordered,
                               cudaStream_t stream);
template <int D>
cudaError_t launch_single_pass_ordered(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                       const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                                       const BwdKParams& kp, dim3 grid, long n_dq, bool f16, cudaStream_t stream);

}  // namespace bwd
}  // namespace attn
