// Backward attention, bf16 or fp16, head_dim 64/128, on the sm_103a tensor cores.
//
// Method (probjax "Attention performance", section "When to use which",
// backward pass): the probabilities are recomputed from the forward's
// log-sum-exp, P = 2^(s * scale * log2(e) - lse * log2(e)), with
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - delta),  delta = rowsum(dO * O),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
// This file holds the deterministic two-pass backward: a dK/dV kernel per KV
// tile, then a separate dQ kernel per query tile; every sum runs in a fixed
// order, so the result is bitwise reproducible.  The single-pass variant
// (atomic dQ) is in bwd_atomic_sm103.cu and shares the launcher below.
// KV tiles past a batch element's length store zeros without running the
// pipeline; query tiles that see none of a key tile (causal) are skipped.
//
// dK/dV kernel: CTA = (batch, KV head, 128 keys); thread = key row = TMEM
// lane.  It walks the G query heads of the group and their 128-row query
// tiles.  Per step: S^T = K Q^T and dP^T = V dO^T (tcgen05, fp32 in TMEM),
// the softmax warps turn them into P^T and dS^T (bf16, written back to TMEM
// over the first half of each warpgroup's columns), then dV += P^T dO and
// dK += dS^T Q take those as the A operand straight from TMEM.
// TMEM: dK [0,128) dV [128,256) S^T [256,384) dP^T [384,512).
//
// dQ kernel: CTA = (batch, head, 128 queries); thread = query row.  Per
// 128-key step: S = Q K^T, dP = dO V^T, dS (bf16, into TMEM), dQ += dS K.
// TMEM: dQ [0,128), S double-buffered at [128,256) and [384,512), dP [256,384).
#include "bwd_common.cuh"

namespace attn {
namespace {

using namespace bwd;

// ============================================================================
// dK / dV kernel, deterministic two-pass variant
// ============================================================================
// CTA = (batch, KV head, 128 keys); thread = key row = TMEM lane.  Each step
// takes 128 queries so every tcgen05.mma is 128 x 128 (64-wide operands run
// the tensor core at two thirds of its rate or less).  TMEM holds one stage:
// dK [0,128) dV [128,256) S^T [256,384) dP^T [384,512).
//
// The two score GEMMs are separate, and so is the softmax work:
//   tensor pipe:  S^T(t) | dP^T(t)           | dV += P^T dO | dK += dS^T Q | S^T(t+1) ...
//   softmax:             | P^T = 2^(S^T - L)  | dS^T = P^T (dP^T - delta)   |
// The P half needs only S^T and runs while dP^T is computed; the dS half runs
// while dV accumulates.  Warpgroup w owns queries [64w, 64w + 64) of the step
// and keeps its 64 probabilities in fp32 registers between the halves; the
// packed bf16 P^T / dS^T go over the first 32 of its 64 S^T / dP^T columns.
// Warps 0-7 softmax, warp 8 TMA producer, warp 9 MMA issuer.
template <int D>
struct DkdvCfg2 {
  static constexpr int kBN = 128, kBM = 128;
  static constexpr int kKVBytes = kBN * D * 2;
  static constexpr int kBox = 128 * 128;      // one 64-column box of a 128-row tile
  static constexpr int kQBytes = kBM * D * 2;
  // Q (with its lse2 rows) in a ring of 3: S^T(t+1) is issued right after
  // dV(t), before dK(t) has released Q(t).  dO (with its delta rows) in a ring
  // of 2: dP^T(t+1) comes after dK(t).  Both release a slot after dK.
  static constexpr int kQSlots = 3, kDOSlots = 2;
  static constexpr int kOffV = kKVBytes;
  static constexpr int kOffQ = 2 * kKVBytes;
  static constexpr int kOffDO = kOffQ + kQSlots * kQBytes;
  static constexpr int kOffLse = kOffDO + kDOSlots * kQBytes;
  static constexpr int kOffDelta = kOffLse + kQSlots * kBM * 4;
  static constexpr int kOffBars = kOffDelta + kDOSlots * kBM * 4;
  static constexpr int kNumBars = 2 * kQSlots + 2 * kDOSlots + 6;
  // No alignment slack: the dynamic shared window starts 1024-aligned (checked
  // at run time; a misaligned base makes the kernel report and do nothing).
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16;
  static constexpr int kThreads = 320;
};

// TMEM column (relative to the step's S^T / S block) of the packed A operand
// for query (or key) k-step k of half h, when NWG warpgroups each convert
// 64 / NWG columns of a half.
template <int NWG>
__device__ __forceinline__ constexpr uint32_t packed_col(int h, int k) {
  constexpr int kC = 64 / NWG;
  return 64 * h + kC * ((16 * k) / kC) + ((16 * k) % kC) / 2;
}

// dS^T = P^T (dP^T - delta) for the same 64 queries, written packed over
// columns [c0, c0 + 32) of dP^T.
template <bool kF16>
__device__ __forceinline__ void dkdv_dscores(uint32_t dp_col, int c0, const float* dlt, const float (&pr)[64]) {
  uint32_t da[32], db[32];
  tmem_ld32_pair(dp_col + c0, dp_col + c0 + 32, da, db);
  uint32_t dk[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 d4 = *reinterpret_cast<const float4*>(dlt + c0 + 4 * i);
    const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
    float ds[4];
#pragma unroll
    for (int e = 0; e < 4; e += 2) {  // P^T (dP^T - delta), two columns per paired instruction
      const int c = 4 * i + e;
      const uint32_t r0 = c < 32 ? da[c] : db[c - 32], r1 = c + 1 < 32 ? da[c + 1] : db[c + 1 - 32];
      f2_unpack(f2_mul(f2_pack(pr[c], pr[c + 1]),
                       f2_sub(f2_pack(__uint_as_float(r0), __uint_as_float(r1)), f2_pack(dv[e], dv[e + 1]))),
                ds[e], ds[e + 1]);
    }
    dk[2 * i] = pack2<kF16>(ds[0], ds[1]);
    dk[2 * i + 1] = pack2<kF16>(ds[2], ds[3]);
  }
  tmem_st32(dp_col + c0, dk);
}

template <int D, bool kLeftBound, bool kF16, bool kSeg>
__global__ void __launch_bounds__(320, 1)
    bwd_dkdv_kernel2(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv, const BwdKParams p) {
  using C = DkdvCfg2<D>;
  constexpr int NQ = C::kQSlots, NO = C::kDOSlots, BM = C::kBM;
  constexpr uint32_t kColS = 256, kColDP = 384;
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // never expected: see kSmemBytes
    if (threadIdx.x == 0) report_status(p.status, 2, 60);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDO = smem + C::kOffDO;
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sDelta = reinterpret_cast<float*>(smem + C::kOffDelta);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* full_q = bars;
  uint64_t* empty_q = bars + NQ;
  uint64_t* full_do = bars + 2 * NQ;
  uint64_t* empty_do = bars + 2 * NQ + NO;
  uint64_t* kv_full = bars + 2 * NQ + 2 * NO;
  uint64_t* s_ready = kv_full + 1;   // S^T(t) computed
  uint64_t* dp_ready = kv_full + 2;  // dP^T(t) computed
  uint64_t* p_ready = kv_full + 3;   // P^T(t) written (256 arrivals)
  uint64_t* ds_ready = kv_full + 4;  // dS^T(t) written (256 arrivals)
  uint64_t* acc_full = kv_full + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  // 1-D grid over (b, hkv) pairs x key tiles in L2 groups; with causal masking
  // the tiles that see the most queries (the first ones) start first.
  const TileCoord tc = grouped_tile(blockIdx.x, p.n_pairs, p.n_tiles, p.pair_group);
  const int j0 = tc.rank * C::kBN, hk = tc.pair % p.Hkv, b = tc.pair / p.Hkv;
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);
  // query tiles that see some key of this tile: from the first row that sees
  // key j0 to the last row that sees the tile's last valid key
  int i_begin = 0, steps_per_head = 0;
  if (j0 < kvl) {
    int q_lo = query_span(j0, p.Lq, kvl, p.wl, p.wr).lo;
    int q_hi = query_span(min(j0 + C::kBN, kvl) - 1, p.Lq, kvl, p.wl, p.wr).hi;
    if (kSeg && p.seg_kblk != nullptr) {  // queries whose blocks may share an id with this key block
      const int4 r = seg_block(p.seg_kblk, b, p.nkb, j0 / kSegBlock);
      q_lo = max(q_lo, r.z);
      q_hi = min(q_hi, r.w);
    }
    if (q_hi > q_lo) {
      i_begin = q_lo / BM;
      steps_per_head = (q_hi + BM - 1) / BM - i_begin;
    }
  }
  const int T = steps_per_head * p.G;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < NQ; ++s) {
      mbar_init(&full_q[s], 1);
      mbar_init(&empty_q[s], 1);
    }
    for (int s = 0; s < NO; ++s) {
      mbar_init(&full_do[s], 1);
      mbar_init(&empty_do[s], 1);
    }
    mbar_init(kv_full, 1);
    mbar_init(s_ready, 1);
    mbar_init(dp_ready, 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // Launched to overlap the preprocess: delta and lse2 are complete from here
  // on.  The dQ pass reads nothing this kernel writes, so its CTAs may then
  // take the SMs that this grid's finished CTAs leave.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 8) {
    if (lane == 0 && T > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(kv_full, 2 * C::kKVBytes);
      for (int h = 0; h < D / 64; ++h) {
        tma_load_4d(sK + h * C::kBox, &tm_k, kv_full, h * 64, j0, hk, b);
        tma_load_4d(sV + h * C::kBox, &tm_v, kv_full, h * 64, j0, hk, b);
      }
      for (int t = 0; t < T; ++t) {
        const int h = hk * p.G + t / steps_per_head;
        const int q0 = (i_begin + t % steps_per_head) * BM;
        const size_t row = (static_cast<size_t>(b) * p.Hq + h) * p.Lq_pad + q0;
        const int sq = t % NQ, rq = t / NQ;
        if (rq > 0 && !mbar_wait(&empty_q[sq], (rq - 1) & 1, abort_flag, p.status, 61)) break;
        mbar_arrive_expect_tx(&full_q[sq], C::kQBytes + BM * 4);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sQ + sq * C::kQBytes + c * C::kBox, &tm_q, &full_q[sq], c * 64, q0, h, b);
        bulk_load(sLse + sq * BM, p.lse2 + row, BM * 4, &full_q[sq]);
        const int so = t % NO, ro = t / NO;
        if (ro > 0 && !mbar_wait(&empty_do[so], (ro - 1) & 1, abort_flag, p.status, 59)) break;
        mbar_arrive_expect_tx(&full_do[so], C::kQBytes + BM * 4);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sDO + so * C::kQBytes + c * C::kBox, &tm_do, &full_do[so], c * 64, q0, h, b);
        bulk_load(sDelta + so * BM, p.delta + row, BM * 4, &full_do[so]);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_st = idesc_16_f32<kF16>(128, BM, 0, 0);  // K x Q^T, V x dO^T
      constexpr uint32_t idesc_acc = idesc_16_f32<kF16>(128, D, 0, 1);  // (P^T|dS^T from TMEM) x (dO|Q MN-major)
      const uint32_t k_addr = smem_u32(sK), v_addr = smem_u32(sV), q_addr = smem_u32(sQ), o_addr = smem_u32(sDO);
      const SDesc dk_base = sdesc_split(k_addr, 16, 1024), dv_base = sdesc_split(v_addr, 16, 1024);
      const SDesc dq_base = sdesc_split(q_addr, 16, 1024), ddo_base = sdesc_split(o_addr, 16, 1024);
      const SDesc bq_base = sdesc_split(q_addr, C::kBox, 1024), bdo_base = sdesc_split(o_addr, C::kBox, 1024);
      constexpr uint32_t kSlot16 = C::kQBytes >> 4;
      auto issue_s = [&](int t) {  // S^T(t) = K Q(t)^T
        const uint32_t qo = (t % NQ) * kSlot16;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * C::kBox + (k & 3) * 32) >> 4;
          mma_ss_d(tbase + kColS, dk_base, off, dq_base, qo + off, idesc_st, k > 0);
        }
        mma_commit(s_ready);
      };
      auto issue_dp = [&](int t) {  // dP^T(t) = V dO(t)^T
        const uint32_t oo = (t % NO) * kSlot16;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * C::kBox + (k & 3) * 32) >> 4;
          mma_ss_d(tbase + kColDP, dv_base, off, ddo_base, oo + off, idesc_st, k > 0);
        }
        mma_commit(dp_ready);
      };
      // Order per step: dV(t), S^T(t+1), dK(t), dP^T(t+1).  S^T(t+1) overwrites
      // P^T(t) right after dV(t) has read it (one thread issues all MMAs; the
      // tensor pipe runs them in order), so the probabilities of step t+1 run
      // while dK(t) and dP^T(t+1) are on the tensor core.
      bool ok = mbar_wait(kv_full, 0, abort_flag, p.status, 62);
      if (ok) ok = mbar_wait(&full_q[0], 0, abort_flag, p.status, 63);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = mbar_wait(&full_do[0], 0, abort_flag, p.status, 58);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(0);
      }
      for (int t = 0; t < T && ok; ++t) {
        const uint32_t qo = (t % NQ) * kSlot16, oo = (t % NO) * kSlot16;
        // query k-step k (16 queries) of warpgroup w = k / 4 sits packed at 64 w + 8 (k - 4 w)
        ok = mbar_wait(p_ready, t & 1, abort_flag, p.status, 64);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // dV += P^T dO
          const uint32_t acol = 64 * (k >> 2) + 8 * (k & 3);
          mma_ts_d(tbase + 128, tbase + kColS + acol, bdo_base, oo + ((16 * k * 128) >> 4), idesc_acc,
                   (t > 0 || k > 0) ? 1u : 0u);
        }
        if (t + 1 < T) {
          ok = mbar_wait(&full_q[(t + 1) % NQ], ((t + 1) / NQ) & 1, abort_flag, p.status, 66);
          if (!ok) break;
          tc_fence_after();
          issue_s(t + 1);
        }
        ok = mbar_wait(ds_ready, t & 1, abort_flag, p.status, 65);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // dK += dS^T Q
          const uint32_t acol = 64 * (k >> 2) + 8 * (k & 3);
          mma_ts_d(tbase + 0, tbase + kColDP + acol, bq_base, qo + ((16 * k * 128) >> 4), idesc_acc,
                   (t > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&empty_q[t % NQ]);
        mma_commit(&empty_do[t % NO]);
        if (t + 1 < T) {
          ok = mbar_wait(&full_do[(t + 1) % NO], ((t + 1) / NO) & 1, abort_flag, p.status, 57);
          if (!ok) break;
          tc_fence_after();
          issue_dp(t + 1);
        }
      }
      if (ok) mma_commit(acc_full);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (thread = key row)
    const int w = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const int j = j0 + r;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(wq * 32) << 16);
    const bool key_ok = j < kvl;
    const Span qs = key_ok ? query_span(j, p.Lq, kvl, p.wl, p.wr) : Span{0, 0};
    // segment masks: the key's id, and the queries' ids of this sequence
    const int my_seg = (kSeg && j < p.Lkv) ? __ldg(p.kv_seg + static_cast<size_t>(b) * p.Lkv + j) : 0;
    const int32_t* qid = kSeg ? p.q_seg + static_cast<size_t>(b) * p.Lq : nullptr;
    const bool qid_vec = kSeg && ((static_cast<size_t>(b) * p.Lq) & 3) == 0;
    // this key block's summary; (0, -1) never counts as a single id
    const int4 krec = (kSeg && p.seg_kblk != nullptr) ? seg_block(p.seg_kblk, b, p.nkb, j0 / kSegBlock)
                                                      : make_int4(0, -1, 0, 0);
    const float sl2 = p.scale_log2;
    const int c0 = 64 * w;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int q0 = (i_begin + t % steps_per_head) * BM;
      uint32_t sg0 = ~0u, sg1 = ~0u;  // segment bits of this warpgroup's 64 queries (before S is ready)
      // query and key block hold one and the same id: every pair matches
      const bool seg_all =
          kSeg && p.seg_qblk != nullptr && seg_same_single_id(seg_block(p.seg_qblk, b, p.nqb, q0 / kSegBlock), krec);
      if (kSeg && !seg_all) {
        sg0 = segment_bits32(qid, q0 + c0, p.Lq, qid_vec, my_seg);
        sg1 = segment_bits32(qid, q0 + c0 + 32, p.Lq, qid_vec, my_seg);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(s_ready, t & 1, abort_flag, p.status, 67));
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = sLse + (t % NQ) * BM;
      const float* dlt = sDelta + (t % NO) * BM;
      float pr[64];
      // without a left window bound every row after the first that sees the
      // key sees it too, so only the lower end needs checking
      if ((!kSeg || seg_all) &&
          __all_sync(0xffffffffu, key_ok && q0 + c0 >= qs.lo && (!kLeftBound || q0 + c0 + 64 <= qs.hi)))
        dkdv_probs<false, kLeftBound, kF16>(t_lane + kColS, c0, lse2, sl2, key_ok, q0, qs.lo, qs.hi, pr);
      else
        dkdv_probs<true, kLeftBound, kF16, kSeg>(t_lane + kColS, c0, lse2, sl2, key_ok, q0, qs.lo, qs.hi, pr, sg0,
                                                 sg1);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_ready);
      ok = __all_sync(0xffffffffu, mbar_wait(dp_ready, t & 1, abort_flag, p.status, 69));
      if (!ok) break;
      tc_fence_after();
      dkdv_dscores<kF16>(t_lane + kColDP, c0, dlt, pr);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ds_ready);
    }
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, p.status, 68));
    // dK (warpgroup 0, times scale) and dV (warpgroup 1) go through the Q ring,
    // idle once every MMA has completed, and out with TMA stores, which clip
    // the rows past Lkv and the columns past the stored head_dim.  (Each thread
    // storing its own row would put 32 rows, a row stride apart, into every
    // store instruction: the epilogue took ~2.9 us per CTA that way.)
    if (ok) {
      tc_fence_after();
      stage_row16<D, kF16>(t_lane + (w == 0 ? 0 : 128), sQ + w * (D / 64) * C::kBox, r, w == 0 ? p.scale : 1.0f,
                           T == 0);
      fence_proxy_async_smem();
    }
    named_barrier_sync(1, 256);
    if (threadIdx.x == 0 && *abort_flag == 0) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_store_4d(&tm_dk, sQ + c * C::kBox, c * 64, j0, hk, b);
        tma_store_4d(&tm_dv, sQ + (D / 64 + c) * C::kBox, c * 64, j0, hk, b);
      }
      tma_store_commit();
      tma_store_wait_read();  // the shared memory is released when the CTA exits
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ============================================================================
// dQ kernel
// ============================================================================
template <int D>
struct DqCfg {
  static constexpr int kNWG = 2;                // softmax warpgroups
  static constexpr int kCols = 64 / kNWG;       // key columns per warpgroup per half-step
  static constexpr int kProducerWarp = 4 * kNWG, kMmaWarp = 4 * kNWG + 1;
  static constexpr int kBM = 128;               // queries per CTA
  static constexpr int kBN = 128;               // keys per step
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kKVBytes = kBN * D * 2;
  static constexpr int kBox = 128 * 128;        // one 64-column box of a 128-row tile
  static constexpr int kKSlots = 3, kVSlots = 2;
  static constexpr int kOffDO = kQBytes;
  static constexpr int kOffK = 2 * kQBytes;
  static constexpr int kOffV = kOffK + kKSlots * kKVBytes;
  static constexpr int kOffBars = kOffV + kVSlots * kKVBytes;
  static constexpr int kNumBars = 2 * kKSlots + 2 * kVSlots + 1 + 3 + 2 + 1;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;
  static constexpr int kThreads = 32 * (4 * kNWG + 2);
};

// Probabilities of the N key columns [c0, c0 + N) of one step (thread =
// query row), from S at s_col; kept in registers until dP is ready.
template <int N, bool MASK, bool kLower = true, bool kSeg = false>
__device__ __forceinline__ void dq_probs(uint32_t s_col, int c0, float l2, float sl2, int kb, Span ks, float* pr,
                                         uint32_t seg = 0u) {
  uint32_t sr[N];
  if constexpr (N == 32)
    tmem_ld32(s_col + c0, *reinterpret_cast<uint32_t(*)[32]>(sr));
  else
    tmem_ld16(s_col + c0, *reinterpret_cast<uint32_t(*)[16]>(sr));
  // 2^(s sl2 - l2), two columns per paired fp32 FMA
  const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(-l2, -l2);
#pragma unroll
  for (int c = 0; c < N; c += 2) {
    float t0, t1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2, nl2), t0, t1);
    float pv[2] = {ex2_approx(t0), ex2_approx(t1)};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (MASK) pv[e] = ((!kLower || kb + c0 + c + e >= ks.lo) && kb + c0 + c + e < ks.hi) ? pv[e] : 0.f;
      if (kSeg) pv[e] = ((seg >> (c + e)) & 1u) ? pv[e] : 0.f;
      pr[c + e] = pv[e];
    }
  }
}

// dS = P (dP - delta) for the same N columns, packed over the first N/2 of
// the S columns they came from.
template <int N, bool kF16>
__device__ __forceinline__ void dq_dscores(uint32_t s_col, uint32_t dp_col, int c0, float dl, const float* pr) {
  uint32_t dr[N];
  if constexpr (N == 32)
    tmem_ld32(dp_col + c0, *reinterpret_cast<uint32_t(*)[32]>(dr));
  else
    tmem_ld16(dp_col + c0, *reinterpret_cast<uint32_t(*)[16]>(dr));
  uint32_t pk[N / 2];
  const uint64_t dl2 = f2_pack(dl, dl);
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {  // P (dP - delta), two columns per paired instruction
    float d0, d1;
    f2_unpack(f2_mul(f2_pack(pr[2 * i], pr[2 * i + 1]),
                     f2_sub(f2_pack(__uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1])), dl2)),
              d0, d1);
    pk[i] = pack2<kF16>(d0, d1);
  }
  if constexpr (N == 32)
    tmem_st16(s_col + c0, *reinterpret_cast<uint32_t(*)[16]>(pk));
  else
    tmem_st8(s_col + c0, *reinterpret_cast<uint32_t(*)[8]>(pk));
}

// dQ kernel: CTA = (batch, head, 128 queries); thread = query row.  Each step
// takes 128 keys (every MMA 128 x 128): S = Q K^T, dP = dO V^T, dS (bf16,
// written back into S's columns), dQ += dS K.  TMEM: dQ [0,128), S in two
// buffers [128,256) and [384,512) (step parity), dP [256,384).  S runs two
// steps ahead, so the softmax warps compute the probabilities of step t+1
// (which need only S) while dQ of step t and dP of step t+1 are on the tensor
// core, and only the cheap dS = P (dP - delta) waits for dP.  dS is released in
// two 64-key halves so the dQ MMAs of half 0 overlap the second half.  K tiles
// use a 3-slot ring (a K tile is read by S and later by dQ), V tiles a 2-slot
// ring.
template <int D, bool kLeftBound, bool kF16, bool kSeg>
__global__ void __launch_bounds__(DqCfg<D>::kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq,
                  const BwdKParams p) {
  using C = DqCfg<D>;
  constexpr int NK = C::kKSlots, NV = C::kVSlots, BN = C::kBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::kOffDO;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* full_k = bars;
  uint64_t* empty_k = bars + NK;
  uint64_t* full_v = bars + 2 * NK;
  uint64_t* empty_v = full_v + NV;
  uint64_t* q_full = empty_v + NV;
  uint64_t* s_ready = q_full + 1;   // [2] S(t) computed, one barrier per S buffer (t & 1)
  uint64_t* dp_ready = q_full + 3;  // dP(t) computed
  uint64_t* p_half = q_full + 4;    // [2] dS(t) halves written
  uint64_t* acc_full = q_full + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  // 1-D grid over (b, hq) pairs x query tiles in L2 groups, longest causal tiles first
  const TileCoord tc = grouped_tile(blockIdx.x, p.n_pairs, p.n_tiles, p.pair_group);
  const int qt = p.causal ? p.n_tiles - 1 - tc.rank : tc.rank;
  const int q0 = qt * C::kBM, h = tc.pair % p.Hq, b = tc.pair / p.Hq;
  const int hk = h / p.G;
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);
  // key tiles [t0, t0 + T): from the first key of row q0 to the last key of
  // the tile's last row (both ends grow with the row index)
  const int last = min(q0 + C::kBM - 1, p.Lq - 1);
  int k_lo = key_span(q0, p.Lq, kvl, p.wl, p.wr).lo;
  int k_hi = key_span(last, p.Lq, kvl, p.wl, p.wr).hi;
  // segment ids: this query block's summary; keys outside its span never match
  const int4 qrec = (kSeg && p.seg_qblk != nullptr) ? seg_block(p.seg_qblk, b, p.nqb, q0 / kSegBlock)
                                                    : make_int4(0, -1, 0, 0);
  if (kSeg && p.seg_qblk != nullptr) {
    k_lo = max(k_lo, qrec.z);
    k_hi = min(k_hi, qrec.w);
  }
  const int t0 = kLeftBound ? k_lo / BN : 0;
  const int T = k_hi > k_lo ? (k_hi + BN - 1) / BN - t0 : 0;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < NK; ++s) {
      mbar_init(&full_k[s], 1);
      mbar_init(&empty_k[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&full_v[s], 1);
      mbar_init(&empty_v[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(&s_ready[0], 1);
    mbar_init(&s_ready[1], 1);
    mbar_init(dp_ready, 1);
    mbar_init(&p_half[0], 128 * C::kNWG);
    mbar_init(&p_half[1], 128 * C::kNWG);
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  griddep_launch_dependents();  // the next kernel waits for this grid before it reads anything

  if (warp == C::kProducerWarp) {
    if (lane == 0 && T > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, 2 * C::kQBytes);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_4d(sQ + c * C::kBox, &tm_q, q_full, c * 64, q0, h, b);
        tma_load_4d(sDO + c * C::kBox, &tm_do, q_full, c * 64, q0, h, b);
      }
      bool ok = true;
      for (int t = 0; t < T && ok; ++t) {
        const int sk = t % NK, rk = t / NK, sv = t % NV, rv = t / NV;
        if (rk > 0 && !(ok = mbar_wait(&empty_k[sk], (rk - 1) & 1, abort_flag, p.status, 31))) break;
        mbar_arrive_expect_tx(&full_k[sk], C::kKVBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sK + sk * C::kKVBytes + c * C::kBox, &tm_k, &full_k[sk], c * 64, (t0 + t) * BN, hk, b);
        if (rv > 0 && !(ok = mbar_wait(&empty_v[sv], (rv - 1) & 1, abort_flag, p.status, 30))) break;
        mbar_arrive_expect_tx(&full_v[sv], C::kKVBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sV + sv * C::kKVBytes + c * C::kBox, &tm_v, &full_v[sv], c * 64, (t0 + t) * BN, hk, b);
      }
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_s = idesc_16_f32<kF16>(128, BN, 0, 0);   // Q x K^T, dO x V^T
      constexpr uint32_t idesc_dq = idesc_16_f32<kF16>(128, D, 0, 1);  // dS (TMEM) x K (MN-major)
      const uint32_t q_addr = smem_u32(sQ), do_addr = smem_u32(sDO);
      const SDesc dq_desc = sdesc_split(q_addr, 16, 1024), ddo_desc = sdesc_split(do_addr, 16, 1024);
      const SDesc dk_desc = sdesc_split(smem_u32(sK), 16, 1024), dv_desc = sdesc_split(smem_u32(sV), 16, 1024);
      const SDesc bk_desc = sdesc_split(smem_u32(sK), C::kBox, 1024);
      constexpr uint32_t kSlot16 = C::kKVBytes >> 4;
      auto s_buf = [](int t) -> uint32_t { return (t & 1) ? 384u : 128u; };
      auto issue_s = [&](int t) {  // S(t) = Q K_t^T into its buffer
        const uint32_t ko = (t % NK) * kSlot16;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * C::kBox + (k & 3) * 32) >> 4;
          mma_ss_d(tbase + s_buf(t), dq_desc, off, dk_desc, ko + off, idesc_s, k > 0);
        }
        mma_commit(&s_ready[t & 1]);
      };
      auto issue_dp = [&](int t) {  // dP(t) = dO V_t^T
        const uint32_t vo = (t % NV) * kSlot16;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * C::kBox + (k & 3) * 32) >> 4;
          mma_ss_d(tbase + 256, ddo_desc, off, dv_desc, vo + off, idesc_s, k > 0);
        }
        mma_commit(dp_ready);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, 32);
      if (ok) ok = mbar_wait(&full_k[0], 0, abort_flag, p.status, 33);
      if (ok) ok = mbar_wait(&full_v[0], 0, abort_flag, p.status, 39);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
        mma_commit(&empty_v[0]);
        if (T > 1) {
          ok = mbar_wait(&full_k[1 % NK], 0, abort_flag, p.status, 33);
          if (ok) {
            tc_fence_after();
            issue_s(1);
          }
        }
      }
      for (int t = 0; t < T && ok; ++t) {
        const uint32_t ko = (t % NK) * kSlot16;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          ok = mbar_wait(&p_half[hh], t & 1, abort_flag, p.status, 34 + hh);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // dQ += dS[:, keys 64hh + 16k ..] K[keys 64hh + 16k ..]
            const uint32_t acol = s_buf(t) + packed_col<C::kNWG>(hh, k);
            const uint32_t boff = ((64 * hh + 16 * k) * 128) >> 4;
            mma_ts_d(tbase, tbase + acol, bk_desc, ko + boff, idesc_dq, (t > 0 || hh > 0 || k > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
        mma_commit(&empty_k[t % NK]);
        if (t + 1 < T) {  // dP(t+1): the softmax has read all of dP(t)
          ok = mbar_wait(&full_v[(t + 1) % NV], ((t + 1) / NV) & 1, abort_flag, p.status, 36);
          if (!ok) break;
          tc_fence_after();
          issue_dp(t + 1);
          mma_commit(&empty_v[(t + 1) % NV]);
        }
        if (t + 2 < T) {  // S(t+2) into the buffer dQ(t) has just consumed
          ok = mbar_wait(&full_k[(t + 2) % NK], ((t + 2) / NK) & 1, abort_flag, p.status, 38);
          if (!ok) break;
          tc_fence_after();
          issue_s(t + 2);
        }
      }
      if (ok) mma_commit(acc_full);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (thread = query row)
    const int w = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const int i = q0 + r;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(wq * 32) << 16);
    const size_t srow = (static_cast<size_t>(b) * p.Hq + h) * p.Lq_pad + i;  // i < Lq_pad always
    const float l2 = p.lse2[srow];
    const float dl = p.delta[srow];
    Span ks = key_span(i, p.Lq, kvl, p.wl, p.wr);
    if (!kLeftBound) ks.lo = 0;
    if (i >= p.Lq) ks.lo = ks.hi = 0;
    const float sl2 = p.scale_log2;
    // segment masks: the row's id, and the keys' ids of this sequence
    const int my_seg = (kSeg && i < p.Lq) ? __ldg(p.q_seg + static_cast<size_t>(b) * p.Lq + i) : 0;
    const int32_t* kid = kSeg ? p.kv_seg + static_cast<size_t>(b) * p.Lkv : nullptr;
    const bool kid_vec = kSeg && ((static_cast<size_t>(b) * p.Lkv) & 3) == 0;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int kb = (t0 + t) * BN;
      uint32_t sg[2] = {~0u, ~0u};  // segment bits of this thread's two key column groups
      // query and key block hold one and the same id: every pair matches
      const bool seg_all =
          kSeg && p.seg_kblk != nullptr && seg_same_single_id(qrec, seg_block(p.seg_kblk, b, p.nkb, t0 + t));
      if (kSeg && !seg_all) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) sg[hh] = segment_bits32(kid, kb + 64 * hh + C::kCols * w, kvl, kid_vec, my_seg);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&s_ready[t & 1], (t >> 1) & 1, abort_flag, p.status, 37));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_col = t_lane + ((t & 1) ? 384u : 128u);
      const uint32_t dp_col = t_lane + 256;
      float pr[2 * C::kCols];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int c0 = 64 * hh + C::kCols * w;
        if ((!kSeg || seg_all) &&
            __all_sync(0xffffffffu, (!kLeftBound || kb + c0 >= ks.lo) && kb + c0 + C::kCols <= ks.hi))
          dq_probs<C::kCols, false, kLeftBound>(s_col, c0, l2, sl2, kb, ks, pr + hh * C::kCols);
        else
          dq_probs<C::kCols, true, kLeftBound, kSeg>(s_col, c0, l2, sl2, kb, ks, pr + hh * C::kCols, sg[hh]);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(dp_ready, t & 1, abort_flag, p.status, 39));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        dq_dscores<C::kCols, kF16>(s_col, dp_col, 64 * hh + C::kCols * w, dl, pr + hh * C::kCols);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_half[hh]);
      }
    }
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, p.status, 38));
    // dQ goes through the K ring, idle once every MMA has completed, and out
    // with TMA stores (rows past Lq and columns past the stored head_dim are
    // clipped); warpgroup w stages head-dim columns [w D / NWG, (w + 1) D / NWG)
    if (ok) {
      tc_fence_after();
      constexpr int kPer = D / C::kNWG;
      stage_row16<kPer, kF16>(t_lane + w * kPer, sK, r, p.scale, T == 0, w * kPer);
      fence_proxy_async_smem();
    }
    named_barrier_sync(1, 128 * C::kNWG);
    if (threadIdx.x == 0 && *abort_flag == 0) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_store_4d(&tm_dq, sK + c * C::kBox, c * 64, q0, h, b);
      tma_store_commit();
      tma_store_wait_read();  // the shared memory is released when the CTA exits
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // Launched to overlap the dK/dV pass (it reads nothing that pass writes).
  // One CTA waits for that grid before it exits, so this grid completes after
  // it and whatever follows in the stream sees dK and dV.
  if (blockIdx.x == gridDim.x - 1) griddep_wait();
}

template <int D, bool kLeftBound, bool kF16, bool kSeg>
cudaError_t launch_dkdv_inst(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                             const BwdKParams& kp, dim3 grid, cudaStream_t stream) {
  using C = DkdvCfg2<D>;
  cudaError_t e = ensure_dynamic_smem<bwd_dkdv_kernel2<D, kLeftBound, kF16, kSeg>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  KernelTimer kt("bwd_dkdv", stream);
  return launch_overlapping(bwd_dkdv_kernel2<D, kLeftBound, kF16, kSeg>, grid, C::kThreads, C::kSmemBytes, stream, tq,
                            tk, tv, tdo, tdk, tdv, kp);
}

template <int D, bool kLeftBound, bool kF16, bool kSeg>
cudaError_t launch_dq_inst(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdKParams& kp, dim3 grid,
                           cudaStream_t stream) {
  using C = DqCfg<D>;
  cudaError_t e = ensure_dynamic_smem<bwd_dq_kernel<D, kLeftBound, kF16, kSeg>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  KernelTimer kt("bwd_dq", stream);
  return launch_overlapping(bwd_dq_kernel<D, kLeftBound, kF16, kSeg>, grid, C::kThreads, C::kSmemBytes, stream, tq, tk,
                            tv, tdo, tdq, kp);
}

// The kernel build for a problem: format x (no left bound | two-sided span |
// two-sided span + segment ids).
template <template <int, bool, bool, bool> class L, int D, typename... A>
cudaError_t dispatch_build(const Problem& pb, A&&... args) {
  const bool left = pb.wl < kWinInf;
  if (pb.q_seg != nullptr)
    return pb.f16 ? L<D, true, true, true>::run(args...) : L<D, true, false, true>::run(args...);
  if (pb.f16) return left ? L<D, true, true, false>::run(args...) : L<D, false, true, false>::run(args...);
  return left ? L<D, true, false, false>::run(args...) : L<D, false, false, false>::run(args...);
}

template <int D, bool kL, bool kF, bool kS>
struct DkdvLaunch {
  template <typename... A>
  static cudaError_t run(A&&... args) { return launch_dkdv_inst<D, kL, kF, kS>(args...); }
};
template <int D, bool kL, bool kF, bool kS>
struct DqLaunch {
  template <typename... A>
  static cudaError_t run(A&&... args) { return launch_dq_inst<D, kL, kF, kS>(args...); }
};

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, DeviceStatus* st, cudaStream_t stream) {
  const Problem& pb = a.pb;
  const int elem = pb.f16 ? kElemF16 : kElemBF16;
  PreprocessArgs pa;
  pa.o = a.o;
  pa.dout = a.dout;
  pa.lse = a.lse;
  pa.delta = a.delta;
  pa.lse2 = a.lse2;
  pa.dq_acc = a.deterministic == 1 ? nullptr : a.dq_acc;  // the single-pass variants sum into it
  pa.B = pb.B;
  pa.Lq = pb.Lq;
  pa.Lq_pad = a.Lq_pad;
  pa.Hq = pb.Hq;
  pa.d = pb.d;  // stored head_dim: the preprocess reads O and dO rows of this width
  pa.elem = elem;
  cudaError_t e = launch_bwd_preprocess(pa, stream);
  if (e != cudaSuccess) return e;

  BwdKParams kp;
  kp.lse2 = a.lse2;
  kp.delta = a.delta;
  kp.dq = a.dq;
  kp.dk = a.dk;
  kp.dv = a.dv;
  kp.dq_acc = a.dq_acc;
  kp.dq_turn = a.dq_turn;
  kp.ticket = a.ticket;
  kp.nq = (pb.Lq + 127) / 128;
  kp.rev = pb.causal;  // later rows see more keys: the light key tiles (the last ones) start the turns
  kp.kv_lens = pb.kv_lens;
  kp.Lq = pb.Lq;
  kp.Lkv = pb.Lkv;
  kp.Hq = pb.Hq;
  kp.Hkv = pb.Hkv;
  kp.G = pb.G;
  kp.causal = pb.causal;
  kp.wl = pb.wl;
  kp.wr = pb.wr;
  kp.Lq_pad = a.Lq_pad;
  kp.dh = pb.d;
  kp.q_seg = pb.q_seg;
  kp.kv_seg = pb.kv_seg;
  kp.seg_qblk = pb.seg_qblk;
  kp.seg_kblk = pb.seg_kblk;
  kp.nqb = (pb.Lq + kSegBlock - 1) / kSegBlock;
  kp.nkb = (pb.Lkv + kSegBlock - 1) / kSegBlock;
  kp.scale = pb.scale;
  kp.scale_log2 = pb.scale * kLog2e;
  kp.status = st;

  // both passes read Q/dO and K/V in boxes of 64 columns x 128 rows
  CUtensorMap tk, tv, tq128, tdo128;
  if (!make_bshd_tmap(&tq128, a.q, elem, pb.B, pb.Lq, pb.Hq, pb.d, 64, 128) ||
      !make_bshd_tmap(&tdo128, a.dout, elem, pb.B, pb.Lq, pb.Hq, pb.d, 64, 128) ||
      !make_bshd_tmap(&tk, a.k, elem, pb.B, pb.Lkv, pb.Hkv, pb.d, 64, 128) ||
      !make_bshd_tmap(&tv, a.v, elem, pb.B, pb.Lkv, pb.Hkv, pb.d, 64, 128))
    return cudaErrorInvalidValue;
  // dK/dV pass (both variants)
  {
    kp.n_tiles = (pb.Lkv + 127) / 128;
    kp.n_pairs = pb.B * pb.Hkv;
    kp.pair_group = l2_pair_group(2l * pb.G * pb.Lq * D * 2, kp.n_pairs, 1);
    dim3 grid(kp.n_pairs * kp.n_tiles);
    // dK and dV leave through TMA stores of the same 64-column x 128-row boxes
    CUtensorMap tdk, tdv;
    if (!make_bshd_tmap(&tdk, a.dk, elem, pb.B, pb.Lkv, pb.Hkv, pb.d, 64, 128) ||
        !make_bshd_tmap(&tdv, a.dv, elem, pb.B, pb.Lkv, pb.Hkv, pb.d, 64, 128))
      return cudaErrorInvalidValue;
    if (a.deterministic != 1) {
      if (a.deterministic == 2) {  // turn counters and the work-item ticket start at zero
        e = cudaMemsetAsync(a.dq_turn, 0, a.turn_bytes, stream);
        if (e != cudaSuccess) return e;
      }
      return launch_single_pass<D>(tq128, tk, tv, tdo128, tdk, tdv, kp, grid,
                                   static_cast<long>(pb.B) * pb.Lq * pb.Hq * pb.d, pb.f16 != 0, a.deterministic == 2,
                                   stream);
    }
    e = dispatch_build<DkdvLaunch, D>(pb, tq128, tk, tv, tdo128, tdk, tdv, kp, grid, stream);
    if (e != cudaSuccess) return e;
  }
  // dQ pass
  {
    kp.n_tiles = (pb.Lq + 127) / 128;
    kp.n_pairs = pb.B * pb.Hq;
    kp.pair_group = l2_pair_group(2l * pb.Lkv * D * 2, kp.n_pairs, pb.G);
    dim3 grid(kp.n_pairs * kp.n_tiles);
    CUtensorMap tdq;
    if (!make_bshd_tmap(&tdq, a.dq, elem, pb.B, pb.Lq, pb.Hq, pb.d, 64, 128)) return cudaErrorInvalidValue;
    return dispatch_build<DqLaunch, D>(pb, tq128, tk, tv, tdo128, tdq, kp, grid, stream);
  }
}

}  // namespace

cudaError_t launch_bwd_16(const BwdArgs& a, DeviceStatus* st, cudaStream_t s) {
  if (a.pb.d == 256) return launch_bwd_d256(a, st, s);
  return a.pb.d <= 64 ? launch_bwd_d<64>(a, st, s) : launch_bwd_d<128>(a, st, s);  // head_dim 32 runs as 64
}

}  // namespace attn
