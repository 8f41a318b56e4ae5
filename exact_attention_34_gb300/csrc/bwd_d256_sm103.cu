// Backward attention at head_dim 256 (bf16 or fp16), deterministic, on the
// sm_103a tensor cores.
//
// Method as in the head_dim 64/128 backward (probjax "Attention performance",
// "When to use which": the split backward with the LSE and delta = rowsum(dO O)
// residuals): with P = 2^(S scale log2e - LSE log2e), dS = P (dP - delta),
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
// At d = 256 one 128-row accumulator pair (dK and dV, 512 TMEM columns) leaves
// no room for the score tiles, and one K/V/Q/dO tile set is 256 KB of shared
// memory, so the work is split three ways, each kernel owning one output:
//   dv kernel  per 128 keys:    S^T = K Q^T,  dV += P^T dO             (2 GEMMs)
//   dk kernel  per 128 keys:    S^T, dP^T = V dO^T,  dK += dS^T Q      (3 GEMMs)
//   dq kernel  per 128 queries: S = Q K^T, dP = dO V^T,  dQ += dS K    (3 GEMMs)
// Steps are 64 wide (64 queries for the key-stationary kernels, 64 keys for
// dq); score tiles are double-buffered in TMEM and the 256-column accumulator
// sits at columns [256, 512).  Warps 0-7 compute P / dS (thread = TMEM lane =
// the stationary row; warps w and w + 4 share a lane quadrant and take 32
// columns of the step each), warp 8 loads with TMA, warp 9 issues the MMAs.  Every
// output element is accumulated in a fixed order, so results repeat bitwise.
#include "bwd_common.cuh"

namespace attn {
namespace bwd {
namespace {

constexpr int kD = 256;
constexpr int kRows = 128;  // stationary rows per CTA (= TMEM lanes)
constexpr int kStep = 64;   // streamed rows per step
constexpr int kBigBox = kRows * 64 * 2;    // 16 KB: 128 rows x 64 columns
constexpr int kSmallBox = kStep * 64 * 2;  // 8 KB: 64 rows x 64 columns
constexpr int kBig = 4 * kBigBox;          // 64 KB: a stationary 128 x 256 tile
constexpr int kSmall = 4 * kSmallBox;      // 32 KB: a streamed 64 x 256 tile
constexpr int kThreads = 320;  // warps 0-7 P/dS (two column halves), 8 TMA, 9 MMA

// S(buf) = A B^T over d: A a stationary 128 x 256 tile, B a streamed 64 x 256
// tile, both K-major; 16 k-steps, each 64-column block of d its own box.
__device__ __forceinline__ void issue_scores(uint32_t d_tmem, SDesc a, SDesc b, uint32_t b_base, uint32_t idesc) {
#pragma unroll
  for (int k = 0; k < kD / 16; ++k) {
    const uint32_t ao = ((k >> 2) * kBigBox + (k & 3) * 32) >> 4;
    const uint32_t bo = (b_base + (k >> 2) * kSmallBox + (k & 3) * 32) >> 4;
    mma_ss_d(d_tmem, a, ao, b, bo, idesc, k > 0);
  }
}

// ACC (+)= A X: A a 128 x 64 16-bit tile in TMEM, X a streamed 64 x 256 tile
// read MN-major (64-column atoms 8 KB apart); 4 k-steps of 16.  A's columns
// 32h..32h+31 (written by softmax warpgroup h) sit packed in TMEM columns
// [32h, 32h + 16) of the score buffer, so k-step k reads 32 (k/2) + 8 (k%2).
__device__ __forceinline__ void issue_accumulate(uint32_t acc_tmem, uint32_t a_tmem, SDesc x, uint32_t x_base,
                                                 uint32_t idesc, bool acc) {
#pragma unroll
  for (int k = 0; k < kStep / 16; ++k)
    mma_ts_d(acc_tmem, a_tmem + (k >> 1) * 32 + (k & 1) * 8, x, (x_base + k * 2048) >> 4, idesc,
             (acc || k > 0) ? 1u : 0u);
}

// Pack 32 fp32 values (columns [32 wg, 32 wg + 32) of a step) to 16-bit and
// write them over the first 16 of the TMEM columns they were read from, so
// the two warpgroups never write where the other still reads.
template <bool kF16>
__device__ __forceinline__ void store_operand32(uint32_t taddr, const float (&v)[32]) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack2<kF16>(v[2 * i], v[2 * i + 1]);
  tmem_st16(taddr, pk);
}

// ---------------------------------------------------------------------------
// dQ: CTA = 128 queries of one (batch, head), 64-key steps.
// TMEM: S [0,64) [64,128), dP [128,192) [192,256), dQ [256,512).
// smem: Q, dO (64 KB each, resident), K ring 2 x 32 KB (a K tile serves S and
// then dQ), one 32 KB V slot (V serves dP only).  MMA issue order:
//   S(0) dP(0) S(1) dP(1) | dQ(0) dP(2) S(2) | dQ(1) dP(3) S(3) | ...
// dP(j+2) runs while K(j+2) is loaded into the slot dQ(j) released.
// ---------------------------------------------------------------------------
struct DqCfg256 {
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kBig;
  static constexpr int kOffK = 2 * kBig;
  static constexpr int kOffV = kOffK + 2 * kSmall;
  static constexpr int kOffBars = kOffV + kSmall;
  static constexpr int kNumBars = 12;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;
};

template <bool kF16, bool kSeg>
__global__ void __launch_bounds__(kThreads, 1)
    dq256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_out, const BwdKParams p) {
  using C = DqCfg256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDO = smem + C::kOffDO;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* q_full = bars;        // Q and dO landed
  uint64_t* full_k = bars + 1;    // [2]
  uint64_t* empty_k = bars + 3;   // [2] dQ(j) done with K(j)
  uint64_t* full_v = bars + 5;
  uint64_t* empty_v = bars + 6;   // dP(j) done with V(j)
  uint64_t* sd_full = bars + 7;   // [2] S(j) and dP(j) computed, per buffer
  uint64_t* ds_full = bars + 9;   // [2] dS(j) written, per buffer (256 arrivals)
  uint64_t* acc_full = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const TileCoord tc = grouped_tile(blockIdx.x, p.n_pairs, p.n_tiles, p.pair_group);
  const int qt = p.causal ? p.n_tiles - 1 - tc.rank : tc.rank;
  const int q0 = qt * kRows, h = tc.pair % p.Hq, b = tc.pair / p.Hq;
  const int hk = h / p.G;
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);
  // key steps [t0, t0 + T)
  int k_lo = key_span(q0, p.Lq, kvl, p.wl, p.wr).lo;
  int k_hi = key_span(min(q0 + kRows - 1, p.Lq - 1), p.Lq, kvl, p.wl, p.wr).hi;
  const int4 qrec = (kSeg && p.seg_qblk != nullptr) ? seg_block(p.seg_qblk, b, p.nqb, q0 / kSegBlock)
                                                    : make_int4(0, -1, 0, 0);
  if (kSeg && p.seg_qblk != nullptr) {
    k_lo = max(k_lo, qrec.z);
    k_hi = min(k_hi, qrec.w);
  }
  const int t0 = k_hi > k_lo ? k_lo / kStep : 0;
  const int T = k_hi > k_lo ? (k_hi + kStep - 1) / kStep - t0 : 0;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::kNumBars; ++i) mbar_init(&bars[i], (i == 9 || i == 10) ? 256 : 1);
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
  griddep_launch_dependents();  // the next kernel waits for this grid before it reads anything

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && T > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, 2 * kBig);
      for (int c = 0; c < 4; ++c) {
        tma_load_4d(sQ + c * kBigBox, &tm_q, q_full, c * 64, q0, h, b);
        tma_load_4d(sDO + c * kBigBox, &tm_do, q_full, c * 64, q0, h, b);
      }
      auto load_k = [&](int u) -> bool {
        const int st = u & 1;
        if (u >= 2 && !mbar_wait(&empty_k[st], ((u >> 1) - 1) & 1, abort_flag, p.status, 110)) return false;
        mbar_arrive_expect_tx(&full_k[st], kSmall);
        for (int c = 0; c < 4; ++c)
          tma_load_4d(sK + st * kSmall + c * kSmallBox, &tm_k, &full_k[st], c * 64, (t0 + u) * kStep, hk, b);
        return true;
      };
      auto load_v = [&](int u) -> bool {
        if (u >= 1 && !mbar_wait(empty_v, (u - 1) & 1, abort_flag, p.status, 111)) return false;
        mbar_arrive_expect_tx(full_v, kSmall);
        for (int c = 0; c < 4; ++c)
          tma_load_4d(sV + c * kSmallBox, &tm_v, full_v, c * 64, (t0 + u) * kStep, hk, b);
        return true;
      };
      // K(0) V(0) K(1) V(1), then V(u) before K(u): V(u) is free once dP(u-1)
      // completed, K(u) only once dQ(u-2) did, which comes later
      bool ok = load_k(0) && load_v(0);
      if (ok && T > 1) ok = load_k(1) && load_v(1);
      for (int u = 2; u < T && ok; ++u) ok = load_v(u) && load_k(u);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_s = idesc_16_f32<kF16>(kRows, kStep, 0, 0);
      constexpr uint32_t idesc_acc = idesc_16_f32<kF16>(kRows, kD, 0, 1);
      const SDesc dq = sdesc_split(smem_u32(sQ), 16, 1024);
      const SDesc ddo = sdesc_split(smem_u32(sDO), 16, 1024);
      const SDesc dk = sdesc_split(smem_u32(sK), 16, 1024);
      const SDesc dv = sdesc_split(smem_u32(sV), 16, 1024);
      const SDesc dk_mn = sdesc_split(smem_u32(sK), kSmallBox, 1024);
      auto issue_s = [&](int buf, int st) { issue_scores(tbase + buf * kStep, dq, dk, st * kSmall, idesc_s); };
      auto issue_dp = [&](int buf) { issue_scores(tbase + 128 + buf * kStep, ddo, dv, 0, idesc_s); };
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, 112);
      for (int u = 0; u < 2 && u < T && ok; ++u) {
        ok = mbar_wait(&full_k[u], 0, abort_flag, p.status, 113);
        if (!ok) break;
        tc_fence_after();
        issue_s(u, u);
        ok = mbar_wait(full_v, u & 1, abort_flag, p.status, 114);
        if (!ok) break;
        tc_fence_after();
        issue_dp(u);
        mma_commit(empty_v);
        mma_commit(&sd_full[u]);
      }
      for (int j = 0; j < T && ok; ++j) {
        const int buf = j & 1;
        ok = mbar_wait(&ds_full[buf], (j >> 1) & 1, abort_flag, p.status, 115);
        if (!ok) break;
        tc_fence_after();
        issue_accumulate(tbase + 256, tbase + buf * kStep, dk_mn, buf * kSmall, idesc_acc, j > 0);
        mma_commit(&empty_k[buf]);
        if (j == T - 1) mma_commit(acc_full);
        if (j + 2 < T) {
          // dP(j+2) then S(j+2) into buffer j&1: after dQ(j) has read dS(j)
          // from it (one thread's tcgen05.mma execute in issue order)
          ok = mbar_wait(full_v, j & 1, abort_flag, p.status, 116);
          if (!ok) break;
          tc_fence_after();
          issue_dp(buf);
          mma_commit(empty_v);
          ok = mbar_wait(&full_k[buf], ((j + 2) >> 1) & 1, abort_flag, p.status, 117);
          if (!ok) break;
          tc_fence_after();
          issue_s(buf, buf);
          mma_commit(&sd_full[buf]);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ dS (thread = query row)
    const int wg = warp >> 2, wq = warp & 3;
    const int i = q0 + wq * 32 + lane;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(wq * 32) << 16);
    const size_t srow = (static_cast<size_t>(b) * p.Hq + h) * p.Lq_pad + i;  // i < Lq_pad always
    const float l2 = p.lse2[srow];
    const float dl = p.delta[srow];
    Span ks = key_span(i, p.Lq, kvl, p.wl, p.wr);
    if (i >= p.Lq) ks.lo = ks.hi = 0;
    const float sl2 = p.scale_log2;
    const int my_seg = (kSeg && i < p.Lq) ? __ldg(p.q_seg + static_cast<size_t>(b) * p.Lq + i) : 0;
    const int32_t* kid = kSeg ? p.kv_seg + static_cast<size_t>(b) * p.Lkv : nullptr;
    const bool kid_vec = kSeg && ((static_cast<size_t>(b) * p.Lkv) & 3) == 0;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int buf = j & 1;
      const int col0 = (t0 + j) * kStep + 32 * wg;  // this warpgroup's 32 keys
      uint32_t sg = ~0u;
      const bool seg_all = kSeg && p.seg_kblk != nullptr &&
                           seg_same_single_id(qrec, seg_block(p.seg_kblk, b, p.nkb, col0 / kSegBlock));
      if (kSeg && !seg_all) sg = segment_bits32(kid, col0, kvl, kid_vec, my_seg);
      ok = __all_sync(0xffffffffu, mbar_wait(&sd_full[buf], (j >> 1) & 1, abort_flag, p.status, 118));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_col = t_lane + buf * kStep + 32 * wg, dp_col = t_lane + 128 + buf * kStep + 32 * wg;
      const bool edge = col0 < ks.lo || col0 + 32 > ks.hi;
      uint32_t sa[32], da[32];
      tmem_ld32_pair(s_col, dp_col, sa, da);
      float ds[32];
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(-l2, -l2), dl2 = f2_pack(dl, dl);
#pragma unroll
      for (int c = 0; c < 32; c += 2) {  // two columns per paired fp32 instruction
        float t[2], pv[2];
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sa[c]), __uint_as_float(sa[c + 1])), sl2x2, nl2), t[0], t[1]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = col0 + c + e;
          pv[e] = ex2_approx(t[e]);
          if (edge && (key < ks.lo || key >= ks.hi)) pv[e] = 0.f;
          if (kSeg && !((sg >> (c + e)) & 1u)) pv[e] = 0.f;
        }
        f2_unpack(f2_mul(f2_pack(pv[0], pv[1]),
                         f2_sub(f2_pack(__uint_as_float(da[c]), __uint_as_float(da[c + 1])), dl2)),
                  ds[c], ds[c + 1]);
      }
      store_operand32<kF16>(s_col, ds);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ds_full[buf]);
    }
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, p.status, 119));
    // dQ goes through the Q tile, idle once every MMA has completed, and out
    // with TMA stores that clip the rows past Lq; warpgroup wg stages
    // columns [128 wg, 128 wg + 128)
    if (ok) {
      tc_fence_after();
      stage_row16<128, kF16>(t_lane + 256 + 128 * wg, sQ, wq * 32 + lane, p.scale, T == 0, 128 * wg);
      fence_proxy_async_smem();
    }
    named_barrier_sync(1, 256);  // every P/dS thread gets here (a failed wait only skips work)
    if (threadIdx.x == 0 && *abort_flag == 0) {
#pragma unroll
      for (int c = 0; c < kD / 64; ++c) tma_store_4d(&tm_out, sQ + c * kBigBox, c * 64, q0, h, b);
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
  // launched to overlap the dK pass (it reads nothing that pass writes): one
  // CTA waits for it, so this grid completes after it
  if (blockIdx.x == gridDim.x - 1) griddep_wait();
}

// ---------------------------------------------------------------------------
// dV (kDK = false) and dK (kDK = true): CTA = 128 keys of one (batch, KV head),
// steps of 64 queries over the G query heads of the group.
// TMEM: S^T [0,64) [64,128), dP^T [128,192) [192,256) (dK only), ACC [256,512).
// smem, dV: K, Q ring 2 x 32 KB (Q serves S^T only), dO ring 2 x 32 KB (dO
//           serves dV); the softmax threads read the step's lse2 from global
//           memory before waiting for S^T (a dO slot frees too late to carry it);
//       dK: K, V, Q ring 2 x 32 KB with the step's lse2 and delta (Q serves
//           S^T and then dK), one 32 KB dO slot (dO serves dP^T only).
// MMA issue order, dV: S(0) S(1) | dV(0) S(2) | dV(1) S(3) | ...
//                  dK: S(0) dP(0) S(1) dP(1) | dK(0) dP(2) S(2) | dK(1) ...
// ---------------------------------------------------------------------------
template <bool kDK>
struct KeyCfg256 {
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kBig;  // dK only
  static constexpr int kOffQ = kDK ? 2 * kBig : kBig;
  static constexpr int kOffDO = kOffQ + 2 * kSmall;
  static constexpr int kDOSlots = kDK ? 1 : 2;
  static constexpr int kOffStat = kOffDO + kDOSlots * kSmall;  // 2 slots x (lse2[64], delta[64])
  static constexpr int kOffBars = kOffStat + 2 * 2 * kStep * 4;
  static constexpr int kNumBars = 14;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;
};

template <bool kDK, bool kF16, bool kSeg>
__global__ void __launch_bounds__(kThreads, 1)
    key256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_out,
                  const BwdKParams p) {
  using C = KeyCfg256<kDK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDO = smem + C::kOffDO;
  float* sStat = reinterpret_cast<float*>(smem + C::kOffStat);  // slot s: lse2 at s*128, delta at s*128 + 64
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* kv_full = bars;
  uint64_t* full_q = bars + 1;    // [2]
  uint64_t* empty_q = bars + 3;   // [2]
  uint64_t* full_do = bars + 5;   // [2] (dK: [0] only)
  uint64_t* empty_do = bars + 7;  // [2] (dK: [0] only)
  uint64_t* st_full = bars + 9;   // [2] scores of step t computed, per buffer
  uint64_t* p_full = bars + 11;   // [2] P^T / dS^T of step t written (256 arrivals)
  uint64_t* acc_full = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const TileCoord tc = grouped_tile(blockIdx.x, p.n_pairs, p.n_tiles, p.pair_group);
  const int j0 = tc.rank * kRows, hk = tc.pair % p.Hkv, b = tc.pair / p.Hkv;
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);
  const int4 krec = (kSeg && p.seg_kblk != nullptr) ? seg_block(p.seg_kblk, b, p.nkb, j0 / kSegBlock)
                                                    : make_int4(0, -1, 0, 0);
  // query steps of each head: from the first row that sees key j0 to the last
  // row that sees the tile's last valid key
  int i_begin = 0, sph = 0;
  if (j0 < kvl) {
    int q_lo = query_span(j0, p.Lq, kvl, p.wl, p.wr).lo;
    int q_hi = query_span(min(j0 + kRows, kvl) - 1, p.Lq, kvl, p.wl, p.wr).hi;
    if (kSeg && p.seg_kblk != nullptr) {
      q_lo = max(q_lo, krec.z);
      q_hi = min(q_hi, krec.w);
    }
    if (q_hi > q_lo) {
      i_begin = q_lo / kStep;
      sph = (q_hi + kStep - 1) / kStep - i_begin;
    }
  }
  const int T = sph * p.G;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::kNumBars; ++i) mbar_init(&bars[i], (i == 11 || i == 12) ? 256 : 1);
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
  // The dV pass runs first after the preprocess and waits for it here
  // (delta and lse2); the dK pass, launched to overlap the dV pass, starts
  // only once every dV CTA got past that wait, so it reads them at once.
  if (!kDK) griddep_wait();
  griddep_launch_dependents();

  auto step_head = [&](int t) { return hk * p.G + t / sph; };
  auto step_q0 = [&](int t) { return (i_begin + t % sph) * kStep; };
  auto stat_row = [&](int t) { return (static_cast<size_t>(b) * p.Hq + step_head(t)) * p.Lq_pad + step_q0(t); };

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && T > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      if (kDK) tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(kv_full, kDK ? 2 * kBig : kBig);
      for (int c = 0; c < 4; ++c) {
        tma_load_4d(sK + c * kBigBox, &tm_k, kv_full, c * 64, j0, hk, b);
        if (kDK) tma_load_4d(sV + c * kBigBox, &tm_v, kv_full, c * 64, j0, hk, b);
      }
      // Q(u) [+ lse2, delta for dK] into slot u&1, free once S^T(u-2) (dV) or
      // dK(u-2) (dK) completed
      auto load_q = [&](int u) -> bool {
        const int st = u & 1;
        if (u >= 2 && !mbar_wait(&empty_q[st], ((u >> 1) - 1) & 1, abort_flag, p.status, 120)) return false;
        mbar_arrive_expect_tx(&full_q[st], kSmall + (kDK ? 2 * kStep * 4 : 0));
        for (int c = 0; c < 4; ++c)
          tma_load_4d(sQ + st * kSmall + c * kSmallBox, &tm_q, &full_q[st], c * 64, step_q0(u), step_head(u), b);
        if (kDK) {
          bulk_load(sStat + st * 2 * kStep, p.lse2 + stat_row(u), kStep * 4, &full_q[st]);
          bulk_load(sStat + st * 2 * kStep + kStep, p.delta + stat_row(u), kStep * 4, &full_q[st]);
        }
        return true;
      };
      // dO(u): dV keeps two slots, free once dV(u-2) completed; dK keeps one,
      // free once dP^T(u-1) completed
      auto load_do = [&](int u) -> bool {
        const int st = kDK ? 0 : (u & 1);
        const int use = kDK ? u : (u >> 1);
        if (use >= 1 && !mbar_wait(&empty_do[st], (use - 1) & 1, abort_flag, p.status, 121)) return false;
        mbar_arrive_expect_tx(&full_do[st], kSmall);
        for (int c = 0; c < 4; ++c)
          tma_load_4d(sDO + st * kSmall + c * kSmallBox, &tm_do, &full_do[st], c * 64, step_q0(u), step_head(u), b);
        return true;
      };
      bool ok = load_q(0) && load_do(0);
      if (ok && T > 1) ok = load_q(1) && load_do(1);
      for (int u = 2; u < T && ok; ++u) ok = kDK ? (load_do(u) && load_q(u)) : (load_q(u) && load_do(u));
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_s = idesc_16_f32<kF16>(kRows, kStep, 0, 0);
      constexpr uint32_t idesc_acc = idesc_16_f32<kF16>(kRows, kD, 0, 1);
      const SDesc dk = sdesc_split(smem_u32(sK), 16, 1024);
      const SDesc dv = sdesc_split(smem_u32(sV), 16, 1024);
      const SDesc dq = sdesc_split(smem_u32(sQ), 16, 1024);
      const SDesc ddo = sdesc_split(smem_u32(sDO), 16, 1024);
      const SDesc dq_mn = sdesc_split(smem_u32(sQ), kSmallBox, 1024);
      const SDesc ddo_mn = sdesc_split(smem_u32(sDO), kSmallBox, 1024);
      auto issue_st = [&](int buf) { issue_scores(tbase + buf * kStep, dk, dq, buf * kSmall, idesc_s); };
      auto issue_dpt = [&](int buf) { issue_scores(tbase + 128 + buf * kStep, dv, ddo, 0, idesc_s); };
      bool ok = mbar_wait(kv_full, 0, abort_flag, p.status, 122);
      for (int u = 0; u < 2 && u < T && ok; ++u) {
        ok = mbar_wait(&full_q[u], 0, abort_flag, p.status, 123);
        if (!ok) break;
        tc_fence_after();
        issue_st(u);
        if (kDK) {
          ok = mbar_wait(&full_do[0], u & 1, abort_flag, p.status, 124);
          if (!ok) break;
          tc_fence_after();
          issue_dpt(u);
          mma_commit(&empty_do[0]);
        } else {
          mma_commit(&empty_q[u]);
        }
        mma_commit(&st_full[u]);
      }
      for (int t = 0; t < T && ok; ++t) {
        const int buf = t & 1;
        ok = mbar_wait(&p_full[buf], (t >> 1) & 1, abort_flag, p.status, 125);
        if (!ok) break;
        if (!kDK) {
          ok = mbar_wait(&full_do[buf], (t >> 1) & 1, abort_flag, p.status, 126);
          if (!ok) break;
        }
        tc_fence_after();
        if (kDK) {
          issue_accumulate(tbase + 256, tbase + buf * kStep, dq_mn, buf * kSmall, idesc_acc, t > 0);
          mma_commit(&empty_q[buf]);
        } else {
          issue_accumulate(tbase + 256, tbase + buf * kStep, ddo_mn, buf * kSmall, idesc_acc, t > 0);
          mma_commit(&empty_do[buf]);
        }
        if (t == T - 1) mma_commit(acc_full);
        if (t + 2 < T) {
          // the scores of step t+2 go into buffer t&1 after the accumulation
          // of step t has read its operand from there (issue order)
          if (kDK) {
            ok = mbar_wait(&full_do[0], t & 1, abort_flag, p.status, 127);
            if (!ok) break;
            tc_fence_after();
            issue_dpt(buf);
            mma_commit(&empty_do[0]);
          }
          ok = mbar_wait(&full_q[buf], ((t + 2) >> 1) & 1, abort_flag, p.status, 128);
          if (!ok) break;
          tc_fence_after();
          issue_st(buf);
          if (!kDK) mma_commit(&empty_q[buf]);
          mma_commit(&st_full[buf]);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ P^T / dS^T (thread = key row)
    const int wg = warp >> 2, wq = warp & 3;
    const int j = j0 + wq * 32 + lane;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(wq * 32) << 16);
    const bool key_ok = j < kvl;
    const Span qs = key_ok ? query_span(j, p.Lq, kvl, p.wl, p.wr) : Span{0, 0};
    const int my_seg = (kSeg && j < p.Lkv) ? __ldg(p.kv_seg + static_cast<size_t>(b) * p.Lkv + j) : 0;
    const int32_t* qid = kSeg ? p.q_seg + static_cast<size_t>(b) * p.Lq : nullptr;
    const bool qid_vec = kSeg && ((static_cast<size_t>(b) * p.Lq) & 3) == 0;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int buf = t & 1;
      const int q0 = step_q0(t) + 32 * wg;  // this warpgroup's 32 queries
      // dV reads the 32 lse2 values from global memory (the same for every
      // thread: L1 broadcasts); dK's lse2 and delta arrive with Q
      float4 lg[8];
      if (!kDK) {
        const float4* src = reinterpret_cast<const float4*>(p.lse2 + stat_row(t) + 32 * wg);
#pragma unroll
        for (int i = 0; i < 8; ++i) lg[i] = __ldg(src + i);
      }
      uint32_t sg = ~0u;
      const bool seg_all = kSeg && p.seg_qblk != nullptr &&
                           seg_same_single_id(seg_block(p.seg_qblk, b, p.nqb, q0 / kSegBlock), krec);
      if (kSeg && !seg_all) sg = segment_bits32(qid, q0, p.Lq, qid_vec, my_seg);
      if (kDK) {
        ok = __all_sync(0xffffffffu, mbar_wait(&full_q[buf], (t >> 1) & 1, abort_flag, p.status, 129));
        if (!ok) break;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&st_full[buf], (t >> 1) & 1, abort_flag, p.status, 130));
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = sStat + buf * 2 * kStep + 32 * wg;
      const float* dlt = lse2 + kStep;
      const uint32_t s_col = t_lane + buf * kStep + 32 * wg, dp_col = t_lane + 128 + buf * kStep + 32 * wg;
      const bool edge = !key_ok || q0 < qs.lo || q0 + 32 > qs.hi;
      uint32_t sa[32], da[32];
      if (kDK) {
        tmem_ld32_pair(s_col, dp_col, sa, da);
      } else {
        tmem_ld32(s_col, sa);
      }
      float val[32];
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 l4 = kDK ? *reinterpret_cast<const float4*>(lse2 + 4 * c4) : lg[c4];
        float4 d4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kDK) d4 = *reinterpret_cast<const float4*>(dlt + 4 * c4);
        const float nlv[4] = {-l4.x, -l4.y, -l4.z, -l4.w};
        const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int e = 0; e < 4; e += 2) {  // two columns per paired fp32 instruction
          const int c = 4 * c4 + e;
          float t[2], pv[2];
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sa[c]), __uint_as_float(sa[c + 1])), f2_pack(sl2, sl2),
                           f2_pack(nlv[e], nlv[e + 1])),
                    t[0], t[1]);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int q = q0 + c + u;
            pv[u] = ex2_approx(t[u]);
            if (edge && (!key_ok || q < qs.lo || q >= qs.hi)) pv[u] = 0.f;
            if (kSeg && !((sg >> (c + u)) & 1u)) pv[u] = 0.f;
          }
          if (kDK) {
            f2_unpack(f2_mul(f2_pack(pv[0], pv[1]), f2_sub(f2_pack(__uint_as_float(da[c]), __uint_as_float(da[c + 1])),
                                                            f2_pack(dv4[e], dv4[e + 1]))),
                      val[c], val[c + 1]);
          } else {
            val[c] = pv[0];
            val[c + 1] = pv[1];
          }
        }
      }
      store_operand32<kF16>(s_col, val);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[buf]);
    }
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, p.status, 131));
    // dK or dV goes through the K tile, idle once every MMA has completed,
    // and out with TMA stores that clip the rows past Lkv; warpgroup wg
    // stages columns [128 wg, 128 wg + 128)
    if (ok) {
      tc_fence_after();
      stage_row16<128, kF16>(t_lane + 256 + 128 * wg, sK, wq * 32 + lane, kDK ? p.scale : 1.0f, T == 0, 128 * wg);
      fence_proxy_async_smem();
    }
    named_barrier_sync(1, 256);  // every P/dS thread gets here (a failed wait only skips work)
    if (threadIdx.x == 0 && *abort_flag == 0) {
#pragma unroll
      for (int c = 0; c < kD / 64; ++c) tma_store_4d(&tm_out, sK + c * kBigBox, c * 64, j0, hk, b);
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
  // launched to overlap the dV pass: one CTA waits for it, so this grid
  // completes after it
  if (kDK && blockIdx.x == gridDim.x - 1) griddep_wait();
}

template <bool kF16, bool kSeg>
cudaError_t launch_dq256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                         const CUtensorMap& tout, const BwdKParams& kp, dim3 grid, cudaStream_t stream) {
  cudaError_t e = ensure_dynamic_smem<dq256_kernel<kF16, kSeg>>(DqCfg256::kSmemBytes);
  if (e != cudaSuccess) return e;
  KernelTimer kt("bwd_dq", stream);
  return launch_overlapping(dq256_kernel<kF16, kSeg>, grid, kThreads, DqCfg256::kSmemBytes, stream, tq, tk, tv, tdo,
                            tout, kp);
}

template <bool kDK, bool kF16, bool kSeg>
cudaError_t launch_key256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                          const CUtensorMap& tout, const BwdKParams& kp, dim3 grid, cudaStream_t stream) {
  using C = KeyCfg256<kDK>;
  cudaError_t e = ensure_dynamic_smem<key256_kernel<kDK, kF16, kSeg>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  KernelTimer kt(kDK ? "bwd_dk" : "bwd_dv", stream);
  return launch_overlapping(key256_kernel<kDK, kF16, kSeg>, grid, kThreads, C::kSmemBytes, stream, tq, tk, tv, tdo,
                            tout, kp);
}

template <bool kF16, bool kSeg>
cudaError_t run_bwd256(const BwdArgs& a, BwdKParams kp, cudaStream_t stream) {
  const Problem& pb = a.pb;
  const int elem = kF16 ? kElemF16 : kElemBF16;
  cudaError_t e;
  {  // dV and dK: stationary K/V tiles of 128 rows, streamed Q/dO tiles of 64
    CUtensorMap tq, tdo, tk, tv;
    if (!make_bshd_tmap(&tq, a.q, elem, pb.B, pb.Lq, pb.Hq, kD, 64, kStep) ||
        !make_bshd_tmap(&tdo, a.dout, elem, pb.B, pb.Lq, pb.Hq, kD, 64, kStep) ||
        !make_bshd_tmap(&tk, a.k, elem, pb.B, pb.Lkv, pb.Hkv, kD, 64, kRows) ||
        !make_bshd_tmap(&tv, a.v, elem, pb.B, pb.Lkv, pb.Hkv, kD, 64, kRows))
      return cudaErrorInvalidValue;
    kp.n_tiles = (pb.Lkv + kRows - 1) / kRows;
    kp.n_pairs = pb.B * pb.Hkv;
    kp.pair_group = l2_pair_group(2l * pb.G * pb.Lq * kD * 2, kp.n_pairs, 1);
    // dV and dK leave through TMA stores of 64-column x 128-row boxes
    CUtensorMap tdv, tdk;
    if (!make_bshd_tmap(&tdv, a.dv, elem, pb.B, pb.Lkv, pb.Hkv, kD, 64, kRows) ||
        !make_bshd_tmap(&tdk, a.dk, elem, pb.B, pb.Lkv, pb.Hkv, kD, 64, kRows))
      return cudaErrorInvalidValue;
    const dim3 grid(kp.n_pairs * kp.n_tiles);
    e = launch_key256<false, kF16, kSeg>(tq, tk, tv, tdo, tdv, kp, grid, stream);
    if (e != cudaSuccess) return e;
    e = launch_key256<true, kF16, kSeg>(tq, tk, tv, tdo, tdk, kp, grid, stream);
    if (e != cudaSuccess) return e;
  }
  {  // dQ: stationary Q/dO tiles of 128 rows, streamed K/V tiles of 64
    CUtensorMap tq, tdo, tk, tv;
    if (!make_bshd_tmap(&tq, a.q, elem, pb.B, pb.Lq, pb.Hq, kD, 64, kRows) ||
        !make_bshd_tmap(&tdo, a.dout, elem, pb.B, pb.Lq, pb.Hq, kD, 64, kRows) ||
        !make_bshd_tmap(&tk, a.k, elem, pb.B, pb.Lkv, pb.Hkv, kD, 64, kStep) ||
        !make_bshd_tmap(&tv, a.v, elem, pb.B, pb.Lkv, pb.Hkv, kD, 64, kStep))
      return cudaErrorInvalidValue;
    kp.n_tiles = (pb.Lq + kRows - 1) / kRows;
    kp.n_pairs = pb.B * pb.Hq;
    kp.pair_group = l2_pair_group(2l * pb.Lkv * kD * 2, kp.n_pairs, pb.G);
    CUtensorMap tdq;
    if (!make_bshd_tmap(&tdq, a.dq, elem, pb.B, pb.Lq, pb.Hq, kD, 64, kRows)) return cudaErrorInvalidValue;
    const dim3 grid(kp.n_pairs * kp.n_tiles);
    return launch_dq256<kF16, kSeg>(tq, tk, tv, tdo, tdq, kp, grid, stream);
  }
}

}  // namespace
}  // namespace bwd

// head_dim 256 backward (deterministic at either setting of `deterministic`:
// the three kernels each own one output and accumulate it in a fixed order).
cudaError_t launch_bwd_d256(const BwdArgs& a, DeviceStatus* st, cudaStream_t stream) {
  using namespace bwd;
  const Problem& pb = a.pb;
  PreprocessArgs pa;
  pa.o = a.o;
  pa.dout = a.dout;
  pa.lse = a.lse;
  pa.delta = a.delta;
  pa.lse2 = a.lse2;
  pa.dq_acc = nullptr;
  pa.B = pb.B;
  pa.Lq = pb.Lq;
  pa.Lq_pad = a.Lq_pad;
  pa.Hq = pb.Hq;
  pa.d = kD;
  pa.elem = pb.f16 ? kElemF16 : kElemBF16;
  cudaError_t e = launch_bwd_preprocess(pa, stream);
  if (e != cudaSuccess) return e;
  BwdKParams kp;
  kp.lse2 = a.lse2;
  kp.delta = a.delta;
  kp.dq = a.dq;
  kp.dk = a.dk;
  kp.dv = a.dv;
  kp.dq_acc = nullptr;
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
  kp.dh = kD;
  kp.q_seg = pb.q_seg;
  kp.kv_seg = pb.kv_seg;
  kp.seg_qblk = pb.seg_qblk;
  kp.seg_kblk = pb.seg_kblk;
  kp.nqb = (pb.Lq + kSegBlock - 1) / kSegBlock;
  kp.nkb = (pb.Lkv + kSegBlock - 1) / kSegBlock;
  kp.scale = pb.scale;
  kp.scale_log2 = pb.scale * kLog2e;
  kp.status = st;
  kp.n_tiles = kp.n_pairs = kp.pair_group = 0;
  const bool seg = pb.q_seg != nullptr;
  if (pb.f16) return seg ? run_bwd256<true, true>(a, kp, stream) : run_bwd256<true, false>(a, kp, stream);
  return seg ? run_bwd256<false, true>(a, kp, stream) : run_bwd256<false, false>(a, kp, stream);
}

}  // namespace attn
