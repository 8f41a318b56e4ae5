// Single-pass backward, bf16 or fp16, head_dim 64/128: dK and dV as in the
// two-pass variant, while dQ = scale * dS K is summed over key tiles in a
// float32 buffer that a convert kernel scales and casts to the 16-bit format
// (probjax "Attention performance", section "When to use which", backward
// pass).  Two builds of one kernel:
//
//  * atomic (kOrdered = false): every key tile adds its part of dQ with fp32
//    reductions the moment it has it.  The order of the adds is not fixed, so
//    the result is not bitwise reproducible.
//  * ordered (kOrdered = true): the parts of one 128-row query tile are added
//    in increasing key-tile order.  Each (batch, query head, query tile) has a
//    turn counter; key tile j adds its part only once the counter reads j
//    (its predecessor, key tile j - 1, has added and published), then
//    publishes j + 1.  Every sum then runs in one fixed order and the result
//    repeats bit for bit.  A CTA takes its key tile from a ticket counter when
//    it starts, so the tiles of one head are claimed in increasing order and a
//    CTA only ever waits on a tile that a running (or finished) CTA holds: the
//    lowest unfinished tile never waits, so the waits always end.  Every wait
//    is still bounded (an expired wait reports in the status word).
//
// CTA = (batch, KV head, 128 keys); thread = key row = TMEM lane; 128-query
// steps, every MMA 128 x 128 x 16.  Five GEMMs per step instead of the
// two-pass backward's seven:
//   tensor pipe:  S^T | dP^T | dV += P^T dO | dQ^T = K^T dS^T | dK += dS^T Q | S^T(t+1) | dP^T(t+1) ...
//   softmax:          | P^T  | dS^T        |
//   reduction:                              | dQ^T -> registers -> fp32 adds (overlaps the next step)
// TMEM: dK [0,128) dV [128,256) S^T [256,384) dP^T [384,512); dQ^T reuses the
// dP^T columns once the softmax has read them.  P^T goes back to TMEM (A of
// dV); dS^T goes to 128B-swizzled shared memory, where it is the K-major A of
// dK and the MN-major B of dQ^T.  For head_dim 64 the M = 128 rows of dQ^T
// repeat the 64 head-dim rows (the second A block points at the first) and
// only the first 64 lanes are read out.
//
// The adds into the fp32 dQ buffer (64 KB per step and CTA) run at the L2's
// reduction rate, well below the SM's, so four reduction warps own them: each
// thread copies its head-dim row of dQ^T (128 queries) out of TMEM, releases
// the columns for dP^T(t+1) at once, and then issues its 128 adds while the
// next step's GEMMs and softmax run.  In the ordered build two more warps
// (one for even, one for odd steps) wait for the turn of their step, hand it
// to the reduction warps through a named barrier, wait for the adds to be
// issued, then fence and publish the next turn; the fence (the time until
// 64 KB of adds are performed in L2) runs beside the next step's adds.
//
// Step order: the atomic build walks the G query heads, each over its query
// tiles upwards.  The ordered build visits the G heads of one query tile in a
// row, and its turn order follows the mask:
//  * masks where later rows see more keys (causal): the turns of a query tile
//    go from its last key tile down to key tile 0, key tiles are claimed from
//    the last down, and each walks its query tiles upwards.  Key tile j then
//    reaches a query tile one step after tile j + 1 did, and its first query
//    tile (the diagonal) waits for nobody, so the tiles that start together
//    hardly wait on one another (a tile lags its predecessor only by the part
//    of a turn's latency that exceeds a step);
//  * other masks: turns go from key tile 0 up, key tiles are claimed from the
//    first up, and each walks its query tiles downwards, so neighbouring tiles
//    visit every query tile at the same step index and tile j runs a fixed lag
//    behind tile j - 1.
//
// Warps 0-7 softmax (warpgroup w owns queries [64w, 64w + 64) of the step),
// 8-11 reduction (warp 8 + i reads TMEM lanes [32i, 32i + 32)), 12 TMA
// producer, 13 MMA issuer, 14-15 turn keepers (ordered build; idle otherwise);
// the control warpgroup gives its registers to the other three.
#pragma once
#include "bwd_common.cuh"

namespace attn {
namespace bwd {
namespace {  // each translation unit that includes this builds its own copies

template <int D>
struct DkdvAtomicCfg {
  static constexpr int kBN = 128, kBM = 128;
  static constexpr int kKVBytes = kBN * D * 2;
  static constexpr int kBox = 128 * 128;      // one 64-column box of a 128-row tile
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kOffV = kKVBytes;
  static constexpr int kOffQ = 2 * kKVBytes;  // stage s: Q at s * 2 * kQBytes, dO right after
  static constexpr int kOffDS = kOffQ + kStages * 2 * kQBytes;
  static constexpr int kOffStat = kOffDS + kBN * kBM * 2;
  static constexpr int kOffBars = kOffStat + kStages * 2 * kBM * 4;
  static constexpr int kNumBars = 2 * kStages + 1 + 7;
  // No alignment slack: the dynamic shared window starts right after the
  // 1 KB the system reserves per block, which is 1024-aligned (checked at run
  // time; a misaligned base makes the kernel report and do nothing).  After
  // the barriers: TMEM address, abort flag, claimed work item.
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16;
  static constexpr int kThreads = 512;
  // Registers per thread after the split (launch: 512 x 128).  Each SM
  // sub-partition holds one warp of each warpgroup: 3 x kRegsWork + kRegsCtl
  // must equal 4 x 128.
  static constexpr int kRegsWork = 144, kRegsCtl = 80;
};

// Named barriers of the ordered build (id 0 is __syncthreads): per step
// parity, "turn granted" and "adds issued", each over the four reduction
// warps and that parity's turn keeper.
constexpr int kBarTurn = 1, kBarDone = 3, kBarThreads = 160;
// Named barrier of the epilogue: the eight softmax warps, before the dK/dV
// TMA stores.
constexpr int kBarStore = 5;

// Query tiles [i_begin, i_begin + steps) that see some key of the key tile
// starting at j0 (of a sequence with kvl valid keys): from the first row that
// sees key j0 to the last row that sees the tile's last valid key.  With
// `narrow`, also cut to the rows whose segment blocks may share an id with
// this key block.
__device__ __forceinline__ void key_tile_queries(const BwdKParams& p, int b, int j0, int kvl, bool narrow,
                                                 int& i_begin, int& steps) {
  i_begin = 0;
  steps = 0;
  if (j0 < 0 || j0 >= kvl) return;
  int q_lo = query_span(j0, p.Lq, kvl, p.wl, p.wr).lo;
  int q_hi = query_span(min(j0 + 128, kvl) - 1, p.Lq, kvl, p.wl, p.wr).hi;
  if (narrow) {
    const int4 r = seg_block(p.seg_kblk, b, p.nkb, j0 / kSegBlock);
    q_lo = max(q_lo, r.z);
    q_hi = min(q_hi, r.w);
  }
  if (q_hi > q_lo) {
    i_begin = q_lo / 128;
    steps = (q_hi + 127) / 128 - i_begin;
  }
}

// (query head, query tile) of step t.
struct StepCoord {
  int h, it;
};
template <bool kOrdered>
__device__ __forceinline__ StepCoord step_coord(int t, int hk, int G, int i_begin, int steps_per_head, bool rev) {
  if (kOrdered) return {hk * G + t % G, rev ? i_begin + t / G : i_begin + steps_per_head - 1 - t / G};
  return {hk * G + t / steps_per_head, i_begin + t % steps_per_head};
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Make every write this thread has observed (here: the reduction warps' adds,
// ordered before it by a named barrier) visible GPU-wide, then publish `v`.
__device__ __forceinline__ void publish_gpu(int* p, int v) {
  asm volatile("fence.acq_rel.gpu;\n\tst.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until *turn == want.  Gives up after kWaitTimeoutNs (records the site,
// raises the CTA's abort flag) or at once when the CTA is already aborting.
__device__ __forceinline__ bool wait_turn(const int* turn, int want, volatile int* abort, DeviceStatus* st,
                                          int site) {
  if (ld_acquire_gpu(turn) == want) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_gpu(turn) == want) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      *abort = 1;
      report_timeout(st, site);
      return false;
    }
  }
}

template <int D, bool kLeftBound, bool kF16, bool kSeg, bool kOrdered>
__global__ void __launch_bounds__(512, 1)
    bwd_dkdv_single_pass_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                                const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                                const BwdKParams p) {
  using C = DkdvAtomicCfg<D>;
  constexpr int NS = C::kStages, BM = C::kBM;
  constexpr uint32_t kColS = 256, kColDP = 384;
  constexpr int kSite = kOrdered ? 100 : 70;  // status sites of this build
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // never expected: see kSmemBytes
    if (threadIdx.x == 0) report_status(p.status, 2, kSite + 29);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDS = smem + C::kOffDS;
  float* sStat = reinterpret_cast<float*>(smem + C::kOffStat);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* full = bars;
  uint64_t* empty = bars + NS;
  uint64_t* kv_full = bars + 2 * NS;
  uint64_t* s_ready = kv_full + 1;   // S^T(t) computed
  uint64_t* dp_ready = kv_full + 2;  // dP^T(t) computed
  uint64_t* p_ready = kv_full + 3;   // P^T(t) in TMEM (256 arrivals)
  uint64_t* ds_ready = kv_full + 4;  // dS^T(t) in shared memory (256 arrivals)
  uint64_t* dq_ready = kv_full + 5;  // dQ^T(t) computed
  uint64_t* dq_free = kv_full + 6;   // dQ^T(t) copied out of TMEM (128 arrivals)
  uint64_t* acc_full = kv_full + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    // ordered: the key tile comes from the ticket counter, so tiles are
    // claimed (by running CTAs) in the order the turns go
    if (kOrdered) *item_slot = atomicAdd(p.ticket, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(kv_full, 1);
    mbar_init(s_ready, 1);
    mbar_init(dp_ready, 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(dq_ready, 1);
    mbar_init(dq_free, 128);
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // the atomic build is launched to overlap the preprocess: the zeroed dQ
  // buffer, delta and lse2 are complete from here on (the ordered build
  // follows a memset and starts after it)
  griddep_wait();
  griddep_launch_dependents();
  static_assert(3 * C::kRegsWork + C::kRegsCtl == 4 * 128, "register split must match the launch allocation");

  const int linear = kOrdered ? *item_slot : static_cast<int>(blockIdx.x);
  const bool rev = kOrdered && p.rev != 0;
  const TileCoord tc = grouped_tile(linear, p.n_pairs, p.n_tiles, p.pair_group);
  // claimed in rank order; with reversed turns the last key tile has rank 0
  const int tile = rev ? p.n_tiles - 1 - tc.rank : tc.rank;
  const int j0 = tile * C::kBN, hk = tc.pair % p.Hkv, b = tc.pair / p.Hkv;
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);
  // The ordered build keeps each key tile's query range a position span (no
  // segment-block narrowing), so the key tiles that add into one query tile
  // are consecutive and a tile's predecessor is the tile before it.
  const bool narrow = kSeg && !kOrdered && p.seg_kblk != nullptr;
  int i_begin, steps_per_head;
  key_tile_queries(p, b, j0, kvl, narrow, i_begin, steps_per_head);
  const int T = steps_per_head * p.G;

  if (warp >= 12) {
    setmaxnreg_dec<C::kRegsCtl>();
    if (warp == 12 && lane == 0 && T > 0) {
      // ---------------------------------------------------------------- TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(kv_full, 2 * C::kKVBytes);
      for (int h = 0; h < D / 64; ++h) {
        tma_load_4d(sK + h * C::kBox, &tm_k, kv_full, h * 64, j0, hk, b);
        tma_load_4d(sV + h * C::kBox, &tm_v, kv_full, h * 64, j0, hk, b);
      }
      for (int t = 0; t < T; ++t) {
        const int s = t % NS, r = t / NS;
        if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, abort_flag, p.status, kSite + 1)) break;
        const StepCoord sc = step_coord<kOrdered>(t, hk, p.G, i_begin, steps_per_head, rev);
        const int q0 = sc.it * BM;
        mbar_arrive_expect_tx(&full[s], 2 * C::kQBytes + 2 * BM * 4);
        uint8_t* q_dst = sQ + s * 2 * C::kQBytes;
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(q_dst + c * C::kBox, &tm_q, &full[s], c * 64, q0, sc.h, b);
          tma_load_4d(q_dst + C::kQBytes + c * C::kBox, &tm_do, &full[s], c * 64, q0, sc.h, b);
        }
        const size_t row = (static_cast<size_t>(b) * p.Hq + sc.h) * p.Lq_pad + q0;
        bulk_load(sStat + s * 2 * BM, p.lse2 + row, BM * 4, &full[s]);
        bulk_load(sStat + s * 2 * BM + BM, p.delta + row, BM * 4, &full[s]);
      }
    } else if (warp == 13 && lane == 0 && T > 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_st = idesc_16_f32<kF16>(128, BM, 0, 0);   // K x Q^T, V x dO^T
      constexpr uint32_t idesc_acc = idesc_16_f32<kF16>(128, D, 0, 1);   // A (K-major or TMEM) x (dO|Q MN-major)
      constexpr uint32_t idesc_dq = idesc_16_f32<kF16>(128, BM, 1, 1);   // K^T (MN-major) x dS^T (MN-major)
      const uint32_t k_addr = smem_u32(sK), v_addr = smem_u32(sV), q_addr = smem_u32(sQ), ds_addr = smem_u32(sDS);
      const SDesc dk_base = sdesc_split(k_addr, 16, 1024), dv_base = sdesc_split(v_addr, 16, 1024);
      const SDesc dq_base = sdesc_split(q_addr, 16, 1024), ddo_base = sdesc_split(q_addr + C::kQBytes, 16, 1024);
      const SDesc bq_base = sdesc_split(q_addr, C::kBox, 1024), bdo_base = sdesc_split(q_addr + C::kQBytes, C::kBox, 1024);
      const SDesc ads = sdesc_split(ds_addr, 16, 1024);              // dS^T as K-major A (keys x queries)
      const SDesc bds = sdesc_split(ds_addr, C::kBox, 1024);         // dS^T as MN-major B (keys x queries)
      const SDesc akt = sdesc_split(k_addr, D == 128 ? C::kBox : 0, 1024);  // K^T as MN-major A (d x keys)
      constexpr uint32_t kStage16 = (2 * C::kQBytes) >> 4;
      auto issue_s = [&](int t) {
        const uint32_t so = (t % NS) * kStage16;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * C::kBox + (k & 3) * 32) >> 4;
          mma_ss_d(tbase + kColS, dk_base, off, dq_base, so + off, idesc_st, k > 0);
        }
        mma_commit(s_ready);
      };
      auto issue_dp = [&](int t) {
        const uint32_t so = (t % NS) * kStage16;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * C::kBox + (k & 3) * 32) >> 4;
          mma_ss_d(tbase + kColDP, dv_base, off, ddo_base, so + off, idesc_st, k > 0);
        }
        mma_commit(dp_ready);
      };
      bool ok = mbar_wait(kv_full, 0, abort_flag, p.status, kSite + 2);
      if (ok) ok = mbar_wait(&full[0], 0, abort_flag, p.status, kSite + 3);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int t = 0; t < T && ok; ++t) {
        const uint32_t so = (t % NS) * kStage16;
        ok = mbar_wait(p_ready, t & 1, abort_flag, p.status, kSite + 4);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // dV += P^T dO ; query k-step k of warpgroup k/4 is packed at 64(k/4) + 8(k%4)
          const uint32_t acol = 64 * (k >> 2) + 8 * (k & 3);
          mma_ts_d(tbase + 128, tbase + kColS + acol, bdo_base, so + ((16 * k * 128) >> 4), idesc_acc,
                   (t > 0 || k > 0) ? 1u : 0u);
        }
        ok = mbar_wait(ds_ready, t & 1, abort_flag, p.status, kSite + 5);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // dQ^T = K^T dS^T into the dP^T columns (the softmax has read dP^T(t))
          const uint32_t off = (16 * k * 128) >> 4;
          mma_ss_d(tbase + kColDP, akt, off, bds, off, idesc_dq, k > 0);
        }
        mma_commit(dq_ready);
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // dK += dS^T Q (dS^T from shared memory)
          const uint32_t aoff = ((k >> 2) * C::kBox + (k & 3) * 32) >> 4;
          mma_ss_d(tbase + 0, ads, aoff, bq_base, so + ((16 * k * 128) >> 4), idesc_acc, (t > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&empty[t % NS]);
        if (t + 1 < T) {
          ok = mbar_wait(&full[(t + 1) % NS], ((t + 1) / NS) & 1, abort_flag, p.status, kSite + 7);
          if (!ok) break;
          tc_fence_after();
          issue_s(t + 1);
          ok = mbar_wait(dq_free, t & 1, abort_flag, p.status, kSite + 8);
          if (!ok) break;
          tc_fence_after();
          issue_dp(t + 1);
        }
      }
      if (ok) mma_commit(acc_full);
    } else if (kOrdered && warp >= 14) {
      // ---------------------------------------------------------------- turn keepers (even / odd steps)
      const int par = warp - 14;
      // The tile before this one in turn order (key tile j - 1, or j + 1 when
      // reversed) adds first wherever it adds; a turn counter holds the turn
      // position (tc.rank) of the next tile to add.
      int pb = 0, ps = 0;
      if (tc.rank > 0) key_tile_queries(p, b, rev ? j0 + C::kBN : j0 - C::kBN, kvl, false, pb, ps);
      for (int t = par; t < T; t += 2) {
        const StepCoord sc = step_coord<kOrdered>(t, hk, p.G, i_begin, steps_per_head, rev);
        int* turn = p.dq_turn + (static_cast<size_t>(b) * p.Hq + sc.h) * p.nq + sc.it;
        if (lane == 0 && sc.it >= pb && sc.it < pb + ps) (void)wait_turn(turn, tc.rank, abort_flag, p.status, kSite + 14);
        __syncwarp();
        named_barrier_sync(kBarTurn + par, kBarThreads);  // the reduction warps may add
        named_barrier_sync(kBarDone + par, kBarThreads);  // their adds are issued
        // published even when this CTA is giving up, so no later tile waits out its limit
        if (lane == 0) publish_gpu(turn, tc.rank + 1);
        __syncwarp();
      }
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ------------------------------------------------ reduction (thread = head-dim row of dQ^T)
    setmaxnreg_inc<C::kRegsWork>();
    const int quarter = warp - 8;
    const int dr = quarter * 32 + lane;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool active = quarter * 32 < p.dh;  // lanes past the stored head_dim hold copies or padding
    const size_t qstride = static_cast<size_t>(p.Hq) * p.dh;
    for (int t = 0; t < T; ++t) {
      // the ordered build keeps taking part in the turn barriers after a
      // failed wait (the waits return at once then), so no warp is left
      // waiting at a named barrier
      const bool ok = __all_sync(0xffffffffu, mbar_wait(dq_ready, t & 1, abort_flag, p.status, kSite + 13));
      if (!ok && !kOrdered) break;
      uint32_t v[128];
      if (ok) {
        tc_fence_after();
        if (active) {
          tmem_ld32_pair(t_lane + kColDP, t_lane + kColDP + 32, *reinterpret_cast<uint32_t(*)[32]>(v),
                         *reinterpret_cast<uint32_t(*)[32]>(v + 32));
          tmem_ld32_pair(t_lane + kColDP + 64, t_lane + kColDP + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 64),
                         *reinterpret_cast<uint32_t(*)[32]>(v + 96));
        }
        tc_fence_before();
        mbar_arrive(dq_free);
      }
      if (kOrdered) named_barrier_sync(kBarTurn + (t & 1), kBarThreads);
      if (ok && active) {
        const StepCoord sc = step_coord<kOrdered>(t, hk, p.G, i_begin, steps_per_head, rev);
        const int q0 = sc.it * BM;
        float* dst = p.dq_acc + ((static_cast<size_t>(b) * p.Lq + q0) * p.Hq + sc.h) * p.dh + dr;
        if (q0 + BM <= p.Lq) {
#pragma unroll
          for (int c = 0; c < BM; ++c) atomicAdd(dst + c * qstride, __uint_as_float(v[c]));
        } else {
          const int n = p.Lq - q0;
#pragma unroll
          for (int c = 0; c < BM; ++c)
            if (c < n) atomicAdd(dst + c * qstride, __uint_as_float(v[c]));
        }
      }
      if (kOrdered) named_barrier_sync(kBarDone + (t & 1), kBarThreads);
    }
  } else {
    // ------------------------------------------------------------ softmax (thread = key row)
    setmaxnreg_inc<C::kRegsWork>();
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
    uint8_t* ds_row = sDS + w * C::kBox + r * 128;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int s = t % NS;
      const int q0 = step_coord<kOrdered>(t, hk, p.G, i_begin, steps_per_head, rev).it * BM;
      uint32_t sg0 = ~0u, sg1 = ~0u;  // segment bits of this warpgroup's 64 queries (before S is ready)
      // query and key block hold one and the same id: every pair matches
      const bool seg_all =
          kSeg && p.seg_qblk != nullptr && seg_same_single_id(seg_block(p.seg_qblk, b, p.nqb, q0 / kSegBlock), krec);
      if (kSeg && !seg_all) {
        sg0 = segment_bits32(qid, q0 + c0, p.Lq, qid_vec, my_seg);
        sg1 = segment_bits32(qid, q0 + c0 + 32, p.Lq, qid_vec, my_seg);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(s_ready, t & 1, abort_flag, p.status, kSite + 9));
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = sStat + s * 2 * BM;
      const float* dlt = lse2 + BM;
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
      ok = __all_sync(0xffffffffu, mbar_wait(dp_ready, t & 1, abort_flag, p.status, kSite + 10));
      if (!ok) break;
      tc_fence_after();
      // dS^T = P^T (dP^T - delta) -> 128B-swizzled shared memory (this row, this
      // warpgroup's 64 queries), 32 columns of dP^T at a time
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t da[32];
        tmem_ld32(t_lane + kColDP + c0 + 32 * hh, da);
#pragma unroll
        for (int ch = 4 * hh; ch < 4 * hh + 4; ++ch) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 8 * ch + 2 * e;
            const float4 d4 = *reinterpret_cast<const float4*>(dlt + c0 + (c & ~3));
            const float dv0 = (c & 3) ? d4.z : d4.x, dv1 = (c & 3) ? d4.w : d4.y;
            pk[e] = pack2<kF16>(pr[c] * (__uint_as_float(da[c - 32 * hh]) - dv0),
                                pr[c + 1] * (__uint_as_float(da[c + 1 - 32 * hh]) - dv1));
          }
          *reinterpret_cast<uint4*>(ds_row + ((ch ^ (r & 7)) * 16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ds_ready);
    }
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, p.status, kSite + 12));
    // dK (warpgroup 0, times scale) and dV (warpgroup 1) go through the Q/dO
    // stages, idle once every MMA has completed (the reduction warps read
    // dQ^T from TMEM only), and out with TMA stores that clip the rows past
    // Lkv and the columns past the stored head_dim
    if (ok) {
      tc_fence_after();
      stage_row16<D, kF16>(t_lane + (w == 0 ? 0 : 128), sQ + w * (D / 64) * C::kBox, r, w == 0 ? p.scale : 1.0f,
                           T == 0);
      fence_proxy_async_smem();
    }
    named_barrier_sync(kBarStore, 256);
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
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// dq = scale * dq_acc cast to the 16-bit format (single-pass variants)
template <bool kF16>
__global__ void dq_convert_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq, long n4,
                                  float scale) {
  griddep_wait();  // launched to overlap the single pass: its adds are complete from here on
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[i];
  uint2 o;
  o.x = pack2<kF16>(a.x * scale, a.y * scale);
  o.y = pack2<kF16>(a.z * scale, a.w * scale);
  reinterpret_cast<uint2*>(dq)[i] = o;
}

template <int D, bool kLeftBound, bool kF16, bool kSeg, bool kOrdered>
cudaError_t launch_single_pass_inst(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                                    const BwdKParams& kp, dim3 grid, long n_dq, cudaStream_t stream) {
  using C = DkdvAtomicCfg<D>;
  constexpr auto kern = bwd_dkdv_single_pass_kernel<D, kLeftBound, kF16, kSeg, kOrdered>;
  cudaError_t e = ensure_dynamic_smem<kern>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  {
    KernelTimer kt(kOrdered ? "bwd_dkdv_ordered" : "bwd_dkdv_atomic", stream);
    if (kOrdered) {
      kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdk, tdv, kp);
      e = cudaGetLastError();
    } else {
      e = launch_overlapping(kern, grid, C::kThreads, C::kSmemBytes, stream, tq, tk, tv, tdo, tdk, tdv, kp);
    }
  }
  if (e != cudaSuccess) return e;
  const long n4 = n_dq / 4;
  KernelTimer kt("dq_convert", stream);
  return launch_overlapping(dq_convert_kernel<kF16>, dim3(static_cast<unsigned>((n4 + 255) / 256)), 256, 0, stream,
                            static_cast<const float*>(kp.dq_acc), static_cast<uint16_t*>(kp.dq), n4, kp.scale);
}

// The kernel build for a problem: format x (no left bound | two-sided span |
// two-sided span + segment ids).
// Compile-time flags of one kernel build: left window bound, fp16, segment ids.
template <bool L, bool F, bool S>
struct Build {
  static constexpr bool kL = L, kF = F, kS = S;
};

template <int D, bool kOrdered>
cudaError_t launch_single_pass_build(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                                     const BwdKParams& kp, dim3 grid, long n_dq, bool f16, cudaStream_t stream) {
  const bool left = kp.wl < kWinInf;
  // (left bound, fp16, segment ids) of the build
  auto run = [&](auto build) {
    return launch_single_pass_inst<D, decltype(build)::kL, decltype(build)::kF, decltype(build)::kS, kOrdered>(
        tq, tk, tv, tdo, tdk, tdv, kp, grid, n_dq, stream);
  };
  if (kp.q_seg != nullptr)  // segment masks run the general (two-sided span) build
    return f16 ? run(Build<true, true, true>{}) : run(Build<true, false, true>{});
  if (f16) return left ? run(Build<true, true, false>{}) : run(Build<false, true, false>{});
  return left ? run(Build<true, false, false>{}) : run(Build<false, false, false>{});
}

}  // namespace
}  // namespace bwd
}  // namespace attn
