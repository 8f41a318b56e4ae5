// Single-pass backward, bf16 or fp16, head_dim 64/128: dK and dV as in the two-pass
// variant, while dQ is summed over key tiles with float32 atomic adds into a
// buffer that a convert kernel scales and casts to bf16 (probjax "Attention
// performance", section "When to use which", backward pass: dQ = scale * dS K).
// The order of the adds is not fixed, so the result is not bitwise
// reproducible; the two-pass backward is.
#include "bwd_common.cuh"

namespace attn {
namespace bwd {
namespace {

// ============================================================================
// dK / dV kernel with atomic dQ (single-pass backward)
// ============================================================================
// CTA = (batch, KV head, 128 keys); thread = key row = TMEM lane; 128-query
// steps, every MMA 128 x 128 x 16.  Five GEMMs per step instead of the
// two-pass backward's seven:
//   tensor pipe:  S^T | dP^T | dV += P^T dO | dQ^T = K^T dS^T | dK += dS^T Q | S^T(t+1) | dP^T(t+1) ...
//   softmax:          | P^T  | dS^T        |
//   reduction:                              | dQ^T -> registers -> fp32 atomic adds (overlaps the next step)
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
// next step's GEMMs and softmax run.  The summation order of dQ over key tiles
// is not fixed, so this variant is not bitwise reproducible.
//
// Warps 0-7 softmax (warpgroup w owns queries [64w, 64w + 64) of the step),
// 8-11 reduction (warp 8 + i reads TMEM lanes [32i, 32i + 32)), 12 TMA
// producer, 13 MMA issuer, 14-15 idle; the control warpgroup gives its
// registers to the other three.
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
  // time; a misaligned base makes the kernel report and do nothing).
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16;
  static constexpr int kThreads = 512;
  // Registers per thread after the split (launch: 512 x 128).  Each SM
  // sub-partition holds one warp of each warpgroup: 3 x kRegsWork + kRegsCtl
  // must equal 4 x 128.
  static constexpr int kRegsWork = 144, kRegsCtl = 80;
};

template <int D, bool kLeftBound, bool kF16, bool kSeg>
__global__ void __launch_bounds__(512, 1)
    bwd_dkdv_atomic_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                           const BwdKParams p) {
  using C = DkdvAtomicCfg<D>;
  constexpr int NS = C::kStages, BM = C::kBM;
  constexpr uint32_t kColS = 256, kColDP = 384;
  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // never expected: see kSmemBytes
    if (threadIdx.x == 0) report_status(p.status, 2, 99);
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

  const int warp = warp_id(), lane = lane_id();
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
  static_assert(3 * C::kRegsWork + C::kRegsCtl == 4 * 128, "register split must match the launch allocation");

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
        if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, abort_flag, p.status, 71)) break;
        const int h = hk * p.G + t / steps_per_head;
        const int q0 = (i_begin + t % steps_per_head) * BM;
        mbar_arrive_expect_tx(&full[s], 2 * C::kQBytes + 2 * BM * 4);
        uint8_t* q_dst = sQ + s * 2 * C::kQBytes;
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(q_dst + c * C::kBox, &tm_q, &full[s], c * 64, q0, h, b);
          tma_load_4d(q_dst + C::kQBytes + c * C::kBox, &tm_do, &full[s], c * 64, q0, h, b);
        }
        const size_t row = (static_cast<size_t>(b) * p.Hq + h) * p.Lq_pad + q0;
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
      bool ok = mbar_wait(kv_full, 0, abort_flag, p.status, 72);
      if (ok) ok = mbar_wait(&full[0], 0, abort_flag, p.status, 73);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int t = 0; t < T && ok; ++t) {
        const uint32_t so = (t % NS) * kStage16;
        ok = mbar_wait(p_ready, t & 1, abort_flag, p.status, 74);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // dV += P^T dO ; query k-step k of warpgroup k/4 is packed at 64(k/4) + 8(k%4)
          const uint32_t acol = 64 * (k >> 2) + 8 * (k & 3);
          mma_ts_d(tbase + 128, tbase + kColS + acol, bdo_base, so + ((16 * k * 128) >> 4), idesc_acc,
                   (t > 0 || k > 0) ? 1u : 0u);
        }
        ok = mbar_wait(ds_ready, t & 1, abort_flag, p.status, 75);
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
          ok = mbar_wait(&full[(t + 1) % NS], ((t + 1) / NS) & 1, abort_flag, p.status, 77);
          if (!ok) break;
          tc_fence_after();
          issue_s(t + 1);
          ok = mbar_wait(dq_free, t & 1, abort_flag, p.status, 78);
          if (!ok) break;
          tc_fence_after();
          issue_dp(t + 1);
        }
      }
      if (ok) mma_commit(acc_full);
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
      if (!__all_sync(0xffffffffu, mbar_wait(dq_ready, t & 1, abort_flag, p.status, 83))) break;
      tc_fence_after();
      uint32_t v[128];
      if (active) {
        tmem_ld32_pair(t_lane + kColDP, t_lane + kColDP + 32, *reinterpret_cast<uint32_t(*)[32]>(v),
                       *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_ld32_pair(t_lane + kColDP + 64, t_lane + kColDP + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 64),
                       *reinterpret_cast<uint32_t(*)[32]>(v + 96));
      }
      tc_fence_before();
      mbar_arrive(dq_free);
      if (active) {
        const int h = hk * p.G + t / steps_per_head;
        const int q0 = (i_begin + t % steps_per_head) * BM;
        float* dst = p.dq_acc + ((static_cast<size_t>(b) * p.Lq + q0) * p.Hq + h) * p.dh + dr;
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
      const int q0 = (i_begin + t % steps_per_head) * BM;
      uint32_t sg0 = ~0u, sg1 = ~0u;  // segment bits of this warpgroup's 64 queries (before S is ready)
      // query and key block hold one and the same id: every pair matches
      const bool seg_all =
          kSeg && p.seg_qblk != nullptr && seg_same_single_id(seg_block(p.seg_qblk, b, p.nqb, q0 / kSegBlock), krec);
      if (kSeg && !seg_all) {
        sg0 = segment_bits32(qid, q0 + c0, p.Lq, qid_vec, my_seg);
        sg1 = segment_bits32(qid, q0 + c0 + 32, p.Lq, qid_vec, my_seg);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(s_ready, t & 1, abort_flag, p.status, 79));
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
      ok = __all_sync(0xffffffffu, mbar_wait(dp_ready, t & 1, abort_flag, p.status, 80));
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
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, p.status, 82));
    if (ok) {
      tc_fence_after();
      const bool st = j < p.Lkv;
      const size_t off = ((static_cast<size_t>(b) * p.Lkv + (st ? j : 0)) * p.Hkv + hk) * p.dh;
      if (w == 0)
        store_row16<D, kF16>(t_lane + 0, reinterpret_cast<uint16_t*>(p.dk) + off, p.scale, st, T == 0, p.dh);
      else
        store_row16<D, kF16>(t_lane + 128, reinterpret_cast<uint16_t*>(p.dv) + off, 1.0f, st, T == 0, p.dh);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// dq = scale * dq_acc cast to bf16 (single-pass variant)
template <bool kF16>
__global__ void dq_convert_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq, long n4,
                                  float scale) {
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[i];
  uint2 o;
  o.x = pack2<kF16>(a.x * scale, a.y * scale);
  o.y = pack2<kF16>(a.z * scale, a.w * scale);
  reinterpret_cast<uint2*>(dq)[i] = o;
}

}  // namespace

namespace {

template <int D, bool kLeftBound, bool kF16, bool kSeg>
cudaError_t launch_single_pass_inst(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const CUtensorMap& tdo, const BwdKParams& kp, dim3 grid, long n_dq,
                                    cudaStream_t stream) {
  using C = DkdvAtomicCfg<D>;
  cudaError_t e = ensure_dynamic_smem<bwd_dkdv_atomic_kernel<D, kLeftBound, kF16, kSeg>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  {
    KernelTimer kt("bwd_dkdv_atomic", stream);
    bwd_dkdv_atomic_kernel<D, kLeftBound, kF16, kSeg>
        <<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, kp);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long n4 = n_dq / 4;
  KernelTimer kt("dq_convert", stream);
  dq_convert_kernel<kF16><<<static_cast<int>((n4 + 255) / 256), 256, 0, stream>>>(
      kp.dq_acc, static_cast<uint16_t*>(kp.dq), n4, kp.scale);
  return cudaGetLastError();
}

}  // namespace

template <int D>
cudaError_t launch_single_pass(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, const BwdKParams& kp, dim3 grid, long n_dq, bool f16,
                               cudaStream_t stream) {
  const bool left = kp.wl < kWinInf;
  if (kp.q_seg != nullptr)  // segment masks run the general (two-sided span) build
    return f16 ? launch_single_pass_inst<D, true, true, true>(tq, tk, tv, tdo, kp, grid, n_dq, stream)
               : launch_single_pass_inst<D, true, false, true>(tq, tk, tv, tdo, kp, grid, n_dq, stream);
  if (f16)
    return left ? launch_single_pass_inst<D, true, true, false>(tq, tk, tv, tdo, kp, grid, n_dq, stream)
                : launch_single_pass_inst<D, false, true, false>(tq, tk, tv, tdo, kp, grid, n_dq, stream);
  return left ? launch_single_pass_inst<D, true, false, false>(tq, tk, tv, tdo, kp, grid, n_dq, stream)
              : launch_single_pass_inst<D, false, false, false>(tq, tk, tv, tdo, kp, grid, n_dq, stream);
}

template cudaError_t launch_single_pass<64>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                            const CUtensorMap&, const BwdKParams&, dim3, long, bool, cudaStream_t);
template cudaError_t launch_single_pass<128>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                             const CUtensorMap&, const BwdKParams&, dim3, long, bool, cudaStream_t);

}  // namespace bwd
}  // namespace attn
