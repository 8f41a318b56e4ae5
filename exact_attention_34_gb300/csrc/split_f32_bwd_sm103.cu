// float32 backward on the bf16 tensor cores by operand splitting (see
// split_f32.cuh): the deterministic two-pass backward of bwd_sm103.cu with
// its products taken as a few bf16 MMAs each and the probabilities and score
// gradients kept in float32 until they are split for the MMAs that use them
// (probjax "Attention performance", section "When to use which", backward
// pass: dV = P^T dO, dP = dO V^T, dS = P (dP - delta), dQ = scale dS K,
// dK = scale dS^T Q).
//
// Precision.  dS = P (dP - delta) cancels wherever a row's probability sits
// on few keys (one key: dP = delta exactly, dS = 0), so dP needs more than the
// two-part split's ~2^-16: dO and V are split into three exact parts and dP
// takes the six products of combined order <= 2 (hi hi, hi mid, mid hi, hi lo,
// lo hi, mid mid; error ~2^-24), the small ones first: each MMA rounds the
// accumulator it adds to (about an ulp of the running sum), so the eight
// large hi hi additions come last.  S = Q K^T and dS^T Q, dS K take three
// products of two-part splits (~2^-16, which moves P by ~1e-6), and
// dV = P^T dO four (P_hi with all of dO's parts, P_lo with dO_hi: a row with
// P = 1 gives dV = dO exactly).
// Both passes split their float32 operands on the fly with four converter
// warps (no workspace beyond the row statistics), so the float32 workspace is
// the same as for the CUDA-core kernels.
//
// dK/dV pass: CTA = (batch, KV head, 128 keys); thread = key row = TMEM lane;
// 32-query steps over the G query heads of the group.  K (two parts) and V
// (three) are split once into shared memory; each step's Q (two parts,
// double-buffered) and dO (three) with their lse2 and delta rows are split by
// the converters.  Per step: S^T = K Q^T and dP^T = V dO^T, P^T and dS^T in
// float32 on the softmax warps, written back as hi and lo parts, then
// dV += P^T dO and dK += dS^T Q with A from TMEM.  MMA order per step: dV(t),
// S^T(t+1), dK(t), dP^T(t+1).  TMEM: dK [0,128) dV [128,256) S^T [256,288)
// dP^T [288,320) P^T lo [320,336) dS^T lo [336,352); the hi parts go over the
// first 16 columns of S^T / dP^T.
//
// dQ pass: CTA = (batch, head, 128 queries); thread = query row; 32-key
// steps.  Q (two parts) and dO (three) are split once; each step's K (two
// parts, double-buffered) and V (three) by the converters.  Per step: S = Q
// K^T (double-buffered in TMEM, two steps ahead) and dP = dO V^T, dS in
// float32, then dQ += dS K with dS from TMEM.  TMEM: dQ [0,128) S [128,160)
// and [160,192) dP [192,224) dS lo [224,240) and [240,256).
//
// Warps 0-3 softmax, 4-7 converters, 8 MMA issuer (owns TMEM); every wait is
// bounded.
#include "bwd_common.cuh"
#include "split_f32.cuh"

namespace attn {
namespace {

using namespace split;
using bwd::BwdKParams;

constexpr int kRowsBig = 128;   // stationary rows per CTA (keys in dK/dV, queries in dQ)
constexpr int kRowsStep = 32;   // streamed rows per step
constexpr float kLog2eB = 1.4426950408889634f;

template <int D>
struct SplitDkdvCfg {
  static constexpr int kBigBox = kRowsBig * 128;         // one 64-column box of a 128-row tile
  static constexpr int kBigPart = kBigBox * (D / 64);    // one part of K or V
  static constexpr int kStepBox = kRowsStep * 128;       // one 64-column box of a 32-row tile
  static constexpr int kStepPart = kStepBox * (D / 64);  // one part of Q or dO
  static constexpr int kOffK = 0;                        // K hi, K lo
  static constexpr int kOffV = 2 * kBigPart;             // V hi, V mid, V lo
  static constexpr int kOffQ = 5 * kBigPart;             // buffer b: Q hi at kOffQ + 2b kStepPart, lo after
  static constexpr int kOffDO = kOffQ + 4 * kStepPart;   // dO hi, mid, lo
  static constexpr int kOffLse = kOffDO + 3 * kStepPart; // [2][32] lse2 rows of the Q buffers
  static constexpr int kOffDelta = kOffLse + 2 * kRowsStep * 4;  // [2][32] delta rows
  static constexpr int kOffBars = kOffDelta + 2 * kRowsStep * 4;
  static constexpr int kNumBars = 12;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;
  static constexpr int kThreads = 288;
};

template <int D>
struct SplitDqCfg {
  static constexpr int kBigBox = kRowsBig * 128;
  static constexpr int kBigPart = kBigBox * (D / 64);    // one part of Q or dO
  static constexpr int kStepBox = kRowsStep * 128;
  static constexpr int kStepPart = kStepBox * (D / 64);  // one part of K or V
  static constexpr int kOffQ = 0;                        // Q hi, Q lo
  static constexpr int kOffDO = 2 * kBigPart;            // dO hi, mid, lo
  static constexpr int kOffK = 5 * kBigPart;             // buffer b: K hi at kOffK + 2b kStepPart, lo after
  static constexpr int kOffV = kOffK + 4 * kStepPart;    // V hi, mid, lo
  static constexpr int kOffBars = kOffV + 3 * kStepPart;
  static constexpr int kNumBars = 12;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;
  static constexpr int kThreads = 288;
};

// The three MMAs of one 16-wide k-step of a split product, A and B from
// shared memory: A_hi B_hi + A_hi B_lo + A_lo B_hi.
__device__ __forceinline__ void mma3_ss(uint32_t d, SDesc ah, SDesc al, uint32_t ao, SDesc bh, SDesc bl, uint32_t bo,
                                        uint32_t idesc, uint32_t acc) {
  mma_ss_d(d, ah, ao, bh, bo, idesc, acc);
  mma_ss_d(d, ah, ao, bl, bo, idesc, 1u);
  mma_ss_d(d, al, ao, bh, bo, idesc, 1u);
}

// The five smaller MMAs of one k-step of a product of three-part operands
// (hi mid, mid hi, hi lo, lo hi, mid mid); with the hi hi product that is
// every part pair of combined order <= 2 (error ~2^-24 of |A||B|).  A whole
// product issues these for all k-steps first and the hi hi products last:
// each MMA rounds the accumulator it adds to, so the large additions should
// come last and be few.
__device__ __forceinline__ void mma5_small_ss(uint32_t d, SDesc ah, SDesc am, SDesc al, uint32_t ao, SDesc bh,
                                              SDesc bm, SDesc bl, uint32_t bo, uint32_t idesc, uint32_t acc) {
  mma_ss_d(d, ah, ao, bm, bo, idesc, acc);
  mma_ss_d(d, am, ao, bh, bo, idesc, 1u);
  mma_ss_d(d, ah, ao, bl, bo, idesc, 1u);
  mma_ss_d(d, al, ao, bh, bo, idesc, 1u);
  mma_ss_d(d, am, ao, bm, bo, idesc, 1u);
}

// The same with A (hi and lo parts) from TMEM.
__device__ __forceinline__ void mma3_ts(uint32_t d, uint32_t ah, uint32_t al, SDesc bh, SDesc bl, uint32_t bo,
                                        uint32_t idesc, uint32_t acc) {
  mma_ts_d(d, ah, bh, bo, idesc, acc);
  mma_ts_d(d, ah, bl, bo, idesc, 1u);
  mma_ts_d(d, al, bh, bo, idesc, 1u);
}

// 32 float32 values -> packed bf16 hi (16 columns) and lo (16 columns) parts.
__device__ __forceinline__ void split32(const float (&x)[32], uint32_t (&hi)[16], uint32_t (&lo)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    hi[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
    lo[i] = pack_bf16x2(x[2 * i] - __uint_as_float(hi[i] << 16), x[2 * i + 1] - __uint_as_float(hi[i] & 0xffff0000u));
  }
}

// Store D float32 values of one TMEM row, times `mul` (zeros when `zero`).
template <int D>
__device__ __forceinline__ void store_row_f32(uint32_t taddr, float* dst, float mul, bool do_store, bool zero) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t r[32];
    if (!zero) {
      tmem_ld32(taddr + c * 32, r);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = 0u;
    }
    if (do_store) {
      float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        d4[i] = make_float4(__uint_as_float(r[4 * i]) * mul, __uint_as_float(r[4 * i + 1]) * mul,
                            __uint_as_float(r[4 * i + 2]) * mul, __uint_as_float(r[4 * i + 3]) * mul);
    }
  }
}

// ============================================================================
// dK / dV pass
// ============================================================================
template <int D, bool kLeftBound>
__global__ void __launch_bounds__(288, 1) bwd_split_dkdv_kernel(const BwdKParams p, const float* __restrict__ q,
                                                                const float* __restrict__ k,
                                                                const float* __restrict__ v,
                                                                const float* __restrict__ dout) {
  using C = SplitDkdvCfg<D>;
  constexpr int RS = kRowsStep;
  constexpr uint32_t kColS = 256, kColDP = 288, kColPlo = 320, kColDSlo = 336;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sDelta = reinterpret_cast<float*>(smem + C::kOffDelta);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* kv_full = bars;        // converters split K and V (4 warp arrivals)
  uint64_t* q_full = bars + 1;     // [2] Q(t) and its lse2 rows split
  uint64_t* q_empty = bars + 3;    // [2] dK(t) done with the Q buffer
  uint64_t* do_full = bars + 5;    // dO(t) and its delta rows split
  uint64_t* do_empty = bars + 6;   // dV(t) done with the dO buffer
  uint64_t* s_ready = bars + 7;    // S^T(t) computed
  uint64_t* dp_ready = bars + 8;   // dP^T(t) computed
  uint64_t* p_ready = bars + 9;    // P^T(t) written (4 warp arrivals)
  uint64_t* ds_ready = bars + 10;  // dS^T(t) written (4 warp arrivals)
  uint64_t* acc_full = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const TileCoord tc = grouped_tile(blockIdx.x, p.n_pairs, p.n_tiles, p.pair_group);
  const int j0 = tc.rank * kRowsBig, hk = tc.pair % p.Hkv, b = tc.pair / p.Hkv;
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);
  // 32-row query tiles that see some key of this tile
  int i_begin = 0, steps_per_head = 0;
  if (j0 < kvl) {
    const int q_lo = query_span(j0, p.Lq, kvl, p.wl, p.wr).lo;
    const int q_hi = query_span(min(j0 + kRowsBig, kvl) - 1, p.Lq, kvl, p.wl, p.wr).hi;
    if (q_hi > q_lo) {
      i_begin = q_lo / RS;
      steps_per_head = (q_hi + RS - 1) / RS - i_begin;
    }
  }
  const int T = steps_per_head * p.G;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(kv_full, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 4);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(do_full, 4);
    mbar_init(do_empty, 1);
    mbar_init(s_ready, 1);
    mbar_init(dp_ready, 1);
    mbar_init(p_ready, 4);
    mbar_init(ds_ready, 4);
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // launched to overlap the preprocess: delta and lse2 are complete from here
  // on; the dQ pass reads nothing this kernel writes
  griddep_wait();
  griddep_launch_dependents();

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ converters
    const int t = threadIdx.x - 128;
    if (T > 0) {
      for (int half = 0; half < 2; ++half) {
        const int r0 = half * (kRowsBig / 2);
        convert_tile<D, kRowsBig / 2, kRowsBig>(k, b, p.Lkv, p.Hkv, hk, j0 + r0, kvl, smem + C::kOffK,
                                                smem + C::kOffK + C::kBigPart, r0, t);
        convert_tile<D, kRowsBig / 2, kRowsBig, true>(v, b, p.Lkv, p.Hkv, hk, j0 + r0, kvl, smem + C::kOffV,
                                                      smem + C::kOffV + 2 * C::kBigPart, r0, t,
                                                      smem + C::kOffV + C::kBigPart);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(kv_full);
    }
    bool ok = true;
    for (int s = 0; s < T && ok; ++s) {
      const int h = hk * p.G + s / steps_per_head;
      const int q0 = (i_begin + s % steps_per_head) * RS;
      const size_t row = (static_cast<size_t>(b) * p.Hq + h) * p.Lq_pad + q0;  // q0 + 32 <= Lq_pad
      const int qb = s & 1;
      if (s >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&q_empty[qb], ((s - 2) >> 1) & 1, abort_flag, p.status, 141));
      if (!ok) break;
      uint8_t* qh = smem + C::kOffQ + 2 * qb * C::kStepPart;
      convert_tile<D, RS, RS>(q, b, p.Lq, p.Hq, h, q0, p.Lq, qh, qh + C::kStepPart, 0, t);
      if (t < RS) sLse[qb * RS + t] = p.lse2[row + t];
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[qb]);
      if (s >= 1) ok = __all_sync(0xffffffffu, mbar_wait(do_empty, (s - 1) & 1, abort_flag, p.status, 142));
      if (!ok) break;
      convert_tile<D, RS, RS, true>(dout, b, p.Lq, p.Hq, h, q0, p.Lq, smem + C::kOffDO,
                                    smem + C::kOffDO + 2 * C::kStepPart, 0, t, smem + C::kOffDO + C::kStepPart);
      if (t < RS) sDelta[qb * RS + t] = p.delta[row + t];
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(do_full);
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_st = idesc_bf16_f32(kRowsBig, RS, 0, 0);  // K x Q^T, V x dO^T
      constexpr uint32_t idesc_acc = idesc_bf16_f32(kRowsBig, D, 0, 1);  // (P^T | dS^T from TMEM) x (dO | Q)
      const uint32_t k_addr = smem_u32(smem + C::kOffK), v_addr = smem_u32(smem + C::kOffV);
      const SDesc kh = sdesc_split(k_addr, 16, 1024), kl = sdesc_split(k_addr + C::kBigPart, 16, 1024);
      const SDesc vh = sdesc_split(v_addr, 16, 1024), vm = sdesc_split(v_addr + C::kBigPart, 16, 1024),
                  vl = sdesc_split(v_addr + 2 * C::kBigPart, 16, 1024);
      const uint32_t do_addr = smem_u32(smem + C::kOffDO);
      auto q_addr = [&](int s) { return smem_u32(smem + C::kOffQ + 2 * (s & 1) * C::kStepPart); };
      auto issue_st = [&](int s) {  // S^T(s) = K Q(s)^T
        const uint32_t qa = q_addr(s);
        const SDesc qh = sdesc_split(qa, 16, 1024), ql = sdesc_split(qa + C::kStepPart, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * C::kBigBox + (kk & 3) * 32) >> 4;
          const uint32_t bo = ((kk >> 2) * C::kStepBox + (kk & 3) * 32) >> 4;
          mma3_ss(tbase + kColS, kh, kl, ao, qh, ql, bo, idesc_st, kk > 0);
        }
        mma_commit(s_ready);
      };
      auto issue_dpt = [&]() {  // dP^T = V dO^T, three-part operands
        const SDesc oh = sdesc_split(do_addr, 16, 1024), om = sdesc_split(do_addr + C::kStepPart, 16, 1024),
                    ol = sdesc_split(do_addr + 2 * C::kStepPart, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * C::kBigBox + (kk & 3) * 32) >> 4;
          const uint32_t bo = ((kk >> 2) * C::kStepBox + (kk & 3) * 32) >> 4;
          mma5_small_ss(tbase + kColDP, vh, vm, vl, ao, oh, om, ol, bo, idesc_st, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * C::kBigBox + (kk & 3) * 32) >> 4;
          const uint32_t bo = ((kk >> 2) * C::kStepBox + (kk & 3) * 32) >> 4;
          mma_ss_d(tbase + kColDP, vh, ao, oh, bo, idesc_st, 1u);
        }
        mma_commit(dp_ready);
      };
      bool ok = mbar_wait(kv_full, 0, abort_flag, p.status, 143);
      if (ok) ok = mbar_wait(&q_full[0], 0, abort_flag, p.status, 144);
      if (ok) {
        tc_fence_after();
        issue_st(0);
        ok = mbar_wait(do_full, 0, abort_flag, p.status, 145);
      }
      if (ok) {
        tc_fence_after();
        issue_dpt();
      }
      for (int s = 0; s < T && ok; ++s) {
        ok = mbar_wait(p_ready, s & 1, abort_flag, p.status, 146);
        if (!ok) break;
        tc_fence_after();
        {  // dV += P^T dO: P_hi with dO's three parts, P_lo with dO_hi
          const SDesc oh = sdesc_split(do_addr, C::kStepBox, 1024),
                      om = sdesc_split(do_addr + C::kStepPart, C::kStepBox, 1024),
                      ol = sdesc_split(do_addr + 2 * C::kStepPart, C::kStepBox, 1024);
#pragma unroll
          for (int kk = 0; kk < RS / 16; ++kk) {
            const uint32_t bo = (16 * kk * 128) >> 4;
            const uint32_t ph = tbase + kColS + kk * 8, pl = tbase + kColPlo + kk * 8;
            mma_ts_d(tbase + 128, ph, oh, bo, idesc_acc, (s > 0 || kk > 0) ? 1u : 0u);
            mma_ts_d(tbase + 128, ph, om, bo, idesc_acc, 1u);
            mma_ts_d(tbase + 128, ph, ol, bo, idesc_acc, 1u);
            mma_ts_d(tbase + 128, pl, oh, bo, idesc_acc, 1u);
          }
        }
        mma_commit(do_empty);
        if (s + 1 < T) {  // S^T(s+1) over P^T(s), which dV(s) has just read
          ok = mbar_wait(&q_full[(s + 1) & 1], ((s + 1) >> 1) & 1, abort_flag, p.status, 147);
          if (!ok) break;
          tc_fence_after();
          issue_st(s + 1);
        }
        ok = mbar_wait(ds_ready, s & 1, abort_flag, p.status, 148);
        if (!ok) break;
        tc_fence_after();
        {  // dK += dS^T Q
          const uint32_t qa = q_addr(s);
          const SDesc qh = sdesc_split(qa, C::kStepBox, 1024), ql = sdesc_split(qa + C::kStepPart, C::kStepBox, 1024);
#pragma unroll
          for (int kk = 0; kk < RS / 16; ++kk)
            mma3_ts(tbase + 0, tbase + kColDP + kk * 8, tbase + kColDSlo + kk * 8, qh, ql, (16 * kk * 128) >> 4,
                    idesc_acc, (s > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&q_empty[s & 1]);
        if (s + 1 < T) {  // dP^T(s+1) over dS^T(s), which dK(s) has just read
          ok = mbar_wait(do_full, (s + 1) & 1, abort_flag, p.status, 149);
          if (!ok) break;
          tc_fence_after();
          issue_dpt();
        }
      }
      if (ok) mma_commit(acc_full);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (thread = key row)
    const int r = warp * 32 + lane;
    const int j = j0 + r;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    const bool key_ok = j < kvl;
    const Span qs = key_ok ? query_span(j, p.Lq, kvl, p.wl, p.wr) : Span{0, 0};
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int s = 0; s < T; ++s) {
      const int q0 = (i_begin + s % steps_per_head) * RS;
      const float* lse2 = sLse + (s & 1) * RS;
      const float* dlt = sDelta + (s & 1) * RS;
      ok = __all_sync(0xffffffffu, mbar_wait(s_ready, s & 1, abort_flag, p.status, 150));
      if (!ok) break;
      tc_fence_after();
      float pr[RS];
      {
        uint32_t sa[32];
        tmem_ld32(t_lane + kColS, sa);
#pragma unroll
        for (int c = 0; c < RS; ++c) {
          const int qq = q0 + c;
          const bool valid = key_ok && qq >= qs.lo && qq < qs.hi;  // qs.hi <= Lq
          pr[c] = valid ? ex2_approx(fmaf(__uint_as_float(sa[c]), sl2, -lse2[c])) : 0.f;
        }
        uint32_t hi[16], lo[16];
        split32(pr, hi, lo);
        tmem_st16(t_lane + kColS, hi);
        tmem_st16(t_lane + kColPlo, lo);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
      ok = __all_sync(0xffffffffu, mbar_wait(dp_ready, s & 1, abort_flag, p.status, 151));
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t da[32];
        tmem_ld32(t_lane + kColDP, da);
        float ds[RS];
#pragma unroll
        for (int c = 0; c < RS; ++c) ds[c] = pr[c] * (__uint_as_float(da[c]) - dlt[c]);
        uint32_t hi[16], lo[16];
        split32(ds, hi, lo);
        tmem_st16(t_lane + kColDP, hi);
        tmem_st16(t_lane + kColDSlo, lo);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
    }
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, p.status, 152));
    if (ok) {
      tc_fence_after();
      const bool st = j < p.Lkv;
      const size_t off = ((static_cast<size_t>(b) * p.Lkv + (st ? j : 0)) * p.Hkv + hk) * D;
      store_row_f32<D>(t_lane + 0, static_cast<float*>(p.dk) + off, p.scale, st, T == 0);
      store_row_f32<D>(t_lane + 128, static_cast<float*>(p.dv) + off, 1.0f, st, T == 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ============================================================================
// dQ pass
// ============================================================================
template <int D, bool kLeftBound>
__global__ void __launch_bounds__(288, 1) bwd_split_dq_kernel(const BwdKParams p, const float* __restrict__ q,
                                                              const float* __restrict__ k,
                                                              const float* __restrict__ v,
                                                              const float* __restrict__ dout) {
  using C = SplitDqCfg<D>;
  constexpr int RS = kRowsStep;
  constexpr uint32_t kColS = 128, kColDP = 192, kColDSlo = 224;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* qdo_full = bars;       // converters split Q and dO (4 warp arrivals)
  uint64_t* k_full = bars + 1;     // [2]
  uint64_t* k_empty = bars + 3;    // [2] dQ(t) done with the K buffer
  uint64_t* v_full = bars + 5;
  uint64_t* v_empty = bars + 6;    // dP(t) done with the V buffer
  uint64_t* s_ready = bars + 7;    // [2] S(t) computed, one barrier per S buffer
  uint64_t* dp_ready = bars + 9;   // dP(t) computed
  uint64_t* ds_ready = bars + 10;  // dS(t) written (4 warp arrivals)
  uint64_t* acc_full = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const TileCoord tc = grouped_tile(blockIdx.x, p.n_pairs, p.n_tiles, p.pair_group);
  const int qt = p.causal ? p.n_tiles - 1 - tc.rank : tc.rank;
  const int q0 = qt * kRowsBig, h = tc.pair % p.Hq, b = tc.pair / p.Hq;
  const int hk = h / p.G;
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);
  // 32-key steps [t0, t0 + T): from the first key of row q0 to the last key of
  // the tile's last row (both ends grow with the row index)
  const int last = min(q0 + kRowsBig - 1, p.Lq - 1);
  const int k_lo = key_span(q0, p.Lq, kvl, p.wl, p.wr).lo;
  const int k_hi = key_span(last, p.Lq, kvl, p.wl, p.wr).hi;
  const int t0 = kLeftBound ? k_lo / RS : 0;
  const int T = k_hi > k_lo ? (k_hi + RS - 1) / RS - t0 : 0;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(qdo_full, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 4);
      mbar_init(&k_empty[i], 1);
      mbar_init(&s_ready[i], 1);
    }
    mbar_init(v_full, 4);
    mbar_init(v_empty, 1);
    mbar_init(dp_ready, 1);
    mbar_init(ds_ready, 4);
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  griddep_launch_dependents();  // the next kernel waits for this grid before it reads anything

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ converters
    const int t = threadIdx.x - 128;
    if (T > 0) {
      for (int half = 0; half < 2; ++half) {
        const int r0 = half * (kRowsBig / 2);
        convert_tile<D, kRowsBig / 2, kRowsBig>(q, b, p.Lq, p.Hq, h, q0 + r0, p.Lq, smem + C::kOffQ,
                                                smem + C::kOffQ + C::kBigPart, r0, t);
        convert_tile<D, kRowsBig / 2, kRowsBig, true>(dout, b, p.Lq, p.Hq, h, q0 + r0, p.Lq, smem + C::kOffDO,
                                                      smem + C::kOffDO + 2 * C::kBigPart, r0, t,
                                                      smem + C::kOffDO + C::kBigPart);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(qdo_full);
    }
    bool ok = true;
    for (int s = 0; s < T && ok; ++s) {
      const int key0 = (t0 + s) * RS;
      const int kb = s & 1;
      if (s >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&k_empty[kb], ((s - 2) >> 1) & 1, abort_flag, p.status, 161));
      if (!ok) break;
      uint8_t* kh = smem + C::kOffK + 2 * kb * C::kStepPart;
      convert_tile<D, RS, RS>(k, b, p.Lkv, p.Hkv, hk, key0, kvl, kh, kh + C::kStepPart, 0, t);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&k_full[kb]);
      if (s >= 1) ok = __all_sync(0xffffffffu, mbar_wait(v_empty, (s - 1) & 1, abort_flag, p.status, 162));
      if (!ok) break;
      convert_tile<D, RS, RS, true>(v, b, p.Lkv, p.Hkv, hk, key0, kvl, smem + C::kOffV,
                                    smem + C::kOffV + 2 * C::kStepPart, 0, t, smem + C::kOffV + C::kStepPart);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(v_full);
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kRowsBig, RS, 0, 0);  // Q x K^T, dO x V^T
      constexpr uint32_t idesc_dq = idesc_bf16_f32(kRowsBig, D, 0, 1);  // dS (TMEM) x K (MN-major)
      const uint32_t qa = smem_u32(smem + C::kOffQ), oa = smem_u32(smem + C::kOffDO);
      const SDesc qh = sdesc_split(qa, 16, 1024), ql = sdesc_split(qa + C::kBigPart, 16, 1024);
      const SDesc oh = sdesc_split(oa, 16, 1024), om = sdesc_split(oa + C::kBigPart, 16, 1024),
                  ol = sdesc_split(oa + 2 * C::kBigPart, 16, 1024);
      const uint32_t va = smem_u32(smem + C::kOffV);
      auto k_addr = [&](int s) { return smem_u32(smem + C::kOffK + 2 * (s & 1) * C::kStepPart); };
      auto issue_s = [&](int s) {  // S(s) = Q K(s)^T into S buffer s & 1
        const uint32_t ka = k_addr(s);
        const SDesc kh = sdesc_split(ka, 16, 1024), kl = sdesc_split(ka + C::kStepPart, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * C::kBigBox + (kk & 3) * 32) >> 4;
          const uint32_t bo = ((kk >> 2) * C::kStepBox + (kk & 3) * 32) >> 4;
          mma3_ss(tbase + kColS + (s & 1) * RS, qh, ql, ao, kh, kl, bo, idesc_s, kk > 0);
        }
        mma_commit(&s_ready[s & 1]);
      };
      auto issue_dp = [&]() {  // dP = dO V^T, three-part operands
        const SDesc vh = sdesc_split(va, 16, 1024), vm = sdesc_split(va + C::kStepPart, 16, 1024),
                    vl = sdesc_split(va + 2 * C::kStepPart, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * C::kBigBox + (kk & 3) * 32) >> 4;
          const uint32_t bo = ((kk >> 2) * C::kStepBox + (kk & 3) * 32) >> 4;
          mma5_small_ss(tbase + kColDP, oh, om, ol, ao, vh, vm, vl, bo, idesc_s, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * C::kBigBox + (kk & 3) * 32) >> 4;
          const uint32_t bo = ((kk >> 2) * C::kStepBox + (kk & 3) * 32) >> 4;
          mma_ss_d(tbase + kColDP, oh, ao, vh, bo, idesc_s, 1u);
        }
        mma_commit(dp_ready);
        mma_commit(v_empty);
      };
      bool ok = mbar_wait(qdo_full, 0, abort_flag, p.status, 163);
      for (int s = 0; s < 2 && s < T && ok; ++s) {
        ok = mbar_wait(&k_full[s], 0, abort_flag, p.status, 164);
        if (!ok) break;
        tc_fence_after();
        issue_s(s);
      }
      if (ok) ok = mbar_wait(v_full, 0, abort_flag, p.status, 165);
      if (ok) {
        tc_fence_after();
        issue_dp();
      }
      for (int s = 0; s < T && ok; ++s) {
        ok = mbar_wait(ds_ready, s & 1, abort_flag, p.status, 166);
        if (!ok) break;
        tc_fence_after();
        {  // dQ += dS K (dS hi over the S buffer's first 16 columns, lo in its own buffer)
          const uint32_t ka = k_addr(s);
          const SDesc kh = sdesc_split(ka, C::kStepBox, 1024), kl = sdesc_split(ka + C::kStepPart, C::kStepBox, 1024);
          const uint32_t ah = tbase + kColS + (s & 1) * RS, al = tbase + kColDSlo + (s & 1) * (RS / 2);
#pragma unroll
          for (int kk = 0; kk < RS / 16; ++kk)
            mma3_ts(tbase + 0, ah + kk * 8, al + kk * 8, kh, kl, (16 * kk * 128) >> 4, idesc_dq,
                    (s > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&k_empty[s & 1]);
        if (s + 1 < T) {  // dP(s+1): the softmax has read dP(s)
          ok = mbar_wait(v_full, (s + 1) & 1, abort_flag, p.status, 167);
          if (!ok) break;
          tc_fence_after();
          issue_dp();
        }
        if (s + 2 < T) {  // S(s+2) into the buffer dQ(s) has just read
          ok = mbar_wait(&k_full[s & 1], ((s + 2) >> 1) & 1, abort_flag, p.status, 168);
          if (!ok) break;
          tc_fence_after();
          issue_s(s + 2);
        }
      }
      if (ok) mma_commit(acc_full);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (thread = query row)
    const int i = q0 + warp * 32 + lane;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    const size_t srow = (static_cast<size_t>(b) * p.Hq + h) * p.Lq_pad + i;  // i < Lq_pad always
    const float l2 = p.lse2[srow];
    const float dl = p.delta[srow];
    Span ks = key_span(i, p.Lq, kvl, p.wl, p.wr);
    if (!kLeftBound) ks.lo = 0;
    if (i >= p.Lq) ks.lo = ks.hi = 0;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int s = 0; s < T; ++s) {
      const int kb0 = (t0 + s) * RS;
      const uint32_t s_col = t_lane + kColS + (s & 1) * RS;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_ready[s & 1], (s >> 1) & 1, abort_flag, p.status, 169));
      if (!ok) break;
      tc_fence_after();
      float pr[RS];
      {
        uint32_t sa[32];
        tmem_ld32(s_col, sa);
#pragma unroll
        for (int c = 0; c < RS; ++c) {
          const int kk = kb0 + c;
          pr[c] = (kk >= ks.lo && kk < ks.hi) ? ex2_approx(fmaf(__uint_as_float(sa[c]), sl2, -l2)) : 0.f;
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(dp_ready, s & 1, abort_flag, p.status, 170));
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t da[32];
        tmem_ld32(t_lane + kColDP, da);
        float ds[RS];
#pragma unroll
        for (int c = 0; c < RS; ++c) ds[c] = pr[c] * (__uint_as_float(da[c]) - dl);
        uint32_t hi[16], lo[16];
        split32(ds, hi, lo);
        tmem_st16(s_col, hi);
        tmem_st16(t_lane + kColDSlo + (s & 1) * (RS / 2), lo);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
    }
    if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, p.status, 171));
    if (ok) {
      tc_fence_after();
      const bool st = i < p.Lq;
      float* dst = static_cast<float*>(p.dq) + ((static_cast<size_t>(b) * p.Lq + (st ? i : 0)) * p.Hq + h) * D;
      store_row_f32<D>(t_lane + 0, dst, p.scale, st, T == 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // launched to overlap the dK/dV pass: one CTA waits for that grid before it
  // exits, so this grid completes after it
  if (blockIdx.x == gridDim.x - 1) griddep_wait();
}

template <int D, bool kLeftBound>
cudaError_t run_split_bwd(BwdKParams kp, const BwdArgs& a, cudaStream_t s) {
  const Problem& pb = a.pb;
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  const float* dout = static_cast<const float*>(a.dout);
  {
    using C = SplitDkdvCfg<D>;
    cudaError_t e = ensure_dynamic_smem<bwd_split_dkdv_kernel<D, kLeftBound>>(C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kp.n_tiles = (pb.Lkv + kRowsBig - 1) / kRowsBig;
    kp.n_pairs = pb.B * pb.Hkv;
    kp.pair_group = l2_pair_group(2l * pb.G * pb.Lq * D * 4, kp.n_pairs, 1);
    KernelTimer kt("bwd_dkdv_split_f32", s);
    e = launch_overlapping(bwd_split_dkdv_kernel<D, kLeftBound>, dim3(kp.n_pairs * kp.n_tiles), C::kThreads,
                           C::kSmemBytes, s, kp, q, k, v, dout);
    if (e != cudaSuccess) return e;
  }
  using C = SplitDqCfg<D>;
  cudaError_t e = ensure_dynamic_smem<bwd_split_dq_kernel<D, kLeftBound>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kp.n_tiles = (pb.Lq + kRowsBig - 1) / kRowsBig;
  kp.n_pairs = pb.B * pb.Hq;
  kp.pair_group = l2_pair_group(2l * pb.Lkv * D * 4, kp.n_pairs, pb.G);
  KernelTimer kt("bwd_dq_split_f32", s);
  return launch_overlapping(bwd_split_dq_kernel<D, kLeftBound>, dim3(kp.n_pairs * kp.n_tiles), C::kThreads,
                            C::kSmemBytes, s, kp, q, k, v, dout);
}

}  // namespace

cudaError_t launch_bwd_split_f32(const BwdArgs& a, DeviceStatus* st, cudaStream_t s) {
  const Problem& pb = a.pb;
  PreprocessArgs pa;
  pa.o = a.o;
  pa.dout = a.dout;
  pa.lse = a.lse;
  pa.delta = a.delta;  // padded [B, Hq, Lq_pad] rows, as the 16-bit backward
  pa.lse2 = a.lse2;
  pa.dq_acc = nullptr;
  pa.B = pb.B;
  pa.Lq = pb.Lq;
  pa.Lq_pad = a.Lq_pad;
  pa.Hq = pb.Hq;
  pa.d = pb.d;
  pa.elem = kElemF32;
  cudaError_t e = launch_bwd_preprocess(pa, s);
  if (e != cudaSuccess) return e;
  BwdKParams kp{};
  kp.lse2 = a.lse2;
  kp.delta = a.delta;
  kp.dq = a.dq;
  kp.dk = a.dk;
  kp.dv = a.dv;
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
  kp.scale = pb.scale;
  kp.scale_log2 = pb.scale * kLog2eB;
  kp.status = st;
  const bool left = pb.wl < kWinInf;
  if (pb.d == 64) return left ? run_split_bwd<64, true>(kp, a, s) : run_split_bwd<64, false>(kp, a, s);
  return left ? run_split_bwd<128, true>(kp, a, s) : run_split_bwd<128, false>(kp, a, s);
}

}  // namespace attn
