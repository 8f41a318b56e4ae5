// Forward attention at head_dim 256, bf16 or fp16, on the sm_103a tensor cores.
//
// Same method as the head_dim 64/128 forward (probjax "Attention performance",
// "When to use which" and "Memory"): exact softmax attention tile by tile with
// an online softmax in base 2, O and the per-row LSE as outputs.  At d = 256
// two query tiles no longer fit the 512 TMEM columns (S_A, S_B, O_A, O_B would
// need 768) and a 128-key K/V stage is 128 KB, so this kernel takes one
// 128-row query tile per CTA and 64-key steps:
//   TMEM  S(0) [0,64)  S(1) [64,128)  (double-buffered scores; P over their
//         first 32 columns)  O [256,512)
//   smem  Q 64 KB (four 64-column boxes), K ring 2 x 32 KB, V ring 2 x 32 KB
// Warps 0-3 run the softmax (thread = query row = TMEM lane), warp 4 the TMA
// producer, warp 5 issues the MMAs.  Issue order per step j:
//   PV(j) into O (P(j) from TMEM, V(j) from smem), then S(j+2) into buffer j&1,
// so the softmax of step j+1 runs while PV(j) and S(j+2) execute.  K slots are
// released when their S completes and V slots when their PV completes, so the
// loads of K(j+2) overlap step j.  O is rescaled lazily (threshold 2^8) by the
// softmax warps, after waiting for the PV that last wrote it.
#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kBM = 128;  // query rows per CTA (= TMEM lanes)
constexpr int kBN = 64;   // keys per step
constexpr int kD = 256;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

struct Cfg256 {
  static constexpr int kQBox = kBM * 64 * 2;   // 16 KB: 128 rows x 64 columns
  static constexpr int kKVBox = kBN * 64 * 2;  // 8 KB: 64 rows x 64 columns
  static constexpr int kQBytes = 4 * kQBox;    // 64 KB
  static constexpr int kSlotBytes = 4 * kKVBox;  // 32 KB: one K or V tile
  static constexpr int kSlots = 2;
  static constexpr int kOffK = kQBytes;
  static constexpr int kOffV = kOffK + kSlots * kSlotBytes;
  static constexpr int kOffBars = kOffV + kSlots * kSlotBytes;
  // full_k[2] empty_k[2] full_v[2] empty_v[2] q_full s_full[2] p_full[2] o_step o_final
  static constexpr int kNumBars = 4 * kSlots + 7;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;  // + alignment slack
  static constexpr int kThreads = 192;
};

struct Fwd256Params {
  void* o;
  float* lse;
  const int32_t* kv_lens;
  int Lq, Lkv, Hq, Hkv, G, causal, wl, wr, n_qtiles, n_pairs, pair_group;
  const int32_t* q_seg;  // [B, Lq] segment ids (kSeg builds)
  const int32_t* kv_seg;
  const int4* seg_qblk;  // segment block summary or nullptr
  const int4* seg_kblk;
  int nqb, nkb;
  float scale_log2;
  DeviceStatus* status;
};

template <bool kF16, bool kSeg>
__global__ void __launch_bounds__(Cfg256::kThreads, 1)
    fwd_d256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const Fwd256Params p) {
  using C = Cfg256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* full_k = bars;
  uint64_t* empty_k = bars + 2;
  uint64_t* full_v = bars + 4;
  uint64_t* empty_v = bars + 6;
  uint64_t* q_full = bars + 8;
  uint64_t* s_full = bars + 9;   // [2] S(j) computed, one per buffer (j & 1)
  uint64_t* p_full = bars + 11;  // [2] P(j) written, one per buffer (128 arrivals)
  uint64_t* o_step = bars + 13;  // PV(j) completed (one phase per step)
  uint64_t* o_final = bars + 14;  // the last PV completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  // 1-D grid over (b, hq) pairs x query tiles in L2 groups, the longest causal
  // tiles of a group first
  const TileCoord tc = grouped_tile(blockIdx.x, p.n_pairs, p.n_qtiles, p.pair_group);
  const int qt = p.causal ? p.n_qtiles - 1 - tc.rank : tc.rank;
  const int row0 = qt * kBM;
  const int hq = tc.pair % p.Hq, b = tc.pair / p.Hq;
  const int hkv = hq / p.G;
  // launched to overlap the tail of the kernel before it: nothing in global
  // memory is read before that grid has completed
  griddep_wait();
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);

  // key steps [t0, t0 + n): from the first key of row row0 to the last key of
  // the tile's last row, narrowed to the keys whose blocks may share an id
  int t0 = 0, n = 0;
  {
    const int last = min(row0 + kBM - 1, p.Lq - 1);
    int lo = key_span(row0, p.Lq, kvl, p.wl, p.wr).lo;
    int hi = key_span(last, p.Lq, kvl, p.wl, p.wr).hi;
    if (kSeg && p.seg_qblk != nullptr) {
      const int4 r = seg_block(p.seg_qblk, b, p.nqb, row0 / kSegBlock);
      lo = max(lo, r.z);
      hi = min(hi, r.w);
    }
    if (hi > lo) {
      t0 = lo / kBN;
      n = (hi + kBN - 1) / kBN - t0;
    }
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < 8; ++s) mbar_init(&bars[s], 1);
    mbar_init(q_full, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 128);
    }
    mbar_init(o_step, 1);
    mbar_init(o_final, 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  griddep_launch_dependents();  // the next kernel waits for this grid before it reads anything

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, C::kQBytes);
      for (int h = 0; h < 4; ++h) tma_load_4d(sQ + h * C::kQBox, &tm_q, q_full, h * 64, row0, hq, b);
      // K(u) and V(u) in step order; a K slot is free once its S completed, a
      // V slot once its PV completed
      for (int u = 0; u < n; ++u) {
        const int st = u & 1, r = u >> 1;
        const int key0 = (t0 + u) * kBN;
        if (r > 0 && !mbar_wait(&empty_k[st], (r - 1) & 1, abort_flag, p.status, 100)) break;
        mbar_arrive_expect_tx(&full_k[st], C::kSlotBytes);
        for (int h = 0; h < 4; ++h)
          tma_load_4d(sK + st * C::kSlotBytes + h * C::kKVBox, &tm_k, &full_k[st], h * 64, key0, hkv, b);
        if (r > 0 && !mbar_wait(&empty_v[st], (r - 1) & 1, abort_flag, p.status, 101)) break;
        mbar_arrive_expect_tx(&full_v[st], C::kSlotBytes);
        for (int h = 0; h < 4; ++h)
          tma_load_4d(sV + st * C::kSlotBytes + h * C::kKVBox, &tm_v, &full_v[st], h * 64, key0, hkv, b);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = idesc_16_f32<kF16>(kBM, kBN, 0, 0);  // Q (K-major) x K^T (K-major)
      constexpr uint32_t idesc_o = idesc_16_f32<kF16>(kBM, kD, 0, 1);   // P (TMEM) x V (MN-major)
      const SDesc dq = sdesc_split(smem_u32(sQ), 16, 1024);
      const SDesc dk = sdesc_split(smem_u32(sK), 16, 1024);
      const SDesc dv = sdesc_split(smem_u32(sV), C::kKVBox, 1024);  // 64-column atoms of V along N
      // S(buf) = Q K^T: 16 k-steps of 16 along d; d column block h is its own box
      auto issue_s = [&](int buf, int st) {
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint32_t qo = ((k >> 2) * C::kQBox + (k & 3) * 32) >> 4;
          const uint32_t ko = (st * C::kSlotBytes + (k >> 2) * C::kKVBox + (k & 3) * 32) >> 4;
          mma_ss_d(tbase + buf * kBN, dq, qo, dk, ko, idesc_s, k > 0);
        }
      };
      // O (+)= P V: 4 k-steps of 16 keys; P advances 8 TMEM columns, V 16 rows (2 KB)
      auto issue_pv = [&](int buf, int st, int acc) {
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          mma_ts_d(tbase + 256, tbase + buf * kBN + k * 8, dv, (st * C::kSlotBytes + k * 2048) >> 4, idesc_o,
                   (acc || k > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, 102);
      for (int u = 0; u < 2 && u < n && ok; ++u) {
        ok = mbar_wait(&full_k[u], 0, abort_flag, p.status, 103);
        if (!ok) break;
        tc_fence_after();
        issue_s(u, u);
        mma_commit(&s_full[u]);
        mma_commit(&empty_k[u]);
      }
      for (int j = 0; j < n && ok; ++j) {
        const int buf = j & 1, st = j & 1;
        ok = mbar_wait(&p_full[buf], (j >> 1) & 1, abort_flag, p.status, 104);
        if (!ok) break;
        ok = mbar_wait(&full_v[st], (j >> 1) & 1, abort_flag, p.status, 105);
        if (!ok) break;
        tc_fence_after();
        issue_pv(buf, st, j > 0);
        mma_commit(o_step);
        mma_commit(&empty_v[st]);
        if (j == n - 1) mma_commit(o_final);
        if (j + 2 < n) {
          // S(j+2) overwrites buffer j&1 after PV(j) has read P(j) from it
          // (tcgen05.mma of one thread execute in issue order)
          ok = mbar_wait(&full_k[st], ((j + 2) >> 1) & 1, abort_flag, p.status, 106);
          if (!ok) break;
          tc_fence_after();
          issue_s(buf, st);
          mma_commit(&s_full[buf]);
          mma_commit(&empty_k[st]);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int row = row0 + warp * 32 + lane;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t o_addr = t_lane + 256;
    Span span = key_span(row, p.Lq, kvl, p.wl, p.wr);
    if (row >= p.Lq) span.lo = span.hi = 0;
    const int my_seg = (kSeg && row < p.Lq) ? __ldg(p.q_seg + static_cast<size_t>(b) * p.Lq + row) : 0;
    const int32_t* kid = kSeg ? p.kv_seg + static_cast<size_t>(b) * p.Lkv : nullptr;
    const bool kid_vec = kSeg && ((static_cast<size_t>(b) * p.Lkv) & 3) == 0;
    const int4 qrec = (kSeg && p.seg_qblk != nullptr) ? seg_block(p.seg_qblk, b, p.nqb, row0 / kSegBlock)
                                                      : make_int4(0, -1, 0, 0);
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int buf = j & 1;
      const int col0 = (t0 + j) * kBN;
      const uint32_t s_addr = t_lane + buf * kBN;
      // segment ids of the step's 64 keys (before S is ready); a tile whose
      // query and key blocks hold one and the same id needs no compare
      uint32_t segbits[2] = {~0u, ~0u};
      const bool seg_all = kSeg && p.seg_kblk != nullptr &&
                           seg_same_single_id(qrec, seg_block(p.seg_kblk, b, p.nkb, col0 / kSegBlock));
      if (kSeg && !seg_all) {
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
          uint32_t bits = 0u;
#pragma unroll 2
          for (int i = 0; i < 32; i += 4) {
            const int4 id = load_ids4(kid, col0 + 32 * w2 + i, kvl, kid_vec);
            bits |= (static_cast<uint32_t>(id.x == my_seg) | (static_cast<uint32_t>(id.y == my_seg) << 1) |
                     (static_cast<uint32_t>(id.z == my_seg) << 2) | (static_cast<uint32_t>(id.w == my_seg) << 3))
                    << i;
          }
          segbits[w2] = bits;
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[buf], (j >> 1) & 1, abort_flag, p.status, 107));
      if (!ok) break;
      tc_fence_after();
      uint32_t sa[32], sb[32];
      tmem_ld32_pair(s_addr, s_addr + 32, sa, sb);
      float s[kBN];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(sa[i]);
        s[32 + i] = __uint_as_float(sb[i]);
      }
      if (col0 < span.lo || col0 + kBN > span.hi) {
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (col0 + i < span.lo || col0 + i >= span.hi) s[i] = -INFINITY;
      }
      if (kSeg && !seg_all) {
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (!((segbits[i / 32] >> (i % 32)) & 1u)) s[i] = -INFINITY;
      }
      // row max: 8 chains of three-input max, then a short tree
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(s[k], s[8 + k]);  // columns 0..15
#pragma unroll
      for (int i = 16; i < kBN; i += 16)  // then 16 more a step: the last reads column kBN - 1
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = max3f(mx8[k], s[i + k], s[i + 8 + k]);
      const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
      const float m_tile = mx * sl2;
      const bool grow = m_tile > m_used + kRescaleThreshold;
      const float m_new = grow ? m_tile : m_used;
      const float alpha = grow ? ex2_approx(m_used - m_new) : 1.0f;
      l_sum *= alpha;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O was last written by PV(j-1), which may still run: wait for it.
        // At this point PV(j-2) has completed (it precedes S(j) in issue
        // order) and PV(j) is not issued, so the phase query is unambiguous.
        ok = __all_sync(0xffffffffu, mbar_wait(o_step, (j - 1) & 1, abort_flag, p.status, 108));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(o_addr + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(o_addr + c * 32, r);
        }
      }
      m_used = m_new;
      const float mb = (m_used == -INFINITY) ? 0.f : m_used;
      // P = 2^(s sl2 - mb), two columns per paired fp32 instruction
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nmb2 = f2_pack(-mb, -mb);
      uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), sl2x2, nmb2), t0, t1);
          const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
          ls2[i & 1] = f2_add(ls2[i & 1], f2_pack(p0, p1));
          pk[i] = pack2<kF16>(p0, p1);
        }
        tmem_st16(s_addr + c * 16, pk);
      }
      float la, lb, lc, ld;
      f2_unpack(ls2[0], la, lb);
      f2_unpack(ls2[1], lc, ld);
      l_sum += (la + lb) + (lc + ld);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[buf]);
    }
    // epilogue: O / l -> 16-bit, LSE
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_final, 0, abort_flag, p.status, 109));
    if (ok) {
      tc_fence_after();
      const float inv_l = l_sum > 0.f ? 1.0f / l_sum : 0.f;
      // O goes through the Q buffer, idle once o_final has completed (every
      // MMA is done), and out with TMA stores that clip the rows past Lq
#pragma unroll 1
      for (int h = 0; h < kD / 64; ++h)
        stage_row16<64, kF16>(o_addr + h * 64, sQ, warp * 32 + lane, inv_l, n == 0, h * 64);
      fence_proxy_async_smem();
      if (row < p.Lq)
        p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Lq + row] =
            l_sum > 0.f ? (m_used + lg2_approx(l_sum)) * kLn2 : -INFINITY;
    }
    named_barrier_sync(1, kBM);  // every softmax thread gets here (a failed wait only skips work)
    if (threadIdx.x == 0 && *abort_flag == 0 && row0 < p.Lq) {
#pragma unroll
      for (int h = 0; h < kD / 64; ++h) tma_store_4d(&tm_o, sQ + h * C::kQBox, h * 64, row0, hq, b);
      tma_store_commit();
      tma_store_wait_read();  // the shared memory is released when the CTA exits
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <bool kF16, bool kSeg>
cudaError_t launch_fwd256_inst(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& to, const Fwd256Params& kp, dim3 grid, cudaStream_t stream) {
  cudaError_t e = ensure_dynamic_smem<fwd_d256_kernel<kF16, kSeg>>(Cfg256::kSmemBytes);
  if (e != cudaSuccess) return e;
  KernelTimer kt("fwd", stream);
  return launch_overlapping(fwd_d256_kernel<kF16, kSeg>, grid, Cfg256::kThreads, Cfg256::kSmemBytes, stream, tq, tk, tv,
                            to, kp);
}

}  // namespace

cudaError_t launch_fwd_d256(const FwdArgs& a, DeviceStatus* st, cudaStream_t stream) {
  const Problem& pb = a.pb;
  const int elem = pb.f16 ? kElemF16 : kElemBF16;
  CUtensorMap tq, tk, tv;
  if (!make_bshd_tmap(&tq, a.q, elem, pb.B, pb.Lq, pb.Hq, kD, 64, kBM)) return cudaErrorInvalidValue;
  if (!make_bshd_tmap(&tk, a.k, elem, pb.B, pb.Lkv, pb.Hkv, kD, 64, kBN)) return cudaErrorInvalidValue;
  if (!make_bshd_tmap(&tv, a.v, elem, pb.B, pb.Lkv, pb.Hkv, kD, 64, kBN)) return cudaErrorInvalidValue;
  CUtensorMap to;  // the output leaves through TMA stores of the query tile's boxes
  if (!make_bshd_tmap(&to, a.o, elem, pb.B, pb.Lq, pb.Hq, kD, 64, kBM)) return cudaErrorInvalidValue;
  Fwd256Params kp;
  kp.o = a.o;
  kp.lse = a.lse;
  kp.kv_lens = pb.kv_lens;
  kp.Lq = pb.Lq;
  kp.Lkv = pb.Lkv;
  kp.Hq = pb.Hq;
  kp.Hkv = pb.Hkv;
  kp.G = pb.G;
  kp.causal = pb.causal;
  kp.wl = pb.wl;
  kp.wr = pb.wr;
  kp.n_qtiles = (pb.Lq + kBM - 1) / kBM;
  kp.n_pairs = pb.B * pb.Hq;
  kp.pair_group = l2_pair_group(2l * pb.Lkv * kD * 2, kp.n_pairs, pb.G);
  kp.q_seg = pb.q_seg;
  kp.kv_seg = pb.kv_seg;
  kp.seg_qblk = pb.seg_qblk;
  kp.seg_kblk = pb.seg_kblk;
  kp.nqb = (pb.Lq + kSegBlock - 1) / kSegBlock;
  kp.nkb = (pb.Lkv + kSegBlock - 1) / kSegBlock;
  kp.scale_log2 = pb.scale * kLog2e;
  kp.status = st;
  const dim3 grid(kp.n_pairs * kp.n_qtiles);
  if (pb.q_seg != nullptr)
    return pb.f16 ? launch_fwd256_inst<true, true>(tq, tk, tv, to, kp, grid, stream)
                  : launch_fwd256_inst<false, true>(tq, tk, tv, to, kp, grid, stream);
  return pb.f16 ? launch_fwd256_inst<true, false>(tq, tk, tv, to, kp, grid, stream)
                : launch_fwd256_inst<false, false>(tq, tk, tv, to, kp, grid, stream);
}

}  // namespace attn
