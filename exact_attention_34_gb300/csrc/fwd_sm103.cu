// Forward attention, bf16 or fp16, head_dim 64/128, on the sm_103a tensor cores.
//
// Method (probjax "Attention performance", sections "When to use which" and
// "Memory"): exact softmax attention computed tile by tile with an online
// softmax, so memory stays linear in the sequence length; the output and the
// per-row log-sum-exp are the residuals of the backward.  The softmax is
// evaluated in base 2: t = s * scale * log2(e), P = 2^(t - m), and
// LSE = ln(2) * (m + log2(l)).
//
// One CTA owns two 128-row query tiles (A and B) of one (batch, head) and
// streams the K/V tiles of the head's KV head (GQA: h / G) through a ring of
// shared-memory slots filled by TMA.  Warp roles:
//   warps 0-3  softmax of tile A (thread = query row = TMEM lane)
//   warps 4-7  softmax of tile B
//   warp  8    TMA producer (one lane)
//   warp  9    tcgen05.mma issuer (one lane); owns the TMEM allocation
// TMEM (512 columns): S_A [0,128) S_B [128,256) O_A [256,256+d) O_B [384,384+d).
// P (bf16) is written over the first 64 columns of its S tile and is the A
// operand of O += P V straight from TMEM.  The MMA issue order per KV tile j is
//   PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
// so each softmax group has the other tile's two MMAs to hide behind, and
// S_X(j+1) is issued after the PV_X(j) that reads the P stored in S_X's
// columns (tcgen05.mma ops of one thread execute in issue order).  O is
// rescaled lazily: only when a row's running maximum grows by more than
// 2^8 (kRescaleThreshold), done by the softmax warps in TMEM.
//
// Split key ranges (left-bounded builds, n_split > 1): every tile pair gets
// n_split programs and program sp takes piece sp of the pair's key stream,
// cut into pieces = min(n_split, ceil(n / split_chunk)) near-equal parts;
// programs past the last piece exit at once.  A pair left whole writes o and
// lse as usual.  A piece of a cut pair writes O / l of its keys in fp32 and
// its own log-sum-exp to the partial buffers ([B, Hq, n_split, Lq, dh] and
// [B, Hq, n_split, Lq]), then takes a ticket from the pair's counter; the
// piece that draws the last ticket merges all pieces by their log-sum-exps
// (from L2, no wait on anyone) and writes o and lse, and resets the counter.
// So a KV-length mask that puts most keys in a few batch elements still
// spreads them over every SM.
#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kBM = 128;  // rows per query tile (= TMEM lanes)
constexpr int kBN = 128;  // keys per KV tile
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct FwdCfg {
  static constexpr int kQTileBytes = kBM * D * 2;     // one query tile, bf16
  static constexpr int kSlotBytes = kBN * D * 2;      // one K or V tile
  static constexpr int kBoxBytes = 128 * 64 * 2;      // one TMA box (128 rows x 64 cols)
  static constexpr int kSlots = (D == 128) ? 2 : 4;   // ring depth in (K, V) stages
  static constexpr int kStageBytes = 2 * kSlotBytes;  // K at 0, V at kSlotBytes
  static constexpr int kOffSlots = 2 * kQTileBytes;
  static constexpr int kOffBars = kOffSlots + kSlots * kStageBytes;
  static constexpr int kNumBars = 2 * kSlots + 7;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;  // + alignment slack
  static constexpr int kThreads = 320;
};

struct FwdKParams {
  void* o;
  float* lse;
  const int32_t* kv_lens;
  int Lq, Lkv, Hq, Hkv, G, causal, wl, wr, n_qblocks, n_pairs, pair_group;
  int dh;  // stored head_dim (32 runs as D = 64 with zero-filled columns)
  const int32_t* q_seg;   // [B, Lq] segment ids (kSeg builds)
  const int32_t* kv_seg;  // [B, Lkv]
  const int4* seg_qblk;   // segment block summary (kSeg builds; nullptr: none)
  const int4* seg_kblk;
  int nqb, nkb;           // 128-position blocks per sequence: ceil(Lq/128), ceil(Lkv/128)
  float scale_log2;
  DeviceStatus* status;
  int n_split;            // 1, or copies of the tile-pair grid (split key ranges)
  int split_chunk;        // KV tiles a piece may hold before the stream is cut further
  float* o_part;          // [B, Hq, n_split, Lq, dh] fp32 (n_split > 1)
  float* lse_part;        // [B, Hq, n_split, Lq]
  int* counters;          // [n_pairs * n_qblocks] tickets, zero on entry and on exit
};

template <int D, bool kLeftBound, bool kF16, bool kSeg>
__global__ void __launch_bounds__(320, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdKParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem;  // tile A at 0, tile B at kQTileBytes
  uint8_t* sSlots = smem + C::kOffSlots;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kSlots;
  uint64_t* q_full = bars + 2 * C::kSlots;
  uint64_t* s_full = q_full + 1;  // [2]
  uint64_t* p_full = q_full + 3;  // [2]
  uint64_t* o_full = q_full + 5;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_piece = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = warp_id(), lane = lane_id();
  // 1-D grid over (b, hq) pairs x query blocks in L2 groups; the longest
  // causal blocks of a group start first.
  // split key ranges: the pieces of one pair are neighbours in the grid, so
  // the longest pairs' pieces all start in the first wave
  const int sp = kLeftBound ? static_cast<int>(blockIdx.x) % p.n_split : 0;  // key-range piece
  const int item = kLeftBound ? static_cast<int>(blockIdx.x) / p.n_split : static_cast<int>(blockIdx.x);
  const TileCoord tc = grouped_tile(item, p.n_pairs, p.n_qblocks, p.pair_group);
  const int qb = p.causal ? p.n_qblocks - 1 - tc.rank : tc.rank;
  const int hq = tc.pair % p.Hq, b = tc.pair / p.Hq;
  const int hkv = hq / p.G;
  // launched to overlap the tail of the kernel before it: nothing in global
  // memory is read before that grid has completed
  griddep_wait();
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);

  // KV tiles [first, first + count) query tile x needs: both ends of a row's
  // valid keys grow with the row index.  The two tiles share one K/V stream
  // over the union of their ranges, [jlo, jlo + n) (consecutive rows: no gap).
  auto tile_range = [&](int x, int& first, int& count) {
    const int row0 = qb * 2 * kBM + x * kBM;
    first = 0;
    count = 0;
    if (row0 >= p.Lq) return;
    const int last = min(row0 + kBM - 1, p.Lq - 1);
    int lo = key_span(row0, p.Lq, kvl, p.wl, p.wr).lo;
    int hi = key_span(last, p.Lq, kvl, p.wl, p.wr).hi;
    if (kSeg && p.seg_qblk != nullptr) {  // keys whose blocks may share an id with this block
      const int4 r = seg_block(p.seg_qblk, b, p.nqb, row0 / kSegBlock);
      lo = max(lo, r.z);
      hi = min(hi, r.w);
    }
    if (hi <= lo) return;
    first = lo / kBN;
    count = (hi + kBN - 1) / kBN - first;
  };
  int jlo_a, n_a, jlo_b, n_b;
  tile_range(0, jlo_a, n_a);
  tile_range(1, jlo_b, n_b);
  // without a left bound every range starts at key tile 0 (compile-time);
  // otherwise the stream is the hull of the two ranges (with segment ids the
  // ranges need not grow with the row index, and tiles between two disjoint
  // ranges are streamed and released unused)
  int jlo = 0, n = max(n_a, n_b);
  if (kLeftBound) {
    jlo = n_a == 0 ? jlo_b : n_b == 0 ? jlo_a : min(jlo_a, jlo_b);
    n = n_a == 0 ? n_b : n_b == 0 ? n_a : max(jlo_a + n_a, jlo_b + n_b) - jlo;
  }
  int pieces = 1;
  if (kLeftBound && p.n_split > 1) {
    pieces = n == 0 ? 1 : min(p.n_split, (n + p.split_chunk - 1) / p.split_chunk);
    if (sp >= pieces) return;  // nothing of this pair's stream left
    // piece sp is the stream's tiles [c0, c1); each tile keeps its part of it
    const int c0 = jlo + static_cast<int>(static_cast<long>(sp) * n / pieces);
    const int c1 = jlo + static_cast<int>(static_cast<long>(sp + 1) * n / pieces);
    auto clip = [&](int& first, int& count) {
      const int a = max(first, c0), e = min(first + count, c1);
      first = e > a ? a : c0;
      count = e > a ? e - a : 0;
    };
    clip(jlo_a, n_a);
    clip(jlo_b, n_b);
    jlo = c0;
    n = (n_a == 0 && n_b == 0) ? 0 : c1 - c0;
  }
  const bool split = pieces > 1;  // this pair is cut: partials, then a ticket
  const int lo_a = kLeftBound ? jlo_a - jlo : 0, lo_b = kLeftBound ? jlo_b - jlo : 0;  // tile starts in the stream

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 128);
      mbar_init(&o_full[x], 1);
    }
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
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t qbytes = (n_a > 0 ? C::kQTileBytes : 0) + (n_b > 0 ? C::kQTileBytes : 0);
      mbar_arrive_expect_tx(q_full, qbytes);
      for (int x = 0; x < 2; ++x) {
        if ((x == 0 ? n_a : n_b) == 0) continue;
        const int row0 = qb * 2 * kBM + x * kBM;
        for (int h = 0; h < D / 64; ++h)
          tma_load_4d(sQ + x * C::kQTileBytes + h * C::kBoxBytes, &tm_q, q_full, h * 64, row0, hq, b);
      }
      for (int u = 0; u < n; ++u) {
        const int st = u % C::kSlots, r = u / C::kSlots;
        if (r > 0 && !mbar_wait(&empty[st], (r - 1) & 1, abort_flag, p.status, 1)) break;
        mbar_arrive_expect_tx(&full[st], C::kStageBytes);
        uint8_t* dst = sSlots + st * C::kStageBytes;
        const int key0 = (jlo + u) * kBN;
        for (int h = 0; h < D / 64; ++h) {
          tma_load_4d(dst + h * C::kBoxBytes, &tm_k, &full[st], h * 64, key0, hkv, b);
          tma_load_4d(dst + C::kSlotBytes + h * C::kBoxBytes, &tm_v, &full[st], h * 64, key0, hkv, b);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = idesc_16_f32<kF16>(kBM, kBN, 0, 0);  // Q (K-major) x K^T (K-major)
      constexpr uint32_t idesc_o = idesc_16_f32<kF16>(kBM, D, 0, 1);    // P (TMEM) x V (MN-major)
      const SDesc dq[2] = {sdesc_split(smem_u32(sQ), 16, 1024), sdesc_split(smem_u32(sQ) + C::kQTileBytes, 16, 1024)};
      const SDesc dk0 = sdesc_split(smem_u32(sSlots), 16, 1024);
      const SDesc dv0 = sdesc_split(smem_u32(sSlots) + C::kSlotBytes, C::kBoxBytes, 1024);
      constexpr uint32_t kStage16 = C::kStageBytes >> 4;
      // S_x = Q_x K^T : 16-wide k-steps along d; each 64-column half of d is its own TMA box.
      auto issue_s = [&](int x, int st) {
        const uint32_t so = st * kStage16;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * C::kBoxBytes + (k & 3) * 32) >> 4;
          mma_ss_d(tbase + x * 128, dq[x], off, dk0, so + off, idesc_s, k > 0);
        }
      };
      // O_x (+)= P_x V : 16-key k-steps; P advances 8 TMEM columns, V 16 rows (2 KB).
      auto issue_pv = [&](int x, int st, int acc) {
        const uint32_t so = st * kStage16;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          mma_ts_d(tbase + 256 + x * 128, tbase + x * 128 + k * 8, dv0, so + k * 128, idesc_o, (acc || k > 0) ? 1u : 0u);
      };
      // stream step u serves tile x when lo_x <= u < lo_x + n_x; the tile's own
      // step index u - lo_x drives its barrier parities
      auto in_a = [&](int u) { return u >= lo_a && u < lo_a + n_a; };
      auto in_b = [&](int u) { return u >= lo_b && u < lo_b + n_b; };
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, 2);
      if (ok) ok = mbar_wait(&full[0], 0, abort_flag, p.status, 3);
      if (ok) {
        tc_fence_after();
        if (in_a(0)) { issue_s(0, 0); mma_commit(&s_full[0]); }
        if (in_b(0)) { issue_s(1, 0); mma_commit(&s_full[1]); }
      }
      for (int u = 0; u < n && ok; ++u) {
        const int st = u % C::kSlots;
        const int stn = (u + 1) % C::kSlots;
        const bool has_next = u + 1 < n;
        if (in_a(u)) {
          const int ja = u - lo_a;
          ok = mbar_wait(&p_full[0], ja & 1, abort_flag, p.status, 5);
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, st, ja > 0);
          if (ja == n_a - 1) mma_commit(&o_full[0]);
        }
        if (has_next) {
          ok = mbar_wait(&full[stn], ((u + 1) / C::kSlots) & 1, abort_flag, p.status, 6);
          if (!ok) break;
          tc_fence_after();
          if (in_a(u + 1)) { issue_s(0, stn); mma_commit(&s_full[0]); }
        }
        if (in_b(u)) {
          const int jb = u - lo_b;
          ok = mbar_wait(&p_full[1], jb & 1, abort_flag, p.status, 7);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, st, jb > 0);
          if (jb == n_b - 1) mma_commit(&o_full[1]);
        }
        mma_commit(&empty[st]);
        if (has_next && in_b(u + 1)) { issue_s(1, stn); mma_commit(&s_full[1]); }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2, wq = warp & 3;
    const int row = qb * 2 * kBM + x * kBM + wq * 32 + lane;
    const int n_x = x == 0 ? n_a : n_b;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t s_addr = t_lane + x * 128;
    const uint32_t o_addr = t_lane + 256 + x * 128;
    // a row's valid keys [span.lo, span.hi); without a left window bound the
    // lower end is 0 (kept out of the registers of the causal/unmasked build)
    Span span = key_span(row, p.Lq, kvl, p.wl, p.wr);
    if (!kLeftBound) span.lo = 0;
    if (row >= p.Lq) span.lo = span.hi = 0;
    // segment masks: a key counts only if its id equals the row's
    const int my_seg = (kSeg && row < p.Lq) ? __ldg(p.q_seg + static_cast<size_t>(b) * p.Lq + row) : 0;
    const int32_t* kid = kSeg ? p.kv_seg + static_cast<size_t>(b) * p.Lkv : nullptr;
    const bool kid_vec = kSeg && ((static_cast<size_t>(b) * p.Lkv) & 3) == 0;
    // this query block's summary; (0, -1) never counts as a single id
    const int row0x = qb * 2 * kBM + x * kBM;
    const int4 qrec = (kSeg && p.seg_qblk != nullptr && row0x < p.Lq)
                          ? seg_block(p.seg_qblk, b, p.nqb, row0x / kSegBlock)
                          : make_int4(0, -1, 0, 0);
    const int jbase = kLeftBound ? (x == 0 ? jlo_a : jlo_b) : 0;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n_x; ++j) {
      const int col0 = (jbase + j) * kBN;
      // segment masks: bit i says key col0 + i has the row's id (loaded while
      // the tensor core computes S, so the ids are not live next to S)
      uint32_t segbits[kBN / 32];
      // query and key block hold one and the same id: every pair matches
      const bool seg_all =
          kSeg && p.seg_kblk != nullptr && seg_same_single_id(qrec, seg_block(p.seg_kblk, b, p.nkb, jbase + j));
      if (kSeg && !seg_all) {
#pragma unroll
        for (int w4 = 0; w4 < kBN / 32; ++w4) {
          uint32_t bits = 0u;
#pragma unroll 2
          for (int i = 0; i < 32; i += 4) {
            const int4 id = load_ids4(kid, col0 + 32 * w4 + i, kvl, kid_vec);
            bits |= (static_cast<uint32_t>(id.x == my_seg) | (static_cast<uint32_t>(id.y == my_seg) << 1) |
                     (static_cast<uint32_t>(id.z == my_seg) << 2) | (static_cast<uint32_t>(id.w == my_seg) << 3))
                    << i;
          }
          segbits[w4] = bits;
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[x], j & 1, abort_flag, p.status, 8));
      if (!ok) break;
      tc_fence_after();
      uint32_t sraw[kBN];
      tmem_ld128(s_addr, sraw);
      float s[kBN];
#pragma unroll
      for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(sraw[i]);
      if ((kLeftBound && col0 < span.lo) || col0 + kBN > span.hi) {
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if ((kLeftBound && col0 + i < span.lo) || col0 + i >= span.hi) s[i] = -INFINITY;
      }
      if (kSeg && !seg_all) {
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (!((segbits[i / 32] >> (i % 32)) & 1u)) s[i] = -INFINITY;
      }
      // row max: 8 independent chains of three-input max, then a short tree
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(s[k], s[8 + k]);  // columns 0..15
#pragma unroll
      for (int i = 16; i < kBN; i += 16)  // then 16 more a step: the last reads column kBN - 1
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = max3f(mx8[k], s[i + k], s[i + 8 + k]);
      const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
      const float m_tile = mx * sl2;  // scale > 0, so the max commutes with the scaling
      const bool grow = m_tile > m_used + kRescaleThreshold;
      const float m_new = grow ? m_tile : m_used;
      const float alpha = grow ? ex2_approx(m_used - m_new) : 1.0f;
      l_sum *= alpha;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
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
      mbar_arrive(&p_full[x]);
    }
    // epilogue: O / l -> bf16, LSE
    if (ok && n_x > 0) ok = __all_sync(0xffffffffu, mbar_wait(&o_full[x], 0, abort_flag, p.status, 9));
    if (ok) {
      tc_fence_after();
      const float inv_l = l_sum > 0.f ? 1.0f / l_sum : 0.f;
      // a piece of a split stream writes fp32 partials, a whole stream the output
      const size_t prow = ((static_cast<size_t>(b) * p.Hq + hq) * p.n_split + sp) * p.Lq + row;
      if (split) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          if (c * 32 >= p.dh) break;
          uint32_t r[32];
          if (n_x > 0) {
            tmem_ld32(o_addr + c * 32, r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          if (row < p.Lq) {
            float4* dst = reinterpret_cast<float4*>(p.o_part + prow * p.dh + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv_l, __uint_as_float(r[4 * i + 1]) * inv_l,
                                   __uint_as_float(r[4 * i + 2]) * inv_l, __uint_as_float(r[4 * i + 3]) * inv_l);
          }
        }
      } else {
        // O goes through this tile's Q buffer, idle once o_full[x] has
        // completed (every MMA of the tile is done), and out with TMA stores
        // below, which clip the rows past Lq and the columns past the stored
        // head_dim (a store of each thread's own row would put 32 rows, a row
        // stride apart, into every store instruction)
        stage_row16<D, kF16>(o_addr, sQ + x * C::kQTileBytes, wq * 32 + lane, inv_l, n_x == 0);
        fence_proxy_async_smem();
      }
      if (row < p.Lq) {
        const float lv = l_sum > 0.f ? (m_used + lg2_approx(l_sum)) * kLn2 : -INFINITY;
        if (split)
          p.lse_part[prow] = lv;
        else
          p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Lq + row] = lv;
      }
    }
    if (!split) {
      // every thread of this softmax warpgroup reaches this point (a failed
      // wait only skips work)
      const int row0 = qb * 2 * kBM + x * kBM;
      named_barrier_sync(2 + x, kBM);
      if ((threadIdx.x & (kBM - 1)) == 0 && *abort_flag == 0 && row0 < p.Lq) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_store_4d(&tm_o, sQ + x * C::kQTileBytes + c * C::kBoxBytes, c * 64, row0, hq, b);
        tma_store_commit();
        tma_store_wait_read();  // the shared memory is released when the CTA exits
      }
    }
    if (split) {
      // every softmax thread of the CTA reaches this point (a failed wait only
      // skips work), so the 256-thread named barrier always completes
      __threadfence();  // this row's partial is visible device-wide
      named_barrier_sync(1, 2 * kBM);
      if (threadIdx.x == 0) {
        const int ticket = atomicAdd(p.counters + item, 1);
        const int last = ticket == pieces - 1;
        if (last) p.counters[item] = 0;  // ready for the next call
        *last_piece = last;
      }
      named_barrier_sync(1, 2 * kBM);
      if (*last_piece && row < p.Lq) {
        __threadfence();
        // merge the pieces of this row by their log-sum-exps (natural log)
        const size_t row0p = (static_cast<size_t>(b) * p.Hq + hq) * p.n_split * p.Lq + row;
        const size_t lstride = p.Lq;
        float m = -INFINITY;
        for (int t = 0; t < pieces; ++t) m = fmaxf(m, __ldcg(p.lse_part + row0p + t * lstride));
        float tot = 0.f;
        if (m != -INFINITY)
          for (int t = 0; t < pieces; ++t) {
            const float ls = __ldcg(p.lse_part + row0p + t * lstride);
            if (ls != -INFINITY) tot += expf(ls - m);
          }
        const float inv = m == -INFINITY ? 0.f : 1.0f / tot;
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) +
                         ((static_cast<size_t>(b) * p.Lq + row) * p.Hq + hq) * p.dh;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          if (c * 32 >= p.dh) break;
          float acc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = 0.f;
          // two pieces a step, their 16 loads in flight together
          for (int t0 = 0; t0 < pieces && m != -INFINITY; t0 += 2) {
            float w[2];
            float4 v4[2][8];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int t = t0 + u;
              const float ls = t < pieces ? __ldcg(p.lse_part + row0p + t * lstride) : -INFINITY;
              w[u] = ls == -INFINITY ? 0.f : expf(ls - m) * inv;
              const float4* src = reinterpret_cast<const float4*>(p.o_part + (row0p + t * lstride) * p.dh + c * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i) v4[u][i] = w[u] != 0.f ? __ldcg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              if (w[u] == 0.f) continue;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                acc[4 * i] = fmaf(w[u], v4[u][i].x, acc[4 * i]);
                acc[4 * i + 1] = fmaf(w[u], v4[u][i].y, acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(w[u], v4[u][i].z, acc[4 * i + 2]);
                acc[4 * i + 3] = fmaf(w[u], v4[u][i].w, acc[4 * i + 3]);
              }
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack2<kF16>(acc[2 * i], acc[2 * i + 1]);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Lq + row] = m == -INFINITY ? -INFINITY : m + logf(tot);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool kLeftBound, bool kF16, bool kSeg = false>
cudaError_t launch_fwd_inst(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const FwdKParams& kp, dim3 grid, cudaStream_t stream) {
  using C = FwdCfg<D>;
  cudaError_t e = ensure_dynamic_smem<fwd_tc_kernel<D, kLeftBound, kF16, kSeg>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  KernelTimer kt("fwd", stream);
  return launch_overlapping(fwd_tc_kernel<D, kLeftBound, kF16, kSeg>, grid, C::kThreads, C::kSmemBytes, stream, tq, tk,
                            tv, to, kp);
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs& a, DeviceStatus* st, cudaStream_t stream) {
  const Problem& pb = a.pb;
  const int elem = pb.f16 ? kElemF16 : kElemBF16;
  CUtensorMap tq, tk, tv;
  if (!make_bshd_tmap(&tq, a.q, elem, pb.B, pb.Lq, pb.Hq, pb.d, 64, kBM)) return cudaErrorInvalidValue;
  if (!make_bshd_tmap(&tk, a.k, elem, pb.B, pb.Lkv, pb.Hkv, pb.d, 64, kBN)) return cudaErrorInvalidValue;
  if (!make_bshd_tmap(&tv, a.v, elem, pb.B, pb.Lkv, pb.Hkv, pb.d, 64, kBN)) return cudaErrorInvalidValue;
  CUtensorMap to;  // the output leaves through TMA stores of the query tiles' boxes
  if (!make_bshd_tmap(&to, a.o, elem, pb.B, pb.Lq, pb.Hq, pb.d, 64, kBM)) return cudaErrorInvalidValue;
  FwdKParams kp;
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
  kp.dh = pb.d;
  kp.q_seg = pb.q_seg;
  kp.kv_seg = pb.kv_seg;
  kp.seg_qblk = pb.seg_qblk;
  kp.seg_kblk = pb.seg_kblk;
  kp.nqb = (pb.Lq + kSegBlock - 1) / kSegBlock;
  kp.nkb = (pb.Lkv + kSegBlock - 1) / kSegBlock;
  kp.n_qblocks = (pb.Lq + 2 * kBM - 1) / (2 * kBM);
  kp.n_pairs = pb.B * pb.Hq;
  kp.pair_group = l2_pair_group(2l * pb.Lkv * D * 2, kp.n_pairs, pb.G);
  kp.scale_log2 = pb.scale * kLog2e;
  kp.status = st;
  kp.n_split = a.n_split > 1 ? a.n_split : 1;
  kp.split_chunk = a.split_chunk > 0 ? a.split_chunk : 1;
  kp.o_part = a.o_part;
  kp.lse_part = a.lse_part;
  kp.counters = a.counters;
  const dim3 grid(kp.n_pairs * kp.n_qblocks * kp.n_split);
  // split key ranges run in the left-bounded builds (their streams start anywhere)
  const bool left = pb.wl < kWinInf || kp.n_split > 1;
  if (pb.q_seg != nullptr)  // segment masks run the general (two-sided span) build
    return pb.f16 ? launch_fwd_inst<D, true, true, true>(tq, tk, tv, to, kp, grid, stream)
                  : launch_fwd_inst<D, true, false, true>(tq, tk, tv, to, kp, grid, stream);
  if (pb.f16)
    return left ? launch_fwd_inst<D, true, true>(tq, tk, tv, to, kp, grid, stream)
                : launch_fwd_inst<D, false, true>(tq, tk, tv, to, kp, grid, stream);
  return left ? launch_fwd_inst<D, true, false>(tq, tk, tv, to, kp, grid, stream)
              : launch_fwd_inst<D, false, false>(tq, tk, tv, to, kp, grid, stream);
}

}  // namespace

cudaError_t launch_fwd_16(const FwdArgs& a, DeviceStatus* st, cudaStream_t s) {
  // head_dim 32 runs through the 64-column kernel: TMA zero-fills columns
  // 32..63 of Q, K and V, so S and the first 32 columns of O are exact
  if (a.pb.d <= 64) return launch_fwd_d<64>(a, st, s);
  if (a.pb.d == 256) return launch_fwd_d256(a, st, s);
  return launch_fwd_d<128>(a, st, s);
}

}  // namespace attn
