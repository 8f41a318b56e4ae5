// Split-KV decode forward, bf16 or fp16, head_dim 64/128/256, on the sm_103a tensor cores.
//
// Method (probjax "Attention performance", section "Grouped-query attention
// and decoding"): for few queries over a long KV cache the keys are split
// across programs, the query heads of a GQA group are packed into one tile,
// and each program writes its partial result with its log-sum-exp for a
// later combine.  CTA = (split, KV head, batch).  Tile row r = i * G + g holds
// query i of head hkv * G + g (G * Lq <= 128 rows; the rest of the 128-row MMA
// tile is zero).  The split covers keys [s * chunk, min((s+1) * chunk, kvl)).
// With the causal offset, row i sees keys j <= i + kvl - Lq.
//
// The KV stream is the whole cost (HBM-bound), so K/V tiles flow through a
// deep TMA ring; S is double-buffered in TMEM (S0 [0,128) S1 [128,256),
// O [256,256+d)) so the softmax of tile j+1 runs while PV of tile j is on the
// tensor core.  Key tiles are 128 keys wide, 64 at d = 256 (a 128 x 256 K or V
// tile would be 64 KB and leave room for only two ring slots).  Warps: 0-3 softmax (only the warps holding real rows work),
// 4 TMA producer, 5 MMA issuer.
#include "attn_internal.h"

namespace attn {
namespace {

constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DecCfg {
  static constexpr int kBN = (D == 256) ? 64 : 128;  // keys per tile
  static constexpr int kQBytes = 128 * D * 2;
  static constexpr int kBox = 128 * 128;      // query tile box: 128 rows x 64 cols, 16-bit
  static constexpr int kKVBox = kBN * 128;    // K/V tile box: kBN rows x 64 cols
  static constexpr int kSlotBytes = kBN * D * 2;
  static constexpr int kSlots = (D == 256) ? 5 : (D == 128) ? 5 : 10;
  static constexpr int kOffSlots = kQBytes;
  static constexpr int kOffBars = kOffSlots + kSlots * kSlotBytes;
  static constexpr int kNumBars = 2 * kSlots + 1 + 2 + 2 + 2;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;
};

struct DecKParams {
  float* o_part;
  float* lse_part;
  const int32_t* kv_lens;
  int Lq, Lkv, Hq, Hkv, G, causal, num_splits, chunk;
  int dh;  // stored head_dim (32 runs as D = 64 with zero-filled columns)
  float scale_log2;
  DeviceStatus* status;
};

template <int D, bool kF16>
__global__ void __launch_bounds__(192, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const DecKParams p) {
  using C = DecCfg<D>;
  constexpr int NS = C::kSlots;
  constexpr int kBN = C::kBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem;
  uint8_t* sSlots = smem + C::kOffSlots;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* full = bars;
  uint64_t* empty = bars + NS;
  uint64_t* q_full = bars + 2 * NS;
  uint64_t* s_full = q_full + 1;  // [2]
  uint64_t* p_full = q_full + 3;  // [2]
  uint64_t* o_done = q_full + 5;  // one phase per PV
  uint64_t* o_full = q_full + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int R = p.G * p.Lq;  // real rows
  const int n_active = (R + 31) / 32;
  // launched to overlap the tail of the kernel before it: nothing in global
  // memory is read before that grid has completed
  griddep_wait();
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);
  const int lo = split * p.chunk;
  const int hi = min(kvl, lo + p.chunk);
  const int n = hi > lo ? (hi - lo + kBN - 1) / kBN : 0;

  // zero the query tile: rows >= R stay zero, rows < R are overwritten by TMA
  for (int idx = threadIdx.x; idx < C::kQBytes / 16; idx += blockDim.x)
    reinterpret_cast<uint4*>(sQ)[idx] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 32 * n_active);
    }
    mbar_init(o_done, 1);
    mbar_init(o_full, 1);
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
  griddep_launch_dependents();  // the combine waits for this grid before it reads the partials

  if (warp == 4) {
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(R * 128 * (D / 64)));
      for (int c = 0; c < D / 64; ++c) tma_load_4d(sQ + c * C::kBox, &tm_q, q_full, c * 64, hkv * p.G, 0, b);
      const int t0 = lo / kBN;
      for (int j = 0; j < n; ++j) {
        bool ok = true;
        for (int t = 0; t < 2 && ok; ++t) {
          const int ld = 2 * j + t, s = ld % NS, r = ld / NS;
          if (r > 0) ok = mbar_wait(&empty[s], (r - 1) & 1, abort_flag, p.status, 41);
          if (!ok) break;
          mbar_arrive_expect_tx(&full[s], C::kSlotBytes);
          uint8_t* dst = sSlots + s * C::kSlotBytes;
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(dst + c * C::kKVBox, t == 0 ? &tm_k : &tm_v, &full[s], c * 64, (t0 + j) * kBN, hkv, b);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = idesc_16_f32<kF16>(128, kBN, 0, 0);
      constexpr uint32_t idesc_o = idesc_16_f32<kF16>(128, D, 0, 1);
      const uint32_t q_addr = smem_u32(sQ), slot_addr = smem_u32(sSlots);
      auto issue_s = [&](int j) {
        const uint32_t ka = slot_addr + ((2 * j) % NS) * C::kSlotBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t qoff = (k >> 2) * C::kBox + (k & 3) * 32;
          const uint32_t koff = (k >> 2) * C::kKVBox + (k & 3) * 32;
          mma_ss(tbase + (j & 1) * 128, sdesc_sw128(q_addr + qoff, 16, 1024), sdesc_sw128(ka + koff, 16, 1024),
                 idesc_s, k > 0);
        }
        mma_commit(&s_full[j & 1]);
        mma_commit(&empty[(2 * j) % NS]);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, 42);
      for (int j = 0; j < 2 && j < n && ok; ++j) {
        ok = mbar_wait(&full[(2 * j) % NS], ((2 * j) / NS) & 1, abort_flag, p.status, 43);
        if (!ok) break;
        tc_fence_after();
        issue_s(j);
      }
      for (int j = 0; j < n && ok; ++j) {
        const int vl = 2 * j + 1, vs = vl % NS;
        ok = mbar_wait(&full[vs], (vl / NS) & 1, abort_flag, p.status, 44);
        if (!ok) break;
        ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag, p.status, 45);
        if (!ok) break;
        tc_fence_after();
        const uint32_t va = slot_addr + vs * C::kSlotBytes;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          mma_ts(tbase + 256, tbase + (j & 1) * 128 + k * 8, sdesc_sw128(va + k * 2048, C::kKVBox, 1024), idesc_o,
                 (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(o_done);
        mma_commit(&empty[vs]);
        if (j == n - 1) mma_commit(o_full);
        if (j + 2 < n) {
          const int kl = 2 * (j + 2);
          ok = mbar_wait(&full[kl % NS], (kl / NS) & 1, abort_flag, p.status, 46);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 2);
        }
      }
    }
    __syncwarp();
  } else if (warp < n_active) {
    // ------------------------------------------------------------ softmax (thread = packed row)
    const int r = warp * 32 + lane;
    const bool real = r < R;
    const int i = r / p.G, g = r % p.G;
    const int hq = hkv * p.G + g;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    int lim = real ? (p.causal ? min(kvl, i + 1 + kvl - p.Lq) : kvl) : lo;
    lim = min(lim, hi);
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, p.status, 47));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = t_lane + (j & 1) * 128;
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(s_addr + c * 32, rr);
#pragma unroll
        for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(rr[e]);
      }
      const int col0 = lo + j * kBN;
      if (col0 + kBN > lim) {
#pragma unroll
        for (int e = 0; e < kBN; ++e)
          if (col0 + e >= lim) s[e] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int e = 1; e < kBN; ++e) mx = fmaxf(mx, s[e]);
      const float m_tile = mx * sl2;
      const bool grow = m_tile > m_used + kRescaleThreshold;
      const float m_new = grow ? m_tile : m_used;
      const float alpha = grow ? ex2_approx(m_used - m_new) : 1.0f;
      l_sum *= alpha;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O still holds PV of tiles < j; wait until PV(j-1) has landed
        ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag, p.status, 48));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(t_lane + 256 + c * 32, rr);
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
          tmem_st32(t_lane + 256 + c * 32, rr);
        }
      }
      m_used = m_new;
      const float mb = (m_used == -INFINITY) ? 0.f : m_used;
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2_approx(fmaf(s[c * 32 + 2 * e], sl2, -mb));
          const float p1 = ex2_approx(fmaf(s[c * 32 + 2 * e + 1], sl2, -mb));
          l_sum += p0 + p1;
          pk[e] = pack2<kF16>(p0, p1);
        }
        tmem_st16(s_addr + c * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
    }
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_full, 0, abort_flag, p.status, 49));
    if (ok) {
      tc_fence_after();
      const float inv_l = l_sum > 0.f ? 1.0f / l_sum : 0.f;
      const size_t prow = ((static_cast<size_t>(b) * p.Hq + hq) * p.num_splits + split) * p.Lq + i;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        if (c * 32 >= p.dh) break;
        uint32_t rr[32];
        if (n > 0) {
          tmem_ld32(t_lane + 256 + c * 32, rr);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = 0u;
        }
        if (real) {
          float4* dst = reinterpret_cast<float4*>(p.o_part + prow * p.dh + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(rr[4 * e]) * inv_l, __uint_as_float(rr[4 * e + 1]) * inv_l,
                                 __uint_as_float(rr[4 * e + 2]) * inv_l, __uint_as_float(rr[4 * e + 3]) * inv_l);
        }
      }
      if (real) p.lse_part[prow] = l_sum > 0.f ? (m_used + lg2_approx(l_sum)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// TMA map over q viewed as (d, Hq, Lq, B) with box (64, G, Lq, 1): one load
// packs the G heads of a KV head times the Lq queries as rows i * G + g.
bool make_q_group_tmap(CUtensorMap* map, const void* q, int B, int Lq, int Hq, int d, int G, bool f16) {
  typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  // looked up once (a function-local static is initialised thread-safely)
  static const EncodeFn fn = []() -> EncodeFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeFn>(ptr);
  }();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(Lq),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Hq) * d * 2,
                           static_cast<cuuint64_t>(Lq) * Hq * d * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(Lq), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims,
            strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool kF16>
cudaError_t launch_decode_inst(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecKParams& kp, dim3 grid, cudaStream_t stream) {
  using C = DecCfg<D>;
  cudaError_t e = ensure_dynamic_smem<decode_tc_kernel<D, kF16>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  KernelTimer kt("decode", stream);
  return launch_overlapping(decode_tc_kernel<D, kF16>, grid, 192, C::kSmemBytes, stream, tq, tk, tv, kp);
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs& a, DeviceStatus* st, cudaStream_t stream) {
  const Problem& pb = a.pb;
  const int elem = pb.f16 ? kElemF16 : kElemBF16;
  CUtensorMap tq, tk, tv;
  if (!make_q_group_tmap(&tq, a.q, pb.B, pb.Lq, pb.Hq, pb.d, pb.G, pb.f16 != 0)) return cudaErrorInvalidValue;
  constexpr int kBN = DecCfg<D>::kBN;
  if (!make_bshd_tmap(&tk, a.k, elem, pb.B, pb.Lkv, pb.Hkv, pb.d, 64, kBN)) return cudaErrorInvalidValue;
  if (!make_bshd_tmap(&tv, a.v, elem, pb.B, pb.Lkv, pb.Hkv, pb.d, 64, kBN)) return cudaErrorInvalidValue;
  DecKParams kp;
  kp.o_part = a.o_part;
  kp.lse_part = a.lse_part;
  kp.kv_lens = pb.kv_lens;
  kp.Lq = pb.Lq;
  kp.Lkv = pb.Lkv;
  kp.Hq = pb.Hq;
  kp.Hkv = pb.Hkv;
  kp.G = pb.G;
  kp.causal = pb.causal;
  kp.dh = pb.d;
  kp.num_splits = a.num_splits;
  kp.chunk = a.chunk;
  kp.scale_log2 = pb.scale * kLog2e;
  kp.status = st;
  const dim3 grid(a.num_splits, pb.Hkv, pb.B);
  return pb.f16 ? launch_decode_inst<D, true>(tq, tk, tv, kp, grid, stream)
                : launch_decode_inst<D, false>(tq, tk, tv, kp, grid, stream);
}

}  // namespace

cudaError_t launch_decode_16(const DecodeArgs& a, DeviceStatus* st, cudaStream_t s) {
  if (a.pb.d == 256) return launch_decode_d<256>(a, st, s);
  return a.pb.d <= 64 ? launch_decode_d<64>(a, st, s) : launch_decode_d<128>(a, st, s);  // head_dim 32 runs as 64
}

}  // namespace attn
