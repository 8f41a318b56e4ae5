// float32 attention on the bf16 tensor cores, by operand splitting.
//
// The pages run float32 attention as TF32 and accept ~1e-3 error ("GPU and
// CPU performance", section "Methodology", TF32); the float32 target here is
// 1e-4.  Each float32 operand x is split into two bf16 parts,
//   x_hi = bf16(x),  x_lo = bf16(x - x_hi),
// which carry 16 of its 24 mantissa bits (|x - x_hi - x_lo| <= 2^-17 |x|),
// and each product is taken as three bf16 MMAs with float32 accumulation:
//   A B ~= A_hi B_hi + A_hi B_lo + A_lo B_hi,
// dropping A_lo B_lo (<= 2^-18 of |A||B|; with the rounding of the lo parts,
// ~2^-16 per product at most, far inside the target), while running on the
// tensor cores instead of the CUDA cores.  V is split into three parts,
// v = v_hi + v_mid + v_lo exactly (8 + 8 + 8 significant bits), and PV takes
// P_hi (V_hi + V_mid + V_lo) + P_lo V_hi: a row whose softmax has one key has
// P = 1 exactly (P_hi = 1, P_lo = 0), so its output is that key's value row
// bit for bit, as in the 16-bit kernels.  Softmax, row sums and the
// log-sum-exp stay in float32.
//
// Forward (this file): CTA = one 128-row query tile of one (batch, head);
// 64-key steps.  The float32 inputs are split on the fly: four converter warps
// read Q once and each step's K and V tiles from global memory (L2) and write
// their hi and lo parts into shared memory in the 128-byte-swizzled layout the
// MMA descriptors read (the forward has no workspace to hold split copies).
// Warp roles:
//   warps 0-3  softmax (thread = query row = TMEM lane)
//   warps 4-7  converters (Q, then K and V of every step)
//   warp  8    MMA issuer (one lane); owns the TMEM allocation
// Per step j: S(j) = Q K^T as three MMAs per 16-wide k-step (into one of two
// S buffers, so S(j + 2) is computed while the softmax works on S(j + 1));
// the softmax turns it into P (float32), writes P_hi over the first 32
// columns of its S buffer and P_lo into a buffer of its own; then
// O += P V as four MMAs per 16-key k-step with P from TMEM.  K and V have two
// buffers each, freed separately (K after S, V after PV), so the converters
// fill step j + 2 while steps j and j + 1 compute.
// TMEM: S [0,64) and [64,128), P_lo [128,160) and [160,192), O [256, 256 + D).
// O is rescaled lazily in TMEM (a row's running maximum grew by more than
// 2^8), after the previous PV has completed.
#include "split_f32.cuh"

namespace attn {
namespace {

using namespace split;

constexpr int kSM = 128;  // query rows per CTA (= TMEM lanes)
constexpr int kSN = 64;   // keys per step
constexpr float kSplitRescale = 8.0f;
constexpr float kLn2f = 0.6931471805599453f;
constexpr float kLog2ef = 1.4426950408889634f;

template <int D>
struct SplitFwdCfg {
  static constexpr int kQBox = kSM * 128;       // one 64-column box of the 128-row Q tile (bf16)
  static constexpr int kQPart = kQBox * (D / 64);  // Q hi or Q lo
  static constexpr int kKVBox = kSN * 128;      // one 64-column box of a 64-row K or V tile
  static constexpr int kKVPart = kKVBox * (D / 64);  // one of K hi, K lo, V hi, V lo
  static constexpr int kOffQ = 0;               // Q hi, then Q lo
  static constexpr int kOffK = 2 * kQPart;      // buffer b: K hi at kOffK + 2b kKVPart, K lo right after
  static constexpr int kOffV = kOffK + 4 * kKVPart;  // buffer b: V hi, mid, lo at kOffV + 3b kKVPart
  static constexpr int kOffBars = kOffV + 6 * kKVPart;
  static constexpr int kNumBars = 1 + 2 * 4 + 2 + 2 + 1 + 1;
  static constexpr int kSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;  // + alignment slack
  static constexpr int kThreads = 288;
};

struct SplitFwdParams {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  const int32_t* kv_lens;
  int Lq, Lkv, Hq, Hkv, G, causal, wl, wr, n_qtiles, n_pairs, pair_group;
  float scale_log2;
  DeviceStatus* status;
};

template <int D, bool kLeftBound>
__global__ void __launch_bounds__(288, 1) fwd_split_kernel(const SplitFwdParams p) {
  using C = SplitFwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQh = smem + C::kOffQ;
  uint8_t* sQl = sQh + C::kQPart;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* q_full = bars;
  uint64_t* full_k = bars + 1;    // [2] converters wrote K(j) hi/lo (4 warp arrivals)
  uint64_t* empty_k = bars + 3;   // [2] S(j) done with the K buffer
  uint64_t* full_v = bars + 5;    // [2]
  uint64_t* empty_v = bars + 7;   // [2] PV(j) done with the V buffer
  uint64_t* s_full = bars + 9;    // [2] S(j) computed
  uint64_t* p_full = bars + 11;   // [2] P(j) written (4 warp arrivals)
  uint64_t* pv_done = bars + 13;  // PV(j) completed (one phase per step)
  uint64_t* o_full = bars + 14;   // the last PV completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const TileCoord tc = grouped_tile(blockIdx.x, p.n_pairs, p.n_qtiles, p.pair_group);
  const int qt = p.causal ? p.n_qtiles - 1 - tc.rank : tc.rank;
  const int hq = tc.pair % p.Hq, b = tc.pair / p.Hq;
  const int hkv = hq / p.G;
  const int q0 = qt * kSM;
  // launched to overlap the tail of the kernel before it: nothing in global
  // memory is read before that grid has completed
  griddep_wait();
  int kvl = p.Lkv;
  if (p.kv_lens != nullptr) kvl = min(max(p.kv_lens[b], 0), p.Lkv);
  // 64-key steps [jlo, jlo + n) the tile's rows need (both ends of a row's
  // span grow with the row)
  int jlo = 0, n = 0;
  {
    const int last = min(q0 + kSM - 1, p.Lq - 1);
    const int lo = key_span(q0, p.Lq, kvl, p.wl, p.wr).lo;
    const int hi = key_span(last, p.Lq, kvl, p.wl, p.wr).hi;
    if (hi > lo) {
      jlo = kLeftBound ? lo / kSN : 0;
      n = (hi + kSN - 1) / kSN - jlo;
    }
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(q_full, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full_k[i], 4);
      mbar_init(&empty_k[i], 1);
      mbar_init(&full_v[i], 4);
      mbar_init(&empty_v[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
    }
    mbar_init(pv_done, 1);
    mbar_init(o_full, 1);
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
    bool ok = true;
    if (n > 0) {
      // in two halves of 64 rows: half the loads in flight, half the registers
      convert_tile<D, kSM / 2, kSM>(p.q, b, p.Lq, p.Hq, hq, q0, p.Lq, sQh, sQl, 0, t);
      convert_tile<D, kSM / 2, kSM>(p.q, b, p.Lq, p.Hq, hq, q0 + kSM / 2, p.Lq, sQh, sQl, kSM / 2, t);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    // K of step u, then V of step u - 1: a K buffer is released when S of
    // its step has run, a V buffer only after PV, so converting K one step
    // ahead keeps S(j + 2) from waiting behind V(j + 1), which waits for PV(j - 1).
    for (int u = 0; u <= n && ok; ++u) {
      if (u < n) {
        const int buf = u & 1, use = u >> 1;
        uint8_t* kh = smem + C::kOffK + 2 * buf * C::kKVPart;
        if (use > 0) ok = __all_sync(0xffffffffu, mbar_wait(&empty_k[buf], (use - 1) & 1, abort_flag, p.status, 121));
        if (!ok) break;
        convert_tile<D, kSN, kSN>(p.k, b, p.Lkv, p.Hkv, hkv, (jlo + u) * kSN, kvl, kh, kh + C::kKVPart, 0, t);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_k[buf]);
      }
      if (u > 0) {
        const int w = u - 1, buf = w & 1, use = w >> 1;
        uint8_t* vh = smem + C::kOffV + 3 * buf * C::kKVPart;
        if (use > 0) ok = __all_sync(0xffffffffu, mbar_wait(&empty_v[buf], (use - 1) & 1, abort_flag, p.status, 122));
        if (!ok) break;
        convert_tile<D, kSN, kSN, true>(p.v, b, p.Lkv, p.Hkv, hkv, (jlo + w) * kSN, kvl, vh, vh + 2 * C::kKVPart, 0,
                                        t, vh + C::kKVPart);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_v[buf]);
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kSM, kSN, 0, 0);  // Q (K-major) x K^T (K-major)
      constexpr uint32_t idesc_o = idesc_bf16_f32(kSM, D, 0, 1);    // P (TMEM) x V (MN-major)
      const SDesc qh = sdesc_split(smem_u32(sQh), 16, 1024), ql = sdesc_split(smem_u32(sQl), 16, 1024);
      auto issue_s = [&](int j) {  // S(j) = Qh Kh^T + Qh Kl^T + Ql Kh^T into S buffer j % 2
        const int buf = j & 1;
        const uint32_t kaddr = smem_u32(smem + C::kOffK + 2 * buf * C::kKVPart);
        const SDesc kh = sdesc_split(kaddr, 16, 1024), kl = sdesc_split(kaddr + C::kKVPart, 16, 1024);
        const uint32_t d_s = tbase + buf * 64;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t qo = ((k >> 2) * C::kQBox + (k & 3) * 32) >> 4;
          const uint32_t ko = ((k >> 2) * C::kKVBox + (k & 3) * 32) >> 4;
          mma_ss_d(d_s, qh, qo, kh, ko, idesc_s, k > 0);
          mma_ss_d(d_s, qh, qo, kl, ko, idesc_s, 1u);
          mma_ss_d(d_s, ql, qo, kh, ko, idesc_s, 1u);
        }
      };
      auto issue_pv = [&](int j) {  // O += Ph Vh + Ph Vm + Ph Vl + Pl Vh
        const int buf = j & 1;
        const uint32_t vaddr = smem_u32(smem + C::kOffV + 3 * buf * C::kKVPart);
        const SDesc vh = sdesc_split(vaddr, C::kKVBox, 1024), vm = sdesc_split(vaddr + C::kKVPart, C::kKVBox, 1024),
                    vl = sdesc_split(vaddr + 2 * C::kKVPart, C::kKVBox, 1024);
        const uint32_t ph = tbase + buf * 64, pl = tbase + 128 + buf * 32;
#pragma unroll
        for (int k = 0; k < kSN / 16; ++k) {
          const uint32_t vo = (16 * k * 128) >> 4;
          mma_ts_d(tbase + 256, ph + k * 8, vh, vo, idesc_o, (j > 0 || k > 0) ? 1u : 0u);
          mma_ts_d(tbase + 256, ph + k * 8, vm, vo, idesc_o, 1u);
          mma_ts_d(tbase + 256, ph + k * 8, vl, vo, idesc_o, 1u);
          mma_ts_d(tbase + 256, pl + k * 8, vh, vo, idesc_o, 1u);
        }
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, 123);
      for (int j = 0; j < 2 && j < n && ok; ++j) {
        ok = mbar_wait(&full_k[j], 0, abort_flag, p.status, 124);
        if (!ok) break;
        tc_fence_after();
        issue_s(j);
        mma_commit(&s_full[j]);
        mma_commit(&empty_k[j]);
      }
      for (int j = 0; j < n && ok; ++j) {
        const int buf = j & 1, use = j >> 1;
        ok = mbar_wait(&p_full[buf], use & 1, abort_flag, p.status, 125);
        if (ok) ok = mbar_wait(&full_v[buf], use & 1, abort_flag, p.status, 126);
        if (!ok) break;
        tc_fence_after();
        issue_pv(j);
        mma_commit(pv_done);
        mma_commit(&empty_v[buf]);
        if (j + 2 < n) {  // S(j + 2) reuses S buffer j % 2, whose P(j) PV(j) has just read
          ok = mbar_wait(&full_k[buf], (use + 1) & 1, abort_flag, p.status, 127);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 2);
          mma_commit(&s_full[buf]);
          mma_commit(&empty_k[buf]);
        }
      }
      if (ok) mma_commit(o_full);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (thread = query row)
    const int row = q0 + warp * 32 + lane;
    const uint32_t t_lane = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    Span span = row < p.Lq ? key_span(row, p.Lq, kvl, p.wl, p.wr) : Span{0, 0};
    if (!kLeftBound) span.lo = 0;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int buf = j & 1, use = j >> 1;
      const int col0 = (jlo + j) * kSN;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[buf], use & 1, abort_flag, p.status, 128));
      if (!ok) break;
      tc_fence_after();
      uint32_t sa[32], sb[32];
      tmem_ld32_pair(t_lane + buf * 64, t_lane + buf * 64 + 32, sa, sb);
      float s[kSN];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(sa[i]);
        s[32 + i] = __uint_as_float(sb[i]);
      }
      if ((kLeftBound && col0 < span.lo) || col0 + kSN > span.hi) {
#pragma unroll
        for (int i = 0; i < kSN; ++i)
          if ((kLeftBound && col0 + i < span.lo) || col0 + i >= span.hi) s[i] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int i = 1; i < kSN; ++i) mx = fmaxf(mx, s[i]);
      const float m_tile = mx * sl2;
      const bool grow = m_tile > m_used + kSplitRescale;
      const float m_new = grow ? m_tile : m_used;
      const float alpha = grow ? ex2_approx(m_used - m_new) : 1.0f;
      l_sum *= alpha;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O may still be accumulating PV(j - 1): wait for it first
        ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1, abort_flag, p.status, 129));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(t_lane + 256 + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(t_lane + 256 + c * 32, r);
        }
      }
      m_used = m_new;
      const float mb = (m_used == -INFINITY) ? 0.f : m_used;
      // t = s sl2 rounded before the subtraction: rounding is monotonic, so the
      // row's largest t is exactly mb and its probability exactly 2^0 (an FMA
      // would expose the rounding residual of s sl2 and leave P at 1 +- ulp)
      uint32_t ph[32], pl[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = ex2_approx(__fmul_rn(s[2 * i], sl2) - mb), p1 = ex2_approx(__fmul_rn(s[2 * i + 1], sl2) - mb);
        l_sum += p0 + p1;
        ph[i] = pack_bf16x2(p0, p1);
        pl[i] = pack_bf16x2(p0 - __uint_as_float(ph[i] << 16), p1 - __uint_as_float(ph[i] & 0xffff0000u));
      }
      tmem_st32(t_lane + buf * 64, ph);
      tmem_st32(t_lane + 128 + buf * 32, pl);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[buf]);
    }
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_full, 0, abort_flag, p.status, 130));
    if (ok) {
      // every lane takes part in the TMEM loads (warp-collective); rows past Lq
      // only skip their stores
      tc_fence_after();
      const float inv_l = l_sum > 0.f ? 1.0f / l_sum : 0.f;
      float* orow = p.o + ((static_cast<size_t>(b) * p.Lq + (row < p.Lq ? row : 0)) * p.Hq + hq) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(t_lane + 256 + c * 32, r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (row < p.Lq) {
          float4* dst = reinterpret_cast<float4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv_l, __uint_as_float(r[4 * i + 1]) * inv_l,
                                 __uint_as_float(r[4 * i + 2]) * inv_l, __uint_as_float(r[4 * i + 3]) * inv_l);
        }
      }
      if (row < p.Lq)
        p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Lq + row] =
            l_sum > 0.f ? (m_used + lg2_approx(l_sum)) * kLn2f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool kLeftBound>
cudaError_t launch_split_fwd_inst(const SplitFwdParams& kp, dim3 grid, cudaStream_t stream) {
  using C = SplitFwdCfg<D>;
  cudaError_t e = ensure_dynamic_smem<fwd_split_kernel<D, kLeftBound>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  KernelTimer kt("fwd_split_f32", stream);
  return launch_overlapping(fwd_split_kernel<D, kLeftBound>, grid, C::kThreads, C::kSmemBytes, stream, kp);
}

}  // namespace

bool split_f32_applies(const Problem& pb) { return (pb.d == 64 || pb.d == 128) && pb.q_seg == nullptr; }

cudaError_t launch_fwd_split_f32(const FwdArgs& a, DeviceStatus* st, cudaStream_t s) {
  const Problem& pb = a.pb;
  SplitFwdParams kp;
  kp.q = static_cast<const float*>(a.q);
  kp.k = static_cast<const float*>(a.k);
  kp.v = static_cast<const float*>(a.v);
  kp.o = static_cast<float*>(a.o);
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
  kp.n_qtiles = (pb.Lq + kSM - 1) / kSM;
  kp.n_pairs = pb.B * pb.Hq;
  kp.pair_group = l2_pair_group(2l * pb.Lkv * pb.d * 4, kp.n_pairs, pb.G);
  kp.scale_log2 = pb.scale * kLog2ef;
  kp.status = st;
  const dim3 grid(kp.n_pairs * kp.n_qtiles);
  const bool left = pb.wl < kWinInf;
  if (pb.d == 64) return left ? launch_split_fwd_inst<64, true>(kp, grid, s) : launch_split_fwd_inst<64, false>(kp, grid, s);
  return left ? launch_split_fwd_inst<128, true>(kp, grid, s) : launch_split_fwd_inst<128, false>(kp, grid, s);
}

}  // namespace attn
