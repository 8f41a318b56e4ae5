// HBM-bound helper kernels: the backward preprocess (delta = rowsum(dO * O)),
// the log-sum-exp combine of split-KV partials and the per-block summary of
// segment ids that lets the tensor-core kernels skip tiles.
#include <climits>
#include <cstring>
#include <type_traits>

#include "attn_internal.h"

namespace attn {
namespace {

// Eight consecutive elements as loaded (16 bytes of 16-bit values, 32 of
// float32), converted to float32 only when used, so that several rows' loads
// can be in flight before the first is needed.
template <typename T>
struct Raw8 {
  uint4 v[sizeof(T) / 2];
};

template <typename T>
__device__ __forceinline__ void raw_load8(const T* p, Raw8<T>& r) {
#pragma unroll
  for (int j = 0; j < static_cast<int>(sizeof(T) / 2); ++j) r.v[j] = reinterpret_cast<const uint4*>(p)[j];
}

template <typename T>
__device__ __forceinline__ void unpack8(const Raw8<T>& r, float (&f)[8]);

template <>
__device__ __forceinline__ void unpack8<__nv_bfloat16>(const Raw8<__nv_bfloat16>& r, float (&f)[8]) {
  const uint32_t w[4] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <>
__device__ __forceinline__ void unpack8<__half>(const Raw8<__half>& r, float (&f)[8]) {
  const uint32_t w[4] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h;
    memcpy(&h, &w[i], sizeof(h));
    const float2 v = __half22float2(h);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

template <>
__device__ __forceinline__ void unpack8<float>(const Raw8<float>& r, float (&f)[8]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    f[4 * j] = __uint_as_float(r.v[j].x);
    f[4 * j + 1] = __uint_as_float(r.v[j].y);
    f[4 * j + 2] = __uint_as_float(r.v[j].z);
    f[4 * j + 3] = __uint_as_float(r.v[j].w);
  }
}

// delta[b, h, i] = sum_c dO[b, i, h, c] * O[b, i, h, c]  (float32 accumulate
// for 16-bit inputs; for float32 inputs a compensated float32 sum, whose
// backward subtracts delta from dP values accurate to about 2^-24, so a plain
// float32 sum's rounding would dominate dP - delta where a row's probability
// sits on one key).  The compensated sum follows Ogita, Rump and Oishi's
// Dot2: each product's rounding error is recovered exactly with an FMA and
// each addition's with Knuth's TwoSum, and the errors are summed beside the
// result, which is then as accurate as a sum in twice the working precision
// (float64 arithmetic runs at a small fraction of the float32 rate here).
// Rows are walked in the padded [B, Hq, Lq_pad] order of the outputs: the
// grid's (z, y) indices give the (b, h) pair (65535 pairs per z slice), its x
// index a run of rows, so that no thread divides its index in 64 bits; D/8
// threads share a row, each reducing 8 consecutive elements, and each thread
// takes kPreRows rows, whose loads it issues before the first sum.  Optionally it
// also writes lse2 = lse * log2(e) (+inf where lse = -inf, so that every
// recomputed probability of such a row is 0), fills the pad rows
// Lq <= i < Lq_pad with delta = 0 and lse2 = +inf, and zeroes the float32 dQ
// accumulator of the atomic backward.
// s += x with the rounding error of the addition added to err (Knuth's
// TwoSum: exact for any ordering of the magnitudes).
__device__ __forceinline__ void two_sum_add(float& s, float& err, float x) {
  const float t = s + x;
  const float z = t - s;
  err += (s - (t - z)) + (x - z);
  s = t;
}

// One thread's share of row i of pair bh = b * Hq + h, from its loaded
// elements of O (ra) and dO (rg).
template <typename T, int D>
__device__ __forceinline__ void preprocess_row(const Raw8<T>& ra, const Raw8<T>& rg, const float* __restrict__ lse,
                                               float* __restrict__ delta, float* __restrict__ lse2,
                                               float* __restrict__ dq_acc, long b, long h, long bh, int i, int part,
                                               int Lq, int Lq_pad, int Hq) {
  constexpr int kTPR = D / 8;
  const long prow = bh * Lq_pad + i;
  const bool real = i < Lq;
  constexpr bool kComp = std::is_same<T, float>::value;
  float acc = 0.f, err = 0.f;  // err: the compensation of the float32 path
  if (real) {
    const long row = (b * Lq + i) * Hq + h;  // row of the [B, Lq, Hq, D] tensors
    float a[8], g[8];
    unpack8<T>(ra, a);
    unpack8<T>(rg, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (kComp) {
        const float pr = a[e] * g[e];
        const float pe = fmaf(a[e], g[e], -pr);  // exact: a g = pr + pe
        two_sum_add(acc, err, pr);
        err += pe;
      } else {
        acc = fmaf(a[e], g[e], acc);
      }
    }
    if (dq_acc != nullptr) {
      float4* z = reinterpret_cast<float4*>(dq_acc + row * D + part * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int off = kTPR / 2; off > 0; off >>= 1) {
    const float other = __shfl_xor_sync(0xffffffffu, acc, off);
    const float other_err = __shfl_xor_sync(0xffffffffu, err, off);
    if (kComp) {
      two_sum_add(acc, err, other);
      err += other_err;
    } else {
      acc += other;
    }
  }
  if (i < Lq_pad && part == 0) {
    delta[prow] = acc + err;  // 0 on pad rows
    if (lse2 != nullptr) {
      const float l = real ? lse[bh * Lq + i] : -INFINITY;
      lse2[prow] = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
    }
  }
}

constexpr int kPreRows = 2;  // rows per thread in the preprocess (1 and 4 measured slower)

template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                             const float* __restrict__ lse, float* __restrict__ delta,
                                                             float* __restrict__ lse2, float* __restrict__ dq_acc,
                                                             long n_bh, int Lq, int Lq_pad, int Hq) {
  constexpr int kTPR = D / 8;  // threads per row
  griddep_wait();  // launched to overlap the forward's tail: O is complete from here on
  griddep_launch_dependents();
  constexpr int kRows = 256 / kTPR;  // rows of one pass of the block
  const int part = static_cast<int>(threadIdx.x % kTPR);
  const int i0 = static_cast<int>(blockIdx.x) * kRows * kPreRows + static_cast<int>(threadIdx.x / kTPR);
  const long bh = static_cast<long>(blockIdx.z) * 65535 + blockIdx.y;
  if (bh >= n_bh) return;  // whole block: the last z slice is partly empty
  long b, h;
  if (n_bh <= 0x7fffffffL) {  // 32-bit division where the pair index fits
    const unsigned q = static_cast<unsigned>(bh) / static_cast<unsigned>(Hq);
    b = q;
    h = static_cast<long>(static_cast<unsigned>(bh) - q * static_cast<unsigned>(Hq));
  } else {
    b = bh / Hq;
    h = bh - b * Hq;
  }
  Raw8<T> ra[kPreRows], rg[kPreRows];
#pragma unroll
  for (int r = 0; r < kPreRows; ++r) {  // every row's loads in flight before the first sum
    const int i = i0 + r * kRows;
    ra[r] = rg[r] = Raw8<T>{};
    if (i < Lq) {
      const long row = (b * Lq + i) * Hq + h;
      raw_load8<T>(o + row * D + part * 8, ra[r]);
      raw_load8<T>(dout + row * D + part * 8, rg[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < kPreRows; ++r)
    preprocess_row<T, D>(ra[r], rg[r], lse, delta, lse2, dq_acc, b, h, bh, i0 + r * kRows, part, Lq, Lq_pad, Hq);
}

// Log-sum-exp combine of split partials, for output rows (b, h, i):
// lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.  Empty splits
// (lse_s = -inf) weigh 0 and their o_s is never read.  A warp takes kRows
// consecutive rows, lane l the elements [l*kPer, (l+1)*kPer) of each; lane s
// keeps split s's log-sum-exp (the first 32 in registers).  The partial rows
// are fetched kU splits of every row at a time, all those loads in flight
// before the adds.  The row index is split into (b, h, i) once per warp, in
// 32-bit arithmetic where it fits: 64-bit divisions per row made the kernel
// instruction-bound.  Many rows (a split forward) run four to a warp, few
// rows with many splits (a decode) one to a warp.
template <typename T, int D, int kRows>
__global__ void __launch_bounds__(256, 2) combine_kernel(const float* __restrict__ o_part,
                                                      const float* __restrict__ lse_part, T* __restrict__ o,
                                                      float* __restrict__ lse, int B, int Lq, int Hq, int S) {
  constexpr int kPer = D / 32;             // elements per lane
  constexpr int kU = kPer >= 8 ? 1 : kPer >= 4 ? 2 : 4;  // splits per row fetched together
  const long warp = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long n_rows = static_cast<long>(B) * Hq * Lq;
  griddep_wait();  // launched to overlap the split kernel: its partials are complete from here on
  griddep_launch_dependents();
  if (warp * kRows >= n_rows) return;
  long bh[kRows];
  int ri[kRows];
  bool live[kRows];
  float l0[kRows], m[kRows], tot[kRows], inv[kRows];
  {
    const long row0 = warp * kRows;  // row = (b * Hq + h) * Lq + i
    long bhc;
    int ic;
    if (n_rows <= 0x7fffffffL) {
      const unsigned r0 = static_cast<unsigned>(row0);
      bhc = r0 / static_cast<unsigned>(Lq);
      ic = static_cast<int>(r0 - static_cast<unsigned>(bhc) * static_cast<unsigned>(Lq));
    } else {
      bhc = row0 / Lq;
      ic = static_cast<int>(row0 - bhc * Lq);
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      live[r] = row0 + r < n_rows;
      ri[r] = ic;
      bh[r] = bhc;
      if (++ic == Lq) {
        ic = 0;
        ++bhc;
      }
      l0[r] = (live[r] && lane < S) ? lse_part[(bh[r] * S + lane) * Lq + ri[r]] : -INFINITY;
    }
  }
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    m[r] = l0[r];
    for (int s = 32 + lane; s < S && live[r]; s += 32) m[r] = fmaxf(m[r], lse_part[(bh[r] * S + s) * Lq + ri[r]]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m[r] = fmaxf(m[r], __shfl_xor_sync(0xffffffffu, m[r], off));
    tot[r] = 0.f;
    if (m[r] != -INFINITY) {
      tot[r] = l0[r] == -INFINITY ? 0.f : expf(l0[r] - m[r]);
      for (int s = 32 + lane; s < S; s += 32) {
        const float ls = lse_part[(bh[r] * S + s) * Lq + ri[r]];
        if (ls != -INFINITY) tot[r] += expf(ls - m[r]);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot[r] += __shfl_xor_sync(0xffffffffu, tot[r], off);
    inv[r] = m[r] == -INFINITY ? 0.f : 1.0f / tot[r];
  }
  float acc[kRows][kPer];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[r][e] = 0.f;
  for (int s0 = 0; s0 < S; s0 += 32) {
    float w_lane[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      float ls = l0[r];
      if (s0 > 0) ls = (live[r] && s0 + lane < S) ? lse_part[(bh[r] * S + s0 + lane) * Lq + ri[r]] : -INFINITY;
      w_lane[r] = (m[r] == -INFINITY || ls == -INFINITY) ? 0.f : expf(ls - m[r]) * inv[r];
    }
    const int cnt = min(32, S - s0);
    for (int t0 = 0; t0 < cnt; t0 += kU) {
      float w[kRows][kU], val[kRows][kU][kPer];
#pragma unroll
      for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          w[r][u] = t0 + u < cnt ? __shfl_sync(0xffffffffu, w_lane[r], t0 + u) : 0.f;
#pragma unroll
          for (int e = 0; e < kPer; ++e) val[r][u][e] = 0.f;
          if (w[r][u] != 0.f) {
            const float* src = o_part + ((bh[r] * S + s0 + t0 + u) * Lq + ri[r]) * D + lane * kPer;
            if constexpr (kPer % 4 == 0) {
#pragma unroll
              for (int e = 0; e < kPer; e += 4) {
                const float4 x = *reinterpret_cast<const float4*>(src + e);
                val[r][u][e] = x.x; val[r][u][e + 1] = x.y; val[r][u][e + 2] = x.z; val[r][u][e + 3] = x.w;
              }
            } else if constexpr (kPer % 2 == 0) {
#pragma unroll
              for (int e = 0; e < kPer; e += 2) {
                const float2 x = *reinterpret_cast<const float2*>(src + e);
                val[r][u][e] = x.x; val[r][u][e + 1] = x.y;
              }
            } else {
#pragma unroll
              for (int e = 0; e < kPer; ++e) val[r][u][e] = src[e];
            }
          }
        }
#pragma unroll
      for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (w[r][u] == 0.f) continue;
#pragma unroll
          for (int e = 0; e < kPer; ++e) acc[r][e] = fmaf(w[r][u], val[r][u][e], acc[r][e]);
        }
    }
  }
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    if (!live[r]) continue;
    long b;  // bh = b * Hq + h
    int h;
    if (static_cast<long>(B) * Hq <= 0x7fffffffL) {
      const unsigned bhu = static_cast<unsigned>(bh[r]);
      b = bhu / static_cast<unsigned>(Hq);
      h = static_cast<int>(bhu - static_cast<unsigned>(b) * static_cast<unsigned>(Hq));
    } else {
      b = bh[r] / Hq;
      h = static_cast<int>(bh[r] - b * Hq);
    }
    T* dst = o + ((b * Lq + ri[r]) * Hq + h) * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      if constexpr (std::is_same<T, __nv_bfloat16>::value)
        dst[e] = __float2bfloat16_rn(acc[r][e]);
      else if constexpr (std::is_same<T, __half>::value)
        dst[e] = __float2half_rn(acc[r][e]);
      else
        dst[e] = acc[r][e];
    }
    if (lane == 0) lse[bh[r] * Lq + ri[r]] = (m[r] == -INFINITY) ? -INFINITY : m[r] + logf(tot[r]);
  }
}

template <typename T, int D>
cudaError_t run_preprocess(const PreprocessArgs& a, cudaStream_t s) {
  constexpr int kRows = 256 / (D / 8) * kPreRows;  // rows per block
  const long n_bh = static_cast<long>(a.B) * a.Hq;
  const dim3 grid((a.Lq_pad + kRows - 1) / kRows, static_cast<unsigned>(n_bh < 65535 ? n_bh : 65535),
                  static_cast<unsigned>((n_bh + 65534) / 65535));
  KernelTimer kt("bwd_preprocess", s);
  return launch_overlapping(bwd_preprocess_kernel<T, D>, grid, 256, 0, s, static_cast<const T*>(a.o),
                            static_cast<const T*>(a.dout), a.lse, a.delta, a.lse2, a.dq_acc, n_bh, a.Lq, a.Lq_pad,
                            a.Hq);
}

template <typename T, int D>
cudaError_t run_combine(const float* o_part, const float* lse_part, void* o, float* lse, int B, int Lq, int Hq,
                        int S, cudaStream_t s) {
  const long n_rows = static_cast<long>(B) * Hq * Lq;
  KernelTimer kt("combine", s);
  if (n_rows >= 16384) {  // four rows a warp
    const long warps = (n_rows + 3) / 4;
    const int blocks = static_cast<int>((warps * 32 + 255) / 256);
    return launch_overlapping(combine_kernel<T, D, 4>, dim3(blocks), 256, 0, s, o_part, lse_part, static_cast<T*>(o),
                              lse, B, Lq, Hq, S);
  } else {
    const int blocks = static_cast<int>((n_rows * 32 + 255) / 256);
    return launch_overlapping(combine_kernel<T, D, 1>, dim3(blocks), 256, 0, s, o_part, lse_part, static_cast<T*>(o),
                              lse, B, Lq, Hq, S);
  }
}

// ---- segment summary -----------------------------------------------------------
// Pass 1: one warp per 128-position block (query blocks of every batch
// element first, then key blocks) writes the block's smallest and largest id.
__global__ void __launch_bounds__(256) seg_minmax_kernel(const int32_t* __restrict__ q_seg,
                                                         const int32_t* __restrict__ kv_seg, int B, int Lq, int Lkv,
                                                         int nq, int nk, int4* __restrict__ info) {
  const long rec = static_cast<long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long nqr = static_cast<long>(B) * nq;
  if (rec >= nqr + static_cast<long>(B) * nk) return;
  const bool is_q = rec < nqr;
  const long r = is_q ? rec : rec - nqr;
  const int nblk = is_q ? nq : nk, L = is_q ? Lq : Lkv;
  const int b = static_cast<int>(r / nblk), blk = static_cast<int>(r % nblk);
  const int32_t* ids = (is_q ? q_seg : kv_seg) + static_cast<size_t>(b) * L;
  int mn = INT_MAX, mx = INT_MIN;
#pragma unroll
  for (int i = 0; i < kSegBlock / 32; ++i) {
    const int pos = blk * kSegBlock + i * 32 + lane;
    if (pos < L) {
      const int id = __ldg(ids + pos);
      mn = min(mn, id);
      mx = max(mx, id);
    }
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) info[rec] = make_int4(mn, mx, 0, 0);
}

// Pass 2: one thread per block record finds the first and last block of the
// other side (same batch element) whose id range meets its own; the other
// side's ranges are staged through shared memory 256 at a time.
__global__ void __launch_bounds__(256) seg_span_kernel(int B, int Lq, int Lkv, int nq, int nk, int4* __restrict__ info) {
  __shared__ int2 other[256];
  const int side = blockIdx.z;  // 0: query blocks look at key blocks, 1: the reverse
  const int n_mine = side == 0 ? nq : nk, n_other = side == 0 ? nk : nq;
  const int L_other = side == 0 ? Lkv : Lq;
  const int idx = blockIdx.x * 256 + threadIdx.x;
  for (int b = blockIdx.y; b < B; b += gridDim.y) {
    int4* mine =
        info + (side == 0 ? static_cast<size_t>(b) * nq : static_cast<size_t>(B) * nq + static_cast<size_t>(b) * nk);
    const int4* theirs =
        info + (side == 0 ? static_cast<size_t>(B) * nq + static_cast<size_t>(b) * nk : static_cast<size_t>(b) * nq);
    int4 me = make_int4(0, -1, 0, 0);
    if (idx < n_mine) me = mine[idx];
    int first = INT_MAX, last = -1;
    for (int c0 = 0; c0 < n_other; c0 += 256) {
      __syncthreads();
      if (c0 + static_cast<int>(threadIdx.x) < n_other) {
        const int4 o = theirs[c0 + threadIdx.x];
        other[threadIdx.x] = make_int2(o.x, o.y);
      }
      __syncthreads();
      const int cn = min(256, n_other - c0);
      for (int c = 0; c < cn; ++c) {
        const int2 o = other[c];
        if (o.x <= me.y && o.y >= me.x) {
          first = min(first, c0 + c);
          last = c0 + c;
        }
      }
    }
    // the other side's records are read for their id range only, which this
    // pass never changes, so writing z and w concurrently is harmless
    if (idx < n_mine) {
      me.z = last >= 0 ? first * kSegBlock : 0;
      me.w = last >= 0 ? min(L_other, (last + 1) * kSegBlock) : 0;
      mine[idx] = me;
    }
  }
}

}  // namespace

cudaError_t launch_segment_info(const int32_t* q_seg, const int32_t* kv_seg, int B, int Lq, int Lkv, int4* info,
                                cudaStream_t s) {
  const int nq = (Lq + kSegBlock - 1) / kSegBlock, nk = (Lkv + kSegBlock - 1) / kSegBlock;
  const long recs = static_cast<long>(B) * (nq + nk);
  seg_minmax_kernel<<<static_cast<unsigned>((recs + 7) / 8), 256, 0, s>>>(q_seg, kv_seg, B, Lq, Lkv, nq, nk, info);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((max(nq, nk) + 255) / 256, min(B, 65535), 2);
  seg_span_kernel<<<grid, 256, 0, s>>>(B, Lq, Lkv, nq, nk, info);
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(const PreprocessArgs& a, cudaStream_t s) {
  auto run = [&](auto tag) -> cudaError_t {
    using T = decltype(tag);
    if (a.d == 32) return run_preprocess<T, 32>(a, s);
    if (a.d == 64) return run_preprocess<T, 64>(a, s);
    if (a.d == 256) return run_preprocess<T, 256>(a, s);
    return run_preprocess<T, 128>(a, s);
  };
  if (a.elem == kElemBF16) return run(__nv_bfloat16{});
  if (a.elem == kElemF16) return run(__half{});
  return run(float{});
}

cudaError_t launch_decode_combine(const float* o_part, const float* lse_part, void* o, float* lse, int B, int Lq,
                                  int Hq, int d, int num_splits, int elem, cudaStream_t s) {
  auto run = [&](auto tag) -> cudaError_t {
    using T = decltype(tag);
    if (d == 32) return run_combine<T, 32>(o_part, lse_part, o, lse, B, Lq, Hq, num_splits, s);
    if (d == 64) return run_combine<T, 64>(o_part, lse_part, o, lse, B, Lq, Hq, num_splits, s);
    if (d == 256) return run_combine<T, 256>(o_part, lse_part, o, lse, B, Lq, Hq, num_splits, s);
    return run_combine<T, 128>(o_part, lse_part, o, lse, B, Lq, Hq, num_splits, s);
  };
  if (elem == kElemBF16) return run(__nv_bfloat16{});
  if (elem == kElemF16) return run(__half{});
  return run(float{});
}

}  // namespace attn
