// HBM-bound helper kernels: the backward preprocess (delta = rowsum(dO * O))
// and the log-sum-exp combine of split-KV partials.
#include <cstring>
#include <type_traits>

#include "attn_internal.h"

namespace attn {
namespace {

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&f)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <>
__device__ __forceinline__ void load8<__half>(const __half* p, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
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
__device__ __forceinline__ void load8<float>(const float* p, float (&f)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// delta[b, h, i] = sum_c dO[b, i, h, c] * O[b, i, h, c]  (float32 accumulate).
// Rows are walked in the padded [B, Hq, Lq_pad] order of the outputs; D/8
// threads share a row, each reducing 8 consecutive elements.  Optionally it
// also writes lse2 = lse * log2(e) (+inf where lse = -inf, so that every
// recomputed probability of such a row is 0), fills the pad rows
// Lq <= i < Lq_pad with delta = 0 and lse2 = +inf, and zeroes the float32 dQ
// accumulator of the atomic backward.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                             const float* __restrict__ lse, float* __restrict__ delta,
                                                             float* __restrict__ lse2, float* __restrict__ dq_acc,
                                                             long n_rows_pad, int Lq, int Lq_pad, int Hq) {
  constexpr int kTPR = D / 8;  // threads per row
  const long tid = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long prow = tid / kTPR;  // (b * Hq + h) * Lq_pad + i
  const int part = static_cast<int>(tid % kTPR);
  const long bh = prow / Lq_pad;
  const int i = static_cast<int>(prow % Lq_pad);
  const long b = bh / Hq, h = bh % Hq;
  const bool real = prow < n_rows_pad && i < Lq;
  float acc = 0.f;
  if (real) {
    const long row = (b * Lq + i) * Hq + h;  // row of the [B, Lq, Hq, D] tensors
    float a[8], g[8];
    load8<T>(o + row * D + part * 8, a);
    load8<T>(dout + row * D + part * 8, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(a[e], g[e], acc);
    if (dq_acc != nullptr) {
      float4* z = reinterpret_cast<float4*>(dq_acc + row * D + part * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int off = kTPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (prow < n_rows_pad && part == 0) {
    delta[prow] = acc;  // 0 on pad rows
    if (lse2 != nullptr) {
      const float l = real ? lse[bh * Lq + i] : -INFINITY;
      lse2[prow] = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
    }
  }
}

// One warp per output row (b, h, i): lse = log sum_s exp(lse_s),
// o = sum_s exp(lse_s - lse) o_s.  Empty splits (lse_s = -inf) weigh 0.
template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ o_part,
                                                      const float* __restrict__ lse_part, T* __restrict__ o,
                                                      float* __restrict__ lse, int B, int Lq, int Hq, int S) {
  const long warp = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long n_rows = static_cast<long>(B) * Hq * Lq;
  if (warp >= n_rows) return;
  // warp = (b * Hq + h) * Lq + i
  const int i = static_cast<int>(warp % Lq);
  const long bh = warp / Lq;
  const int h = static_cast<int>(bh % Hq);
  const int b = static_cast<int>(bh / Hq);
  const float* lrow = lse_part + bh * S * Lq + i;  // stride Lq between splits
  float m = -INFINITY;
  for (int s = lane; s < S; s += 32) m = fmaxf(m, lrow[static_cast<long>(s) * Lq]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float tot = 0.f;
  if (m != -INFINITY)
    for (int s = lane; s < S; s += 32) tot += expf(lrow[static_cast<long>(s) * Lq] - m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
  constexpr int kPer = D / 32;  // elements per lane
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  if (m != -INFINITY) {
    const float inv = 1.0f / tot;
    for (int s = 0; s < S; ++s) {
      const float ls = lrow[static_cast<long>(s) * Lq];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - m) * inv;
      const float* src = o_part + ((bh * S + s) * Lq + i) * D + lane * kPer;
      if constexpr (kPer % 2 == 0) {
#pragma unroll
        for (int e = 0; e < kPer; e += 2) {
          const float2 v = *reinterpret_cast<const float2*>(src + e);
          acc[e] = fmaf(w, v.x, acc[e]);
          acc[e + 1] = fmaf(w, v.y, acc[e + 1]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, src[e], acc[e]);
      }
    }
  }
  T* dst = o + ((static_cast<long>(b) * Lq + i) * Hq + h) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
      dst[e] = __float2bfloat16_rn(acc[e]);
    else if constexpr (std::is_same<T, __half>::value)
      dst[e] = __float2half_rn(acc[e]);
    else
      dst[e] = acc[e];
  }
  if (lane == 0) lse[bh * Lq + i] = (m == -INFINITY) ? -INFINITY : m + logf(tot);
}

template <typename T, int D>
cudaError_t run_preprocess(const PreprocessArgs& a, cudaStream_t s) {
  const long n_rows = static_cast<long>(a.B) * a.Hq * a.Lq_pad;
  const long threads = n_rows * (D / 8);
  const int blocks = static_cast<int>((threads + 255) / 256);
  KernelTimer kt("bwd_preprocess", s);
  bwd_preprocess_kernel<T, D><<<blocks, 256, 0, s>>>(static_cast<const T*>(a.o), static_cast<const T*>(a.dout),
                                                     a.lse, a.delta, a.lse2, a.dq_acc, n_rows, a.Lq, a.Lq_pad, a.Hq);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t run_combine(const float* o_part, const float* lse_part, void* o, float* lse, int B, int Lq, int Hq,
                        int S, cudaStream_t s) {
  const long n_rows = static_cast<long>(B) * Hq * Lq;
  const int blocks = static_cast<int>((n_rows * 32 + 255) / 256);
  KernelTimer kt("combine", s);
  combine_kernel<T, D><<<blocks, 256, 0, s>>>(o_part, lse_part, static_cast<T*>(o), lse, B, Lq, Hq, S);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const PreprocessArgs& a, cudaStream_t s) {
  if (a.elem == kElemBF16)
    return a.d == 32   ? run_preprocess<__nv_bfloat16, 32>(a, s)
           : a.d == 64 ? run_preprocess<__nv_bfloat16, 64>(a, s)
                       : run_preprocess<__nv_bfloat16, 128>(a, s);
  if (a.elem == kElemF16)
    return a.d == 32   ? run_preprocess<__half, 32>(a, s)
           : a.d == 64 ? run_preprocess<__half, 64>(a, s)
                       : run_preprocess<__half, 128>(a, s);
  return a.d == 32 ? run_preprocess<float, 32>(a, s)
         : a.d == 64 ? run_preprocess<float, 64>(a, s)
                     : run_preprocess<float, 128>(a, s);
}

cudaError_t launch_decode_combine(const float* o_part, const float* lse_part, void* o, float* lse, int B, int Lq,
                                  int Hq, int d, int num_splits, int elem, cudaStream_t s) {
  auto run = [&](auto tag) -> cudaError_t {
    using T = decltype(tag);
    if (d == 32) return run_combine<T, 32>(o_part, lse_part, o, lse, B, Lq, Hq, num_splits, s);
    if (d == 64) return run_combine<T, 64>(o_part, lse_part, o, lse, B, Lq, Hq, num_splits, s);
    return run_combine<T, 128>(o_part, lse_part, o, lse, B, Lq, Hq, num_splits, s);
  };
  if (elem == kElemBF16) return run(__nv_bfloat16{});
  if (elem == kElemF16) return run(__half{});
  return run(float{});
}

}  // namespace attn
