// Operand splitting for float32 attention on the bf16 tensor cores: a float32
// value x becomes bf16 parts whose sum approximates it (two parts: 16
// significant bits, |x - hi - lo| <= 2^-17 |x|) or equals it (three parts,
// 8 + 8 + 8 bits), so a product A B can be taken as a few bf16 MMAs with
// float32 accumulation (A_hi B_hi + A_hi B_lo + A_lo B_hi).  The kernels read
// float32 tiles from global memory with four converter warps and write the
// parts into shared memory in the 128-byte-swizzled layout that the MMA
// descriptors (and TMA, in the 16-bit kernels) use: one box per 64 columns,
// 128 bytes a row, 16-byte chunk c of row r at chunk c ^ (r % 8).
#pragma once
#include "attn_internal.h"

namespace attn {
namespace split {

// Split 8 consecutive floats into packed bf16 hi and lo parts.
__device__ __forceinline__ void split8(const float4& a, const float4& b, uint4& hi, uint4& lo) {
  const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
    const float h0 = __uint_as_float(h[i] << 16), h1 = __uint_as_float(h[i] & 0xffff0000u);
    l[i] = pack_bf16x2(x[2 * i] - h0, x[2 * i + 1] - h1);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Split 8 consecutive floats into three packed bf16 parts whose sum is exact.
__device__ __forceinline__ void split8x3(const float4& a, const float4& b, uint4& hi, uint4& mid, uint4& lo) {
  const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t h[4], m[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
    const float r0 = x[2 * i] - __uint_as_float(h[i] << 16), r1 = x[2 * i + 1] - __uint_as_float(h[i] & 0xffff0000u);
    m[i] = pack_bf16x2(r0, r1);
    l[i] = pack_bf16x2(r0 - __uint_as_float(m[i] << 16), r1 - __uint_as_float(m[i] & 0xffff0000u));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  mid = make_uint4(m[0], m[1], m[2], m[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Converters: rows [row0, row0 + R) of a [B, L, H, D] float32 tensor (head
// h, batch b; rows past `valid` read as zero) -> rows [r0, r0 + R) of bf16 hi
// and lo tiles in the 128-byte-swizzled box layout (one box per 64 columns,
// RB rows of 128 bytes each).  128 threads; thread t takes 8-column chunks
// t, t + 128, ...
// With kThree, a third (mid) tile at mid_tile takes the middle part and lo_tile
// the exact remainder.
template <int D, int R, int RB, bool kThree = false>
__device__ __forceinline__ void convert_tile(const float* __restrict__ src, int b, int L, int H, int h, int row0,
                                             int valid, uint8_t* hi_tile, uint8_t* lo_tile, int r0, int t,
                                             uint8_t* mid_tile = nullptr) {
  constexpr int kChunks = R * (D / 8);
  constexpr int kPer = kChunks / 128;
  static_assert(kChunks % 128 == 0, "tile must split evenly over the converter threads");
  float4 va[kPer], vb[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {  // all loads in flight before the conversions
    const int c = t + 128 * i;
    const int r = c / (D / 8), c8 = c % (D / 8);
    const int row = row0 + r;
    if (row < valid) {
      const float4* p = reinterpret_cast<const float4*>(src + ((static_cast<size_t>(b) * L + row) * H + h) * D + c8 * 8);
      va[i] = __ldg(p);
      vb[i] = __ldg(p + 1);
    } else {
      va[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      vb[i] = va[i];
    }
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int c = t + 128 * i;
    const int r = c / (D / 8), c8 = c % (D / 8);
    uint4 hi, mid, lo;
    if (kThree)
      split8x3(va[i], vb[i], hi, mid, lo);
    else
      split8(va[i], vb[i], hi, lo);
    const int rr = r0 + r;
    const int off = (c8 >> 3) * RB * 128 + rr * 128 + (((c8 & 7) ^ (rr & 7)) << 4);
    *reinterpret_cast<uint4*>(hi_tile + off) = hi;
    if (kThree) *reinterpret_cast<uint4*>(mid_tile + off) = mid;
    *reinterpret_cast<uint4*>(lo_tile + off) = lo;
  }
}


}  // namespace split
}  // namespace attn
