// float32 attention in true fp32 arithmetic on the CUDA cores (FFMA).
//
// The pages run fp32 attention with TF32 matmuls and note it costs about three
// decimal digits ("GPU and CPU performance", section "Methodology", TF32);
// these kernels keep full fp32 products so float32 inputs match the exact
// result to ~1e-6.  Same method as the tensor-core path: tiled exact
// attention with an online softmax in base 2 (forward, also used for the
// split-KV partials), a delta = rowsum(dO * O) preprocess, and a two-pass
// backward (dK/dV per KV tile, then dQ per query tile) or a single pass with
// float32 atomic dQ accumulation ("Attention performance", section "When to
// use which", backward pass).
//
// Tiles are 64 x 64; 256 threads form a 16 x 16 grid.  Thread (ty, tx) owns
// tile rows 4*ty .. 4*ty+3 and the tile columns tx, tx+16, tx+32, tx+48 (and
// head-dim columns tx + 16*e), so shared-memory rows padded by one float are
// read without bank conflicts.  The forward at head_dim >= 64 instead pads
// rows by four floats, reads them with 16-byte loads, owns head-dim columns
// 4*tx + 64*g + e, and double-buffers its K/V tiles with asynchronous copies.
#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kT = 64;    // tile rows and columns
constexpr int kPad = 1;   // shared-memory row padding (floats)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ int seq_len_of(const int32_t* kv_lens, int b, int Lkv) {
  return kv_lens == nullptr ? Lkv : min(max(kv_lens[b], 0), Lkv);
}

// Copy `rows` x D floats of a [., L, H, D] tensor (rows l0.. of head h) into a
// padded shared tile; rows past L are zero-filled.
template <int D>
__device__ __forceinline__ void load_tile(float* __restrict__ dst, const float* __restrict__ src, int b, int l0,
                                          int h, int L, int H) {
  constexpr int kW = D / 4;  // float4 per row
  for (int idx = threadIdx.x; idx < kT * kW; idx += blockDim.x) {
    const int r = idx / kW, c4 = idx % kW;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (l0 + r < L) v = *reinterpret_cast<const float4*>(src + ((static_cast<size_t>(b) * L + l0 + r) * H + h) * D + c4 * 4);
    float* d = dst + r * (D + kPad) + c4 * 4;
    d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
  }
}

// acc[a][c] = sum_k A[4*ty + a][k] * Bm[tx + 16*c][k]   (both padded, D wide)
template <int D>
__device__ __forceinline__ void tile_dot(const float* __restrict__ A, const float* __restrict__ Bm, int ty, int tx,
                                         float (&acc)[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
#pragma unroll 4
  for (int k = 0; k < D; ++k) {
    float av[4], bv[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) av[a] = A[(4 * ty + a) * (D + kPad) + k];
#pragma unroll
    for (int c = 0; c < 4; ++c) bv[c] = Bm[(tx + 16 * c) * (D + kPad) + k];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(av[a], bv[c], acc[a][c]);
  }
}

// out[a][e] += sum_j P[4*ty + a][j] * M[j][tx + 16*e]  (P is kT x kT padded, M is kT x D padded)
template <int D>
__device__ __forceinline__ void tile_pv(const float* __restrict__ P, const float* __restrict__ M, int ty, int tx,
                                        float (&out)[4][D / 16]) {
#pragma unroll 4
  for (int j = 0; j < kT; ++j) {
    float pv[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) pv[a] = P[(4 * ty + a) * (kT + kPad) + j];
#pragma unroll
    for (int e = 0; e < D / 16; ++e) {
      const float m = M[j * (D + kPad) + tx + 16 * e];
#pragma unroll
      for (int a = 0; a < 4; ++a) out[a][e] = fmaf(pv[a], m, out[a][e]);
    }
  }
}

// out[a][e] += sum_j P[j][4*ty + a] * M[j][tx + 16*e]  (transposed P)
template <int D>
__device__ __forceinline__ void tile_ptv(const float* __restrict__ P, const float* __restrict__ M, int ty, int tx,
                                         float (&out)[4][D / 16]) {
#pragma unroll 4
  for (int j = 0; j < kT; ++j) {
    float pv[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) pv[a] = P[j * (kT + kPad) + 4 * ty + a];
#pragma unroll
    for (int e = 0; e < D / 16; ++e) {
      const float m = M[j * (D + kPad) + tx + 16 * e];
#pragma unroll
      for (int a = 0; a < 4; ++a) out[a][e] = fmaf(pv[a], m, out[a][e]);
    }
  }
}

// ---- forward tiles: rows padded by 4 floats so 16-byte shared loads are
// aligned and conflict-free (row stride 16 bytes past a multiple of 128) ----
constexpr int kPadV = 4;

// Like load_tile, into rows of D + kPadV floats (16-byte stores).
template <int D>
__device__ __forceinline__ void load_tile_v(float* __restrict__ dst, const float* __restrict__ src, int b, int l0,
                                            int h, int L, int H) {
  constexpr int kW = D / 4;
  for (int idx = threadIdx.x; idx < kT * kW; idx += blockDim.x) {
    const int r = idx / kW, c4 = idx % kW;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (l0 + r < L) v = *reinterpret_cast<const float4*>(src + ((static_cast<size_t>(b) * L + l0 + r) * H + h) * D + c4 * 4);
    *reinterpret_cast<float4*>(dst + r * (D + kPadV) + c4 * 4) = v;
  }
}

// Like load_tile_v, but with asynchronous 16-byte copies (rows past L are
// zero-filled by a zero source size); the caller commits and waits.
template <int D>
__device__ __forceinline__ void load_tile_async(float* __restrict__ dst, const float* __restrict__ src, int b, int l0,
                                                int h, int L, int H) {
  constexpr int kW = D / 4;
  for (int idx = threadIdx.x; idx < kT * kW; idx += blockDim.x) {
    const int r = idx / kW, c4 = idx % kW;
    const bool in = l0 + r < L;
    const float* g = src + ((static_cast<size_t>(b) * L + (in ? l0 + r : 0)) * H + h) * D + c4 * 4;
    const uint32_t d = smem_u32(dst + r * (D + kPadV) + c4 * 4);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(g), "r"(in ? 16 : 0) : "memory");
  }
}

__device__ __forceinline__ void async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// acc[a][c] = sum_k A[4*ty + a][k] * Bm[tx + 16*c][k], four k at a time
// (A reads are broadcast across tx, B reads hit 16 distinct rows).
template <int D>
__device__ __forceinline__ void tile_dot_v(const float* __restrict__ A, const float* __restrict__ Bm, int ty, int tx,
                                           float (&acc)[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
#pragma unroll 2
  for (int k = 0; k < D; k += 4) {
    float4 av[4], bv[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) av[a] = *reinterpret_cast<const float4*>(A + (4 * ty + a) * (D + kPadV) + k);
#pragma unroll
    for (int c = 0; c < 4; ++c) bv[c] = *reinterpret_cast<const float4*>(Bm + (tx + 16 * c) * (D + kPadV) + k);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[a][c] = fmaf(av[a].x, bv[c].x, acc[a][c]);
        acc[a][c] = fmaf(av[a].y, bv[c].y, acc[a][c]);
        acc[a][c] = fmaf(av[a].z, bv[c].z, acc[a][c]);
        acc[a][c] = fmaf(av[a].w, bv[c].w, acc[a][c]);
      }
  }
}

// out[a][4*g + e] += sum_j P[4*ty + a][j] * M[j][4*tx + 64*g + e] for
// g < D/64, e < 4: each thread owns two (D = 128) or one (D = 64) groups of
// four adjacent output columns, read from M with 16-byte loads.  P rows are
// padded to kT + kPadV floats, M rows to D + kPadV.
template <int D>
__device__ __forceinline__ void tile_pv_v(const float* __restrict__ P, const float* __restrict__ M, int ty, int tx,
                                          float (&out)[4][D / 16]) {
  constexpr int kGroups = D / 64;  // groups of 4 contiguous columns per thread
#pragma unroll 2
  for (int j = 0; j < kT; j += 4) {
    float4 pv[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) pv[a] = *reinterpret_cast<const float4*>(P + (4 * ty + a) * (kT + kPadV) + j);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {
        const float4 m = *reinterpret_cast<const float4*>(M + (j + jj) * (D + kPadV) + 4 * tx + 64 * g);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float pa = jj == 0 ? pv[a].x : jj == 1 ? pv[a].y : jj == 2 ? pv[a].z : pv[a].w;
          out[a][4 * g + 0] = fmaf(pa, m.x, out[a][4 * g + 0]);
          out[a][4 * g + 1] = fmaf(pa, m.y, out[a][4 * g + 1]);
          out[a][4 * g + 2] = fmaf(pa, m.z, out[a][4 * g + 2]);
          out[a][4 * g + 3] = fmaf(pa, m.w, out[a][4 * g + 3]);
        }
      }
    }
  }
}

__device__ __forceinline__ float row_reduce_max(float v) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float row_reduce_sum(float v) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

struct F32FwdParams {
  const float* q;
  const float* k;
  const float* v;
  float* o;          // final mode: [B, Lq, Hq, D]
  float* lse;        // final mode: [B, Hq, Lq]
  float* o_part;     // partial mode: [B, Hq, S, Lq, D]
  float* lse_part;   // partial mode: [B, Hq, S, Lq]
  const int32_t* kv_lens;
  int B, Lq, Lkv, Hq, Hkv, G, causal, wl, wr, num_splits, chunk;
  const int32_t* q_seg;   // [B, Lq] segment ids or nullptr
  const int32_t* kv_seg;  // [B, Lkv]
  float scale_log2;
};

// grid (ceil(Lq/64), Hq, B * num_splits).  num_splits == 1 and o != nullptr:
// ordinary forward; otherwise split s covers keys [s*chunk, (s+1)*chunk).
template <int D>
__global__ void __launch_bounds__(256) f32_fwd_kernel(const F32FwdParams p) {
  // head_dim >= 64 reads its tiles with 16-byte loads (rows padded by
  // kPadV); head_dim 32 keeps scalar loads (rows padded by kPad)
  constexpr bool kVec = D >= 64;
  constexpr int kP = kVec ? kPadV : kPad;
  // K and V tiles are double-buffered (head_dim >= 64): tile j+1 is copied
  // asynchronously while tile j is computed
  constexpr int kBufs = kVec ? 2 : 1;
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Kb = Qs + kT * (D + kP);
  float* Vb = Kb + kBufs * kT * (D + kP);
  float* Ps = Vb + kBufs * kT * (D + kP);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int q0 = blockIdx.x * kT, h = blockIdx.y;
  const int b = blockIdx.z % p.B, split = blockIdx.z / p.B;
  const int hk = h / p.G;
  const int kvl = seq_len_of(p.kv_lens, b, p.Lkv);
  const int k_lo = split * p.chunk;
  const int k_hi = min(kvl, k_lo + p.chunk);
  const int last_row = min(q0 + kT - 1, p.Lq - 1);
  const int hi_all = min(k_hi, key_span(last_row, p.Lq, kvl, p.wl, p.wr).hi);
  // first key tile (a multiple of kT past k_lo) holding a key of row q0
  const int lo_first = max(k_lo, key_span(q0, p.Lq, kvl, p.wl, p.wr).lo);
  const int j_start = k_lo + ((lo_first - k_lo) / kT) * kT;

  if (kVec) load_tile_v<D>(Qs, p.q, b, q0, h, p.Lq, p.Hq);
  else load_tile<D>(Qs, p.q, b, q0, h, p.Lq, p.Hq);
  float m[4], l[4], acc[4][D / 16];
  int klo[4], khi[4], qseg[4];
  const bool seg = p.q_seg != nullptr;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m[a] = -INFINITY;
    l[a] = 0.f;
    const int i = q0 + 4 * ty + a;
    const Span ks = key_span(i, p.Lq, kvl, p.wl, p.wr);
    klo[a] = i < p.Lq ? ks.lo : 0;
    khi[a] = i < p.Lq ? min(k_hi, ks.hi) : 0;
    qseg[a] = (seg && i < p.Lq) ? p.q_seg[static_cast<size_t>(b) * p.Lq + i] : 0;
#pragma unroll
    for (int e = 0; e < D / 16; ++e) acc[a][e] = 0.f;
  }
  auto issue_kv = [&](int j, int buf) {
    load_tile_async<D>(Kb + buf * kT * (D + kP), p.k, b, j, hk, p.Lkv, p.Hkv);
    load_tile_async<D>(Vb + buf * kT * (D + kP), p.v, b, j, hk, p.Lkv, p.Hkv);
    async_commit();
  };
  if (kVec && j_start < hi_all) issue_kv(j_start, 0);
  for (int j0 = j_start, it = 0; j0 < hi_all; j0 += kT, ++it) {
    const int buf = kVec ? (it & 1) : 0;
    float* Ks = Kb + buf * kT * (D + kP);
    float* Vs = Vb + buf * kT * (D + kP);
    if (kVec) {
      // buffer buf ^ 1 was last read in the previous iteration, which every
      // thread has left (barrier at its end)
      if (j0 + kT < hi_all) {
        issue_kv(j0 + kT, buf ^ 1);
        async_wait<1>();
      } else {
        async_wait<0>();
      }
      __syncthreads();
    } else {
      __syncthreads();
      load_tile<D>(Ks, p.k, b, j0, hk, p.Lkv, p.Hkv);
      load_tile<D>(Vs, p.v, b, j0, hk, p.Lkv, p.Hkv);
      __syncthreads();
    }
    float s[4][4];
    if (kVec) tile_dot_v<D>(Qs, Ks, ty, tx, s);
    else tile_dot<D>(Qs, Ks, ty, tx, s);
    int kseg[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = j0 + tx + 16 * c;
      kseg[c] = (seg && j < kvl) ? p.kv_seg[static_cast<size_t>(b) * p.Lkv + j] : 0;
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = j0 + tx + 16 * c;
        const bool ok = j >= klo[a] && j < khi[a] && (!seg || kseg[c] == qseg[a]);
        s[a][c] = ok ? s[a][c] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[a][c]);
      }
      mx = row_reduce_max(mx);
      const float m_new = fmaxf(m[a], mx);
      const float mb = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m[a] - mb);
      m[a] = m_new;
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float pv = ex2_approx(s[a][c] - mb);
        ls += pv;
        Ps[(4 * ty + a) * (kT + kP) + tx + 16 * c] = pv;
      }
      l[a] = l[a] * alpha + row_reduce_sum(ls);
#pragma unroll
      for (int e = 0; e < D / 16; ++e) acc[a][e] *= alpha;
    }
    __syncthreads();
    if (kVec) tile_pv_v<D>(Ps, Vs, ty, tx, acc);
    else tile_pv<D>(Ps, Vs, ty, tx, acc);
    if (kVec) __syncthreads();  // Ps, Ks and Vs are rewritten next iteration
  }
  const bool partial = p.o == nullptr;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = q0 + 4 * ty + a;
    if (i >= p.Lq) continue;
    const float inv = l[a] > 0.f ? 1.0f / l[a] : 0.f;
    const float lse_v = l[a] > 0.f ? (m[a] + log2f(l[a])) * kLn2 : -INFINITY;
    float* orow;
    if (!partial) {
      orow = p.o + ((static_cast<size_t>(b) * p.Lq + i) * p.Hq + h) * D;
      if (tx == 0) p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.Lq + i] = lse_v;
    } else {
      const size_t r = ((static_cast<size_t>(b) * p.Hq + h) * p.num_splits + split) * p.Lq + i;
      orow = p.o_part + r * D;
      if (tx == 0) p.lse_part[r] = lse_v;
    }
    if (kVec) {  // columns 4*tx + 64*g + e
#pragma unroll
      for (int g = 0; g < D / 64; ++g)
        *reinterpret_cast<float4*>(orow + 4 * tx + 64 * g) =
            make_float4(acc[a][4 * g] * inv, acc[a][4 * g + 1] * inv, acc[a][4 * g + 2] * inv, acc[a][4 * g + 3] * inv);
    } else {  // columns tx + 16*e
#pragma unroll
      for (int e = 0; e < D / 16; ++e) orow[tx + 16 * e] = acc[a][e] * inv;
    }
  }
}

struct F32BwdParams {
  const float* q;
  const float* k;
  const float* v;
  const float* lse;
  const float* dout;
  const float* delta;
  float* dq;
  float* dk;
  float* dv;
  float* dq_acc;  // atomic variant: [B, Lq, Hq, D] (unscaled)
  const int32_t* kv_lens;
  int B, Lq, Lkv, Hq, Hkv, G, causal, wl, wr;
  const int32_t* q_seg;   // [B, Lq] segment ids or nullptr
  const int32_t* kv_seg;  // [B, Lkv]
  float scale, scale_log2;
};

// Recompute P and dS for one (query tile, key tile) pair in "key-major" form:
// element [a][c] is key 4*ty + a (of the key tile) and query tx + 16*c.
// kVec: tiles with rows padded by kPadV, read with 16-byte loads.
template <int D, bool kVec = false>
__device__ __forceinline__ void kt_probs(const float* Ks, const float* Vs, const float* Qs, const float* dOs,
                                         const float* lse2_s, const float* delta_s, const int* klo_s,
                                         const int* khi_s, const int* qseg_s, const int (&kseg)[4], bool seg,
                                         int j0, int ty,
                                         int tx, float scale_log2, float (&P)[4][4], float (&dS)[4][4]) {
  float s[4][4], dp[4][4];
  if constexpr (kVec) {
    tile_dot_v<D>(Ks, Qs, ty, tx, s);
    tile_dot_v<D>(Vs, dOs, ty, tx, dp);
  } else {
    tile_dot<D>(Ks, Qs, ty, tx, s);
    tile_dot<D>(Vs, dOs, ty, tx, dp);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int qi = tx + 16 * c;
    const float l2 = lse2_s[qi];
    const int klo = klo_s[qi], khi = khi_s[qi];
    const float dl = delta_s[qi];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = j0 + 4 * ty + a;
      const bool ok = j >= klo && j < khi && (!seg || qseg_s[qi] == kseg[a]);
      const float pv = ok ? ex2_approx(fmaf(s[a][c], scale_log2, -l2)) : 0.f;
      P[a][c] = pv;
      dS[a][c] = pv * (dp[a][c] - dl);
    }
  }
}

// dK/dV for one 64-key tile of one KV head, summed over the G query heads and
// every query tile that sees it (fixed order: deterministic).  In the atomic
// variant it also adds dS K into the float32 dQ accumulator.
template <int D>
__global__ void __launch_bounds__(256) f32_bwd_dkdv_kernel(const F32BwdParams p) {
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = Ks + kT * (D + kPad);
  float* Qs = Vs + kT * (D + kPad);
  float* dOs = Qs + kT * (D + kPad);
  float* Pt = dOs + kT * (D + kPad);  // [key][query]
  float* dSt = Pt + kT * (kT + kPad);
  float* lse2_s = dSt + kT * (kT + kPad);
  float* delta_s = lse2_s + kT;
  int* klo_s = reinterpret_cast<int*>(delta_s + kT);
  int* khi_s = klo_s + kT;
  int* qseg_s = khi_s + kT;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int j0 = blockIdx.x * kT, hk = blockIdx.y, b = blockIdx.z;
  const int kvl = seq_len_of(p.kv_lens, b, p.Lkv);
  const bool seg = p.q_seg != nullptr;
  int kseg[4];  // segment ids of this thread's 4 keys
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int j = j0 + 4 * ty + a;
    kseg[a] = (seg && j < p.Lkv) ? p.kv_seg[static_cast<size_t>(b) * p.Lkv + j] : 0;
  }
  float dk[4][D / 16], dv[4][D / 16];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int e = 0; e < D / 16; ++e) dk[a][e] = dv[a][e] = 0.f;
  if (j0 < kvl) {
    load_tile<D>(Ks, p.k, b, j0, hk, p.Lkv, p.Hkv);
    load_tile<D>(Vs, p.v, b, j0, hk, p.Lkv, p.Hkv);
    // rows that see some key of this tile: [q_first, q_end)
    const int q_first = query_span(j0, p.Lq, kvl, p.wl, p.wr).lo;
    const int q_end = query_span(min(j0 + kT, kvl) - 1, p.Lq, kvl, p.wl, p.wr).hi;
    for (int g = 0; g < p.G; ++g) {
      const int h = hk * p.G + g;
      for (int q0 = (q_first / kT) * kT; q0 < q_end; q0 += kT) {
        __syncthreads();
        load_tile<D>(Qs, p.q, b, q0, h, p.Lq, p.Hq);
        load_tile<D>(dOs, p.dout, b, q0, h, p.Lq, p.Hq);
        if (threadIdx.x < kT) {
          const int i = q0 + threadIdx.x;
          const bool in = i < p.Lq;
          const float ls = in ? p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.Lq + i] : -INFINITY;
          lse2_s[threadIdx.x] = ls * kLog2e;
          delta_s[threadIdx.x] = in ? p.delta[(static_cast<size_t>(b) * p.Hq + h) * p.Lq + i] : 0.f;
          const Span ks = key_span(i, p.Lq, kvl, p.wl, p.wr);
          const bool any = in && ls != -INFINITY;
          klo_s[threadIdx.x] = any ? ks.lo : 0;
          khi_s[threadIdx.x] = any ? ks.hi : 0;
          qseg_s[threadIdx.x] = (seg && in) ? p.q_seg[static_cast<size_t>(b) * p.Lq + i] : 0;
        }
        __syncthreads();
        float P[4][4], dS[4][4];
        kt_probs<D>(Ks, Vs, Qs, dOs, lse2_s, delta_s, klo_s, khi_s, qseg_s, kseg, seg, j0, ty, tx, p.scale_log2, P,
                    dS);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            Pt[(4 * ty + a) * (kT + kPad) + tx + 16 * c] = P[a][c];
            dSt[(4 * ty + a) * (kT + kPad) + tx + 16 * c] = dS[a][c];
          }
        __syncthreads();
        tile_pv<D>(Pt, dOs, ty, tx, dv);
        tile_pv<D>(dSt, Qs, ty, tx, dk);
        if (p.dq_acc != nullptr) {
          // dQacc[query 4*ty + a][tx + 16e] += sum_key dS^T[key][query] K[key][...]
          float dq[4][D / 16];
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int e = 0; e < D / 16; ++e) dq[a][e] = 0.f;
          tile_ptv<D>(dSt, Ks, ty, tx, dq);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const int i = q0 + 4 * ty + a;
            if (i >= p.Lq) continue;
            float* dst = p.dq_acc + ((static_cast<size_t>(b) * p.Lq + i) * p.Hq + h) * D;
#pragma unroll
            for (int e = 0; e < D / 16; ++e) atomicAdd(dst + tx + 16 * e, dq[a][e]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int j = j0 + 4 * ty + a;
    if (j >= p.Lkv) continue;
    const size_t off = ((static_cast<size_t>(b) * p.Lkv + j) * p.Hkv + hk) * D;
#pragma unroll
    for (int e = 0; e < D / 16; ++e) {
      p.dk[off + tx + 16 * e] = dk[a][e] * p.scale;
      p.dv[off + tx + 16 * e] = dv[a][e];
    }
  }
}

// Row data of query tile q0 of head h for the dK/dV pass, one query row per
// thread threadIdx.x < kT: log2-domain LSE, delta, the row's key span (empty
// for rows past Lq or without a valid key) and its segment id.
__device__ __forceinline__ void dkdv_row_data(const F32BwdParams& p, int b, int h, int q0, int kvl, bool seg,
                                              float* lse2_s, float* delta_s, int* klo_s, int* khi_s, int* qseg_s) {
  if (threadIdx.x < kT) {
    const int i = q0 + threadIdx.x;
    const bool in = i < p.Lq;
    const float ls = in ? p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.Lq + i] : -INFINITY;
    lse2_s[threadIdx.x] = ls * kLog2e;
    delta_s[threadIdx.x] = in ? p.delta[(static_cast<size_t>(b) * p.Hq + h) * p.Lq + i] : 0.f;
    const Span ks = key_span(i, p.Lq, kvl, p.wl, p.wr);
    const bool any = in && ls != -INFINITY;
    klo_s[threadIdx.x] = any ? ks.lo : 0;
    khi_s[threadIdx.x] = any ? ks.hi : 0;
    qseg_s[threadIdx.x] = (seg && in) ? p.q_seg[static_cast<size_t>(b) * p.Lq + i] : 0;
  }
}

// dK/dV of the deterministic backward at head_dim >= 64: the steps of
// f32_bwd_dkdv_kernel (G heads x the query tiles that see the key tile, in
// that order) with tiles read by 16-byte shared loads (rows padded by kPadV)
// and each step's Q, dO and row data double-buffered: step s+1's copies run
// asynchronously while step s computes.  P and dS take turns in one shared
// tile (dV += P^T dO first, then dK += dS^T Q).
template <int D>
__global__ void __launch_bounds__(256) f32_bwd_dkdv_v_kernel(const F32BwdParams p) {
  constexpr int kRow = D + kPadV;
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = Ks + kT * kRow;
  float* Qb = Vs + kT * kRow;         // [2][kT][kRow]
  float* dOb = Qb + 2 * kT * kRow;    // [2][kT][kRow]
  float* PdS = dOb + 2 * kT * kRow;   // [key][query], rows of kT + kPadV
  float* meta = PdS + kT * (kT + kPadV);  // [2] x {lse2, delta, klo, khi, qseg} x kT
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int j0 = blockIdx.x * kT, hk = blockIdx.y, b = blockIdx.z;
  const int kvl = seq_len_of(p.kv_lens, b, p.Lkv);
  const bool seg = p.q_seg != nullptr;
  int kseg[4];  // segment ids of this thread's 4 keys
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int j = j0 + 4 * ty + a;
    kseg[a] = (seg && j < p.Lkv) ? p.kv_seg[static_cast<size_t>(b) * p.Lkv + j] : 0;
  }
  float dk[4][D / 16], dv[4][D / 16];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int e = 0; e < D / 16; ++e) dk[a][e] = dv[a][e] = 0.f;
  if (j0 < kvl) {
    load_tile_v<D>(Ks, p.k, b, j0, hk, p.Lkv, p.Hkv);
    load_tile_v<D>(Vs, p.v, b, j0, hk, p.Lkv, p.Hkv);
    // rows that see some key of this tile: [q_first, q_end)
    const int q_first = query_span(j0, p.Lq, kvl, p.wl, p.wr).lo;
    const int q_end = query_span(min(j0 + kT, kvl) - 1, p.Lq, kvl, p.wl, p.wr).hi;
    const int qt0 = (q_first / kT) * kT;
    const int n_qt = q_end > qt0 ? (q_end - qt0 + kT - 1) / kT : 0;
    const int n_steps = n_qt * p.G;
    auto row_data = [&](int buf) { return meta + buf * 5 * kT; };
    // copies of step `step` into buffer `buf`: Q and dO asynchronously, the
    // row data directly (made visible by the barrier that precedes its use)
    auto issue = [&](int step, int buf) {
      const int h = hk * p.G + step / n_qt, q0 = qt0 + (step % n_qt) * kT;
      load_tile_async<D>(Qb + buf * kT * kRow, p.q, b, q0, h, p.Lq, p.Hq);
      load_tile_async<D>(dOb + buf * kT * kRow, p.dout, b, q0, h, p.Lq, p.Hq);
      async_commit();
      float* m = row_data(buf);
      dkdv_row_data(p, b, h, q0, kvl, seg, m, m + kT, reinterpret_cast<int*>(m + 2 * kT),
                    reinterpret_cast<int*>(m + 3 * kT), reinterpret_cast<int*>(m + 4 * kT));
    };
    if (n_steps > 0) issue(0, 0);
    for (int step = 0; step < n_steps; ++step) {
      const int buf = step & 1;
      // buffer buf ^ 1 was last read in the previous step, which every thread
      // has left (barrier at its end)
      if (step + 1 < n_steps) {
        issue(step + 1, buf ^ 1);
        async_wait<1>();
      } else {
        async_wait<0>();
      }
      __syncthreads();
      const float* Qs = Qb + buf * kT * kRow;
      const float* dOs = dOb + buf * kT * kRow;
      const float* m = row_data(buf);
      float P[4][4], dS[4][4];
      kt_probs<D, true>(Ks, Vs, Qs, dOs, m, m + kT, reinterpret_cast<const int*>(m + 2 * kT),
                        reinterpret_cast<const int*>(m + 3 * kT), reinterpret_cast<const int*>(m + 4 * kT), kseg, seg,
                        j0, ty, tx, p.scale_log2, P, dS);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) PdS[(4 * ty + a) * (kT + kPadV) + tx + 16 * c] = P[a][c];
      __syncthreads();
      tile_pv_v<D>(PdS, dOs, ty, tx, dv);
      __syncthreads();
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) PdS[(4 * ty + a) * (kT + kPadV) + tx + 16 * c] = dS[a][c];
      __syncthreads();
      tile_pv_v<D>(PdS, Qs, ty, tx, dk);
      __syncthreads();  // PdS and this step's buffers are rewritten next step
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int j = j0 + 4 * ty + a;
    if (j >= p.Lkv) continue;
    const size_t off = ((static_cast<size_t>(b) * p.Lkv + j) * p.Hkv + hk) * D;
#pragma unroll
    for (int g = 0; g < D / 64; ++g) {  // columns 4*tx + 64*g + e
      *reinterpret_cast<float4*>(p.dk + off + 4 * tx + 64 * g) =
          make_float4(dk[a][4 * g] * p.scale, dk[a][4 * g + 1] * p.scale, dk[a][4 * g + 2] * p.scale,
                      dk[a][4 * g + 3] * p.scale);
      *reinterpret_cast<float4*>(p.dv + off + 4 * tx + 64 * g) =
          make_float4(dv[a][4 * g], dv[a][4 * g + 1], dv[a][4 * g + 2], dv[a][4 * g + 3]);
    }
  }
}

// dQ for one 64-row query tile: loops over the key tiles it sees.  At
// head_dim >= 64 (as in the forward) tiles are read with 16-byte shared loads
// (rows padded by kPadV) and the K/V tiles are double-buffered: tile j+1 is
// copied asynchronously while tile j is computed.
template <int D>
__global__ void __launch_bounds__(256) f32_bwd_dq_kernel(const F32BwdParams p) {
  constexpr bool kVec = D >= 64;
  constexpr int kP = kVec ? kPadV : kPad;
  constexpr int kBufs = kVec ? 2 : 1;
  extern __shared__ float sm[];
  float* Qs = sm;
  float* dOs = Qs + kT * (D + kP);
  float* Kb = dOs + kT * (D + kP);
  float* Vb = Kb + kBufs * kT * (D + kP);
  float* dSs = Vb + kBufs * kT * (D + kP);  // [query][key]
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int q0 = blockIdx.x * kT, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / p.G;
  const int kvl = seq_len_of(p.kv_lens, b, p.Lkv);
  if (kVec) {
    load_tile_v<D>(Qs, p.q, b, q0, h, p.Lq, p.Hq);
    load_tile_v<D>(dOs, p.dout, b, q0, h, p.Lq, p.Hq);
  } else {
    load_tile<D>(Qs, p.q, b, q0, h, p.Lq, p.Hq);
    load_tile<D>(dOs, p.dout, b, q0, h, p.Lq, p.Hq);
  }
  float l2[4], dl[4];
  int klo[4], khi[4], qseg[4];
  const bool seg = p.q_seg != nullptr;
  float acc[4][D / 16];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = q0 + 4 * ty + a;
    const bool in = i < p.Lq;
    const float ls = in ? p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.Lq + i] : -INFINITY;
    l2[a] = ls * kLog2e;
    dl[a] = in ? p.delta[(static_cast<size_t>(b) * p.Hq + h) * p.Lq + i] : 0.f;
    const Span ks = key_span(i, p.Lq, kvl, p.wl, p.wr);
    const bool any = in && ls != -INFINITY;
    klo[a] = any ? ks.lo : 0;
    khi[a] = any ? ks.hi : 0;
    qseg[a] = (seg && in) ? p.q_seg[static_cast<size_t>(b) * p.Lq + i] : 0;
#pragma unroll
    for (int e = 0; e < D / 16; ++e) acc[a][e] = 0.f;
  }
  const int last_row = min(q0 + kT - 1, p.Lq - 1);
  const int hi_all = key_span(last_row, p.Lq, kvl, p.wl, p.wr).hi;
  const int lo_all = key_span(min(q0, p.Lq - 1), p.Lq, kvl, p.wl, p.wr).lo;
  const int j_start = (lo_all / kT) * kT;
  auto issue_kv = [&](int j, int buf) {
    load_tile_async<D>(Kb + buf * kT * (D + kP), p.k, b, j, hk, p.Lkv, p.Hkv);
    load_tile_async<D>(Vb + buf * kT * (D + kP), p.v, b, j, hk, p.Lkv, p.Hkv);
    async_commit();
  };
  if (kVec && j_start < hi_all) issue_kv(j_start, 0);
  for (int j0 = j_start, it = 0; j0 < hi_all; j0 += kT, ++it) {
    const int buf = kVec ? (it & 1) : 0;
    float* Ks = Kb + buf * kT * (D + kP);
    float* Vs = Vb + buf * kT * (D + kP);
    if (kVec) {
      // buffer buf ^ 1 was last read in the previous iteration, which every
      // thread has left (barrier at its end)
      if (j0 + kT < hi_all) {
        issue_kv(j0 + kT, buf ^ 1);
        async_wait<1>();
      } else {
        async_wait<0>();
      }
      __syncthreads();
    } else {
      __syncthreads();
      load_tile<D>(Ks, p.k, b, j0, hk, p.Lkv, p.Hkv);
      load_tile<D>(Vs, p.v, b, j0, hk, p.Lkv, p.Hkv);
      __syncthreads();
    }
    float s[4][4], dp[4][4];
    if (kVec) {
      tile_dot_v<D>(Qs, Ks, ty, tx, s);
      tile_dot_v<D>(dOs, Vs, ty, tx, dp);
    } else {
      tile_dot<D>(Qs, Ks, ty, tx, s);
      tile_dot<D>(dOs, Vs, ty, tx, dp);
    }
    int kseg[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = j0 + tx + 16 * c;
      kseg[c] = (seg && j < kvl) ? p.kv_seg[static_cast<size_t>(b) * p.Lkv + j] : 0;
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = j0 + tx + 16 * c;
        const bool ok = j >= klo[a] && j < khi[a] && (!seg || kseg[c] == qseg[a]);
        const float pv = ok ? ex2_approx(fmaf(s[a][c], p.scale_log2, -l2[a])) : 0.f;
        dSs[(4 * ty + a) * (kT + kP) + tx + 16 * c] = pv * (dp[a][c] - dl[a]);
      }
    __syncthreads();
    if (kVec) {
      tile_pv_v<D>(dSs, Ks, ty, tx, acc);
      __syncthreads();  // dSs, Ks and Vs are rewritten next iteration
    } else {
      tile_pv<D>(dSs, Ks, ty, tx, acc);
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = q0 + 4 * ty + a;
    if (i >= p.Lq) continue;
    float* dst = p.dq + ((static_cast<size_t>(b) * p.Lq + i) * p.Hq + h) * D;
    if (kVec) {  // columns 4*tx + 64*g + e
#pragma unroll
      for (int g = 0; g < D / 64; ++g)
        *reinterpret_cast<float4*>(dst + 4 * tx + 64 * g) =
            make_float4(acc[a][4 * g] * p.scale, acc[a][4 * g + 1] * p.scale, acc[a][4 * g + 2] * p.scale,
                        acc[a][4 * g + 3] * p.scale);
    } else {  // columns tx + 16*e
#pragma unroll
      for (int e = 0; e < D / 16; ++e) dst[tx + 16 * e] = acc[a][e] * p.scale;
    }
  }
}

// dq = scale * dq_acc  (atomic variant, float32 output)
__global__ void f32_dq_convert_kernel(const float* __restrict__ acc, float* __restrict__ dq, long n, float scale) {
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) dq[i] = acc[i] * scale;
}

template <int D>
constexpr int fwd_smem() {
  constexpr int kP = D >= 64 ? kPadV : kPad;
  constexpr int kBufs = D >= 64 ? 2 : 1;
  return ((1 + 2 * kBufs) * kT * (D + kP) + kT * (kT + kP)) * 4;
}
template <int D>
constexpr int dkdv_smem() {
  return (4 * kT * (D + kPad) + 2 * kT * (kT + kPad) + 5 * kT) * 4;  // + lse2, delta, span lo/hi, segment ids
}
template <int D>
constexpr int dkdv_v_smem() {
  return (6 * kT * (D + kPadV) + kT * (kT + kPadV) + 2 * 5 * kT) * 4;
}
template <int D>
constexpr int dq_smem() {
  constexpr int kP = D >= 64 ? kPadV : kPad;
  constexpr int kBufs = D >= 64 ? 2 : 1;
  return ((2 + 2 * kBufs) * kT * (D + kP) + kT * (kT + kP)) * 4;
}

template <int D>
cudaError_t run_fwd(const F32FwdParams& p, int splits, cudaStream_t s) {
  cudaError_t e = ensure_dynamic_smem<f32_fwd_kernel<D>>(fwd_smem<D>());
  if (e != cudaSuccess) return e;
  dim3 grid((p.Lq + kT - 1) / kT, p.Hq, p.B * splits);
  {
    KernelTimer kt(splits > 1 || p.o == nullptr ? "decode_f32" : "fwd_f32", s);
    f32_fwd_kernel<D><<<grid, 256, fwd_smem<D>(), s>>>(p);
  }
  return cudaGetLastError();
}

template <int D>
cudaError_t run_bwd(const F32BwdParams& p, bool atomic_dq, cudaStream_t s) {
  dim3 g1((p.Lkv + kT - 1) / kT, p.Hkv, p.B);
  cudaError_t e;
  bool vec = false;
  if constexpr (D >= 64) vec = !atomic_dq;
  if (vec) {  // 16-byte loads, double-buffered query tiles
    if constexpr (D >= 64) {
      e = ensure_dynamic_smem<f32_bwd_dkdv_v_kernel<D>>(dkdv_v_smem<D>());
      if (e != cudaSuccess) return e;
      KernelTimer kt("bwd_dkdv_f32", s);
      f32_bwd_dkdv_v_kernel<D><<<g1, 256, dkdv_v_smem<D>(), s>>>(p);
    }
  } else {
    e = ensure_dynamic_smem<f32_bwd_dkdv_kernel<D>>(dkdv_smem<D>());
    if (e != cudaSuccess) return e;
    KernelTimer kt("bwd_dkdv_f32", s);
    f32_bwd_dkdv_kernel<D><<<g1, 256, dkdv_smem<D>(), s>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (atomic_dq) {
    const long n = static_cast<long>(p.B) * p.Lq * p.Hq * D;
    KernelTimer kt("dq_convert_f32", s);
    f32_dq_convert_kernel<<<static_cast<int>((n + 255) / 256), 256, 0, s>>>(p.dq_acc, p.dq, n, p.scale);
    return cudaGetLastError();
  }
  e = ensure_dynamic_smem<f32_bwd_dq_kernel<D>>(dq_smem<D>());
  if (e != cudaSuccess) return e;
  dim3 g2((p.Lq + kT - 1) / kT, p.Hq, p.B);
  {
    KernelTimer kt("bwd_dq_f32", s);
    f32_bwd_dq_kernel<D><<<g2, 256, dq_smem<D>(), s>>>(p);
  }
  return cudaGetLastError();
}

F32FwdParams fwd_params(const Problem& pb, const void* q, const void* k, const void* v) {
  F32FwdParams p{};
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.kv_lens = pb.kv_lens;
  p.B = pb.B;
  p.Lq = pb.Lq;
  p.Lkv = pb.Lkv;
  p.Hq = pb.Hq;
  p.Hkv = pb.Hkv;
  p.G = pb.G;
  p.causal = pb.causal;
  p.wl = pb.wl;
  p.wr = pb.wr;
  p.q_seg = pb.q_seg;
  p.kv_seg = pb.kv_seg;
  p.scale_log2 = pb.scale * kLog2e;
  return p;
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdArgs& a, DeviceStatus* st, cudaStream_t s) {
  (void)st;
  F32FwdParams p = fwd_params(a.pb, a.q, a.k, a.v);
  p.o = static_cast<float*>(a.o);
  p.lse = a.lse;
  p.num_splits = 1;
  p.chunk = a.pb.Lkv;
  return a.pb.d == 32 ? run_fwd<32>(p, 1, s) : a.pb.d == 64 ? run_fwd<64>(p, 1, s) : run_fwd<128>(p, 1, s);
}

cudaError_t launch_decode_f32(const DecodeArgs& a, DeviceStatus* st, cudaStream_t s) {
  (void)st;
  F32FwdParams p = fwd_params(a.pb, a.q, a.k, a.v);
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.num_splits = a.num_splits;
  p.chunk = a.chunk;
  return a.pb.d == 32   ? run_fwd<32>(p, a.num_splits, s)
         : a.pb.d == 64 ? run_fwd<64>(p, a.num_splits, s)
                        : run_fwd<128>(p, a.num_splits, s);
}

cudaError_t launch_bwd_f32(const BwdArgs& a, DeviceStatus* st, cudaStream_t s) {
  (void)st;
  const Problem& pb = a.pb;
  PreprocessArgs pa;
  pa.o = a.o;
  pa.dout = a.dout;
  pa.lse = nullptr;
  pa.delta = a.delta;  // unpadded [B, Hq, Lq] layout inside the (larger) workspace
  pa.lse2 = nullptr;
  pa.dq_acc = a.deterministic ? nullptr : a.dq_acc;
  pa.B = pb.B;
  pa.Lq = pb.Lq;
  pa.Lq_pad = pb.Lq;
  pa.Hq = pb.Hq;
  pa.d = pb.d;
  pa.elem = kElemF32;
  cudaError_t e = launch_bwd_preprocess(pa, s);
  if (e != cudaSuccess) return e;
  F32BwdParams p{};
  p.q = static_cast<const float*>(a.q);
  p.k = static_cast<const float*>(a.k);
  p.v = static_cast<const float*>(a.v);
  p.lse = a.lse;
  p.dout = static_cast<const float*>(a.dout);
  p.delta = a.delta;
  p.dq = static_cast<float*>(a.dq);
  p.dk = static_cast<float*>(a.dk);
  p.dv = static_cast<float*>(a.dv);
  p.dq_acc = a.deterministic ? nullptr : a.dq_acc;
  p.kv_lens = pb.kv_lens;
  p.B = pb.B;
  p.Lq = pb.Lq;
  p.Lkv = pb.Lkv;
  p.Hq = pb.Hq;
  p.Hkv = pb.Hkv;
  p.G = pb.G;
  p.causal = pb.causal;
  p.wl = pb.wl;
  p.wr = pb.wr;
  p.q_seg = pb.q_seg;
  p.kv_seg = pb.kv_seg;
  p.scale = pb.scale;
  p.scale_log2 = pb.scale * kLog2e;
  return pb.d == 32   ? run_bwd<32>(p, !a.deterministic, s)
         : pb.d == 64 ? run_bwd<64>(p, !a.deterministic, s)
                      : run_bwd<128>(p, !a.deterministic, s);
}

}  // namespace attn
