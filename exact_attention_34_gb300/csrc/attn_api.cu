// C-ABI layer: argument validation, TMA descriptor construction, workspace
// sizing and kernel dispatch.  Everything is checked on the host before a
// launch; nothing here allocates device memory or synchronises (except
// attn_device_status, which is documented to).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <initializer_list>
#include <utility>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace attn {

// Device-side status word (one per device the library is used on).
__device__ DeviceStatus g_status;

namespace {

thread_local char t_last_error[512] = "";

attn_status fail(attn_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
attn_status fail(attn_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return s;
}

attn_status ok() {
  t_last_error[0] = '\0';
  return ATTN_OK;
}

attn_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, "%s: not supported by this build", what);
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::atomic<DeviceStatus*> g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

// Device address of g_status for the current device (looked up once per
// device; later calls read it without taking the lock).
DeviceStatus* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceStatus* known = g_status_ptr[dev].load(std::memory_order_acquire);
  if (known != nullptr) return known;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (g_status_ptr[dev].load(std::memory_order_relaxed) == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev].store(static_cast<DeviceStatus*>(p), std::memory_order_release);
  }
  return g_status_ptr[dev].load(std::memory_order_relaxed);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

bool overlap_launch_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("EXACT_ATTN_NO_PDL");
    return v == nullptr || v[0] == '\0' || v[0] == '0';
  }();
  return on;
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Shape/pointer checks common to the forward, backward and decode.
attn_status check_problem(int B, int Lq, int Lkv, int Hq, int Hkv, int d, float scale, int causal,
                          attn_dtype dtype) {
  if (B <= 0 || Lq <= 0 || Lkv <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "sizes must be positive (B=%d Lq=%d Lkv=%d Hq=%d Hkv=%d d=%d)", B, Lq, Lkv,
                Hq, Hkv, d);
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (!(std::isfinite(scale) && scale > 0.f)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (dtype != ATTN_BF16 && dtype != ATTN_FP32 && dtype != ATTN_FP16)
    return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (d != 32 && d != 64 && d != 128 && d != 256)
    return fail(ATTN_ERR_UNSUPPORTED, "head_dim %d not supported (32, 64, 128 or 256)", d);
  if (d == 256 && dtype == ATTN_FP32)
    return fail(ATTN_ERR_UNSUPPORTED, "head_dim 256 runs on the 16-bit tensor-core path only (bf16 or fp16)");
  // 32-bit index headroom for per-row offsets (elements of one tensor)
  const double big = static_cast<double>(B) * Lq * Hq * d;
  const double bigk = static_cast<double>(B) * Lkv * Hkv * d;
  if (big >= 9.0e15 || bigk >= 9.0e15) return fail(ATTN_ERR_INVALID_ARG, "tensor too large");
  if (Lq > (1 << 30) || Lkv > (1 << 30)) return fail(ATTN_ERR_INVALID_ARG, "sequence too long");
  return ATTN_OK;
}

attn_status need_ptrs(std::initializer_list<std::pair<const void*, const char*>> ptrs) {
  for (auto& pr : ptrs) {
    if (pr.first == nullptr) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", pr.second);
    if (!aligned16(pr.first)) return fail(ATTN_ERR_INVALID_ARG, "%s is not 16-byte aligned", pr.second);
  }
  return ATTN_OK;
}

Problem make_problem(int B, int Lq, int Lkv, int Hq, int Hkv, int d, float scale, int causal, const int32_t* kl) {
  Problem p;
  p.B = B;
  p.Lq = Lq;
  p.Lkv = Lkv;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.d = d;
  p.G = Hq / Hkv;
  p.f16 = 0;
  p.causal = causal;
  p.wl = kWinInf;
  p.wr = causal ? 0 : kWinInf;
  p.scale = scale;
  p.kv_lens = kl;
  p.q_seg = nullptr;
  p.kv_seg = nullptr;
  p.seg_qblk = nullptr;
  p.seg_kblk = nullptr;
  return p;
}

size_t seg_info_bytes(int B, int Lq, int Lkv) {
  const size_t nq = (static_cast<size_t>(Lq) + kSegBlock - 1) / kSegBlock;
  const size_t nk = (static_cast<size_t>(Lkv) + kSegBlock - 1) / kSegBlock;
  return static_cast<size_t>(B) * (nq + nk) * sizeof(int4);
}

// Segment ids (required) and their block summary (optional) on a problem.
attn_status set_segments(Problem& pb, const int32_t* q_segment, const int32_t* kv_segment, const void* info) {
  attn_status s = need_ptrs({{q_segment, "q_segment"}, {kv_segment, "kv_segment"}});
  if (s != ATTN_OK) return s;
  pb.q_seg = q_segment;
  pb.kv_seg = kv_segment;
  if (info != nullptr) {
    if (!aligned16(info)) return fail(ATTN_ERR_INVALID_ARG, "segment_info is not 16-byte aligned");
    pb.seg_qblk = static_cast<const int4*>(info);
    pb.seg_kblk = pb.seg_qblk + static_cast<size_t>(pb.B) * ((pb.Lq + kSegBlock - 1) / kSegBlock);
  }
  return ATTN_OK;
}

// A local window: a negative bound, or one at least as long as the keys (left)
// or the queries (right), is unbounded, so finite bounds stay below 2^30 and
// the span arithmetic cannot overflow.
Problem make_window_problem(int B, int Lq, int Lkv, int Hq, int Hkv, int d, float scale, int window_left,
                            int window_right, const int32_t* kl) {
  Problem p = make_problem(B, Lq, Lkv, Hq, Hkv, d, scale, 0, kl);
  p.wl = (window_left < 0 || window_left >= Lkv) ? kWinInf : window_left;
  p.wr = (window_right < 0 || window_right >= Lq) ? kWinInf : window_right;
  // later rows see more keys only when the left side is open and the right bounded
  p.causal = (p.wl >= kWinInf && p.wr < kWinInf) ? 1 : 0;
  return p;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int lq_padded(int Lq) { return (Lq + 127) / 128 * 128; }

// bytes of one [B, Hq, Lq_pad] float32 row-statistics array of the backward
size_t bwd_rowstat_bytes(int B, int Lq, int Hq) {
  return align256(static_cast<size_t>(B) * Hq * lq_padded(Lq) * sizeof(float));
}

}  // namespace

namespace {

// Descriptors encoded recently on this thread.  An encode takes about a
// microsecond of host time; a training loop or a benchmark calls the library
// with the same tensors again and again, and a short call is host-bound.  The
// descriptor is a pure function of the key, so a hit is exact; the cache is
// per thread, so calls stay thread-safe.
struct TmapKey {
  const void* base;
  int elem, B, L, H, d, box_inner, box_rows;
  bool operator==(const TmapKey& o) const {
    return base == o.base && elem == o.elem && B == o.B && L == o.L && H == o.H && d == o.d &&
           box_inner == o.box_inner && box_rows == o.box_rows;
  }
};
struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kTmapCacheSize = 32;
thread_local TmapEntry t_tmap_cache[kTmapCacheSize];
thread_local int t_tmap_next = 0;

bool encode_bshd_tmap(CUtensorMap* map, const void* base, int elem, int B, int L, int H, int d, int box_inner,
                      int box_rows);

}  // namespace

bool make_bshd_tmap(CUtensorMap* map, const void* base, int elem, int B, int L, int H, int d, int box_inner,
                    int box_rows) {
  const TmapKey key{base, elem, B, L, H, d, box_inner, box_rows};
  for (int i = 0; i < kTmapCacheSize; ++i) {
    if (t_tmap_cache[i].valid && t_tmap_cache[i].key == key) {
      *map = t_tmap_cache[i].map;
      return true;
    }
  }
  if (!encode_bshd_tmap(map, base, elem, B, L, H, d, box_inner, box_rows)) return false;
  TmapEntry& e = t_tmap_cache[t_tmap_next];
  t_tmap_next = (t_tmap_next + 1) % kTmapCacheSize;
  e.key = key;
  e.map = *map;
  e.valid = true;
  return true;
}

namespace {

bool encode_bshd_tmap(CUtensorMap* map, const void* base, int elem, int B, int L, int H, int d, int box_inner,
                      int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t es = elem == kElemF32 ? 4 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(H) * d * es, static_cast<cuuint64_t>(d) * es,
                           static_cast<cuuint64_t>(L) * H * d * es};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty = elem == kElemF32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : elem == kElemF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, ty, 4,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

int device_sm_count() {
  static std::atomic<int> cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

namespace {
struct TimingRecord {
  std::string name;
  cudaEvent_t start, stop;
};
std::mutex g_timing_mu;
bool g_timing_on = false;
std::atomic<bool> g_timing_flag{false};  // g_timing_on, readable without the lock
std::vector<TimingRecord> g_timing;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pooled_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void clear_timing_locked() {
  for (auto& r : g_timing) {
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_timing.clear();
}
}  // namespace

KernelTimer::KernelTimer(const char* name, cudaStream_t s) : slot_(-1), stream_(s) {
  if (!g_timing_flag.load(std::memory_order_relaxed)) return;  // timing off: no lock per launch
  std::lock_guard<std::mutex> lk(g_timing_mu);
  if (!g_timing_on) return;
  TimingRecord r{name, pooled_event(), pooled_event()};
  if (r.start == nullptr || r.stop == nullptr) return;
  if (cudaEventRecord(r.start, s) != cudaSuccess) return;
  g_timing.push_back(r);
  slot_ = static_cast<int>(g_timing.size()) - 1;
}

KernelTimer::~KernelTimer() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lk(g_timing_mu);
  if (slot_ < static_cast<int>(g_timing.size())) cudaEventRecord(g_timing[slot_].stop, stream_);
}

}  // namespace attn

using namespace attn;

namespace attn {
namespace {

// The failure path every pipeline kernel relies on, run on purpose: two warps
// wait for an mbarrier phase that nothing completes.  The first wait to pass
// the time limit records (code 1, site) in the status word and raises the
// abort flag, the other warp's wait then returns at once, and the CTA frees
// the TMEM it holds before it exits, as the real kernels do.
__global__ void __launch_bounds__(64) wait_timeout_selftest_kernel(DeviceStatus* st, int site) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_slot;
  const int warp = static_cast<int>(warp_id());
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);  // one arrival completes the phase; none comes
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  (void)__all_sync(0xffffffffu, mbar_wait(&bar, 0, &abort_flag, st, site));
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_slot, 32);
  }
}

}  // namespace
}  // namespace attn

extern "C" {

attn_status attn_selftest_wait_timeout(int site, attn_stream_t stream) {
  DeviceStatus* st = status_ptr();
  if (st == nullptr) return fail(ATTN_ERR_CUDA, "cannot resolve the device status word");
  attn::wait_timeout_selftest_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(st, site);
  return from_cuda(cudaGetLastError(), "attn_selftest_wait_timeout launch");
}

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE";
  }
  return "ATTN_ERR_UNKNOWN";
}

const char* attn_last_error(void) { return t_last_error; }

// Split key ranges of the forward: pieces per query-tile pair, the KV tiles a
// piece holds before a stream is cut further, the partial buffers and the
// per-pair ticket counters.
struct FwdSplit {
  int n_split;
  int chunk;
  float* o_part;
  float* lse_part;
  int* counters;
  size_t counter_bytes;
};

static attn_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, const Problem& pb,
                     attn_dtype dtype, attn_stream_t stream, const FwdSplit* split = nullptr) {
  attn_status s = need_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}});
  if (s != ATTN_OK) return s;
  if (pb.kv_lens != nullptr && (reinterpret_cast<uintptr_t>(pb.kv_lens) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "kv_lens is not 4-byte aligned");
  FwdArgs a;
  a.pb = pb;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  DeviceStatus* st = status_ptr();
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (split != nullptr) {
    a.n_split = split->n_split;
    a.split_chunk = split->chunk;
    a.o_part = split->o_part;
    a.lse_part = split->lse_part;
    a.counters = split->counters;
    cudaError_t e = cudaMemsetAsync(split->counters, 0, split->counter_bytes, cs);
    if (e != cudaSuccess) return from_cuda(e, "attn_fwd_split counters");
  }
  a.pb.f16 = dtype == ATTN_FP16;
  cudaError_t e = dtype != ATTN_FP32           ? launch_fwd_16(a, st, cs)
                  : split_f32_applies(a.pb) ? launch_fwd_split_f32(a, st, cs)
                                            : launch_fwd_f32(a, st, cs);
  return from_cuda(e, "attn_fwd launch");
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Lq, int Lkv,
                     int Hq, int Hkv, int d, float scale, int causal, const int32_t* kv_lens, attn_dtype dtype,
                     attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lkv, Hq, Hkv, d, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  return fwd_impl(q, k, v, o, lse, make_problem(B, Lq, Lkv, Hq, Hkv, d, scale, causal, kv_lens), dtype, stream);
}

attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Lq, int Lkv,
                            int Hq, int Hkv, int d, float scale, int window_left, int window_right,
                            const int32_t* kv_lens, attn_dtype dtype, attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lkv, Hq, Hkv, d, scale, 0, dtype);
  if (s != ATTN_OK) return s;
  return fwd_impl(q, k, v, o, lse,
                  make_window_problem(B, Lq, Lkv, Hq, Hkv, d, scale, window_left, window_right, kv_lens), dtype,
                  stream);
}

attn_status attn_fwd_segments(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Lq,
                              int Lkv, int Hq, int Hkv, int d, float scale, int window_left, int window_right,
                              const int32_t* q_segment, const int32_t* kv_segment, const void* segment_info,
                              const int32_t* kv_lens, attn_dtype dtype, attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lkv, Hq, Hkv, d, scale, 0, dtype);
  if (s != ATTN_OK) return s;
  Problem pb = make_window_problem(B, Lq, Lkv, Hq, Hkv, d, scale, window_left, window_right, kv_lens);
  s = set_segments(pb, q_segment, kv_segment, segment_info);
  if (s != ATTN_OK) return s;
  return fwd_impl(q, k, v, o, lse, pb, dtype, stream);
}

int attn_fwd_num_splits(int B, int Lq, int Lkv, int Hq, int d, int has_kv_lens, attn_dtype dtype) {
  if (B <= 0 || Lq <= 0 || Lkv <= 0 || Hq <= 0 || d <= 0 || d > 128 || dtype == ATTN_FP32) return 1;
  // The pairs of 128-row query tiles that may be busy: with KV lengths on the
  // device every key may sit in one batch element, so only its pairs count.
  // From one full wave of them on, cutting does not shorten the run.
  const long tiles = (Lkv + 127) / 128;
  const long busy = static_cast<long>(Hq) * ((Lq + 255) / 256) * (has_kv_lens ? 1 : B);
  const long sms = device_sm_count();
  if (busy >= sms) return 1;
  // Cutting each busy pair into s pieces takes ceil(s * busy / sms) rounds of
  // 1/s of a pair; each piece also costs its float32 partial (written, then
  // read by the combine) and a program start, charged at 5 % of a pair.  Each
  // piece keeps at least 8 KV tiles, and at most Lkv / 4096 pieces keep the
  // partials small next to the tensor work when every batch element is full.
  const long cap = std::min({8L, tiles / 8, static_cast<long>(Lkv) / 4096});
  int best = 1;
  double best_cost = 1.05;
  for (long s = 2; s <= cap; ++s) {
    const double cost = static_cast<double>((s * busy + sms - 1) / sms) / s + 0.05 * s;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = static_cast<int>(s);
    }
  }
  return best;
}

// o_part [B, Hq, S, Lq, d] fp32, lse_part [B, Hq, S, Lq] fp32, then one int
// ticket counter per pair of 128-row query tiles; each region 256-byte aligned
static size_t fwd_split_counter_bytes(int B, int Lq, int Hq) {
  return static_cast<size_t>(B) * Hq * ((Lq + 255) / 256) * sizeof(int);
}

size_t attn_fwd_split_workspace_size(int B, int Lq, int Hq, int d, int num_splits) {
  if (B <= 0 || Lq <= 0 || Hq <= 0 || d <= 0 || d > 128 || num_splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * num_splits * Lq;
  return align256(rows * d * sizeof(float)) + align256(rows * sizeof(float)) +
         align256(fwd_split_counter_bytes(B, Lq, Hq));
}

attn_status attn_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Lq, int Lkv,
                           int Hq, int Hkv, int d, float scale, int window_left, int window_right,
                           const int32_t* kv_lens, int num_splits, void* workspace, size_t workspace_bytes,
                           attn_dtype dtype, attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lkv, Hq, Hkv, d, scale, 0, dtype);
  if (s != ATTN_OK) return s;
  if (num_splits < 0) return fail(ATTN_ERR_INVALID_ARG, "num_splits must be >= 0");
  if (num_splits > 1024) return fail(ATTN_ERR_INVALID_ARG, "num_splits must be <= 1024");
  if (num_splits == 0) num_splits = attn_fwd_num_splits(B, Lq, Lkv, Hq, d, kv_lens != nullptr, dtype);
  const Problem pb = make_window_problem(B, Lq, Lkv, Hq, Hkv, d, scale, window_left, window_right, kv_lens);
  if (num_splits == 1 || d > 128 || dtype == ATTN_FP32) return fwd_impl(q, k, v, o, lse, pb, dtype, stream);
  if (static_cast<long>(B) * Hq * ((Lq + 255) / 256) * num_splits > INT_MAX)
    return fail(ATTN_ERR_UNSUPPORTED, "grid of %ld programs too large", static_cast<long>(B) * Hq * ((Lq + 255) / 256) * num_splits);
  const size_t need = attn_fwd_split_workspace_size(B, Lq, Hq, d, num_splits);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(ATTN_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t rows = static_cast<size_t>(B) * Hq * num_splits * Lq;
  FwdSplit sp;
  sp.n_split = num_splits;
  const int tiles = (Lkv + 127) / 128;
  sp.chunk = (tiles + num_splits - 1) / num_splits;
  sp.o_part = static_cast<float*>(workspace);
  sp.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * d * sizeof(float)));
  sp.counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + align256(rows * d * sizeof(float)) +
                                       align256(rows * sizeof(float)));
  sp.counter_bytes = fwd_split_counter_bytes(B, Lq, Hq);
  return fwd_impl(q, k, v, o, lse, pb, dtype, stream, &sp);
}

size_t attn_segment_info_size(int B, int Lq, int Lkv) {
  if (B <= 0 || Lq <= 0 || Lkv <= 0) return 0;
  return seg_info_bytes(B, Lq, Lkv);
}

attn_status attn_segment_info(const int32_t* q_segment, const int32_t* kv_segment, int B, int Lq, int Lkv,
                              void* info, size_t info_bytes, attn_stream_t stream) {
  if (B <= 0 || Lq <= 0 || Lkv <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "sizes must be positive (B=%d Lq=%d Lkv=%d)", B, Lq, Lkv);
  if (Lq > (1 << 30) || Lkv > (1 << 30)) return fail(ATTN_ERR_INVALID_ARG, "sequence too long");
  attn_status s = need_ptrs({{q_segment, "q_segment"}, {kv_segment, "kv_segment"}, {info, "segment_info"}});
  if (s != ATTN_OK) return s;
  const size_t need = seg_info_bytes(B, Lq, Lkv);
  if (info_bytes < need) return fail(ATTN_ERR_WORKSPACE, "segment_info of %zu bytes needed, %zu given", need, info_bytes);
  cudaError_t e = launch_segment_info(q_segment, kv_segment, B, Lq, Lkv, static_cast<int4*>(info),
                                      reinterpret_cast<cudaStream_t>(stream));
  return from_cuda(e, "attn_segment_info launch");
}

attn_status attn_bwd_preprocess(const void* o, const void* dout, float* delta, int B, int Lq, int Hq, int d,
                                attn_dtype dtype, attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lq, Hq, Hq, d, 1.0f, 0, dtype);
  if (s != ATTN_OK) return s;
  s = need_ptrs({{o, "o"}, {dout, "dout"}, {delta, "delta"}});
  if (s != ATTN_OK) return s;
  PreprocessArgs pa;
  pa.o = o;
  pa.dout = dout;
  pa.lse = nullptr;
  pa.delta = delta;
  pa.lse2 = nullptr;
  pa.dq_acc = nullptr;
  pa.B = B;
  pa.Lq = Lq;
  pa.Lq_pad = Lq;
  pa.Hq = Hq;
  pa.d = d;
  pa.elem = dtype == ATTN_FP32 ? kElemF32 : dtype == ATTN_FP16 ? kElemF16 : kElemBF16;
  cudaError_t e = launch_bwd_preprocess(pa, reinterpret_cast<cudaStream_t>(stream));
  return from_cuda(e, "attn_bwd_preprocess launch");
}

// ordered single pass: one turn counter per (batch, query head, 128-row query
// tile), then the work-item ticket
static size_t bwd_turn_bytes(int B, int Lq, int Hq) {
  return (static_cast<size_t>(B) * Hq * ((Lq + 127) / 128) + 1) * sizeof(int);
}

size_t attn_bwd_workspace_size(int B, int Lq, int Hq, int d, int deterministic, attn_dtype dtype) {
  (void)dtype;
  if (B <= 0 || Lq <= 0 || Hq <= 0 || d <= 0) return 0;
  size_t bytes = 2 * bwd_rowstat_bytes(B, Lq, Hq);  // delta and lse2, padded rows
  if (deterministic != 1) bytes += align256(static_cast<size_t>(B) * Lq * Hq * d * sizeof(float));
  if (deterministic == 2) bytes += align256(bwd_turn_bytes(B, Lq, Hq));
  return bytes;
}

static attn_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, const Problem& pb, attn_dtype dtype, int deterministic,
                     void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  const int B = pb.B, Lq = pb.Lq, Hq = pb.Hq, d = pb.d;
  attn_status s = need_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}, {dout, "dout"}, {dq, "dq"},
                             {dk, "dk"}, {dv, "dv"}});
  if (s != ATTN_OK) return s;
  if (pb.kv_lens != nullptr && (reinterpret_cast<uintptr_t>(pb.kv_lens) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "kv_lens is not 4-byte aligned");
  if (deterministic < 0 || deterministic > 2) return fail(ATTN_ERR_INVALID_ARG, "deterministic must be 0, 1 or 2");
  if (deterministic == 2 && (dtype == ATTN_FP32 || d > 128))
    return fail(ATTN_ERR_UNSUPPORTED,
                "the ordered single-pass backward (deterministic = 2) runs on the 16-bit tensor-core path at "
                "head_dim <= 128; use deterministic = 1 (two-pass, also reproducible)");
  const size_t need = attn_bwd_workspace_size(B, Lq, Hq, d, deterministic, dtype);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(ATTN_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  BwdArgs a;
  a.pb = pb;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  const size_t rs = bwd_rowstat_bytes(B, Lq, Hq);
  a.delta = static_cast<float*>(workspace);
  a.lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + rs);
  a.dq_acc = deterministic == 1 ? nullptr : reinterpret_cast<float*>(static_cast<char*>(workspace) + 2 * rs);
  a.dq_turn = nullptr;
  a.ticket = nullptr;
  a.turn_bytes = 0;
  if (deterministic == 2) {
    const size_t acc = align256(static_cast<size_t>(B) * Lq * Hq * d * sizeof(float));
    a.dq_turn = reinterpret_cast<int*>(static_cast<char*>(workspace) + 2 * rs + acc);
    a.turn_bytes = bwd_turn_bytes(B, Lq, Hq);
    a.ticket = a.dq_turn + static_cast<size_t>(B) * Hq * ((Lq + 127) / 128);
  }
  a.Lq_pad = lq_padded(Lq);
  a.deterministic = deterministic;
  DeviceStatus* st = status_ptr();
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  a.pb.f16 = dtype == ATTN_FP16;
  cudaError_t e = dtype != ATTN_FP32                                  ? launch_bwd_16(a, st, cs)
                  : (deterministic == 1 && split_f32_applies(a.pb)) ? launch_bwd_split_f32(a, st, cs)
                                                                     : launch_bwd_f32(a, st, cs);
  return from_cuda(e, "attn_bwd launch");
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, int B, int Lq, int Lkv, int Hq, int Hkv, int d, float scale,
                     int causal, const int32_t* kv_lens, attn_dtype dtype, int deterministic, void* workspace,
                     size_t workspace_bytes, attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lkv, Hq, Hkv, d, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, make_problem(B, Lq, Lkv, Hq, Hkv, d, scale, causal, kv_lens),
                  dtype, deterministic, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int B, int Lq, int Lkv, int Hq, int Hkv,
                            int d, float scale, int window_left, int window_right, const int32_t* kv_lens,
                            attn_dtype dtype, int deterministic, void* workspace, size_t workspace_bytes,
                            attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lkv, Hq, Hkv, d, scale, 0, dtype);
  if (s != ATTN_OK) return s;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv,
                  make_window_problem(B, Lq, Lkv, Hq, Hkv, d, scale, window_left, window_right, kv_lens), dtype,
                  deterministic, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_segments(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int Lq, int Lkv, int Hq,
                              int Hkv, int d, float scale, int window_left, int window_right,
                              const int32_t* q_segment, const int32_t* kv_segment, const void* segment_info,
                              const int32_t* kv_lens, attn_dtype dtype, int deterministic, void* workspace,
                              size_t workspace_bytes, attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lkv, Hq, Hkv, d, scale, 0, dtype);
  if (s != ATTN_OK) return s;
  Problem pb = make_window_problem(B, Lq, Lkv, Hq, Hkv, d, scale, window_left, window_right, kv_lens);
  s = set_segments(pb, q_segment, kv_segment, segment_info);
  if (s != ATTN_OK) return s;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, pb, dtype, deterministic, workspace, workspace_bytes, stream);
}

int attn_decode_num_splits(int B, int Lq, int Lkv, int Hq, int Hkv, int d) {
  (void)d;
  if (B <= 0 || Lq <= 0 || Lkv <= 0 || Hq <= 0 || Hkv <= 0) return 1;
  // Enough (batch, KV head, split) programs to fill every SM about 4 times
  // over while each split keeps at least 2 KV tiles; the lengths themselves
  // live on the device, so the choice uses Lkv only.
  const int max_splits = std::max(1, (Lkv + 255) / 256);
  const long want = 4L * device_sm_count();
  long s = (want + static_cast<long>(B) * Hkv - 1) / (static_cast<long>(B) * Hkv);
  if (s < 1) s = 1;
  if (s > max_splits) s = max_splits;
  if (s > 1024) s = 1024;
  (void)Hq;
  return static_cast<int>(s);
}

size_t attn_decode_workspace_size(int B, int Lq, int Hq, int d, int num_splits) {
  if (B <= 0 || Lq <= 0 || Hq <= 0 || d <= 0 || num_splits <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * num_splits * Lq;
  return align256(rows * d * sizeof(float)) + align256(rows * sizeof(float));
}

attn_status attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, float* o_part,
                                float* lse_part, int B, int Lq, int Lkv, int Hq, int Hkv, int d, float scale,
                                int causal, const int32_t* kv_lens, int num_splits, attn_dtype dtype,
                                attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lkv, Hq, Hkv, d, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  s = need_ptrs({{q, "q"}, {k_cache, "k_cache"}, {v_cache, "v_cache"}, {o_part, "o_part"}, {lse_part, "lse_part"}});
  if (s != ATTN_OK) return s;
  if (kv_lens != nullptr && (reinterpret_cast<uintptr_t>(kv_lens) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "kv_lens is not 4-byte aligned");
  if (num_splits < 0) return fail(ATTN_ERR_INVALID_ARG, "num_splits must be >= 0");
  if (num_splits == 0) num_splits = attn_decode_num_splits(B, Lq, Lkv, Hq, Hkv, d);
  const int G = Hq / Hkv;
  if (static_cast<long>(G) * Lq > 128)
    return fail(ATTN_ERR_UNSUPPORTED, "decode packs G*Lq = %ld rows into one 128-row tile (at most 128)",
                static_cast<long>(G) * Lq);
  const int per = (Lkv + num_splits - 1) / num_splits;
  DecodeArgs a;
  a.pb = make_problem(B, Lq, Lkv, Hq, Hkv, d, scale, causal, kv_lens);
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.num_splits = num_splits;
  a.chunk = 128 * ((per + 127) / 128);
  DeviceStatus* st = status_ptr();
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  a.pb.f16 = dtype == ATTN_FP16;
  cudaError_t e = dtype == ATTN_FP32 ? launch_decode_f32(a, st, cs) : launch_decode_16(a, st, cs);
  return from_cuda(e, "attn_decode_splitkv launch");
}

attn_status attn_decode_combine(const float* o_part, const float* lse_part, void* o, float* lse, int B, int Lq,
                                int Hq, int d, int num_splits, attn_dtype dtype, attn_stream_t stream) {
  attn_status s = check_problem(B, Lq, Lq, Hq, Hq, d, 1.0f, 0, dtype);
  if (s != ATTN_OK) return s;
  s = need_ptrs({{o_part, "o_part"}, {lse_part, "lse_part"}, {o, "o"}, {lse, "lse"}});
  if (s != ATTN_OK) return s;
  if (num_splits <= 0) return fail(ATTN_ERR_INVALID_ARG, "num_splits must be > 0");
  cudaError_t e = launch_decode_combine(o_part, lse_part, o, lse, B, Lq, Hq, d, num_splits,
                                        dtype == ATTN_FP32 ? kElemF32 : dtype == ATTN_FP16 ? kElemF16 : kElemBF16,
                                        reinterpret_cast<cudaStream_t>(stream));
  return from_cuda(e, "attn_decode_combine launch");
}

attn_status attn_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  if (on) clear_timing_locked();
  g_timing_on = on != 0;
  g_timing_flag.store(g_timing_on, std::memory_order_relaxed);
  return ok();
}

attn_status attn_timing_query(const char* kernel, double* total_ms, int* launches) {
  if (kernel == nullptr || total_ms == nullptr || launches == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "attn_timing_query: NULL argument");
  std::lock_guard<std::mutex> lk(g_timing_mu);
  double tot = 0.0;
  int n = 0;
  for (auto& r : g_timing) {
    if (r.name != kernel) continue;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e != cudaSuccess) return from_cuda(e, "attn_timing_query synchronize");
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess) return from_cuda(e, "attn_timing_query elapsed");
    tot += ms;
    ++n;
  }
  *total_ms = tot;
  *launches = n;
  return ok();
}

attn_status attn_device_status(int* code, int* site, int reset) {
  DeviceStatus* p = status_ptr();
  if (p == nullptr) return fail(ATTN_ERR_CUDA, "cannot resolve the device status word");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return from_cuda(e, "attn_device_status synchronize");
  DeviceStatus h;
  e = cudaMemcpy(&h, p, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return from_cuda(e, "attn_device_status read");
  if (code) *code = h.code;
  if (site) *site = h.site;
  if (reset) {
    DeviceStatus z = {0, 0, 0};
    e = cudaMemcpy(p, &z, sizeof(z), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return from_cuda(e, "attn_device_status reset");
  }
  if (h.code != 0) return fail(ATTN_ERR_DEVICE, "device status code %d at site %d (block %d)", h.code, h.site, h.block);
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward without any device allocation by the caller.
//
// Some callers cannot allocate device memory at the point where they need the
// backward: hosts whose device memory is owned by a fixed pool or another
// runtime's allocator, latency-critical loops that must not take cudaMalloc's
// implicit device synchronisation, and plugin or interpreter embeddings that
// hand the library only the tensors they already own.  For
// them the deterministic backward's scratch (delta and lse*log2(e), one float
// each per padded query row) lives in a file-scope device array instead of a
// caller workspace.  Every GPU that loads this library holds the array until
// the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB: B*Hq*roundup(Lq,128) <= 524288
static __device__ __align__(256) unsigned char g_bwd_static_scratch[kStaticScratchBytes];

void* g_static_scratch_ptr[kMaxDevices] = {};
std::mutex g_static_scratch_mu;

}  // namespace

extern "C" attn_status attn_bwd_static_scratch(const void* q, const void* k, const void* v, const void* o,
                                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                               int B, int Lq, int Lkv, int Hq, int Hkv, int d, float scale,
                                               int causal, const int32_t* kv_lens, attn_dtype dtype,
                                               attn_stream_t stream) {
  // sizes first: the scratch size below assumes them in range
  attn_status s = check_problem(B, Lq, Lkv, Hq, Hkv, d, scale, causal, dtype);
  if (s != ATTN_OK) return s;
  const size_t need = attn_bwd_workspace_size(B, Lq, Hq, d, 1, dtype);
  if (need > kStaticScratchBytes)
    return fail(ATTN_ERR_WORKSPACE,
                "attn_bwd_static_scratch: this problem needs %zu bytes of scratch but the static scratch holds %zu "
                "(B*Hq*roundup(Lq,128) must be <= 524288); use attn_bwd with a caller workspace",
                need, kStaticScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e, "attn_bwd_static_scratch: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "attn_bwd_static_scratch: device %d out of range", dev);
  void* ptr = nullptr;
  {
    // First call on a device: look up the device address of the array (with
    // that device current).  Make that first call before any stream capture.
    std::lock_guard<std::mutex> lk(g_static_scratch_mu);
    if (g_static_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_bwd_static_scratch);
      if (e != cudaSuccess) return from_cuda(e, "attn_bwd_static_scratch: cudaGetSymbolAddress");
      g_static_scratch_ptr[dev] = p;
    }
    ptr = g_static_scratch_ptr[dev];
  }
  // The deterministic backward overwrites every scratch entry it reads (the
  // preprocess writes delta and lse2 for all padded rows), so nothing has to be
  // cleared between calls.
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Lq, Lkv, Hq, Hkv, d, scale, causal, kv_lens, dtype, 1, ptr,
                  kStaticScratchBytes, stream);
}
