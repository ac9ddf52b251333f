// C-ABI entry points: argument validation, TMA descriptor encoding, kernel selection.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <vector>

#include "fa.h"
#include "fa_launch.cuh"
#include "fa_kernel_f32.cuh"
#include "fa_merge.cuh"

namespace fa {

FA_DECLARE_LAUNCH(extern, 64, false, false)
FA_DECLARE_LAUNCH(extern, 64, false, true)
FA_DECLARE_LAUNCH(extern, 64, true, false)
FA_DECLARE_LAUNCH(extern, 64, true, true)
FA_DECLARE_LAUNCH(extern, 128, false, false)
FA_DECLARE_LAUNCH(extern, 128, false, true)
FA_DECLARE_LAUNCH(extern, 128, true, false)
FA_DECLARE_LAUNCH(extern, 128, true, true)
FA_DECLARE_LAUNCH_PARTIAL(extern, 64, false, false)
FA_DECLARE_LAUNCH_PARTIAL(extern, 64, false, true)
FA_DECLARE_LAUNCH_PARTIAL(extern, 64, true, false)
FA_DECLARE_LAUNCH_PARTIAL(extern, 64, true, true)
FA_DECLARE_LAUNCH_PARTIAL(extern, 128, false, false)
FA_DECLARE_LAUNCH_PARTIAL(extern, 128, false, true)
FA_DECLARE_LAUNCH_PARTIAL(extern, 128, true, false)
FA_DECLARE_LAUNCH_PARTIAL(extern, 128, true, true)
FA_DECLARE_LAUNCH_PAIR(extern, 64, false, true)
FA_DECLARE_LAUNCH_PAIR(extern, 64, true, true)

// Error bits OR-ed in by kernels of this library on the device they ran on.
__device__ unsigned int g_device_status = 0;

// Split-KV scratch of fa_forward_splitkv_noalloc: module memory, so that entry point needs no
// allocation. One per device; calls that overlap in time on a device share it.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Work schedules of causal multi-wave launches (get_schedule): module memory, filled by a copy
// on the first call of each shape, so fa_forward allocates nothing.
constexpr size_t kSchedulePoolInts = size_t(1) << 20;
static __device__ int g_schedule_pool[kSchedulePoolInts];

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
constexpr long long kL2SectionBytes = 32ll << 20;  // K+V bytes of the heads kept close in time
constexpr int kMaxSplits = 256;                    // split-KV ranges per query tile
constexpr size_t kWorkspaceAlign = 256;

std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_decomposition{FA_DECOMP_AUTO};
std::atomic<int> g_force_stall{0};
thread_local int t_last_cuda_error = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceInfo {
  std::atomic<bool> ready{false};
  int status = FA_OK;  // FA_OK or FA_ERR_UNSUPPORTED
  int num_sms = 0;
  unsigned int* status_word = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return FA_ERR_CUDA;
}

// One-time per-device setup: architecture check, SM count, status word, driver entry point.
int device_setup(int dev, DeviceInfo*& out) {
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  DeviceInfo& d = g_devices[dev];
  if (d.ready.load(std::memory_order_acquire)) {  // fast path after the first call
    out = &d;
    return d.status;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!d.ready.load(std::memory_order_relaxed)) {
    int major = 0, minor = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    d.status = (major == 10 && minor == 3) ? FA_OK : FA_ERR_UNSUPPORTED;
    if (d.status == FA_OK) {
      void* sym = nullptr;
      e = cudaGetSymbolAddress(&sym, g_device_status);
      if (e != cudaSuccess) return cuda_fail(e);
      d.status_word = static_cast<unsigned int*>(sym);
    }
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess) return cuda_fail(e);
      if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cuda_fail(cudaErrorSymbolNotFound);
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready.store(true, std::memory_order_release);
  }
  out = &d;
  return d.status;
}

// [BH, N, D] tensor viewed as 3-D (D, N, BH); box (128 bytes of columns, box_rows, 1), 128-byte
// swizzle, zero fill outside the tensor. dtype: FA_DTYPE_FP16, _BF16 or _FP32.
int encode_map(CUtensorMap* map, const void* base, int dtype, int BH, int N, int D, int box_rows) {
  const cuuint64_t es = dtype == FA_DTYPE_FP32 ? 4 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * es, static_cast<cuuint64_t>(N) * D * es};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType t = dtype == FA_DTYPE_FP32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                : dtype == FA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = g_encode(map, t, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return FA_OK;
}

// Split-KV partial O: fp32 [planes, N, D] viewed as 3-D (D, N, planes); box (32, 32, 1), i.e.
// 32 rows of 128 bytes, 128-byte swizzle.
int encode_map_f32(CUtensorMap* map, void* base, long long planes, int N, int D) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(planes)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(N) * D * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return FA_OK;
}

// Launch parameters (tensor maps included) of recent calls on this host thread: a repeated
// call with the same buffers and sizes skips validation and descriptor encoding.
struct LaunchKey {
  const void* ptr[6];  // q, k, v, o, lse, workspace
  int B, H, N, D, causal, dtype, dev, decomp, stall, splits;
  float scale;
  unsigned long long timeout;
  size_t workspace_bytes;
  bool operator==(const LaunchKey& o) const { return std::memcmp(this, &o, sizeof(LaunchKey)) == 0; }
};
struct ScheduleEntry;
bool schedule_ready(ScheduleEntry& e, cudaStream_t s);
struct LaunchEntry {
  LaunchKey key;
  Params params;
  int grid;
  bool splitk;
  bool pair;       // paired split-K form
  bool f32;        // fp32-I/O (tf32) kernel
  int splits;      // > 1: split-KV partial kernel, then the merge
  void* o;         // merge output
  float* lse;
  long long rows;  // BH * N
  int num_sms;
  ScheduleEntry* sched;  // the work table the params point to, or nullptr
  bool valid;
};
constexpr int kCacheSize = 4;
thread_local LaunchEntry t_cache[kCacheSize];
thread_local int t_cache_next = 0;

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

cudaError_t launch_partial(const Params& p, int grid, int D, bool bf16, bool c, cudaStream_t s) {
  if (D == 64) {
    if (!bf16) return c ? launch_forward<64, false, true, true, true>(p, grid, s) : launch_forward<64, false, false, true, true>(p, grid, s);
    return c ? launch_forward<64, true, true, true, true>(p, grid, s) : launch_forward<64, true, false, true, true>(p, grid, s);
  }
  if (!bf16) return c ? launch_forward<128, false, true, true, true>(p, grid, s) : launch_forward<128, false, false, true, true>(p, grid, s);
  return c ? launch_forward<128, true, true, true, true>(p, grid, s) : launch_forward<128, true, false, true, true>(p, grid, s);
}

cudaError_t launch(const Params& p, int grid, bool splitk, bool pair, int D, bool bf16, bool c, cudaStream_t s) {
  if (pair && c && D == 64)
    return bf16 ? launch_forward<64, true, true, true, false, true>(p, grid, s)
                : launch_forward<64, false, true, true, false, true>(p, grid, s);
#define FA_LAUNCH(DD, BB, CC) \
  (splitk ? launch_forward<DD, BB, CC, true>(p, grid, s) : launch_forward<DD, BB, CC, false>(p, grid, s))
  if (D == 64) {
    if (!bf16) return c ? FA_LAUNCH(64, false, true) : FA_LAUNCH(64, false, false);
    return c ? FA_LAUNCH(64, true, true) : FA_LAUNCH(64, true, false);
  }
  if (!bf16) return c ? FA_LAUNCH(128, false, true) : FA_LAUNCH(128, false, false);
  return c ? FA_LAUNCH(128, true, true) : FA_LAUNCH(128, true, false);
#undef FA_LAUNCH
}

// Split-KV workspace: partial O [splits, BH, N, D] fp32, then partial lse [splits, BH, N] fp32,
// each starting on a kWorkspaceAlign boundary.
size_t workspace_o_bytes(long long BH, int N, int D, int splits) {
  const size_t b = static_cast<size_t>(splits) * static_cast<size_t>(BH) * static_cast<size_t>(N) * D * sizeof(float);
  return (b + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign;
}
size_t workspace_bytes(long long BH, int N, int D, int splits) {
  const size_t l = static_cast<size_t>(splits) * static_cast<size_t>(BH) * static_cast<size_t>(N) * sizeof(float);
  return workspace_o_bytes(BH, N, D, splits) + (l + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign;
}

// Split count for a split-KV forward: a cost model of the whole job in microseconds. Work
// items (one query tile and one K/V range) are dealt to the SMs greedily in the kernel's
// longest-first order; an item costs a fixed overhead plus its K/V tiles. More splits shorten
// the longest items (causal rows near the end, or too few items to fill the GPU) but add
// items, partial-result traffic and the merge kernel.
int choose_splits(long long BH, int N, int D, bool causal, int num_sms) {
  const int nkt = (N + kBN - 1) / kBN;
  const long long base_items = BH * nkt;
  if (base_items >= 4ll * num_sms || nkt < 2) return 1;
  const double t_tile = D == 64 ? 0.8 : 0.85;  // us per 128 x 128 tile on one SM
  const double t_item = 3.0;                   // us of per-item prologue / epilogue
  const double bytes_per_us = 6.0e6;
  const long long rows = BH * static_cast<long long>(N);
  double best_t = 0.0;
  int best = 1;
  const int max_s = std::min(16, nkt);
  std::vector<double> costs;
  for (int S = 1; S <= max_s; ++S) {
    costs.clear();
    for (int qt = 0; qt < nkt; ++qt) {
      const int nk = causal ? qt + 1 : nkt;
      for (int sp = 0; sp < S; ++sp) {
        const int n = (sp + 1) * nk / S - sp * nk / S;
        if (n > 0) costs.push_back(t_item + n * t_tile);
      }
    }
    std::sort(costs.begin(), costs.end(), std::greater<double>());
    std::priority_queue<double, std::vector<double>, std::greater<double>> sm;
    for (int i = 0; i < num_sms; ++i) sm.push(0.0);
    double makespan = 0.0;
    auto deal = [&](double c) {
      const double t = sm.top() + c;
      sm.pop();
      sm.push(t);
      makespan = std::max(makespan, t);
    };
    if (S == 1) {
      // One split is the fused forward, which balances the items of all heads together (in
      // pairs, by its dispatch-order schedule, or longest first): deal them as one list. (Dealt
      // head by head, one split was estimated at 74 us on 1 x 4 x 8192 x 64 causal, which runs in
      // 48 us, and two splits, 62 us, were chosen.)
      for (double c : costs)
        for (long long h = 0; h < BH; ++h) deal(c);
    } else {
      for (long long h = 0; h < BH; ++h)  // heads interleave; each head's items longest-first
        for (double c : costs) deal(c);
    }
    double t = makespan;
    if (S > 1) t += 2.0 + (static_cast<double>(S) * rows * D * 4 + static_cast<double>(rows) * D * 2) / bytes_per_us;
    if (S == 1 || t < best_t) {
      best_t = t;
      best = S;
    }
  }
  return best;
}

// Work decomposition and item order of a forward (the Params fields BH, N, num_mb, num_splits,
// num_items, section). Two query tiles per item halve the K/V traffic per query row; when that
// leaves too few items to fill the GPU (short or few sequences), each item is a single query
// tile whose K/V range is split between the two softmax warpgroups instead. The split-KV
// partial form and the fp32 kernel always use single query tiles.
struct WorkPlan {
  bool splitk;       // single-query-tile items
  bool by_dispatch;  // causal with more than two waves of items: items follow dispatch order
  bool pair;         // causal single-query-tile items, one to two per SM: each CTA runs two at once
};
WorkPlan plan_work(Params& p, long long BH, int N, int D, bool causal, bool f32, int splits, int decomp, int num_sms) {
  const long long items_two = BH * ((static_cast<long long>(N) + item_rows(false) - 1) / item_rows(false));
  bool splitk = decomp == FA_DECOMP_SPLIT_KV || decomp == FA_DECOMP_SPLIT_KV_SERIAL || splits > 1 || f32;
  if (decomp == FA_DECOMP_AUTO && splits == 1 && !f32) {
    if (causal) {
      // Unequal item costs are balanced by dispatch order; split only when the GPU is not full.
      splitk = items_two < num_sms;
    } else {
      // Equal item costs: compare how well each item count fills whole waves of SMs. The
      // split-KV form pays a few percent for its extra K/V traffic and merge.
      auto wave_eff = [&](long long n) {
        const long long waves = (n + num_sms - 1) / num_sms;
        return static_cast<double>(n) / static_cast<double>(waves * num_sms);
      };
      splitk = wave_eff(2 * items_two) * 0.96 > wave_eff(items_two);
    }
  }
  p.BH = static_cast<int>(BH);
  p.N = N;
  p.num_mb = static_cast<int>((static_cast<long long>(N) + item_rows(splitk) - 1) / item_rows(splitk));
  p.num_splits = splits;
  p.num_items = static_cast<int>(BH * p.num_mb * splits);
  const long long kv_head_bytes = 2ll * N * D * (f32 ? 4 : 2);
  const long long section = kL2SectionBytes / (kv_head_bytes > 0 ? kv_head_bytes : 1);
  p.section = static_cast<int>(section < 1 ? 1 : (section > BH ? BH : section));
  // Pairs at D = 64 only: c2 13.25 -> 12.55 us. At D = 128 the paired form measured 2-3% slower
  // (warpgroup 1's store of b, in the middle of its chain, stalls the single MMA issuer).
  const bool pair = splitk && causal && D == 64 && splits == 1 && !f32 && decomp != FA_DECOMP_SPLIT_KV_SERIAL &&
                    p.num_items > num_sms && p.num_items <= 2 * num_sms;
  return WorkPlan{splitk, causal && p.num_items > 2 * num_sms && splits == 1, pair};
}

// Item lists for a persistent grid that follow the one-CTA-per-item dispatch: in item order
// (decode_item), each item goes to the CTA that frees up first under an estimated cost, the
// key tiles of its longer warpgroup chain plus a fixed per-item overhead (in tile units). The
// persistent CTA then prefetches the next item's Q and K/V during the current one, which the
// per-item launch cannot. The device copies live in a fixed pool of module memory (4 MB per
// device, a few KB per shape) for the process lifetime; shapes past its end launch one CTA per
// item (counted in g_schedule_fallbacks, reported by fa_schedule_pool_status).
//
// The first call of a shape copies its table with cudaMemcpyAsync on that call's stream (the
// host table stays alive in the entry, as the copy's source) and records an event after the
// copy. Until that event has been seen complete, every launch that uses the table first makes
// its own stream wait on the event, so a launch on another stream cannot read the table early.
// A launch under stream capture that would need such a wait runs without the table instead.
struct ScheduleKey {
  int dev, BH, N, causal, splitk, f32, section, num_mb, num_items, grid;
  bool operator<(const ScheduleKey& o) const { return std::memcmp(this, &o, sizeof(ScheduleKey)) < 0; }
};
struct ScheduleEntry {
  int* table = nullptr;          // device copy in the pool
  std::vector<int> host;         // source of the asynchronous copy, kept for the process lifetime
  cudaEvent_t copied = nullptr;  // recorded on the first caller's stream after the copy
  std::atomic<bool> done{false}; // the copy is known to be complete
};
std::mutex g_schedule_mutex;
std::map<ScheduleKey, ScheduleEntry> g_schedules;
std::atomic<unsigned long long> g_schedule_fallbacks{0};
constexpr double kScheduleItemOverhead = 1.0;
struct SchedulePool {
  int* base = nullptr;  // g_schedule_pool on this device
  size_t used = 0;      // ints handed out
};
SchedulePool g_schedule_pools[kMaxDevices];

std::vector<int> build_schedule(const Params& p, bool causal, bool splitk, bool f32, int grid) {
  const int n = p.num_items;
  using Slot = std::pair<double, int>;  // (estimated time the CTA frees up, CTA)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < grid; ++c) free_at.push({0.0, c});
  std::vector<std::vector<int>> lists(grid);
  for (int t = 0; t < n; ++t) {
    const Item it = causal ? decode_item<true>(t, p) : decode_item<false>(t, p);
    int nk = 0, n0 = 0, n1 = 0;
    if (f32) {
      if (causal) tile_counts_f32<true>(it.mb, p.N, nk, n0, n1);
      else tile_counts_f32<false>(it.mb, p.N, nk, n0, n1);
    } else if (splitk) {
      if (causal) tile_counts<true, true>(it.mb, p.N, nk, n0, n1);
      else tile_counts<false, true>(it.mb, p.N, nk, n0, n1);
    } else {
      if (causal) tile_counts<true, false>(it.mb, p.N, nk, n0, n1);
      else tile_counts<false, false>(it.mb, p.N, nk, n0, n1);
    }
    const Slot c = free_at.top();
    free_at.pop();
    lists[c.second].push_back(t);
    free_at.push({c.first + kScheduleItemOverhead + std::max(n0, n1), c.second});
  }
  std::vector<int> out(static_cast<size_t>(grid) + 1 + n);
  int off = 0;
  for (int c = 0; c < grid; ++c) {
    out[c] = off;
    for (int t : lists[c]) out[grid + 1 + off++] = t;
  }
  out[grid] = off;
  return out;
}

bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    return true;  // unknown: treat as capturing (no copies, no waits)
  }
  return cap != cudaStreamCaptureStatusNone;
}

// Makes `s` ordered after the copy of the entry's table. False when it cannot (the stream is
// being captured and the copy is not known to be complete, or a CUDA call failed): the caller
// then launches without the table.
bool schedule_ready(ScheduleEntry& e, cudaStream_t s) {
  if (e.done.load(std::memory_order_acquire)) return true;
  std::lock_guard<std::mutex> lock(g_schedule_mutex);
  if (e.done.load(std::memory_order_relaxed)) return true;
  if (stream_capturing(s)) return false;
  const cudaError_t q = cudaEventQuery(e.copied);
  if (q == cudaSuccess) {
    e.done.store(true, std::memory_order_release);
    return true;
  }
  if (q != cudaErrorNotReady) {
    cudaGetLastError();
    return false;
  }
  if (cudaStreamWaitEvent(s, e.copied, 0) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

// The schedule entry of this shape with its table copied (or being copied, in order before
// anything that follows on `s`) to the device; nullptr when there is none: the first call of
// the shape is under stream capture, the pool is full, or a CUDA call failed. The caller then
// launches one CTA per item.
ScheduleEntry* get_schedule(int dev, const Params& p, bool causal, bool splitk, bool f32, int grid, cudaStream_t s) {
  ScheduleKey key{};
  key.dev = dev;
  key.BH = p.BH;
  key.N = p.N;
  key.causal = causal;
  key.splitk = splitk;
  key.f32 = f32;
  key.section = p.section;
  key.num_mb = p.num_mb;
  key.num_items = p.num_items;
  key.grid = grid;
  ScheduleEntry* existing = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_schedule_mutex);
    auto found = g_schedules.find(key);
    if (found != g_schedules.end()) {
      existing = &found->second;  // map nodes are never erased once their copy is enqueued
    } else {
      if (dev < 0 || dev >= kMaxDevices || stream_capturing(s)) return nullptr;
      SchedulePool& pool = g_schedule_pools[dev];
      if (pool.base == nullptr &&
          cudaGetSymbolAddress(reinterpret_cast<void**>(&pool.base), g_schedule_pool) != cudaSuccess) {
        cudaGetLastError();
        pool.base = nullptr;
        return nullptr;
      }
      std::vector<int> host = build_schedule(p, causal, splitk, f32, grid);
      if (pool.used + host.size() > kSchedulePoolInts) return nullptr;
      cudaEvent_t ev = nullptr;
      if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
      }
      ScheduleEntry& e = g_schedules[key];
      e.host = std::move(host);
      e.table = pool.base + pool.used;
      e.copied = ev;
      if (cudaMemcpyAsync(e.table, e.host.data(), e.host.size() * sizeof(int), cudaMemcpyHostToDevice, s) !=
              cudaSuccess ||
          cudaEventRecord(ev, s) != cudaSuccess) {
        cudaGetLastError();
        cudaStreamSynchronize(s);  // whatever was enqueued has finished before the entry goes away
        cudaGetLastError();
        cudaEventDestroy(ev);
        g_schedules.erase(key);
        return nullptr;
      }
      pool.used += e.host.size();
      return &e;  // the copy is in order on `s` before the launch that follows
    }
  }
  return schedule_ready(*existing, s) ? existing : nullptr;
}

// Shared by fa_forward (splits = 1) and fa_forward_splitkv (splits >= 1 after the automatic
// choice). Validation first, then the per-thread launch cache, then descriptor encoding.
int forward_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
                 float scale, int causal, int dtype, int splits, void* workspace, size_t ws_bytes, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const bool f32 = dtype == FA_DTYPE_FP32;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16 && !f32) return FA_ERR_UNSUPPORTED;
  if (f32 && splits != 1) return FA_ERR_UNSUPPORTED;  // fp32 I/O: the fused forward only
  auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (mis16(q) || mis16(k) || mis16(v) || mis16(o)) return FA_ERR_ALIGN;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_ALIGN;

  const long long BH = static_cast<long long>(B) * H;
  const long long num_qt = (static_cast<long long>(N) + kBM - 1) / kBM;  // 128-row query tiles
  if (N > (1 << 30) || BH > 0x7fffffffll || BH * num_qt > 0x7fffffffll) return FA_ERR_TOO_LARGE;
  const size_t tensor_bytes = static_cast<size_t>(BH) * N * D * (f32 ? 4 : 2);
  const size_t lse_bytes = static_cast<size_t>(BH) * N * sizeof(float);
  if (overlaps(o, tensor_bytes, q, tensor_bytes) || overlaps(o, tensor_bytes, k, tensor_bytes) ||
      overlaps(o, tensor_bytes, v, tensor_bytes) || (lse && overlaps(o, tensor_bytes, lse, lse_bytes)))
    return FA_ERR_INVALID_ARG;
  // Split-KV workspace: present, aligned, large enough, disjoint from the other arguments.
  auto check_workspace = [&](int S) -> int {
    if (BH * num_qt * S > 0x7fffffffll) return FA_ERR_TOO_LARGE;
    const size_t need = workspace_bytes(BH, N, D, S);
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kWorkspaceAlign - 1)) != 0 ||
        ws_bytes < need)
      return FA_ERR_WORKSPACE;
    if (overlaps(workspace, need, q, tensor_bytes) || overlaps(workspace, need, k, tensor_bytes) ||
        overlaps(workspace, need, v, tensor_bytes) || overlaps(workspace, need, o, tensor_bytes) ||
        (lse && overlaps(workspace, need, lse, lse_bytes)))
      return FA_ERR_INVALID_ARG;
    return FA_OK;
  };
  int rc = FA_OK;
  if (splits > 1 && (rc = check_workspace(splits)) != FA_OK) return rc;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool bf16 = dtype == FA_DTYPE_BF16;
  const int decomp = g_decomposition.load(std::memory_order_relaxed);
  const unsigned long long timeout = g_timeout_ns.load(std::memory_order_relaxed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  LaunchKey key;
  std::memset(&key, 0, sizeof(key));
  key.ptr[0] = q;
  key.ptr[1] = k;
  key.ptr[2] = v;
  key.ptr[3] = o;
  key.ptr[4] = lse;
  key.ptr[5] = splits != 1 ? workspace : nullptr;
  key.B = B;
  key.H = H;
  key.N = N;
  key.D = D;
  key.causal = causal != 0;
  key.dtype = dtype;
  key.dev = dev;
  key.decomp = decomp;
  key.stall = g_force_stall.load(std::memory_order_relaxed);
  key.splits = splits;
  key.scale = scale;
  key.timeout = timeout;
  key.workspace_bytes = splits != 1 ? ws_bytes : 0;
  for (int i = 0; i < kCacheSize; ++i) {
    const LaunchEntry& c = t_cache[i];
    if (c.valid && c.key == key) {
      const Params* pp = &c.params;
      int grid = c.grid;
      Params p2;
      if (c.sched != nullptr && !schedule_ready(*c.sched, s)) {
        // The table's copy is not known to be complete and this stream cannot wait for it
        // (stream capture): one CTA per item, without the table.
        p2 = c.params;
        p2.schedule = nullptr;
        pp = &p2;
        grid = p2.num_items;
        g_schedule_fallbacks.fetch_add(1, std::memory_order_relaxed);
      }
      if (c.f32) {
        e = launch_forward_f32(*pp, grid, D, key.causal != 0, s);
      } else if (c.splits > 1) {
        e = launch_partial(*pp, grid, D, bf16, key.causal != 0, s);
        if (e == cudaSuccess)
          e = launch_merge(c.params.o_part, kPartsF32, c.params.lse_part, c.splits, c.rows, D, c.o, bf16, c.lse,
                           c.num_sms, s);
      } else {
        e = launch(*pp, grid, c.splitk, c.pair, D, bf16, key.causal != 0, s);
      }
      return e == cudaSuccess ? FA_OK : cuda_fail(e);
    }
  }

  DeviceInfo* info = nullptr;
  if ((rc = device_setup(dev, info)) != FA_OK) return rc;
  if (!(scale > 0.f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt(static_cast<float>(D));
  if (splits == 0) {
    splits = choose_splits(BH, N, D, causal != 0, info->num_sms);
    if (splits > 1 && (rc = check_workspace(splits)) != FA_OK) return rc;
  }

  Params p{};
  const WorkPlan plan = plan_work(p, BH, N, D, causal != 0, f32, splits, decomp, info->num_sms);
  const bool splitk = plan.splitk;
  const int kv_rows = f32 ? kBNf : kBN;
  if ((rc = encode_map(&p.tm_q, q, dtype, static_cast<int>(BH), N, D, kBM)) != FA_OK) return rc;
  if ((rc = encode_map(&p.tm_k, k, dtype, static_cast<int>(BH), N, D, kv_rows)) != FA_OK) return rc;
  if ((rc = encode_map(&p.tm_v, v, dtype, static_cast<int>(BH), N, D, kv_rows)) != FA_OK) return rc;
  if ((rc = encode_map(&p.tm_o, o, dtype, static_cast<int>(BH), N, D, 32)) != FA_OK) return rc;
  p.lse = lse;
  p.status = info->status_word;
  p.timeout_ns = timeout;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.force_stall = key.stall;
  if (splits > 1) {
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + workspace_o_bytes(BH, N, D, splits));
    if ((rc = encode_map_f32(&p.tm_op, workspace, BH * splits, N, D)) != FA_OK) return rc;
  }

  // Grid. Persistent (one CTA per SM, items strided in snake order) unless the items have
  // very unequal cost (causal) and there are several waves of them: then the static snake
  // balances badly (the L2 sections interleave long and short items), and each CTA takes the
  // item list that one-CTA-per-item dispatch would give it (get_schedule), or, without a
  // schedule, one CTA per item. Split-KV items are short and even: persistent. Paired
  // split-K launches also take one CTA per SM: CTA c runs items c and 2 grid - 1 - c.
  int grid = (plan.by_dispatch || p.num_items < info->num_sms) ? p.num_items : info->num_sms;
  p.schedule = nullptr;
  ScheduleEntry* sched = nullptr;
  if (plan.by_dispatch) {
    sched = get_schedule(dev, p, causal != 0, splitk, f32, info->num_sms, s);
    if (sched != nullptr) {
      p.schedule = sched->table;
      grid = info->num_sms;
    } else {
      g_schedule_fallbacks.fetch_add(1, std::memory_order_relaxed);
    }
  }

  LaunchEntry& slot = t_cache[t_cache_next];
  t_cache_next = (t_cache_next + 1) % kCacheSize;
  slot.key = key;
  slot.params = p;
  slot.grid = grid;
  slot.splitk = splitk;
  slot.pair = plan.pair;
  slot.f32 = f32;
  slot.splits = splits;
  slot.o = o;
  slot.lse = lse;
  slot.rows = BH * N;
  slot.num_sms = info->num_sms;
  slot.sched = sched;
  slot.valid = sched != nullptr || !plan.by_dispatch;  // a launch without its table is not cached
  if (f32) {
    e = launch_forward_f32(p, grid, D, causal != 0, s);
  } else if (splits > 1) {
    e = launch_partial(p, grid, D, bf16, causal != 0, s);
    if (e == cudaSuccess)
      e = launch_merge(p.o_part, kPartsF32, p.lse_part, splits, BH * N, D, o, bf16, lse, info->num_sms, s);
  } else {
    e = launch(p, grid, splitk, plan.pair, D, bf16, causal != 0, s);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_version(void) { return 100; }

const char* fa_error_string(int code) {
  switch (code) {
    case FA_OK: return "success";
    case FA_ERR_INVALID_ARG: return "invalid argument (null pointer, non-positive size, or aliasing output)";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration (D must be 64 or 128, dtype fp16/bf16, device sm_103)";
    case FA_ERR_ALIGN: return "misaligned pointer (Q/K/V/O need 16-byte alignment, LSE 4-byte)";
    case FA_ERR_CUDA: return "CUDA call failed (see fa_last_cuda_error)";
    case FA_ERR_TIMEOUT: return "device-side wait exceeded the watchdog limit";
    case FA_ERR_TOO_LARGE: return "sizes exceed the supported index range";
    case FA_ERR_WORKSPACE: return "split-KV workspace missing, not 256-byte aligned, or smaller than fa_splitkv_workspace_bytes";
    case FA_ERR_LIBRARY: return "naive baseline: cuBLAS could not be loaded or a GEMM failed (see fa_naive_last_library_error)";
    case FA_ERR_SCRATCH: return "split-KV partials exceed the built-in 32 MiB scratch of fa_forward_splitkv_noalloc (use fewer splits or fa_forward_splitkv)";
    default: return "unknown error code";
  }
}

int fa_last_cuda_error(void) { return fa::t_last_cuda_error; }

int fa_set_watchdog_ns(unsigned long long ns) {
  fa::g_timeout_ns.store(ns == 0 ? fa::kDefaultTimeoutNs : ns);
  return FA_OK;
}

int fa_set_decomposition(int mode) {
  if (mode != FA_DECOMP_AUTO && mode != FA_DECOMP_TWO_TILES && mode != FA_DECOMP_SPLIT_KV &&
      mode != FA_DECOMP_SPLIT_KV_SERIAL)
    return FA_ERR_INVALID_ARG;
  fa::g_decomposition.store(mode);
  return FA_OK;
}

int fa_debug_force_stall(int on) {
  fa::g_force_stall.store(on != 0 ? 1 : 0);
  return FA_OK;
}

int fa_debug_work_schedule(int B, int H, int N, int D, int causal, int dtype, int num_sms, int* out, int capacity) {
  if (B <= 0 || H <= 0 || N <= 0 || num_sms <= 0 || capacity < 0) return FA_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || dtype < FA_DTYPE_FP16 || dtype > FA_DTYPE_FP32) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((N + fa::kBM - 1) / fa::kBM) > (1ll << 30)) return FA_ERR_TOO_LARGE;
  fa::Params p{};
  const bool f32 = dtype == FA_DTYPE_FP32;
  const fa::WorkPlan plan = fa::plan_work(p, static_cast<long long>(B) * H, N, D, causal != 0, f32, 1,
                                          fa::g_decomposition.load(std::memory_order_relaxed), num_sms);
  if (!plan.by_dispatch) return 0;
  const std::vector<int> sched = fa::build_schedule(p, causal != 0, plan.splitk, f32, num_sms);
  const int len = static_cast<int>(sched.size());
  if (out == nullptr) return len;
  if (capacity < len) return FA_ERR_INVALID_ARG;
  std::memcpy(out, sched.data(), sched.size() * sizeof(int));
  return len;
}

int fa_debug_work_plan(int B, int H, int N, int D, int causal, int dtype, int num_sms, int* plan, int* units,
                       int capacity) {
  if (B <= 0 || H <= 0 || N <= 0 || num_sms <= 0 || capacity < 0 || plan == nullptr) return FA_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || dtype < FA_DTYPE_FP16 || dtype > FA_DTYPE_FP32) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((N + fa::kBM - 1) / fa::kBM) > (1ll << 30)) return FA_ERR_TOO_LARGE;
  fa::Params p{};
  const bool f32 = dtype == FA_DTYPE_FP32;
  const fa::WorkPlan wp = fa::plan_work(p, static_cast<long long>(B) * H, N, D, causal != 0, f32, 1,
                                        fa::g_decomposition.load(std::memory_order_relaxed), num_sms);
  const int grid = (wp.by_dispatch || p.num_items > num_sms) ? num_sms : p.num_items;
  plan[0] = p.num_items;
  plan[1] = wp.splitk ? 1 : 0;
  plan[2] = wp.pair ? 1 : 0;
  plan[3] = wp.by_dispatch ? 1 : 0;
  plan[4] = grid;
  if (!wp.pair) return 0;
  const int len = 6 * grid;
  if (units == nullptr) return len;
  if (capacity < len) return FA_ERR_INVALID_ARG;
  for (int c = 0; c < grid; ++c) {
    fa::Unit U{};
    int ta = -1, tb = -1;
    int* u = units + 6 * c;
    if (!fa::pair_unit<true>(c, grid, p, U, &ta, &tb)) {
      u[0] = u[1] = -1;
      u[2] = u[3] = u[4] = u[5] = 0;
      continue;
    }
    u[0] = ta;
    u[1] = tb;
    u[2] = U.nk - U.nb;
    u[3] = U.nb;
    u[4] = U.n0;
    u[5] = U.n1;
  }
  return len;
}

int fa_schedule_pool_status(size_t* used_bytes, size_t* capacity_bytes, unsigned long long* fallbacks) {
  if (fallbacks != nullptr) *fallbacks = fa::g_schedule_fallbacks.load(std::memory_order_relaxed);
  if (capacity_bytes != nullptr) *capacity_bytes = fa::kSchedulePoolInts * sizeof(int);
  if (used_bytes != nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fa::cuda_fail(e);
    std::lock_guard<std::mutex> lock(fa::g_schedule_mutex);
    *used_bytes = (dev >= 0 && dev < fa::kMaxDevices) ? fa::g_schedule_pools[dev].used * sizeof(int) : 0;
  }
  return FA_OK;
}

int fa_check_device_status(void) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fa::cuda_fail(e);
  fa::DeviceInfo* d = nullptr;
  int rc = fa::device_setup(dev, d);
  if (rc != FA_OK) return rc;
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fa::cuda_fail(e);
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, fa::g_device_status, sizeof(word));
  if (e != cudaSuccess) return fa::cuda_fail(e);
  if (word != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(fa::g_device_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return fa::cuda_fail(e);
  }
  return (word & fa::kStatusTimeout) ? FA_ERR_TIMEOUT : FA_OK;
}

int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
               float scale, int causal, int dtype, void* stream) {
  return fa::forward_impl(q, k, v, o, lse, B, H, N, D, scale, causal, dtype, 1, nullptr, 0, stream);
}

int fa_forward_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                       int D, float scale, int causal, int dtype, int num_splits, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (num_splits < 0 || num_splits > fa::kMaxSplits) return FA_ERR_INVALID_ARG;
  return fa::forward_impl(q, k, v, o, lse, B, H, N, D, scale, causal, dtype, num_splits, workspace, workspace_bytes,
                          stream);
}

size_t fa_splitkv_workspace_bytes(int B, int H, int N, int D, int num_splits) {
  if (B < 1 || H < 1 || N < 1 || (D != 64 && D != 128) || num_splits < 1 || num_splits > fa::kMaxSplits) return 0;
  if (num_splits == 1) return 0;
  return fa::workspace_bytes(static_cast<long long>(B) * H, N, D, num_splits);
}

int fa_debug_num_splits(int B, int H, int N, int D, int causal, int num_sms, int for_noalloc) {
  if (B < 1 || H < 1 || N < 1 || num_sms < 1) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  int splits = fa::choose_splits(BH, N, D, causal != 0, num_sms);
  if (for_noalloc)
    while (splits > 1 && fa::workspace_bytes(BH, N, D, splits) > fa::kNoAllocScratchBytes) --splits;
  return splits;
}

int fa_splitkv_num_splits(int B, int H, int N, int D, int causal) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fa::cuda_fail(e);
  fa::DeviceInfo* info = nullptr;
  const int rc = fa::device_setup(dev, info);
  if (rc != FA_OK) return rc;
  return fa::choose_splits(static_cast<long long>(B) * H, N, D, causal != 0, info->num_sms);
}

int fa_merge_partials(const void* o_parts, const float* lse_parts, int num_parts, int parts_dtype, void* o,
                      float* lse, int B, int H, int N, int D, int dtype, void* stream) {
  using namespace fa;
  if (o_parts == nullptr || lse_parts == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || num_parts < 1) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED;
  if (parts_dtype != FA_DTYPE_FP16 && parts_dtype != FA_DTYPE_BF16 && parts_dtype != FA_DTYPE_FP32)
    return FA_ERR_UNSUPPORTED;
  auto mis = [](const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0; };
  if (mis(o_parts, 16) || mis(o, 16) || mis(lse_parts, 4) || (lse != nullptr && mis(lse, 4))) return FA_ERR_ALIGN;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows > (1ll << 40) || static_cast<long long>(num_parts) * rows > (1ll << 46)) return FA_ERR_TOO_LARGE;
  const size_t elem = parts_dtype == FA_DTYPE_FP32 ? 4 : 2;
  const size_t parts_bytes = static_cast<size_t>(num_parts) * rows * D * elem;
  const size_t plse_bytes = static_cast<size_t>(num_parts) * rows * sizeof(float);
  const size_t o_bytes = static_cast<size_t>(rows) * D * 2, lse_bytes = static_cast<size_t>(rows) * sizeof(float);
  if (overlaps(o, o_bytes, o_parts, parts_bytes) || overlaps(o, o_bytes, lse_parts, plse_bytes) ||
      (lse && (overlaps(lse, lse_bytes, o_parts, parts_bytes) || overlaps(lse, lse_bytes, lse_parts, plse_bytes) ||
               overlaps(lse, lse_bytes, o, o_bytes))))
    return FA_ERR_INVALID_ARG;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceInfo* info = nullptr;
  const int rc = device_setup(dev, info);
  if (rc != FA_OK) return rc;
  const int kind = parts_dtype == FA_DTYPE_FP32 ? kPartsF32 : (parts_dtype == FA_DTYPE_BF16 ? kPartsBF16 : kPartsF16);
  e = launch_merge(o_parts, kind, lse_parts, num_parts, rows, D, o, dtype == FA_DTYPE_BF16, lse, info->num_sms,
                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_forward_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                               int N, int D, float scale, int causal, int dtype, int num_splits, void* stream) {
  using namespace fa;
  if (num_splits < 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || B < 1 || H < 1 || N < 1)
    return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (num_splits > 1 && workspace_bytes(BH, N, D, num_splits) > kNoAllocScratchBytes) return FA_ERR_SCRATCH;
  // The scratch address, once per device (with that device current).
  static std::atomic<void*> scratch[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  void* ptr = scratch[dev].load(std::memory_order_acquire);
  if (ptr == nullptr) {
    DeviceInfo* info = nullptr;
    const int rc = device_setup(dev, info);
    if (rc != FA_OK) return rc;
    std::lock_guard<std::mutex> lock(g_mutex);
    ptr = scratch[dev].load(std::memory_order_relaxed);
    if (ptr == nullptr) {
      e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e);
      scratch[dev].store(ptr, std::memory_order_release);
    }
  }
  int splits = num_splits;
  if (splits == 0) {
    // The cost model's choice, lowered to the largest count whose partials fit the scratch.
    splits = fa_splitkv_num_splits(B, H, N, D, causal);
    if (splits < 0) return splits;
    while (splits > 1 && workspace_bytes(BH, N, D, splits) > kNoAllocScratchBytes) --splits;
  }
  return forward_impl(q, k, v, o, lse, B, H, N, D, scale, causal, dtype, splits, ptr, kNoAllocScratchBytes, stream);
}

}  // extern "C"
