// Merge of partial attention results over disjoint key ranges (split-KV).
//
// A partial result of query row i over a key set K_s is (O_s, lse_s): O_s normalised over K_s
// and lse_s = ln sum_{j in K_s} exp(s_ij). The parts are combined with the online-softmax
// update of "Android Transformer Optimization: Attention and Mobile GPU Bottlenecks", section
// "The Essence of FlashAttention: Reordering the Computation", taking each part as one block
// whose running max is lse_s and whose denominator relative to it is 1:
//   m' = max(m, lse_s), l = l e^(m - m') + e^(lse_s - m'), acc = acc e^(m - m') + e^(lse_s - m') O_s
// then O = acc / l and lse = m + ln l. Parts with lse_s = -inf hold no key and are skipped
// (their O is never read into the sum); a row without any key gets O = 0, lse = -inf.
//
// Memory-bound: every part is read once (D/4 threads per row, 16-byte loads of fp32 parts,
// 8-byte loads of 16-bit parts, consecutive threads on consecutive columns).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_merge.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kMergeThreads = 256;
// Parts whose loads are in flight together. Two (not four) keeps the kernel at 40 registers,
// so six 256-thread blocks fit on an SM: more rows in flight per SM. lc1 with 2 splits: the
// split-KV forward 60.8 -> 59.4 us.
constexpr int kGroup = 2;

struct F4 {
  float x, y, z, w;
};

template <typename T>
__device__ __forceinline__ F4 load4(const T* p);
template <>
__device__ __forceinline__ F4 load4<float>(const float* p) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  return {v.x, v.y, v.z, v.w};
}
template <>
__device__ __forceinline__ F4 load4<__half>(const __half* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return {a.x, a.y, b.x, b.y};
}
template <>
__device__ __forceinline__ F4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return {a.x, a.y, b.x, b.y};
}

template <bool BF16>
__device__ __forceinline__ void store4(void* p, const F4& v) {
  uint2 u;
  u.x = pack2<BF16>(v.x, v.y);
  u.y = pack2<BF16>(v.z, v.w);
  *reinterpret_cast<uint2*>(p) = u;
}

template <int D, typename TP, bool OUT_BF16>
__global__ void __launch_bounds__(kMergeThreads, 6) fa_merge_kernel(const TP* __restrict__ o_parts,
                                                                  const float* __restrict__ lse_parts,
                                                                  int num_parts, long long rows,
                                                                  void* __restrict__ o, float* __restrict__ lse) {
  constexpr int kThreadsPerRow = D / 4;
  constexpr int kRowsPerBlock = kMergeThreads / kThreadsPerRow;
  // The parts are written by the previous kernel on the stream (programmatic launch).
  grid_dependency_wait();
  const int sub = threadIdx.x % kThreadsPerRow;
  const long long step = static_cast<long long>(gridDim.x) * kRowsPerBlock;
  for (long long row = static_cast<long long>(blockIdx.x) * kRowsPerBlock + threadIdx.x / kThreadsPerRow;
       row < rows; row += step) {
    float m = -INFINITY, l = 0.f;
    F4 acc{0.f, 0.f, 0.f, 0.f};
    // Parts in groups of kGroup: the lse and O loads of a group are all issued before any of
    // them is used (the O addresses do not depend on lse), so one memory round trip covers the
    // group. A part whose lse is -inf is skipped below, whatever its O holds.
    for (int s0 = 0; s0 < num_parts; s0 += kGroup) {
      float ms[kGroup];
      F4 v[kGroup];
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const bool in = s0 + u < num_parts;
        ms[u] = in ? __ldg(lse_parts + static_cast<long long>(s0 + u) * rows + row) : -INFINITY;
        v[u] = in ? load4<TP>(o_parts + (static_cast<long long>(s0 + u) * rows + row) * D + 4 * sub) : F4{0.f, 0.f, 0.f, 0.f};
      }
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const float m_s = ms[u];
        if (!(m_s > -INFINITY)) continue;  // no key in this part
        const float m_new = fmaxf(m, m_s);
        const float alpha = expf(m - m_new);  // 0 for the first part (m = -inf)
        const float beta = expf(m_s - m_new);
        l = l * alpha + beta;
        acc.x = acc.x * alpha + beta * v[u].x;
        acc.y = acc.y * alpha + beta * v[u].y;
        acc.z = acc.z * alpha + beta * v[u].z;
        acc.w = acc.w * alpha + beta * v[u].w;
        m = m_new;
      }
    }
    F4 out{0.f, 0.f, 0.f, 0.f};
    float lse_out = -INFINITY;
    if (l > 0.f) {
      const float inv = 1.0f / l;
      out = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
      lse_out = m + logf(l);
    }
    store4<OUT_BF16>(static_cast<uint16_t*>(o) + row * D + 4 * sub, out);
    if (lse != nullptr && sub == 0) lse[row] = lse_out;
  }
  grid_launch_dependents();
}

template <int D, typename TP, bool OUT_BF16>
cudaError_t launch_merge_t(const void* o_parts, const float* lse_parts, int num_parts, long long rows, void* o,
                           float* lse, int num_sms, cudaStream_t stream) {
  constexpr int kRowsPerBlock = kMergeThreads / (D / 4);
  long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const long long cap = static_cast<long long>(num_sms) * 32;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, fa_merge_kernel<D, TP, OUT_BF16>, static_cast<const TP*>(o_parts),
                                     lse_parts, num_parts, rows, o, lse);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_merge_d(const void* o_parts, int parts_kind, const float* lse_parts, int num_parts,
                           long long rows, void* o, bool out_bf16, float* lse, int num_sms, cudaStream_t s) {
  if (parts_kind == kPartsF32)
    return out_bf16 ? launch_merge_t<D, float, true>(o_parts, lse_parts, num_parts, rows, o, lse, num_sms, s)
                    : launch_merge_t<D, float, false>(o_parts, lse_parts, num_parts, rows, o, lse, num_sms, s);
  if (parts_kind == kPartsBF16)
    return out_bf16 ? launch_merge_t<D, __nv_bfloat16, true>(o_parts, lse_parts, num_parts, rows, o, lse, num_sms, s)
                    : launch_merge_t<D, __nv_bfloat16, false>(o_parts, lse_parts, num_parts, rows, o, lse, num_sms, s);
  return out_bf16 ? launch_merge_t<D, __half, true>(o_parts, lse_parts, num_parts, rows, o, lse, num_sms, s)
                  : launch_merge_t<D, __half, false>(o_parts, lse_parts, num_parts, rows, o, lse, num_sms, s);
}

}  // namespace

cudaError_t launch_merge(const void* o_parts, int parts_kind, const float* lse_parts, int num_parts, long long rows,
                         int D, void* o, bool out_bf16, float* lse, int num_sms, cudaStream_t stream) {
  if (D == 64) return launch_merge_d<64>(o_parts, parts_kind, lse_parts, num_parts, rows, o, out_bf16, lse, num_sms, stream);
  return launch_merge_d<128>(o_parts, parts_kind, lse_parts, num_parts, rows, o, out_bf16, lse, num_sms, stream);
}

}  // namespace fa
