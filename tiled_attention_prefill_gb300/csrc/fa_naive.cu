// Naive (unfused) attention forward: the score matrix written out in full, as a baseline for
// the fused kernel. It is the three-step form that "Android Transformer Optimization:
// Attention and Mobile GPU Bottlenecks" (section "The Self-Attention Bottleneck Is Memory
// Traffic, Not Compute") describes and that "Flash Attention on Android: tiled SGEMM with
// RenderScript" (section "Architecture: tiled attention with RenderScript BLAS") runs through
// a BLAS with the scale as the SGEMM alpha:
//
//   1. S = scale * Q K^T       batched library GEMM (cuBLAS), S stored as fp16 [BH, N, N]
//   2. P = softmax(S) row-wise  this file's kernel: causal mask, lse, P written over S
//   3. O = P V                  batched library GEMM, O fp16
//
// Every step reads or writes the N x N matrix in memory; that traffic is what the fused
// kernel removes. cuBLAS is loaded with dlopen on first use, so the library itself has no
// link-time dependency on it.
#include <cublas_v2.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <dlfcn.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <string>

#include "fa.h"

namespace fa {
namespace {

constexpr int kSoftmaxThreads = 256;
constexpr int kMaxDevices = 64;
constexpr float kLog2e = 1.4426950408889634f;
thread_local int t_naive_error = 0;

// ----------------------------------------------------------------------------- softmax
// One warp per score row (bh, i). Pass 1: per lane a running (max, sum) over its columns
// j in J(i), rescaled when the max grows, then combined across the warp. Pass 2: P = e^(s -
// m) / l over the row (0 for masked columns), written over S. lse = m + ln l.
__device__ __forceinline__ void ml_combine(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  l = l * exp2f((m - mn) * kLog2e) + l2 * exp2f((m2 - mn) * kLog2e);
  m = mn;
}

template <bool CAUSAL, bool VEC>
__global__ void __launch_bounds__(kSoftmaxThreads) fa_naive_softmax_kernel(__half* __restrict__ sp,
                                                                           float* __restrict__ lse, long long rows,
                                                                           int N) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kSoftmaxThreads / 32);
  for (long long r = static_cast<long long>(blockIdx.x) * (kSoftmaxThreads / 32) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const int i = static_cast<int>(r % N);
    const int nv = CAUSAL ? i + 1 : N;  // |J(i)|
    __half* row = sp + r * N;
    float m = -INFINITY, l = 0.f;
    if (VEC) {
      for (int c = lane * 8; c < nv; c += 256) {
        const uint4 u = *reinterpret_cast<const uint4*>(row + c);
        const __half* h = reinterpret_cast<const __half*>(&u);
        float x[8];
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          x[e] = c + e < nv ? __half2float(h[e]) : -INFINITY;
          mx = fmaxf(mx, x[e]);
        }
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) s += exp2f((x[e] - mx) * kLog2e);
        ml_combine(m, l, mx, s);
      }
    } else {
      for (int c = lane; c < nv; c += 32) ml_combine(m, l, __half2float(row[c]), 1.f);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
      ml_combine(m, l, m2, l2);
    }
    const float inv_l = 1.0f / l;
    if (VEC) {
      for (int c = lane * 8; c < N; c += 256) {
        uint4 u = *reinterpret_cast<const uint4*>(row + c);
        __half* h = reinterpret_cast<__half*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          h[e] = __float2half_rn(c + e < nv ? exp2f((__half2float(h[e]) - m) * kLog2e) * inv_l : 0.f);
        *reinterpret_cast<uint4*>(row + c) = u;
      }
    } else {
      for (int c = lane; c < N; c += 32)
        row[c] = __float2half_rn(c < nv ? exp2f((__half2float(row[c]) - m) * kLog2e) * inv_l : 0.f);
    }
    if (lse != nullptr && lane == 0) lse[r] = m + logf(l);
  }
}

// ----------------------------------------------------------------------------- cuBLAS
using CreateFn = cublasStatus_t (*)(cublasHandle_t*);
using SetStreamFn = cublasStatus_t (*)(cublasHandle_t, cudaStream_t);
using GemmFn = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int, const void*,
                                  const void*, cudaDataType, int, long long, const void*, cudaDataType, int, long long,
                                  const void*, void*, cudaDataType, int, long long, int, cublasComputeType_t,
                                  cublasGemmAlgo_t);
struct Blas {
  CreateFn create = nullptr;
  SetStreamFn set_stream = nullptr;
  GemmFn gemm = nullptr;
  bool ok = false;
};
std::once_flag g_blas_once;
Blas g_blas;

void load_blas() {
  const char* names[] = {"libcublas.so.13", "/usr/local/cuda/lib64/libcublas.so.13", "libcublas.so"};
  void* h = nullptr;
  for (const char* n : names)
    if ((h = dlopen(n, RTLD_NOW | RTLD_LOCAL)) != nullptr) break;
  if (h == nullptr) return;
  g_blas.create = reinterpret_cast<CreateFn>(dlsym(h, "cublasCreate_v2"));
  g_blas.set_stream = reinterpret_cast<SetStreamFn>(dlsym(h, "cublasSetStream_v2"));
  g_blas.gemm = reinterpret_cast<GemmFn>(dlsym(h, "cublasGemmStridedBatchedEx"));
  g_blas.ok = g_blas.create && g_blas.set_stream && g_blas.gemm;
}

// One cuBLAS handle per host thread and device (a handle must not be shared by threads).
thread_local cublasHandle_t t_handles[kMaxDevices];

int blas_handle(int dev, cublasHandle_t& h) {
  std::call_once(g_blas_once, load_blas);
  if (!g_blas.ok) return FA_ERR_LIBRARY;
  if (t_handles[dev] == nullptr) {
    cublasHandle_t nh = nullptr;
    const cublasStatus_t st = g_blas.create(&nh);
    if (st != CUBLAS_STATUS_SUCCESS) {
      t_naive_error = static_cast<int>(st);
      return FA_ERR_LIBRARY;
    }
    t_handles[dev] = nh;
  }
  h = t_handles[dev];
  return FA_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace fa

extern "C" {

size_t fa_naive_workspace_bytes(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  const size_t b = static_cast<size_t>(B) * H * static_cast<size_t>(N) * N * 2;
  return (b + 255) / 256 * 256;
}

int fa_naive_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
                     float scale, int causal, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  using namespace fa;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || B < 1 || H < 1 || N < 1)
    return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_DTYPE_FP16) return FA_ERR_UNSUPPORTED;
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(q, 16) || mis(k, 16) || mis(v, 16) || mis(o, 16) || (lse != nullptr && mis(lse, 4))) return FA_ERR_ALIGN;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffll || N > (1 << 30)) return FA_ERR_TOO_LARGE;
  const size_t need = fa_naive_workspace_bytes(B, H, N);
  if (workspace == nullptr || mis(workspace, 256) || workspace_bytes < need) return FA_ERR_WORKSPACE;
  const size_t tb = static_cast<size_t>(BH) * N * D * 2, lb = static_cast<size_t>(BH) * N * 4;
  if (overlaps(o, tb, q, tb) || overlaps(o, tb, k, tb) || overlaps(o, tb, v, tb) || overlaps(workspace, need, q, tb) ||
      overlaps(workspace, need, k, tb) || overlaps(workspace, need, v, tb) || overlaps(workspace, need, o, tb) ||
      (lse && (overlaps(lse, lb, o, tb) || overlaps(lse, lb, workspace, need))))
    return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt(static_cast<float>(D));

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  int num_sms = 0;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FA_ERR_CUDA;
  cublasHandle_t h = nullptr;
  int rc = blas_handle(dev, h);
  if (rc != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (g_blas.set_stream(h, s) != CUBLAS_STATUS_SUCCESS) return FA_ERR_LIBRARY;
  __half* sp = static_cast<__half*>(workspace);
  const long long nd = static_cast<long long>(N) * D, nn = static_cast<long long>(N) * N;

  // 1. S (row-major N x N) = scale Q K^T: column-major S^T = K Q^T, i.e. op(A) = K with A the
  //    column-major D x N view of K's memory, B the D x N view of Q's.
  const float alpha = scale, beta = 0.f, one = 1.f;
  cublasStatus_t st = g_blas.gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, N, N, D, &alpha, k, CUDA_R_16F, D, nd, q, CUDA_R_16F, D,
                                  nd, &beta, sp, CUDA_R_16F, N, nn, static_cast<int>(BH), CUBLAS_COMPUTE_32F,
                                  CUBLAS_GEMM_DEFAULT);
  if (st != CUBLAS_STATUS_SUCCESS) {
    t_naive_error = static_cast<int>(st);
    return FA_ERR_LIBRARY;
  }
  // 2. softmax over each row, in place.
  const long long rows = BH * N;
  long long blocks = (rows + kSoftmaxThreads / 32 - 1) / (kSoftmaxThreads / 32);
  if (blocks > static_cast<long long>(num_sms) * 64) blocks = static_cast<long long>(num_sms) * 64;
  const bool vec = (N % 8) == 0;
  const dim3 grid(static_cast<unsigned>(blocks)), block(kSoftmaxThreads);
  if (causal) {
    if (vec) fa_naive_softmax_kernel<true, true><<<grid, block, 0, s>>>(sp, lse, rows, N);
    else fa_naive_softmax_kernel<true, false><<<grid, block, 0, s>>>(sp, lse, rows, N);
  } else {
    if (vec) fa_naive_softmax_kernel<false, true><<<grid, block, 0, s>>>(sp, lse, rows, N);
    else fa_naive_softmax_kernel<false, false><<<grid, block, 0, s>>>(sp, lse, rows, N);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return FA_ERR_CUDA;
  // 3. O (row-major N x D) = P V: column-major O^T = V^T P^T, A = the D x N view of V, B = the
  //    N x N view of P (that is P^T).
  st = g_blas.gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, D, N, N, &one, v, CUDA_R_16F, D, nd, sp, CUDA_R_16F, N, nn, &beta, o,
                   CUDA_R_16F, D, nd, static_cast<int>(BH), CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  if (st != CUBLAS_STATUS_SUCCESS) {
    t_naive_error = static_cast<int>(st);
    return FA_ERR_LIBRARY;
  }
  return FA_OK;
}

int fa_naive_last_library_error(void) { return fa::t_naive_error; }

}  // extern "C"
