// Kernel instances and launcher of the fp32-I/O (tf32) forward.
#include <cuda_runtime.h>

#include <atomic>

#include "fa_kernel_f32.cuh"
#include "fa_launch.cuh"

namespace fa {

template <int D, bool CAUSAL>
cudaError_t launch_forward_f32_t(const Params& p, int grid, cudaStream_t stream) {
  using L = SmemLayoutF32<D>;
  auto kernel = fa_fwd_f32_kernel<D, CAUSAL>;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamicBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kNumThreads);
  cfg.dynamicSmemBytes = L::kDynamicBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_forward_f32(const Params& p, int grid, int D, bool causal, cudaStream_t stream) {
  if (D == 64) return causal ? launch_forward_f32_t<64, true>(p, grid, stream) : launch_forward_f32_t<64, false>(p, grid, stream);
  return causal ? launch_forward_f32_t<128, true>(p, grid, stream) : launch_forward_f32_t<128, false>(p, grid, stream);
}

}  // namespace fa
