// Kernel launcher template, explicitly instantiated in fa_inst_d64.cu, fa_inst_d128.cu,
// fa_inst_partial.cu and fa_inst_pair.cu so that the kernel variants compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "fa_kernel.cuh"

namespace fa {

template <int D, bool BF16, bool CAUSAL, bool SPLITK, bool PARTIAL = false, bool PAIR = false>
cudaError_t launch_forward(const Params& p, int grid, cudaStream_t stream) {
  using L = KernelLayout<D, SPLITK, PAIR>;
  auto kernel = fa_fwd_kernel<D, BF16, CAUSAL, SPLITK, PARTIAL, PAIR>;
  // Opt in to the large dynamic shared-memory carve-out once per device.
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    // The kernel redistributes its launch registers with setmaxnreg; a smaller launch
    // allocation than the split assumes would make setmaxnreg.inc wait forever, so refuse.
    cudaFuncAttributes attr{};
    e = cudaFuncGetAttributes(&attr, kernel);
    if (e != cudaSuccess) return e;
    if (reg_split<D>() && attr.numRegs * kNumThreads < 128 * (kOtherRegs + 2 * kSoftmaxRegs))
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamicBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  // Programmatic dependent launch: the kernel may start (barrier init, TMEM allocation,
  // descriptor prefetch) while the previous kernel on the stream finishes; it waits for that
  // kernel (griddepcontrol.wait) before touching global memory.
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

// fp32-I/O (tf32) kernel: fa_inst_f32.cu.
cudaError_t launch_forward_f32(const Params& p, int grid, int D, bool causal, cudaStream_t stream);

#define FA_DECLARE_LAUNCH(EXT, D, BF16, CAUSAL)                                                              \
  EXT template cudaError_t launch_forward<D, BF16, CAUSAL, false, false>(const Params&, int, cudaStream_t); \
  EXT template cudaError_t launch_forward<D, BF16, CAUSAL, true, false>(const Params&, int, cudaStream_t);
#define FA_DECLARE_LAUNCH_PARTIAL(EXT, D, BF16, CAUSAL) \
  EXT template cudaError_t launch_forward<D, BF16, CAUSAL, true, true>(const Params&, int, cudaStream_t);
#define FA_DECLARE_LAUNCH_PAIR(EXT, D, BF16, CAUSAL) \
  EXT template cudaError_t launch_forward<D, BF16, CAUSAL, true, false, true>(const Params&, int, cudaStream_t);

}  // namespace fa
