// Launcher of the partial-result merge kernel (fa_merge.cu).
#pragma once

#include <cuda_runtime.h>

namespace fa {

// Element type of the partial outputs.
constexpr int kPartsF16 = 0;
constexpr int kPartsBF16 = 1;
constexpr int kPartsF32 = 2;

// Merges num_parts partial results: o_parts [num_parts, rows, D] (parts_kind), lse_parts
// [num_parts, rows] fp32 -> o [rows, D] (fp16, or bf16 when out_bf16), lse [rows] fp32 (may
// be null). D is 64 or 128; all pointers 16-byte aligned (lse 4-byte). Launched with
// programmatic stream serialization: it waits for the previous kernel's writes first.
cudaError_t launch_merge(const void* o_parts, int parts_kind, const float* lse_parts, int num_parts, long long rows,
                         int D, void* o, bool out_bf16, float* lse, int num_sms, cudaStream_t stream);

}  // namespace fa
