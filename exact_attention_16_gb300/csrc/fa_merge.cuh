// Internal: merge fp32 partial outputs (split-KV workspace) into the final O.
#pragma once

#include <cuda_runtime.h>

namespace fa {
// o_parts (n, B, Sq, Hq, D) fp32, lse_parts (n, B, Hq, Sq) fp32 -> o (B, Sq,
// Hq, D) of `dtype` (fa_dtype_t) and lse (B, Hq, Sq) fp32 or null. Launched
// as a programmatic dependent of the split-KV kernel just enqueued on
// `stream`, which wrote the parts.
int merge_f32_parts(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int B, int Sq,
                    int Hq, int D, int dtype, cudaStream_t stream);
}  // namespace fa
