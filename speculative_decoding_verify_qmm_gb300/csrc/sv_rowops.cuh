// Row reductions shared by the fused activation preparation and the standalone
// RMSNorm kernel, so both produce identical bits.
#pragma once

#include <cuda_bf16.h>

namespace sv {

// Block-wide sum of per-thread fp32 partials in a fixed tree order (256 threads).
__device__ __forceinline__ float block_sum_256(float v, float* red) {
  const int tid = threadIdx.x;
  red[tid] = v;
  __syncthreads();
  for (int s = 128; s; s >>= 1) {
    if (tid < s) red[tid] += red[tid + s];
    __syncthreads();
  }
  const float r = red[0];
  __syncthreads();
  return r;
}

// 1 / sqrt(mean(x^2) + eps) of one bf16 row: per-thread fmaf over a 256 stride,
// then the fixed tree.
__device__ __forceinline__ float rms_scale_256(const __nv_bfloat16* row, int H, float eps, float* red) {
  float ss = 0.f;
  for (int k = threadIdx.x; k < H; k += 256) {
    const float v = __bfloat162float(row[k]);
    ss = fmaf(v, v, ss);
  }
  return 1.f / sqrtf(block_sum_256(ss, red) / (float)H + eps);
}

}  // namespace sv
