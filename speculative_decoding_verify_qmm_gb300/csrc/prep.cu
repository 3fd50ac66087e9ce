// Activation preparation for the verify matmul (the per-group arithmetic is
// prep_group in sv_prep.cuh), and the vocab-head row-stat merge.
#include "sv_internal.h"
#include "sv_ptx.cuh"
#include "sv_prep.cuh"

namespace sv {

__device__ unsigned int g_error_word = 0;

// Host access to the error word lives beside its definition.
cudaError_t read_and_clear_error_word(unsigned int* out) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
  *out = v;
  return e;
}

// One warp per (64-wide group, padded row); a block covers 8 groups of one row.
// Every step is local to the group, so the grid covers the whole block at once.
template <int BITS, int MODE>
__global__ void __launch_bounds__(256) prep_kernel(PrepArgs a) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.y;
  const int g = blockIdx.x * 8 + (threadIdx.x >> 5);
  const bool live = m < a.M;
  prep_group<BITS, MODE>(live ? a.x + (size_t)m * a.ldx : nullptr, live && a.x2 ? a.x2 + (size_t)m * a.ldx2 : nullptr,
                         a.w, a.eps, m, g, a.MP, a.K, a.out);
}

cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int BITS, int MODE>
static cudaError_t launch_prep_t(const PrepArgs& a, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(a.K / KC, a.MP), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, prep_kernel<BITS, MODE>, a);
}

cudaError_t launch_prep(const PrepArgs& a, int bits, int mode, cudaStream_t s) {
  if (bits == 8) {
    if (mode == PREP_RMSNORM) return launch_prep_t<8, PREP_RMSNORM>(a, s);
    if (mode == PREP_SWIGLU) return launch_prep_t<8, PREP_SWIGLU>(a, s);
    return launch_prep_t<8, PREP_PLAIN>(a, s);
  }
  if (bits == 2) {
    if (mode == PREP_RMSNORM) return launch_prep_t<2, PREP_RMSNORM>(a, s);
    if (mode == PREP_SWIGLU) return launch_prep_t<2, PREP_SWIGLU>(a, s);
    return launch_prep_t<2, PREP_PLAIN>(a, s);
  }
  if (mode == PREP_RMSNORM) return launch_prep_t<4, PREP_RMSNORM>(a, s);
  if (mode == PREP_SWIGLU) return launch_prep_t<4, PREP_SWIGLU>(a, s);
  return launch_prep_t<4, PREP_PLAIN>(a, s);
}

// One block per row: merge the per-slice (max, argmax, sumexp) triples of the
// 32-column slices in order.  Ties keep the lowest vocabulary index; each
// slice's sum-exp is rescaled to the global maximum (fp32 exp of a
// non-positive argument) and the terms are added in fp64 in a fixed order.
__global__ void __launch_bounds__(256) lmhead_finalize_kernel(const float* __restrict__ ts, int tiles, int MP,
                                                              float inv_temp, float* row_max, float* row_sumexp,
                                                              int32_t* row_argmax) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x, tid = threadIdx.x;
  __shared__ float sb[256];
  __shared__ int si[256];
  __shared__ double sd[256];
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int t = tid; t < tiles; t += 256) {
    const float v = ts[((size_t)t * MP + m) * 3];
    const int i = __float_as_int(ts[((size_t)t * MP + m) * 3 + 1]);
    if (v > best || (v == best && i < bi)) { best = v; bi = i; }
  }
  sb[tid] = best;
  si[tid] = bi;
  __syncthreads();
  for (int w = 128; w; w >>= 1) {
    if (tid < w) {
      const float ob = sb[tid + w];
      const int oi = si[tid + w];
      if (ob > sb[tid] || (ob == sb[tid] && oi < si[tid])) { sb[tid] = ob; si[tid] = oi; }
    }
    __syncthreads();
  }
  best = sb[0];
  bi = si[0];
  if (inv_temp > 0.f) {
    double acc = 0.0;
    for (int t = tid; t < tiles; t += 256) {
      const float v = ts[((size_t)t * MP + m) * 3];
      const float se = ts[((size_t)t * MP + m) * 3 + 2];
      acc += (double)(se * exp_term((v - best) * inv_temp));
    }
    sd[tid] = acc;
    __syncthreads();
    for (int w = 128; w; w >>= 1) {
      if (tid < w) sd[tid] += sd[tid + w];
      __syncthreads();
    }
  }
  if (tid == 0) {
    if (row_max) row_max[m] = best;
    if (row_argmax) row_argmax[m] = bi;
    if (row_sumexp && inv_temp > 0.f) row_sumexp[m] = (float)sd[0];
  }
}

cudaError_t launch_lmhead_finalize(const float* tile_stats, int tiles_n, int MP, int M, float inv_temp,
                                   float* row_max, float* row_sumexp, int32_t* row_argmax, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(M), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, lmhead_finalize_kernel, tile_stats, tiles_n, MP, inv_temp, row_max, row_sumexp,
                            row_argmax);
}

}  // namespace sv
