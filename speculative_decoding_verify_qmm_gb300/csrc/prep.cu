// Activation preparation for the verify matmul, and the vocab-head row-stat merge.
//
// The tensor-core path multiplies fp16 codes by fp16 activations.  A bf16 row
// converts to fp16 without loss once it is scaled by a power of two that puts
// its largest magnitude in [2^14, 2^15): the 8 significant bits of every bf16
// value fit in fp16's 11, and only values 2^-28 below the row maximum (whose
// products vanish against fp32 accumulation anyway) reach fp16's subnormals.
// The scale is undone once per output row in the epilogue.
#include "sv_internal.h"
#include "sv_ptx.cuh"

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

// Physical offset (within a 32-element block) of slot i of quad-thread t, matching
// the order in which the MMA fragments consume codes (see qmm_kernel.cuh).
template <int BITS>
__device__ __forceinline__ int phys_of_slot(int t, int i) {
  if (BITS == 8) return i < 4 ? 4 * t + i : 16 + 4 * t + (i - 4);
  // 4-bit: slots pair nibble j with nibble j + 4 of the thread's word
  const int perm = (i & 1) ? (i >> 1) + 4 : (i >> 1);
  return 8 * t + perm;
}

template <int BITS>
__global__ void __launch_bounds__(256) prep_kernel(const __nv_bfloat16* __restrict__ x, int ldx, int M, int MP, int K,
                                                   __half* __restrict__ xp, float* __restrict__ xsum,
                                                   float* __restrict__ rowscale) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool live = m < M;
  const __nv_bfloat16* row = x + (size_t)m * ldx;
  __shared__ float red[8];
  float mx = 0.f;
  if (live)
    for (int k = tid; k < K; k += 256) mx = fmaxf(mx, fabsf(__bfloat162float(row[k])));
  for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = red[0];
  for (int w = 1; w < 8; ++w) mx = fmaxf(mx, red[w]);
  int e = 0;
  if (mx > 0.f && mx <= 3.0e38f) {
    int E;
    frexpf(mx, &E);  // mx = f * 2^E, f in [0.5, 1)
    e = 15 - E;
    e = e > 100 ? 100 : (e < -100 ? -100 : e);
  }
  const float sc = ldexpf(1.f, e);
  for (int idx = tid; idx < K; idx += 256) {
    const int blk = idx >> 5, slot = idx & 31;
    float v = 0.f;
    if (live) v = __bfloat162float(row[blk * 32 + phys_of_slot<BITS>(slot >> 3, slot & 7)]) * sc;
    xp[((size_t)blk * MP + m) * 32 + slot] = __float2half_rn(v);
  }
  for (int g = warp; g < K / GROUP; g += 8) {
    float a = 0.f;
    if (live) a = __bfloat162float(row[g * GROUP + lane]) * sc + __bfloat162float(row[g * GROUP + 32 + lane]) * sc;
    for (int off = 16; off; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    if (lane == 0) xsum[(size_t)g * MP + m] = a;
  }
  if (tid == 0) rowscale[m] = live ? ldexpf(1.f, -e) : 0.f;
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

cudaError_t launch_prep(const __nv_bfloat16* x, int ldx, int M, int MP, int K, int bits, __half* xp, float* xsum,
                        float* rowscale, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(MP), dim3(256), 0, s, attr);
  if (bits == 8) return cudaLaunchKernelEx(&cfg, prep_kernel<8>, x, ldx, M, MP, K, xp, xsum, rowscale);
  return cudaLaunchKernelEx(&cfg, prep_kernel<4>, x, ldx, M, MP, K, xp, xsum, rowscale);
}

// One block per row: merge the per-tile (max, argmax, sumexp) triples in tile
// order.  Ties keep the lowest vocabulary index; sum-exp is rescaled to the
// global maximum and added in fp64 in a fixed tree order.
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
      acc += (double)se * exp(((double)v - (double)best) * (double)inv_temp);
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
