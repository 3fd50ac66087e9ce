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
// 64-column tiles.  Ties keep the lowest vocabulary index; each tile's sum-exp
// is rescaled to the global maximum (fp32 exp of a non-positive argument) and
// the terms are added in fp64 in a fixed order (each thread its tiles in
// order, then the lanes of a warp by a shuffle tree, then the warps in order).
// A thread loads its tiles FIN_PT at a time, together (each load is an L2
// round trip), and a row of at most FIN_PT * FIN_THREADS tiles stays in
// registers for both passes.
constexpr int FIN_THREADS = 256, FIN_PT = 16, FIN_CHUNK = FIN_PT * FIN_THREADS;
__global__ void __launch_bounds__(FIN_THREADS) lmhead_finalize_kernel(const float* __restrict__ ts, int tiles, int MP,
                                                                      float inv_temp, float* row_max,
                                                                      float* row_sumexp, int32_t* row_argmax) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  __shared__ float s_best[FIN_THREADS / 32];
  __shared__ int s_idx[FIN_THREADS / 32];
  __shared__ double s_sum[FIN_THREADS / 32];
  __shared__ float s_row_best;
  float v[FIN_PT], se[FIN_PT];
  auto load = [&](int base) {  // tiles base + tid + k * FIN_THREADS; returns their lowest-index maximum
    float b = -INFINITY;
    int bi = 0x7fffffff;
    int ix[FIN_PT];
#pragma unroll
    for (int k = 0; k < FIN_PT; ++k) {
      const int t = base + tid + k * FIN_THREADS;
      v[k] = -INFINITY;
      se[k] = 0.f;
      ix[k] = 0x7fffffff;
      if (t < tiles) {
        const float* e = ts + ((size_t)t * MP + m) * 3;
        v[k] = e[0];
        ix[k] = __float_as_int(e[1]);
        se[k] = e[2];
      }
    }
#pragma unroll
    for (int k = 0; k < FIN_PT; ++k)
      if (v[k] > b || (v[k] == b && ix[k] < bi)) { b = v[k]; bi = ix[k]; }
    return make_float2(b, __int_as_float(bi));
  };
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int base = 0; base < tiles; base += FIN_CHUNK) {
    const float2 r = load(base);
    const int ri = __float_as_int(r.y);
    if (r.x > best || (r.x == best && ri < bi)) { best = r.x; bi = ri; }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
  }
  if (lane == 0) {
    s_best[wid] = best;
    s_idx[wid] = bi;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < FIN_THREADS / 32; ++w)
      if (s_best[w] > best || (s_best[w] == best && s_idx[w] < bi)) { best = s_best[w]; bi = s_idx[w]; }
    s_row_best = best;
    if (row_max) row_max[m] = best;
    if (row_argmax) row_argmax[m] = bi;
  }
  __syncthreads();
  if (!(inv_temp > 0.f)) return;
  best = s_row_best;
  double acc = 0.0;
  for (int base = 0; base < tiles; base += FIN_CHUNK) {
    if (tiles > FIN_CHUNK) load(base);  // a single chunk is still in registers
#pragma unroll
    for (int k = 0; k < FIN_PT; ++k)
      if (base + tid + k * FIN_THREADS < tiles) acc += (double)(se[k] * exp_term((v[k] - best) * inv_temp));
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) s_sum[wid] = acc;
  __syncthreads();
  if (tid == 0) {
    double tot = 0.0;
    for (int w = 0; w < FIN_THREADS / 32; ++w) tot += s_sum[w];
    if (row_sumexp) row_sumexp[m] = (float)tot;
  }
}

cudaError_t launch_lmhead_finalize(const float* tile_stats, int tiles_n, int MP, int M, float inv_temp,
                                   float* row_max, float* row_sumexp, int32_t* row_argmax, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(M), dim3(FIN_THREADS), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, lmhead_finalize_kernel, tile_stats, tiles_n, MP, inv_temp, row_max, row_sumexp,
                            row_argmax);
}

}  // namespace sv
