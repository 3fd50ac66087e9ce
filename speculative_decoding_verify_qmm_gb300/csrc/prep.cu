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
#include "sv_rowops.cuh"

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

// One block per (padded) row.  The row's activation values - x itself, its
// RMSNorm, or silu(g) * u - are rounded to bf16 exactly as the standalone glue
// kernels store them, scaled by 2^e and written as fp16 in the order the MMA
// fragments read them, together with the fp32 sum of each 64-wide group.
// Values are recomputed from global memory (L2) in each pass so the kernel
// needs almost no shared memory and fits beside a running matmul CTA.
template <int MODE>
__device__ __forceinline__ float prep_value(const PrepArgs& a, const __nv_bfloat16* row, int m, int k, float r) {
  float v = __bfloat162float(row[k]);
  if (MODE == PREP_RMSNORM) {
    v *= r;
    if (a.w) v *= __bfloat162float(a.w[k]);
    v = __bfloat162float(__float2bfloat16_rn(v));
  } else if (MODE == PREP_SWIGLU) {
    const float u = __bfloat162float(a.x2[(size_t)m * a.ldx2 + k]);
    v = __bfloat162float(__float2bfloat16_rn(v / (1.f + expf(-v)) * u));
  }
  return v;
}

template <int BITS, int MODE>
__global__ void __launch_bounds__(256) prep_kernel(PrepArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[256];
  const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  const bool live = m < a.M;
  const __nv_bfloat16* row = a.x + (size_t)(live ? m : 0) * a.ldx;
  float r = 1.f;
  if (MODE == PREP_RMSNORM && live) r = rms_scale_256(row, K, a.eps, red);
  float mx = 0.f;
  if (live)
    for (int k = tid; k < K; k += 256) mx = fmaxf(mx, fabsf(prep_value<MODE>(a, row, m, k, r)));
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
  // warp per group: lane l fills slot l of the group's two 32-element blocks
  const int phys = phys_of_slot<BITS>(lane >> 3, lane & 7);
  for (int g = warp; g < K / GROUP; g += 8) {
    float v0 = 0.f, v1 = 0.f;
    if (live) {
      v0 = prep_value<MODE>(a, row, m, g * GROUP + phys, r) * sc;
      v1 = prep_value<MODE>(a, row, m, g * GROUP + 32 + phys, r) * sc;
    }
    a.xp[((size_t)(2 * g) * a.MP + m) * 32 + lane] = __float2half_rn(v0);
    a.xp[((size_t)(2 * g + 1) * a.MP + m) * 32 + lane] = __float2half_rn(v1);
    float s = v0 + v1;
    for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) a.xsum[(size_t)g * a.MP + m] = s;
  }
  if (tid == 0) a.rowscale[m] = live ? ldexpf(1.f, -e) : 0.f;
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
  cudaLaunchConfig_t cfg = pdl_config(dim3(a.MP), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, prep_kernel<BITS, MODE>, a);
}

cudaError_t launch_prep(const PrepArgs& a, int bits, int mode, cudaStream_t s) {
  if (bits == 8) {
    if (mode == PREP_RMSNORM) return launch_prep_t<8, PREP_RMSNORM>(a, s);
    if (mode == PREP_SWIGLU) return launch_prep_t<8, PREP_SWIGLU>(a, s);
    return launch_prep_t<8, PREP_PLAIN>(a, s);
  }
  if (mode == PREP_RMSNORM) return launch_prep_t<4, PREP_RMSNORM>(a, s);
  if (mode == PREP_SWIGLU) return launch_prep_t<4, PREP_SWIGLU>(a, s);
  return launch_prep_t<4, PREP_PLAIN>(a, s);
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
