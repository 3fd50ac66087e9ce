// Row-wise glue between the verify projections: RMSNorm, residual add, SwiGLU.
// fp32 arithmetic, one rounding to bf16 per output.
#include <cuda_bf16.h>

#include "sv_kernels.h"
#include "sv_ptx.cuh"
#include "sv_rowops.cuh"

namespace sv {

__global__ void __launch_bounds__(256) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, int ldx, int H,
                                                      const __nv_bfloat16* __restrict__ w, float eps,
                                                      __nv_bfloat16* __restrict__ y, int ldy) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x, tid = threadIdx.x;
  const __nv_bfloat16* row = x + (size_t)m * ldx;
  __shared__ float red[256];
  const float r = rms_scale_256(row, H, eps, red);
  for (int k = tid; k < H; k += 256) {
    float v = __bfloat162float(row[k]) * r;
    if (w) v *= __bfloat162float(w[k]);
    y[(size_t)m * ldy + k] = __float2bfloat16_rn(v);
  }
}

__global__ void __launch_bounds__(256) residual_kernel(__nv_bfloat16* h, int ldh, const __nv_bfloat16* t, int ldt,
                                                       int H) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.y;
  for (int k = blockIdx.x * 256 + threadIdx.x; k < H; k += gridDim.x * 256) {
    const size_t i = (size_t)m * ldh + k;
    h[i] = __float2bfloat16_rn(__bfloat162float(h[i]) + __bfloat162float(t[(size_t)m * ldt + k]));
  }
}

__global__ void __launch_bounds__(256) swiglu_kernel(const __nv_bfloat16* g, int ldg, const __nv_bfloat16* u, int ldu,
                                                     int I, __nv_bfloat16* out, int lds) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.y;
  for (int k = blockIdx.x * 256 + threadIdx.x; k < I; k += gridDim.x * 256) {
    const float gv = __bfloat162float(g[(size_t)m * ldg + k]);
    const float uv = __bfloat162float(u[(size_t)m * ldu + k]);
    out[(size_t)m * lds + k] = __float2bfloat16_rn(silu_f32(gv) * uv);
  }
}

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, int ldx, int M, int H, const __nv_bfloat16* w, float eps,
                           __nv_bfloat16* y, int ldy, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(M), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, x, ldx, H, w, eps, y, ldy);
}

static dim3 elementwise_grid(int M, int H) {
  int bx = (H + 255) / 256;
  if (bx > 64) bx = 64;
  return dim3(bx, M);
}

cudaError_t launch_residual(__nv_bfloat16* h, int ldh, const __nv_bfloat16* t, int ldt, int M, int H,
                            cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(elementwise_grid(M, H), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, residual_kernel, h, ldh, t, ldt, H);
}

cudaError_t launch_swiglu(const __nv_bfloat16* g, int ldg, const __nv_bfloat16* u, int ldu, int M, int I,
                          __nv_bfloat16* out, int lds, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(elementwise_grid(M, I), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, swiglu_kernel, g, ldg, u, ldu, I, out, lds);
}

// Self-test of the bounded-wait error path: one thread waits on an mbarrier
// that nothing arrives at, for at most limit_ns, and records the timeout in
// the device error word as the library's own waits do (no fault, no trap).
__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_ns();
    bool done = mbar_try_wait(&bar, 0);
    while (!done && global_ns() - t0 < limit_ns) done = mbar_try_wait(&bar, 0);
    if (!done) raise_error(ERR_TIMEOUT_FULL);
  }
}

cudaError_t launch_wait_selftest(unsigned int limit_us, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>((unsigned long long)limit_us * 1000ull);
  return cudaGetLastError();
}

}  // namespace sv
