// Activation preparation of one (64-wide group, padded row): shared by the
// input preparation of a projection and the gathered preparation of the
// experts' rows.
//
// The tensor-core path multiplies fp16 codes by fp16 activations.  A bf16 row
// converts to fp16 without loss once it is scaled by a power of two that puts
// its largest magnitude in [2^14, 2^15): the 8 significant bits of every bf16
// value fit in fp16's 11, and only values 2^-28 below the row maximum (whose
// products vanish against fp32 accumulation anyway) reach fp16's subnormals.
// The scale is undone once per output row in the epilogue.  Per group:
//   v   = x, bf16(silu(x) * x2) for SwiGLU, or bf16(x * weight) for RMSNorm
//         (whose row scale 1/sqrt(mean(x^2) + eps) is applied to the matmul
//         output from the group sums of x^2 stored here),
//   e   = 15 - exponent of the group's max |v|, so v * 2^e lies below 2^15 and
//         every bf16 value keeps all its significant bits in fp16,
//   out = fp16(v * 2^e) in the order the MMA fragments read the codes, the
//         fp32 sum of v * 2^e, and 2^-e.
#pragma once

#include "sv_internal.h"
#include "sv_ptx.cuh"
#include "stream_kernel.cuh"

namespace sv {

// One warp: group g of padded row m.  `row` is null for a padding row (zeros).
template <int BITS, int MODE>
__device__ __forceinline__ void prep_group(const __nv_bfloat16* row, const __nv_bfloat16* row2,
                                           const __nv_bfloat16* w, float eps, int m, int g, int MP, int K,
                                           const ActBuf& out) {
  const int lane = threadIdx.x & 31;
  float v[2] = {0.f, 0.f}, sq = 0.f;
  if (row) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int k = g * GROUP + lane + 32 * i;
      float x = __bfloat162float(row[k]);
      if (MODE == PREP_RMSNORM) {
        sq = fmaf(x, x, sq);
        if (w) x = __bfloat162float(__float2bfloat16_rn(x * __bfloat162float(w[k])));
      } else if (MODE == PREP_SWIGLU) {
        const float u = __bfloat162float(row2[k]);
        x = __bfloat162float(__float2bfloat16_rn(silu_f32(x) * u));
      }
      v[i] = x;
    }
  }
  float mx = fmaxf(fabsf(v[0]), fabsf(v[1]));
  for (int off = 16; off; off >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    sq += __shfl_xor_sync(0xffffffffu, sq, off);
  }
  const int e = scale_exponent(mx);
  const float sc = pow2_exact(e);
  float gs = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int pos = act_pos<BITS>(lane + 32 * i);  // element lane + 32 i of the group
    const float y = v[i] * sc;
    gs += y;
    out.xp[((size_t)(2 * g + (pos >> 5)) * MP + m) * 32 + (pos & 31)] = __float2half_rn(y);
  }
  for (int off = 16; off; off >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, off);
  if (lane == 0) {
    float* xs = out.xs + (size_t)g * 2 * MP;
    xs[m] = gs;
    xs[MP + m] = pow2_exact(-e);
    out.sq[(size_t)g * MP + m] = sq;
    if (g == 0) out.sq[(size_t)(K / GROUP) * MP + m] = MODE == PREP_RMSNORM ? eps : -1.f;
  }
}

}  // namespace sv
