// Parameter blocks and launchers of the accept, row-stat, Philox and glue kernels.
#pragma once

#include "sv_internal.h"

namespace sv {

constexpr int MAX_BATCH = 256;

// Exact sums of weights in (0, 1] (probabilities, fp32 exp terms) as 64.64
// fixed-point integers: exact for every weight from 2^-40 up, and the
// integer sum does not depend on the order of the terms.
typedef unsigned __int128 u128;

// w * 2^64 as an integer: exact for normal w >= 2^-40 (a 24-bit mantissa
// shifted left), truncated below; 0 for w <= 0, subnormal or not below 2^40.
__device__ __forceinline__ u128 to_fixed(float w) {
  if (!(w > 0.f) || !(w < 1.0995116e12f)) return 0;
  const uint32_t bits = __float_as_uint(w);
  const int e = (int)((bits >> 23) & 255u);
  if (e == 0) return 0;
  const uint32_t mant = (bits & 0x7fffffu) | 0x800000u;
  const int shift = e - 127 - 23 + 64;  // w = mant * 2^(e - 150)
  if (shift >= 0) return (u128)mant << shift;
  return shift > -24 ? (u128)(mant >> -shift) : (u128)0;
}
__device__ __forceinline__ double fixed_to_double(u128 m) {
  return (double)(unsigned long long)(m >> 64) + ldexp((double)(unsigned long long)m, -64);
}
__device__ __forceinline__ u128 warp_sum_u128(u128 v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const unsigned long long lo = __shfl_xor_sync(0xffffffffu, (unsigned long long)v, off);
    const unsigned long long hi = __shfl_xor_sync(0xffffffffu, (unsigned long long)(v >> 64), off);
    v += ((u128)hi << 64) | lo;
  }
  return v;
}
// Order-preserving 32-bit key of an fp32 value: larger value -> larger key;
// -0 and +0 share a key.  Truncation bounds are expressed in these keys.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

enum : int { SEL_LOGITS = 0, SEL_PROBS = 1, SEL_TOPN = 2 };
struct SelectArgs {
  const float* x; int ldx;      // rows: fp32 logits (SEL_LOGITS, SEL_TOPN) or probabilities (SEL_PROBS)
  float* y; int ldy;            // SEL_PROBS: truncated rows (may alias x)
  int V, mode;
  const float* row_max;         // SEL_LOGITS: row maxima (null: computed in the kernel)
  float temperature;            // SEL_LOGITS: T > 0; SEL_TOPN: T <= 0 means 1
  int top_k; float top_p;
  uint32_t* out_key; int32_t* out_idx; float* out_norm;          // SEL_LOGITS: kept = key > K or (== K and index <= I)
  const int32_t* chosen; float* chosen_lp; int32_t* top_ids; float* top_lp; int top_n;  // SEL_TOPN
};
cudaError_t launch_select(const SelectArgs& a, int rows, cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned int limit_us, cudaStream_t s);

struct AcceptParams {
  int offs[MAX_BATCH + 1];   // logits-row offsets of the requests (copied by value)
  const float* logits; int ldl;
  const float* row_max; const float* row_sumexp; const int32_t* row_argmax;
  const float* q; int ldq;
  const int32_t* draft;
  int V;
  float temperature;
  const float* u;
  int32_t* out_len; int32_t* out_tokens;
  const uint32_t* tkey;      // truncated target (or null): per logits row, kept tokens have
  const int32_t* tidx;       //   order_key(z) > tkey, or == tkey with index <= tidx,
  const float* tnorm;        //   and tnorm is their sum of exp((z - max) / T)
  double* chunk_sums;        // [B][nb][2]
  int* counters;             // [B], zero between calls
  int nb;                    // vocabulary chunks per request
};

cudaError_t launch_accept(const AcceptParams& p, int B, cudaStream_t s);
cudaError_t launch_row_stats(const float* logits, int ldl, int rows, int V, float temperature, float* row_max,
                             float* row_sumexp, int32_t* row_argmax, cudaStream_t s);
cudaError_t launch_philox(uint64_t seed, uint64_t subseq, uint64_t offset, int n, float* out, cudaStream_t s);
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, int ldx, int M, int H, const __nv_bfloat16* w, float eps,
                           __nv_bfloat16* y, int ldy, cudaStream_t s);
cudaError_t launch_residual(__nv_bfloat16* h, int ldh, const __nv_bfloat16* t, int ldt, int M, int H,
                            cudaStream_t s);
cudaError_t launch_swiglu(const __nv_bfloat16* g, int ldg, const __nv_bfloat16* u, int ldu, int M, int I,
                          __nv_bfloat16* out, int lds, cudaStream_t s);

}  // namespace sv
