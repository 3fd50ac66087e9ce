// Parameter blocks and launchers of the accept, row-stat, Philox and glue kernels.
#pragma once

#include "sv_internal.h"

namespace sv {

constexpr int MAX_BATCH = 256;

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
