// Internal interfaces between the C entry points and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "specverify.h"

namespace sv {

// ---------------------------------------------------------------- tiling
constexpr int GROUP = 64;        // weights per quantization group (along K)
constexpr int BN = 64;           // weight rows per CTA tile
constexpr int KC = 512;          // k per pipeline stage (8 groups)
constexpr int GPS = KC / GROUP;  // groups per stage
constexpr int NCW = 8;           // consumer warps per CTA: 2 row halves x 4 k-quarters
constexpr int QMM_THREADS = (NCW + 1) * 32;
constexpr int MAX_M = 32;        // rows per verify block handled by the kernels

enum EpiMode : int { EPI_BF16 = 0, EPI_BF16_RESIDUAL = 1, EPI_LOGITS = 2 };
enum PrepMode : int { PREP_PLAIN = 0, PREP_RMSNORM = 1, PREP_SWIGLU = 2 };
constexpr size_t COUNTER_BYTES = 262144;  // zero-between-calls counter prefix of every workspace
constexpr int MAX_TILES = (int)(COUNTER_BYTES / 8);  // two counters (row halves) per tile

struct PrepArgs {
  const __nv_bfloat16* x; int ldx;      // activations (g for SwiGLU)
  const __nv_bfloat16* x2; int ldx2;    // u for SwiGLU
  const __nv_bfloat16* w; float eps;    // RMSNorm weight (nullable) and epsilon
  int M, MP, K, mode;
  __half* xp;                           // [K/32][MP][32] fp16 (scaled, MMA order)
  float* xsum;                          // [K/512][9][MP]: 8 group sums, then 2^-e of the chunk
  float* rms;                           // [K/512 + 1][MP]: chunk sums of x^2, then eps (or -1: no RMSNorm)
};

// Stream-K schedule shared by host and device.  Work unit = (tile, k-chunk):
// units [c*total/grid, (c+1)*total/grid) belong to CTA c.
struct Schedule {
  int N, K, tiles_n, units_per_tile, total_units, grid;
};

struct QmmParams {
  Schedule sch;
  int M, MP;                       // rows, rows padded to the n8 MMA tile
  // prepared activations (written by the prep kernel into the workspace)
  const __half* xp;                // [K/32][MP][32] fp16, scaled by 2^e per (row, chunk), permuted
  const float* xsum;               // [K/512][9][MP]: group sums of the scaled rows, then 2^-e
  const float* rms;                // [K/512 + 1][MP]: RMSNorm partials and eps (eps < 0: none)
  float* partials;                 // [grid][2 slots][2 halves][32*MP]
  int* counters;                   // [tiles_n][2], zero between calls
  // epilogue
  int mode;
  __nv_bfloat16* y; int ldy;       // EPI_BF16 / EPI_BF16_RESIDUAL
  const __nv_bfloat16* res; int ldres;
  float* logits; int ldl;          // EPI_LOGITS
  float* tile_stats;               // [tiles_n*2][MP][3] per 32-row half (max, argmax bits, sumexp)
  float inv_temp;                  // 1/T, 0 for greedy
};

// Byte offsets of the pieces of a qmm workspace.  The counters always sit in
// the fixed prefix; the prepared activations depend only on (M, K), so a
// prepare call and the run calls that consume it agree on where they are.
struct QmmWorkspace {
  size_t counters, xp, xsum, rms, partials, tile_stats, total;
};

Schedule make_schedule(int N, int K, int grid_limit);
QmmWorkspace qmm_workspace_layout(int M, int N, int K, int grid, bool with_stats);
int device_sm_count();
int fail(int status, const char* fmt, ...);
int check_weight(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                 int group, int M);
int cuda_fail(cudaError_t e, const char* what);
size_t align256(size_t v);
bool aligned(const void* p, size_t a);
size_t prepare_bytes(int M, int K);
size_t qmm_bytes(int M, int N, int K, bool stats);
size_t accept_bytes(int B, int rows);
int qmm_prepare_internal(const uint16_t* x, int ldx, int M, int K, int bits, int mode, const uint16_t* x2, int ldx2,
                         const uint16_t* w, float eps, void* ws, cudaStream_t s);
int qmm_run_internal(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                     int M, int mode, uint16_t* y, int ldy, const uint16_t* residual, int ldr, float* logits,
                     int ldl, float temperature, float* row_max, float* row_sumexp, int32_t* row_argmax, void* ws,
                     cudaStream_t s);
int check_accept(int B, const int32_t* row_offsets, const float* logits, int ldl, const float* row_max,
                 const float* row_sumexp, const int32_t* row_argmax, const float* q, int ldq, const int32_t* draft,
                 int V, float temperature, const float* u, int32_t* out_len, int32_t* out_tokens);
int accept_internal(int B, const int32_t* offs, const float* logits, int ldl, const float* row_max,
                    const float* row_sumexp, const int32_t* row_argmax, const float* q, int ldq, const int32_t* draft,
                    int V, float temperature, const float* u, int32_t* out_len, int32_t* out_tokens, void* ws,
                    cudaStream_t s);
cudaError_t read_and_clear_error_word(unsigned int* out);

// Launchers (return cudaError_t of the launch).
cudaError_t launch_prep(const PrepArgs& a, int bits, int mode, cudaStream_t s);
cudaError_t launch_qmm(int bits, int NT, const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tb,
                       const QmmParams& p, cudaStream_t s);
cudaError_t launch_lmhead_finalize(const float* tile_stats, int tiles_n, int MP, int M, float inv_temp,
                                   float* row_max, float* row_sumexp, int32_t* row_argmax, cudaStream_t s);

// Common launch helper: programmatic-serialization attribute on every launch.
cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr);

}  // namespace sv
