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
constexpr int NCW = 8;           // consumer warps per CTA: 4 row quarters x 2 k halves
constexpr int NEW = 4;           // epilogue warps per CTA: one per row quarter
constexpr int XPW = NCW + 1 + NEW;  // the activation-copy warp
constexpr int QMM_THREADS = (NCW + 1 + NEW + 1) * 32;  // consumers, weight producer, epilogue warps, activation producer
constexpr int MAX_M = 32;        // rows per verify block handled by the weight-streaming kernels
constexpr int WIDE_MAX_M = 512;  // rows per block of the tensor-memory kernel (sv_qmm_verify, M > 32)
constexpr int MAX_PHASES = 272;  // matmuls per launch (64 layers x 4 projections + head, with room)

enum PrepMode : int { PREP_PLAIN = 0, PREP_RMSNORM = 1, PREP_SWIGLU = 2 };

// Workspace prefix of counters that are zero between calls.
constexpr size_t COUNTER_BYTES = 262144;
constexpr size_t ACC_CTR_OFF = 0;             // the accept step's per-request counters
constexpr int MAX_TILES = 32768;
constexpr size_t GRID_BAR_OFF = 196608;       // grid barrier arrivals, one counter per phase transition
constexpr size_t EXIT_CTR_OFF = 200704;       // CTAs finished
constexpr size_t ABORT_OFF = 200708;          // some CTA gave up

// What a phase's finishing epilogue does with its output tile.
enum PhaseKind : int {
  PH_STORE = 0,   // y = bf16(out); tiles < prep_tiles also become the next phase's input
  PH_RESID = 1,   // y (the hidden state) += bf16(out) in place; it becomes the next RMSNorm input
  PH_GATEUP = 2,  // 64-row gate/up blocks interleaved; silu(gate) * up becomes the next input
  PH_LOGITS = 3,  // fp32 logits and per-tile row statistics
};

struct Phase {
  const uint8_t* packed;  // the weight in unit-packed form (sv_qmm_pack), or null: tensor maps
  const uint8_t* wq;
  const uint16_t* scales;
  const uint16_t* biases;
  __nv_bfloat16* y;   // output (PH_RESID: the updated hidden state)
  const __nv_bfloat16* res;  // PH_RESID: hidden state read (may equal y)
  int N, K, ldy, ldr;
  int kind;
  int prep_tiles;     // PH_STORE: output tiles that feed the next phase
  int in_buf, out_buf;
  int half;           // PH_GATEUP: columns per half (gate, then up) of y
};

// Prepared activations of one phase input (K <= the buffer's capacity).
struct ActBuf {
  __half* xp;   // [K/32][MP][32] fp16 x * 2^e, MMA order
  float* xs;    // [K/64][2][MP]: group sum of x * 2^e, then 2^-e
  float* sq;    // [K/64 + 1][MP]: group sums of x^2, then eps (RMSNorm input) or -1
};

struct StreamParams {
  CUtensorMap tm[3];          // weights, scales, biases of a one-phase launch
  const CUtensorMap* maps;    // [n_phases][3] in device memory (a round plan), or null: use tm
  int n_phases, M, MP, grid;
  float rms_eps;
  ActBuf act[2];
  float* partials;        // [grid][2 slots][4 quarters][16*MP]
  float* pair_words;      // PH_GATEUP: [blocks][4 quarters][16*MP] up values, self-announcing words
  unsigned* grid_bar;     // [MAX_PHASES]: arrivals for the transition into phase t
  int* exit_counter;
  int* abort_all;
  float* logits; int ldl;
  float* tile_stats;      // [tiles][MP][3] (max, argmax bits, sum-exp) of the PH_LOGITS phase
  float inv_temp;
  Phase ph[MAX_PHASES];
};

struct PrepArgs {
  const __nv_bfloat16* x; int ldx;      // activations (g for SwiGLU)
  const __nv_bfloat16* x2; int ldx2;    // u for SwiGLU
  const __nv_bfloat16* w; float eps;    // RMSNorm weight (nullable) and epsilon
  int M, MP, K, mode;
  ActBuf out;
};

// Byte offsets of a workspace's pieces: the counter prefix, two activation
// buffers for inputs up to K_cap wide, the stream-K partials, tile statistics.
struct Layout {
  size_t act[2][3], partials, tile_stats, total;
};
Layout workspace_layout(int M, int K_cap, int grid, int stat_tiles, int n_act);
ActBuf act_buf(void* ws, const Layout& L, int a);
void stream_params_init(StreamParams& p, void* ws, const Layout& L, int M, int grid, float rms_eps);
int prepare_into(const uint16_t* x, int ldx, int M, int K, int bits, int mode, const uint16_t* x2, int ldx2,
                 const uint16_t* w, float eps, const ActBuf& out, cudaStream_t s);

int device_sm_count();
bool bits_supported(int bits);  // code widths of the matmul kernels: 2, 4, 8
size_t packed_bytes(int N, int K, int bits);
// Tensor maps of one quantized weight: codes in 128-byte swizzled boxes of
// 64 rows, scales and biases in 8-group x 64-row boxes.
int encode_weight_maps(CUtensorMap (&out)[3], const void* wq, const void* scales, const void* biases, int N, int K,
                       int bits);
int fail(int status, const char* fmt, ...);
int encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw);
// The wide-block matmul (33 <= M <= 512, tcgen05): workspace size and launch.
size_t wide_bytes(int M, int N, int K, int bits);
int wide_qmm(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
             const uint16_t* x, int ldx, int M, uint16_t* y, int ldy, const uint16_t* residual, int ldr, void* ws,
             cudaStream_t s);
int check_weight(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                 int group, int M);
int cuda_fail(cudaError_t e, const char* what);
size_t align256(size_t v);
bool aligned(const void* p, size_t a);
size_t prepare_bytes(int M, int K);
size_t qmm_bytes(int M, int N, int K, int bits, bool stats);
// Offset and size of the split-tile partials in a one-projection workspace
// (zero between calls, like the counter block).
void qmm_partials_region(int M, int N, int K, int bits, size_t* off, size_t* bytes);
size_t accept_bytes(int B, int rows);
int qmm_prepare_internal(const uint16_t* x, int ldx, int M, int K, int bits, int mode, const uint16_t* x2, int ldx2,
                         const uint16_t* w, float eps, void* ws, cudaStream_t s);
// mode: 0 = store bf16, 1 = add to the residual, 2 = logits with row statistics
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
                    cudaStream_t s, int top_k = 0, float top_p = 1.f);
cudaError_t read_and_clear_error_word(unsigned int* out);

// Launchers (return cudaError_t of the launch).
cudaError_t launch_prep(const PrepArgs& a, int bits, int mode, cudaStream_t s);
// cooperative when the launch has more than one phase (grid barriers)
cudaError_t launch_stream(int bits, const StreamParams& p, cudaStream_t s);
int stream_max_grid(int bits, int MP);
cudaError_t launch_lmhead_finalize(const float* tile_stats, int tiles_n, int MP, int M, float inv_temp,
                                   float* row_max, float* row_sumexp, int32_t* row_argmax, cudaStream_t s);

// Common launch helper: programmatic-serialization attribute on every launch.
cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr);

}  // namespace sv
