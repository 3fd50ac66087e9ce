// C entry points of libspecverify: argument validation, workspace layout,
// tensor-map encoding and kernel dispatch.  Nothing here allocates device
// memory and nothing throws across the boundary.
#include <cudaTypedefs.h>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <cstddef>
#include <mutex>

#include "sv_internal.h"
#include "sv_kernels.h"
#include "sv_ptx.cuh"

namespace sv {

cudaError_t launch_stream_b2(const StreamParams& p, cudaStream_t s);
cudaError_t launch_stream_b4(const StreamParams& p, cudaStream_t s);
cudaError_t launch_stream_b8(const StreamParams& p, cudaStream_t s);
int stream_max_grid_b2(int MP);
int stream_max_grid_b4(int MP);
int stream_max_grid_b8(int MP);

cudaError_t launch_stream(int bits, const StreamParams& p, cudaStream_t s) {
  return bits == 8 ? launch_stream_b8(p, s) : (bits == 4 ? launch_stream_b4(p, s) : launch_stream_b2(p, s));
}

bool bits_supported(int bits) { return bits == 2 || bits == 4 || bits == 8; }

int stream_max_grid(int bits, int MP) {
  static std::mutex mu;
  static int cache[64][3][5] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][bits == 8 ? 2 : (bits == 4 ? 1 : 0)][MP / 8];
  if (!c) c = bits == 8 ? stream_max_grid_b8(MP) : (bits == 4 ? stream_max_grid_b4(MP) : stream_max_grid_b2(MP));
  return c;
}

static thread_local char g_last[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last, sizeof(g_last), fmt, ap);
  va_end(ap);
  return status;
}
int cuda_fail(cudaError_t e, const char* what) { return fail(SV_ECUDA, "%s: %s", what, cudaGetErrorString(e)); }

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

Layout workspace_layout(int M, int K_cap, int grid, int stat_tiles, int n_act) {
  const int MP = 8 * ((M + 7) / 8);
  const size_t G = (size_t)K_cap / GROUP;
  Layout L = {};
  size_t off = COUNTER_BYTES;
  for (int a = 0; a < n_act; ++a) {
    L.act[a][0] = off; off = align256(off + (size_t)K_cap * MP * 2);
    L.act[a][1] = off; off = align256(off + G * 2 * MP * 4);
    L.act[a][2] = off; off = align256(off + (G + 1) * MP * 4);
  }
  L.partials = off;   off = align256(off + (size_t)grid * 2 * BN * MP * 4);
  L.tile_stats = off; off = align256(off + (size_t)stat_tiles * MP * 12);
  L.total = off;
  return L;
}

ActBuf act_buf(void* ws, const Layout& L, int a) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  ActBuf b;
  b.xp = reinterpret_cast<__half*>(base + L.act[a][0]);
  b.xs = reinterpret_cast<float*>(base + L.act[a][1]);
  b.sq = reinterpret_cast<float*>(base + L.act[a][2]);
  return b;
}

void stream_params_init(StreamParams& p, void* ws, const Layout& L, int M, int grid, float rms_eps) {
  memset(static_cast<void*>(&p), 0, offsetof(StreamParams, ph));
  uint8_t* base = static_cast<uint8_t*>(ws);
  p.M = M;
  p.MP = 8 * ((M + 7) / 8);
  p.grid = grid;
  p.rms_eps = rms_eps;
  p.act[0] = act_buf(ws, L, 0);
  p.act[1] = L.act[1][0] ? act_buf(ws, L, 1) : p.act[0];
  p.partials = reinterpret_cast<float*>(base + L.partials);
  p.grid_bar = reinterpret_cast<unsigned*>(base + GRID_BAR_OFF);
  p.exit_counter = reinterpret_cast<int*>(base + EXIT_CTR_OFF);
  p.abort_all = reinterpret_cast<int*>(base + ABORT_OFF);
  p.tile_stats = reinterpret_cast<float*>(base + L.tile_stats);
}

// ------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t stride1, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return fail(SV_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SV_ECUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return SV_OK;
}

// Codes as a 3D view (byte within a 128-byte piece, row, piece) so that one
// copy brings all pieces of a stage: shared memory receives [piece][row][128 B]
// with the 128-byte swizzle, the layout the consumers read.
static int encode_codes(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t N, uint32_t pieces) {
  auto fn = encode_fn();
  if (!fn) return fail(SV_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {128, N, row_bytes / 128};
  const cuuint64_t strides[2] = {row_bytes, 128};
  const cuuint32_t box[3] = {128, (cuuint32_t)BN, pieces};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SV_ECUDA, "cuTensorMapEncodeTiled (codes) failed (CUresult %d)", (int)r);
  return SV_OK;
}

int encode_weight_maps(CUtensorMap (&out)[3], const void* wq, const void* scales, const void* biases, int N, int K,
                       int bits) {
  const uint64_t row_bytes = (uint64_t)K * bits / 8, G = (uint64_t)(K / GROUP);
  int st = encode_codes(&out[0], wq, row_bytes, (uint64_t)N, (uint32_t)(KC * bits / 8 / 128));
  if (st) return st;
  st = encode_tiled_2d(&out[1], CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, G, (uint64_t)N, G * 2, GPS, BN,
                 CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st) return st;
  return encode_tiled_2d(&out[2], CU_TENSOR_MAP_DATA_TYPE_UINT16, biases, G, (uint64_t)N, G * 2, GPS, BN,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Shared validation of a quantized weight + activation block.
int check_weight(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                 int group, int M) {
  if (!wq || !scales || !biases) return fail(SV_EINVAL, "weight pointers must be non-null");
  if (!bits_supported(bits)) return fail(SV_EUNSUPPORTED, "bits must be 2, 4 or 8 (got %d)", bits);
  if (group != GROUP) return fail(SV_EUNSUPPORTED, "group size must be 64 (got %d)", group);
  if (N < 1 || N > MAX_TILES * BN) return fail(SV_EINVAL, "N out of range (got %d)", N);
  if (K < 1 || K % GROUP) return fail(SV_EINVAL, "K must be a positive multiple of 64 (got %d)", K);
  if (K % KC) return fail(SV_EUNSUPPORTED, "K must be a multiple of 512 (got %d)", K);
  if (K > (1 << 20)) return fail(SV_EINVAL, "K too large (got %d)", K);
  if (M < 1) return fail(SV_EINVAL, "M must be >= 1 (got %d)", M);
  if (M > MAX_M) return fail(SV_EUNSUPPORTED, "M must be <= 32 (got %d)", M);
  if (!aligned(wq, 16) || !aligned(scales, 16) || !aligned(biases, 16))
    return fail(SV_EINVAL, "wq, scales and biases must be 16-byte aligned");
  return SV_OK;
}

// Validation of a prepare call (everything the host can check).
static int check_prepare(const uint16_t* x, int ldx, int M, int K, int bits, int mode, const uint16_t* x2, int ldx2,
                         void* ws) {
  if (!bits_supported(bits)) return fail(SV_EUNSUPPORTED, "bits must be 2, 4 or 8 (got %d)", bits);
  if (K < 1 || K % GROUP) return fail(SV_EINVAL, "K must be a positive multiple of 64 (got %d)", K);
  if (K % KC) return fail(SV_EUNSUPPORTED, "K must be a multiple of 512 (got %d)", K);
  if (K > (1 << 20)) return fail(SV_EINVAL, "K too large (got %d)", K);
  if (M < 1) return fail(SV_EINVAL, "M must be >= 1 (got %d)", M);
  if (M > MAX_M) return fail(SV_EUNSUPPORTED, "M must be <= 32 (got %d)", M);
  if (mode < PREP_PLAIN || mode > PREP_SWIGLU) return fail(SV_EINVAL, "unknown prepare mode %d", mode);
  if (!x || !ws) return fail(SV_EINVAL, "x and workspace must be non-null");
  if (ldx < K) return fail(SV_EINVAL, "ldx must be >= K");
  if (mode == PREP_SWIGLU && (!x2 || ldx2 < K)) return fail(SV_EINVAL, "SwiGLU needs u with ldu >= K");
  if (!aligned(ws, 256)) return fail(SV_EINVAL, "workspace must be 256-byte aligned");
  return SV_OK;
}

size_t prepare_bytes(int M, int K) { return workspace_layout(M, K, 0, 0, 1).partials; }

int prepare_into(const uint16_t* x, int ldx, int M, int K, int bits, int mode, const uint16_t* x2, int ldx2,
                 const uint16_t* w, float eps, const ActBuf& out, cudaStream_t s) {
  PrepArgs a;
  a.x = reinterpret_cast<const __nv_bfloat16*>(x);
  a.ldx = ldx;
  a.x2 = reinterpret_cast<const __nv_bfloat16*>(x2);
  a.ldx2 = ldx2;
  a.w = reinterpret_cast<const __nv_bfloat16*>(w);
  a.eps = eps;
  a.M = M;
  a.MP = 8 * ((M + 7) / 8);
  a.K = K;
  a.mode = mode;
  a.out = out;
  cudaError_t e = launch_prep(a, bits, mode, s);
  if (e != cudaSuccess) return cuda_fail(e, "prepare launch");
  return SV_OK;
}

int qmm_prepare_internal(const uint16_t* x, int ldx, int M, int K, int bits, int mode, const uint16_t* x2, int ldx2,
                         const uint16_t* w, float eps, void* ws, cudaStream_t s) {
  const Layout L = workspace_layout(M, K, 0, 0, 1);
  return prepare_into(x, ldx, M, K, bits, mode, x2, ldx2, w, eps, act_buf(ws, L, 0), s);
}

static int grid_for(int bits, int M, int total_units) {
  const int cap = stream_max_grid(bits, 8 * ((M + 7) / 8));
  if (cap <= 0) return 0;
  return total_units < cap ? total_units : cap;
}

enum RunMode : int { RUN_STORE = 0, RUN_RESIDUAL = 1, RUN_LOGITS = 2 };

size_t qmm_bytes(int M, int N, int K, int bits, bool stats) {
  const int tiles = (N + BN - 1) / BN;
  const int grid = grid_for(bits, M, tiles * (K / KC));
  if (grid <= 0) return 0;
  return workspace_layout(M, K, grid, stats ? tiles : 0, 1).total;
}

void qmm_partials_region(int M, int N, int K, int bits, size_t* off, size_t* bytes) {
  const int tiles = (N + BN - 1) / BN;
  const int grid = grid_for(bits, M, tiles * (K / KC));
  const Layout L = workspace_layout(M, K, grid > 0 ? grid : 0, 0, 1);
  *off = L.partials;
  *bytes = L.tile_stats - L.partials;
}

int qmm_run_internal(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                     int M, int mode, uint16_t* y, int ldy, const uint16_t* residual, int ldr, float* logits,
                     int ldl, float temperature, float* row_max, float* row_sumexp, int32_t* row_argmax, void* ws,
                     cudaStream_t s) {
  const int tiles = (N + BN - 1) / BN;
  const int grid = grid_for(bits, M, tiles * (K / KC));
  if (grid <= 0) return fail(SV_ECUDA, "no CUDA device");
  const bool stats = mode == RUN_LOGITS;
  const Layout L = workspace_layout(M, K, grid, stats ? tiles : 0, 1);
  static thread_local StreamParams p;  // about 22 KB: kept off the stack
  stream_params_init(p, ws, L, M, grid, 0.f);
  int st = encode_weight_maps(p.tm, wq, scales, biases, N, K, bits);
  if (st) return st;
  p.maps = nullptr;
  p.n_phases = 1;
  Phase& ph = p.ph[0];
  memset(&ph, 0, sizeof(ph));
  ph.wq = reinterpret_cast<const uint8_t*>(wq);
  ph.scales = scales;
  ph.biases = biases;
  ph.N = N;
  ph.K = K;
  ph.in_buf = 0;
  ph.out_buf = -1;
  if (mode == RUN_LOGITS) {
    ph.kind = PH_LOGITS;
    p.logits = logits;
    p.ldl = ldl;
    p.inv_temp = temperature > 0.f ? 1.f / temperature : 0.f;
  } else if (mode == RUN_RESIDUAL) {
    ph.kind = PH_RESID;
    ph.y = reinterpret_cast<__nv_bfloat16*>(y);
    ph.ldy = ldy;
    ph.res = reinterpret_cast<const __nv_bfloat16*>(residual);
    ph.ldr = ldr;
  } else {
    ph.kind = PH_STORE;
    ph.y = reinterpret_cast<__nv_bfloat16*>(y);
    ph.ldy = ldy;
  }
  cudaError_t e = launch_stream(bits, p, s);
  if (e != cudaSuccess) return cuda_fail(e, "qmm launch");
  if (stats && (row_max || row_sumexp || row_argmax)) {
    e = launch_lmhead_finalize(p.tile_stats, tiles, p.MP, M, p.inv_temp, row_max, row_sumexp, row_argmax, s);
    if (e != cudaSuccess) return cuda_fail(e, "lm_head finalize launch");
  }
  return SV_OK;
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t sv_qmm_workspace_bytes(int M, int N, int K, int bits) {
  if (M < 1 || M > WIDE_MAX_M || N < 1 || N > MAX_TILES * BN || K < KC || K % KC || !bits_supported(bits)) return 0;
  if (M > MAX_M) return wide_bytes(M, N, K, bits);
  return qmm_bytes(M, N, K, bits, false);
}

size_t sv_lm_head_workspace_bytes(int M, int V, int K, int bits) {
  if (M < 1 || M > MAX_M || V < 1 || V > MAX_TILES * BN || K < KC || K % KC || !bits_supported(bits)) return 0;
  return qmm_bytes(M, V, K, bits, true);
}

int sv_qmm_prepare(const uint16_t* x, int ldx, int M, int K, int bits, int mode, const uint16_t* x2, int ldx2,
                   const uint16_t* rms_weight, float eps, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_prepare(x, ldx, M, K, bits, mode, x2, ldx2, workspace);
  if (st) return st;
  if (mode == PREP_RMSNORM && !(eps >= 0.f)) return fail(SV_EINVAL, "eps must be >= 0");
  if (workspace_bytes < prepare_bytes(M, K))
    return fail(SV_EINVAL, "workspace too small: %zu < %zu", workspace_bytes, prepare_bytes(M, K));
  return qmm_prepare_internal(x, ldx, M, K, bits, mode, x2, ldx2, rms_weight, eps, workspace,
                              static_cast<cudaStream_t>(stream));
}

static int check_run(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                     int group, int M, void* ws, size_t ws_bytes, bool stats) {
  int st = check_weight(wq, scales, biases, N, K, bits, group, M);
  if (st) return st;
  if (!ws) return fail(SV_EINVAL, "workspace must be non-null");
  if (!aligned(ws, 256)) return fail(SV_EINVAL, "workspace must be 256-byte aligned");
  const size_t need = qmm_bytes(M, N, K, bits, stats);
  if (need == 0) return fail(SV_ECUDA, "no CUDA device");
  if (ws_bytes < need) return fail(SV_EINVAL, "workspace too small: %zu < %zu", ws_bytes, need);
  return SV_OK;
}

int sv_qmm_run(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits, int group,
               int M, uint16_t* y, int ldy, const uint16_t* residual, int ldr, void* workspace,
               size_t workspace_bytes, void* stream) {
  int st = check_run(wq, scales, biases, N, K, bits, group, M, workspace, workspace_bytes, false);
  if (st) return st;
  if (!y) return fail(SV_EINVAL, "y must be non-null");
  if (ldy < N || (residual && ldr < N)) return fail(SV_EINVAL, "ldy and ldr must be >= N");
  if (!aligned(y, 2) || (residual && !aligned(residual, 2))) return fail(SV_EINVAL, "misaligned y or residual");
  return qmm_run_internal(wq, scales, biases, N, K, bits, M, residual ? RUN_RESIDUAL : RUN_STORE, y, ldy,
                          residual, ldr, nullptr, 0, 0.f, nullptr, nullptr, nullptr, workspace,
                          static_cast<cudaStream_t>(stream));
}

static int qmm_verify_wide(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                           int group, const uint16_t* x, int ldx, int M, uint16_t* y, int ldy,
                           const uint16_t* residual, int ldr, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_weight(wq, scales, biases, N, K, bits, group, 1);
  if (st) return st;
  if (!x || !y || !workspace) return fail(SV_EINVAL, "x, y and workspace must be non-null");
  if (ldx < K || ldy < N || (residual && ldr < N)) return fail(SV_EINVAL, "ldx must be >= K, ldy and ldr >= N");
  if (!aligned(x, 2) || !aligned(y, 2) || (residual && !aligned(residual, 2)))
    return fail(SV_EINVAL, "misaligned x, y or residual");
  if (!aligned(workspace, 256)) return fail(SV_EINVAL, "workspace must be 256-byte aligned");
  const size_t need = wide_bytes(M, N, K, bits);
  if (workspace_bytes < need) return fail(SV_EINVAL, "workspace too small: %zu < %zu", workspace_bytes, need);
  return wide_qmm(wq, scales, biases, N, K, bits, x, ldx, M, y, ldy, residual, ldr, workspace,
                  static_cast<cudaStream_t>(stream));
}

int sv_qmm_verify(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                  int group, const uint16_t* x, int ldx, int M, uint16_t* y, int ldy, const uint16_t* residual,
                  int ldr, void* workspace, size_t workspace_bytes, void* stream) {
  if (M > MAX_M && M <= WIDE_MAX_M)
    return qmm_verify_wide(wq, scales, biases, N, K, bits, group, x, ldx, M, y, ldy, residual, ldr, workspace,
                           workspace_bytes, stream);
  int st = check_weight(wq, scales, biases, N, K, bits, group, M);
  if (st) return st;
  st = check_prepare(x, ldx, M, K, bits, PREP_PLAIN, nullptr, 0, workspace);
  if (st) return st;
  if (!y) return fail(SV_EINVAL, "y must be non-null");
  if (ldy < N || (residual && ldr < N)) return fail(SV_EINVAL, "ldy and ldr must be >= N");
  if (!aligned(y, 2) || (residual && !aligned(residual, 2))) return fail(SV_EINVAL, "misaligned y or residual");
  st = check_run(wq, scales, biases, N, K, bits, group, M, workspace, workspace_bytes, false);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = qmm_prepare_internal(x, ldx, M, K, bits, PREP_PLAIN, nullptr, 0, nullptr, 0.f, workspace, s);
  if (st) return st;
  return qmm_run_internal(wq, scales, biases, N, K, bits, M, residual ? RUN_RESIDUAL : RUN_STORE, y, ldy,
                          residual, ldr, nullptr, 0, 0.f, nullptr, nullptr, nullptr, workspace, s);
}

static int check_head_outputs(float temperature, float* logits, int ldl, int V) {
  if (!(temperature >= 0.f) || std::isinf(temperature)) return fail(SV_EINVAL, "temperature must be finite and >= 0");
  if (!logits) return fail(SV_EINVAL, "logits must be non-null");
  if (ldl < V) return fail(SV_EINVAL, "ldl must be >= V");
  if (!aligned(logits, 4)) return fail(SV_EINVAL, "misaligned logits");
  return SV_OK;
}

int sv_lm_head_run(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int V, int K, int bits,
                   int group, int M, float temperature, float* logits, int ldl, float* row_max, float* row_sumexp,
                   int32_t* row_argmax, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_run(wq, scales, biases, V, K, bits, group, M, workspace, workspace_bytes, true);
  if (st) return st;
  st = check_head_outputs(temperature, logits, ldl, V);
  if (st) return st;
  return qmm_run_internal(wq, scales, biases, V, K, bits, M, RUN_LOGITS, nullptr, 0, nullptr, 0, logits, ldl,
                          temperature, row_max, row_sumexp, row_argmax, workspace, static_cast<cudaStream_t>(stream));
}

int sv_lm_head_verify(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int V, int K, int bits,
                      int group, const uint16_t* x, int ldx, int M, float temperature, float* logits, int ldl,
                      float* row_max, float* row_sumexp, int32_t* row_argmax, void* workspace,
                      size_t workspace_bytes, void* stream) {
  int st = check_weight(wq, scales, biases, V, K, bits, group, M);
  if (st) return st;
  st = check_prepare(x, ldx, M, K, bits, PREP_PLAIN, nullptr, 0, workspace);
  if (st) return st;
  st = check_head_outputs(temperature, logits, ldl, V);
  if (st) return st;
  st = check_run(wq, scales, biases, V, K, bits, group, M, workspace, workspace_bytes, true);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = qmm_prepare_internal(x, ldx, M, K, bits, PREP_PLAIN, nullptr, 0, nullptr, 0.f, workspace, s);
  if (st) return st;
  return qmm_run_internal(wq, scales, biases, V, K, bits, M, RUN_LOGITS, nullptr, 0, nullptr, 0, logits, ldl,
                          temperature, row_max, row_sumexp, row_argmax, workspace, s);
}

const char* sv_status_string(int status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_EINVAL: return "invalid argument";
    case SV_EUNSUPPORTED: return "unsupported";
    case SV_ECUDA: return "CUDA error";
    case SV_ETIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

const char* sv_last_error(void) { return g_last; }

int sv_version(void) { return 100; }

int sv_selftest_bounded_wait(unsigned int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000u) return fail(SV_EINVAL, "limit_us must be in [1, 1e6] (got %u)", limit_us);
  cudaError_t e = launch_wait_selftest(limit_us, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return SV_OK;
}

int sv_device_error(unsigned int* bits) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  unsigned int v = 0;
  e = read_and_clear_error_word(&v);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (bits) *bits = v;
  if (v) return fail(SV_ETIMEOUT, "device error bits 0x%x", v);
  return SV_OK;
}

// ---------------------------------------------------------------- accept
}  // extern "C"

namespace sv {

static int accept_chunks(int V) {
  int nb = V / 2048;
  return nb < 1 ? 1 : (nb > 64 ? 64 : nb);
}

// Accept scratch relative to the workspace base: per-request counters in the
// zero prefix, chunk sums after it, then (only when the caller passes no row
// statistics) the statistics of every row.
static size_t accept_sums_offset() { return COUNTER_BYTES; }
static size_t accept_stats_offset(int B) { return COUNTER_BYTES + align256((size_t)B * 64 * 2 * 8); }
// per logits row: truncation key, tie index and kept mass of the target
static size_t accept_trunc_offset(int B, int rows) { return accept_stats_offset(B) + align256((size_t)rows * 12); }
size_t accept_bytes(int B, int rows) { return accept_trunc_offset(B, rows) + align256((size_t)rows * 12); }

int accept_internal(int B, const int32_t* offs, const float* logits, int ldl, const float* row_max,
                    const float* row_sumexp, const int32_t* row_argmax, const float* q, int ldq, const int32_t* draft,
                    int V, float temperature, const float* u, int32_t* out_len, int32_t* out_tokens, void* ws,
                    cudaStream_t s, int top_k, float top_p) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  const int rows = offs[B];
  AcceptParams p;
  memset(&p, 0, sizeof(p));
  for (int b = 0; b <= B; ++b) p.offs[b] = offs[b];
  p.logits = logits;
  p.ldl = ldl;
  if (!row_max && !row_argmax) {
    float* smax = reinterpret_cast<float*>(base + accept_stats_offset(B));
    float* ssum = smax + rows;
    int32_t* sarg = reinterpret_cast<int32_t*>(ssum + rows);
    cudaError_t e = launch_row_stats(logits, ldl, rows, V, temperature, smax, ssum, sarg, s);
    if (e != cudaSuccess) return cuda_fail(e, "row stats launch");
    p.row_max = smax;
    p.row_sumexp = ssum;
    p.row_argmax = sarg;
  } else {
    p.row_max = row_max;
    p.row_sumexp = row_sumexp;
    p.row_argmax = row_argmax;
  }
  if (temperature > 0.f && ((top_k > 0 && top_k < V) || top_p < 1.f)) {
    // truncation bounds of every row's target before the accept decisions
    uint8_t* tb = base + accept_trunc_offset(B, rows);
    SelectArgs a;
    memset(&a, 0, sizeof(a));
    a.x = logits;
    a.ldx = ldl;
    a.V = V;
    a.mode = SEL_LOGITS;
    a.row_max = p.row_max;
    a.temperature = temperature;
    a.top_k = top_k;
    a.top_p = top_p;
    a.out_key = reinterpret_cast<uint32_t*>(tb);
    a.out_idx = reinterpret_cast<int32_t*>(tb + 4 * (size_t)rows);
    a.out_norm = reinterpret_cast<float*>(tb + 8 * (size_t)rows);
    cudaError_t e = launch_select(a, rows, s);
    if (e != cudaSuccess) return cuda_fail(e, "truncation launch");
    p.tkey = a.out_key;
    p.tidx = a.out_idx;
    p.tnorm = a.out_norm;
  }
  p.q = q;
  p.ldq = ldq;
  p.draft = draft;
  p.V = V;
  p.temperature = temperature;
  p.u = u;
  p.out_len = out_len;
  p.out_tokens = out_tokens;
  p.chunk_sums = reinterpret_cast<double*>(base + accept_sums_offset());
  p.counters = reinterpret_cast<int*>(base + ACC_CTR_OFF);
  p.nb = accept_chunks(V);
  cudaError_t e = launch_accept(p, B, s);
  if (e != cudaSuccess) return cuda_fail(e, "accept launch");
  return SV_OK;
}

int check_accept(int B, const int32_t* row_offsets, const float* logits, int ldl, const float* row_max,
                 const float* row_sumexp, const int32_t* row_argmax, const float* q, int ldq, const int32_t* draft,
                 int V, float temperature, const float* u, int32_t* out_len, int32_t* out_tokens) {
  if (B < 1 || B > MAX_BATCH) return fail(SV_EINVAL, "B must be in [1, 256] (got %d)", B);
  if (!row_offsets) return fail(SV_EINVAL, "row_offsets must be non-null");
  if (row_offsets[0] != 0) return fail(SV_EINVAL, "row_offsets[0] must be 0");
  int max_m = 0;
  for (int b = 0; b < B; ++b) {
    const int mb = row_offsets[b + 1] - row_offsets[b] - 1;
    if (mb < 0 || mb > 31) return fail(SV_EINVAL, "request %d has m = %d (must be in [0, 31])", b, mb);
    max_m = mb > max_m ? mb : max_m;
  }
  if (V < 2 || V > (1 << 24)) return fail(SV_EINVAL, "V must be in [2, 2^24] (got %d)", V);
  if (!(temperature >= 0.f) || std::isinf(temperature)) return fail(SV_EINVAL, "temperature must be finite and >= 0");
  const bool sampled = temperature > 0.f;
  if (!logits || !out_len || !out_tokens) return fail(SV_EINVAL, "null pointer argument");
  if (max_m > 0 && !draft) return fail(SV_EINVAL, "draft must be non-null when m > 0");
  if (ldl < V) return fail(SV_EINVAL, "ldl must be >= V");
  if (sampled && (!u || (max_m > 0 && !q))) return fail(SV_EINVAL, "sampled accept needs q and u");
  if (sampled && max_m > 0 && ldq < V) return fail(SV_EINVAL, "ldq must be >= V");
  const int given = (row_max != nullptr) + (row_sumexp != nullptr) + (row_argmax != nullptr);
  const bool ok_stats = given == 0 || given == 3 || (!sampled && row_max && row_argmax && !row_sumexp);
  if (!ok_stats) return fail(SV_EINVAL, "row statistics must be all given or all NULL");
  return SV_OK;
}

}  // namespace sv

extern "C" {

size_t sv_accept_workspace_bytes(int B, int max_rows) {
  if (B < 1 || B > MAX_BATCH || max_rows < 1) return 0;
  return accept_bytes(B, max_rows);
}

int sv_spec_accept_batched(int B, const int32_t* row_offsets, const float* logits, int ldl, const float* row_max,
                           const float* row_sumexp, const int32_t* row_argmax, const float* q, int ldq,
                           const int32_t* draft, int V, float temperature, const float* u, int32_t* out_len,
                           int32_t* out_tokens, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_accept(B, row_offsets, logits, ldl, row_max, row_sumexp, row_argmax, q, ldq, draft, V, temperature,
                        u, out_len, out_tokens);
  if (st) return st;
  if (!workspace) return fail(SV_EINVAL, "workspace must be non-null");
  if (!aligned(workspace, 256)) return fail(SV_EINVAL, "workspace must be 256-byte aligned");
  const size_t need = accept_bytes(B, row_offsets[B]);
  if (workspace_bytes < need) return fail(SV_EINVAL, "workspace too small: %zu < %zu", workspace_bytes, need);
  return accept_internal(B, row_offsets, logits, ldl, row_max, row_sumexp, row_argmax, q, ldq, draft, V,
                         temperature, u, out_len, out_tokens, workspace, static_cast<cudaStream_t>(stream), 0, 1.f);
}

int sv_spec_accept_truncated(int B, const int32_t* row_offsets, const float* logits, int ldl, const float* row_max,
                             const float* row_sumexp, const int32_t* row_argmax, const float* q, int ldq,
                             const int32_t* draft, int V, float temperature, const float* u, int top_k, float top_p,
                             int32_t* out_len, int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                             void* stream) {
  int st = check_accept(B, row_offsets, logits, ldl, row_max, row_sumexp, row_argmax, q, ldq, draft, V, temperature,
                        u, out_len, out_tokens);
  if (st) return st;
  if (top_k < 0) return fail(SV_EINVAL, "top_k must be >= 0 (0 = no limit)");
  if (!(top_p > 0.f && top_p <= 1.f)) return fail(SV_EINVAL, "top_p must be in (0, 1]");
  if (!workspace) return fail(SV_EINVAL, "workspace must be non-null");
  if (!aligned(workspace, 256)) return fail(SV_EINVAL, "workspace must be 256-byte aligned");
  const size_t need = accept_bytes(B, row_offsets[B]);
  if (workspace_bytes < need) return fail(SV_EINVAL, "workspace too small: %zu < %zu", workspace_bytes, need);
  return accept_internal(B, row_offsets, logits, ldl, row_max, row_sumexp, row_argmax, q, ldq, draft, V,
                         temperature, u, out_len, out_tokens, workspace, static_cast<cudaStream_t>(stream), top_k,
                         top_p);
}

int sv_truncate_probs(const float* probs, int ldp, float* out, int ldo, int rows, int V, int top_k, float top_p,
                      void* stream) {
  if (rows < 1 || rows > 65535) return fail(SV_EINVAL, "rows must be in [1, 65535]");
  if (V < 1 || V > (1 << 24)) return fail(SV_EINVAL, "V must be in [1, 2^24]");
  if (!probs || !out) return fail(SV_EINVAL, "probs and out must be non-null");
  if (ldp < V || ldo < V) return fail(SV_EINVAL, "strides must be >= V");
  if (!aligned(probs, 4) || !aligned(out, 4)) return fail(SV_EINVAL, "misaligned rows");
  if (top_k < 0) return fail(SV_EINVAL, "top_k must be >= 0 (0 = no limit)");
  if (!(top_p > 0.f && top_p <= 1.f)) return fail(SV_EINVAL, "top_p must be in (0, 1]");
  if (out != probs && ldo == ldp) {
    const char* a = reinterpret_cast<const char*>(probs);
    const char* b = reinterpret_cast<const char*>(out);
    const size_t span = ((size_t)(rows - 1) * ldp + V) * 4;
    if (a < b + span && b < a + span) return fail(SV_EINVAL, "out must equal probs or not overlap it");
  }
  SelectArgs a;
  memset(&a, 0, sizeof(a));
  a.x = probs;
  a.ldx = ldp;
  a.y = out;
  a.ldy = ldo;
  a.V = V;
  a.mode = SEL_PROBS;
  a.top_k = top_k;
  a.top_p = top_p;
  cudaError_t e = launch_select(a, rows, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "truncation launch");
  return SV_OK;
}

int sv_logprobs(const float* logits, int ldl, int rows, int V, float temperature, const int32_t* chosen, int top_n,
                float* chosen_logprob, int32_t* top_ids, float* top_logprobs, void* stream) {
  if (rows < 1 || rows > 65535) return fail(SV_EINVAL, "rows must be in [1, 65535]");
  if (V < 1 || V > (1 << 24)) return fail(SV_EINVAL, "V must be in [1, 2^24]");
  if (!logits || ldl < V) return fail(SV_EINVAL, "logits must be non-null with ldl >= V");
  if (!(temperature >= 0.f) || std::isinf(temperature)) return fail(SV_EINVAL, "temperature must be finite and >= 0");
  if (top_n < 0 || top_n > 32) return fail(SV_EINVAL, "top_n must be in [0, 32]");
  if (top_n > 0 && (!top_ids || !top_logprobs)) return fail(SV_EINVAL, "top_n > 0 needs top_ids and top_logprobs");
  if (chosen && !chosen_logprob) return fail(SV_EINVAL, "chosen needs chosen_logprob");
  if (!chosen && top_n == 0) return SV_OK;
  SelectArgs a;
  memset(&a, 0, sizeof(a));
  a.x = logits;
  a.ldx = ldl;
  a.V = V;
  a.mode = SEL_TOPN;
  a.temperature = temperature;
  a.chosen = chosen;
  a.chosen_lp = chosen_logprob;
  a.top_ids = top_ids;
  a.top_lp = top_logprobs;
  a.top_n = top_n;
  cudaError_t e = launch_select(a, rows, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "logprobs launch");
  return SV_OK;
}

int sv_spec_accept(const float* logits, int ldl, const float* row_max, const float* row_sumexp,
                   const int32_t* row_argmax, const float* q, int ldq, const int32_t* draft, int m, int V,
                   float temperature, const float* u, int32_t* out_len, int32_t* out_tokens, void* workspace,
                   size_t workspace_bytes, void* stream) {
  if (m < 0 || m > 31) return fail(SV_EINVAL, "m must be in [0, 31] (got %d)", m);
  const int32_t offs[2] = {0, m + 1};
  return sv_spec_accept_batched(1, offs, logits, ldl, row_max, row_sumexp, row_argmax, q, ldq, draft, V,
                                temperature, u, out_len, out_tokens, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- philox
int sv_philox_uniforms(uint64_t seed, uint64_t subsequence, uint64_t offset, int n, float* out, void* stream) {
  if (n < 0) return fail(SV_EINVAL, "n must be >= 0");
  if (n == 0) return SV_OK;
  if (!out) return fail(SV_EINVAL, "out must be non-null");
  cudaError_t e = launch_philox(seed, subsequence, offset, n, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "philox launch");
  return SV_OK;
}

// ------------------------------------------------------------------ glue
static int check_rows(int M, int H) {
  if (M < 1 || M > 4096) return fail(SV_EINVAL, "M must be in [1, 4096] (got %d)", M);
  if (H < 1) return fail(SV_EINVAL, "row length must be >= 1 (got %d)", H);
  return SV_OK;
}

int sv_rmsnorm(const uint16_t* x, int ldx, int M, int H, const uint16_t* weight, float eps, uint16_t* y, int ldy,
               void* stream) {
  int st = check_rows(M, H);
  if (st) return st;
  if (!x || !y) return fail(SV_EINVAL, "x and y must be non-null");
  if (ldx < H || ldy < H) return fail(SV_EINVAL, "strides must be >= H");
  if (!(eps >= 0.f)) return fail(SV_EINVAL, "eps must be >= 0");
  cudaError_t e = launch_rmsnorm(reinterpret_cast<const __nv_bfloat16*>(x), ldx, M, H,
                                 reinterpret_cast<const __nv_bfloat16*>(weight), eps,
                                 reinterpret_cast<__nv_bfloat16*>(y), ldy, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm launch");
  return SV_OK;
}

int sv_residual_add(uint16_t* h, int ldh, const uint16_t* t, int ldt, int M, int H, void* stream) {
  int st = check_rows(M, H);
  if (st) return st;
  if (!h || !t) return fail(SV_EINVAL, "h and t must be non-null");
  if (ldh < H || ldt < H) return fail(SV_EINVAL, "strides must be >= H");
  cudaError_t e = launch_residual(reinterpret_cast<__nv_bfloat16*>(h), ldh, reinterpret_cast<const __nv_bfloat16*>(t),
                                  ldt, M, H, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "residual launch");
  return SV_OK;
}

int sv_swiglu(const uint16_t* g, int ldg, const uint16_t* u, int ldu, int M, int I, uint16_t* s, int lds,
              void* stream) {
  int st = check_rows(M, I);
  if (st) return st;
  if (!g || !u || !s) return fail(SV_EINVAL, "g, u and s must be non-null");
  if (ldg < I || ldu < I || lds < I) return fail(SV_EINVAL, "strides must be >= I");
  cudaError_t e = launch_swiglu(reinterpret_cast<const __nv_bfloat16*>(g), ldg,
                                reinterpret_cast<const __nv_bfloat16*>(u), ldu, M, I,
                                reinterpret_cast<__nv_bfloat16*>(s), lds, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "swiglu launch");
  return SV_OK;
}

}  // extern "C"
