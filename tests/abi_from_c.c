/* A plain C caller of the library: no Python in the process.
 *
 *   abi_from_c host               host-side checks only (no device is touched)
 *   abi_from_c gpu IN OUT         one verify step on device memory it allocates itself
 *
 * The gpu mode reads the inputs a test wrote to IN (little-endian):
 *   int32 N, K, bits, M, V, Kh, m, seed;  float T
 *   uint32 wq[N][K*bits/32]; uint16 scales[N][K/64], biases[N][K/64]; uint16 x[M][K]   (bf16 bits)
 *   uint32 hwq[V][Kh*bits/32]; uint16 hscales[V][Kh/64], hbiases[V][Kh/64]; uint16 hx[m+1][Kh]
 *   float q[m][V]; int32 draft[m]
 * runs sv_qmm_verify, sv_lm_head_verify, sv_philox_uniforms (subsequence 0,
 * offset 0) and sv_spec_accept on the head's rows, and writes to OUT:
 *   int32 status[4]; uint16 y[M][N]; float logits[m+1][V], row_max[m+1], row_sumexp[m+1];
 *   int32 row_argmax[m+1]; float u[m+1]; int32 out_len, out_tokens[m+1]
 * Exit status 0 when every call returned SV_OK and the device error word is clear. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "specverify.h"

static int fail(const char* what) {
  fprintf(stderr, "abi_from_c: %s\n", what);
  return 1;
}

static int host_checks(void) {
  if (!sv_status_string(SV_OK) || !sv_status_string(SV_EINVAL)) return fail("status strings");
  if (sv_version() <= 0) return fail("version");
  /* unit-packed size: 16 tile rows x 2 chunks of (64 x 512 code bytes + 64 x 8 scales and biases) */
  if (sv_qmm_pack_bytes(1000, 1024, 8) != (size_t)16 * 2 * (64 * 512 + 2 * 64 * 8 * 2)) return fail("packed size");
  /* rejected on the host, before any device work: bad width, bad group, null
   * weights.  The other pointers are aligned stand-ins that validation only
   * inspects (the calls are refused before anything could read them). */
  const uint32_t* wq = (const uint32_t*)(uintptr_t)16;
  const uint16_t* h16 = (const uint16_t*)(uintptr_t)16;
  uint16_t* y = (uint16_t*)(uintptr_t)16;
  void* ws = (void*)(uintptr_t)256;
  if (sv_qmm_verify(wq, h16, h16, 64, 512, 3, 64, h16, 512, 4, y, 64, NULL, 0, ws, 1 << 20, NULL) != SV_EUNSUPPORTED)
    return fail("3-bit codes not refused");
  if (sv_qmm_verify(wq, h16, h16, 64, 512, 8, 32, h16, 512, 4, y, 64, NULL, 0, ws, 1 << 20, NULL) != SV_EUNSUPPORTED)
    return fail("group 32 not refused");
  if (sv_qmm_verify(NULL, h16, h16, 64, 512, 8, 64, h16, 512, 4, y, 64, NULL, 0, ws, 1 << 20, NULL) != SV_EINVAL)
    return fail("null weights not refused");
  if (sv_philox_uniforms(1, 0, 0, -1, NULL, NULL) != SV_EINVAL) return fail("negative count not refused");
  /* the draft-cap controller is host-only: a flat cost curve and a high
   * acceptance rate pick the widest cap */
  double verify[8], draft[8];
  for (int i = 0; i < 8; ++i) {
    verify[i] = 1000.0;
    draft[i] = 0.0;
  }
  int cap = -1;
  double rate = 0.0;
  if (sv_best_cap(0.9, 7, verify, draft, 0.0, &cap, &rate) != SV_OK || cap != 7 || !(rate > 0.0))
    return fail("best cap on a flat curve");
  printf("host checks ok\n");
  return 0;
}

static void* read_all(const char* path, size_t* n) {
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  fseek(f, 0, SEEK_END);
  long len = ftell(f);
  fseek(f, 0, SEEK_SET);
  void* buf = malloc(len > 0 ? (size_t)len : 1);
  if (buf && fread(buf, 1, (size_t)len, f) != (size_t)len) {
    free(buf);
    buf = NULL;
  }
  fclose(f);
  *n = (size_t)len;
  return buf;
}

/* a device copy of `bytes` host bytes (NULL on failure) */
static void* to_device(const void* src, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) return NULL;
  if (bytes && cudaMemcpy(d, src, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

static int gpu_step(const char* in_path, const char* out_path) {
  size_t n_in = 0;
  unsigned char* in = (unsigned char*)read_all(in_path, &n_in);
  if (!in || n_in < 36) return fail("cannot read the input file");
  int hdr[8];
  float T;
  memcpy(hdr, in, sizeof hdr);
  memcpy(&T, in + 32, 4);
  const int N = hdr[0], K = hdr[1], bits = hdr[2], M = hdr[3], V = hdr[4], Kh = hdr[5], m = hdr[6], seed = hdr[7];
  const size_t b_wq = (size_t)N * K * bits / 8, b_sb = (size_t)N * (K / 64) * 2, b_x = (size_t)M * K * 2;
  const size_t b_hwq = (size_t)V * Kh * bits / 8, b_hsb = (size_t)V * (Kh / 64) * 2, b_hx = (size_t)(m + 1) * Kh * 2;
  const size_t b_q = (size_t)m * V * 4, b_d = (size_t)m * 4;
  const size_t need = 36 + b_wq + 2 * b_sb + b_x + b_hwq + 2 * b_hsb + b_hx + b_q + b_d;
  if (n_in != need) return fail("input file size does not match its header");
  const unsigned char* p = in + 36;
  void *wq = to_device(p, b_wq), *sc = to_device(p + b_wq, b_sb), *bi = to_device(p + b_wq + b_sb, b_sb);
  p += b_wq + 2 * b_sb;
  void* x = to_device(p, b_x);
  p += b_x;
  void *hwq = to_device(p, b_hwq), *hsc = to_device(p + b_hwq, b_hsb), *hbi = to_device(p + b_hwq + b_hsb, b_hsb);
  p += b_hwq + 2 * b_hsb;
  void* hx = to_device(p, b_hx);
  p += b_hx;
  void* q = to_device(p, b_q);
  void* dr = to_device(p + b_q, b_d);
  const int rows = m + 1;
  const size_t ws_q = sv_qmm_workspace_bytes(M, N, K, bits), ws_h = sv_lm_head_workspace_bytes(rows, V, Kh, bits);
  const size_t ws_a = sv_accept_workspace_bytes(1, rows);
  size_t ws_bytes = ws_q > ws_h ? ws_q : ws_h;
  if (ws_a > ws_bytes) ws_bytes = ws_a;
  void *y = NULL, *logits = NULL, *rmax = NULL, *rse = NULL, *ram = NULL, *u = NULL, *olen = NULL, *otok = NULL;
  void* ws = NULL;
  if (!wq || !sc || !bi || !x || !hwq || !hsc || !hbi || !hx || !q || !dr ||
      cudaMalloc(&y, (size_t)M * N * 2) != cudaSuccess || cudaMalloc(&logits, (size_t)rows * V * 4) != cudaSuccess ||
      cudaMalloc(&rmax, rows * 4) != cudaSuccess || cudaMalloc(&rse, rows * 4) != cudaSuccess ||
      cudaMalloc(&ram, rows * 4) != cudaSuccess || cudaMalloc(&u, rows * 4) != cudaSuccess ||
      cudaMalloc(&olen, 4) != cudaSuccess || cudaMalloc(&otok, rows * 4) != cudaSuccess ||
      cudaMalloc(&ws, ws_bytes) != cudaSuccess)
    return fail("device allocation");
  /* the workspaces start zeroed (the rule the header states for fresh workspaces) */
  if (cudaMemset(ws, 0, ws_bytes) != cudaSuccess) return fail("workspace clear");

  int st[4];
  st[0] = sv_qmm_verify((const uint32_t*)wq, (const uint16_t*)sc, (const uint16_t*)bi, N, K, bits, 64,
                        (const uint16_t*)x, K, M, (uint16_t*)y, N, NULL, 0, ws, ws_bytes, NULL);
  st[1] = sv_lm_head_verify((const uint32_t*)hwq, (const uint16_t*)hsc, (const uint16_t*)hbi, V, Kh, bits, 64,
                            (const uint16_t*)hx, Kh, rows, T, (float*)logits, V, (float*)rmax, (float*)rse,
                            (int32_t*)ram, ws, ws_bytes, NULL);
  st[2] = sv_philox_uniforms((uint64_t)seed, 0, 0, rows, (float*)u, NULL);
  st[3] = sv_spec_accept((const float*)logits, V, (const float*)rmax, (const float*)rse, (const int32_t*)ram,
                         (const float*)q, V, (const int32_t*)dr, m, V, T, (const float*)u, (int32_t*)olen,
                         (int32_t*)otok, ws, ws_bytes, NULL);
  if (cudaDeviceSynchronize() != cudaSuccess) return fail("device synchronize");
  unsigned int err_bits = 0;
  const int dev_status = sv_device_error(&err_bits);

  const size_t b_out = 16 + (size_t)M * N * 2 + (size_t)rows * V * 4 + 5 * (size_t)rows * 4 + 4;
  unsigned char* out = (unsigned char*)malloc(b_out);
  if (!out) return fail("host allocation");
  unsigned char* o = out;
  memcpy(o, st, 16);
  o += 16;
  int ok = cudaMemcpy(o, y, (size_t)M * N * 2, cudaMemcpyDeviceToHost) == cudaSuccess;
  o += (size_t)M * N * 2;
  ok &= cudaMemcpy(o, logits, (size_t)rows * V * 4, cudaMemcpyDeviceToHost) == cudaSuccess;
  o += (size_t)rows * V * 4;
  void* const small[4] = {rmax, rse, ram, u};
  for (int i = 0; i < 4; ++i, o += rows * 4) ok &= cudaMemcpy(o, small[i], rows * 4, cudaMemcpyDeviceToHost) == cudaSuccess;
  ok &= cudaMemcpy(o, olen, 4, cudaMemcpyDeviceToHost) == cudaSuccess;
  o += 4;
  ok &= cudaMemcpy(o, otok, rows * 4, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (!ok) return fail("copy back");
  FILE* f = fopen(out_path, "wb");
  if (!f || fwrite(out, 1, b_out, f) != b_out) return fail("cannot write the output file");
  fclose(f);
  for (int i = 0; i < 4; ++i)
    if (st[i] != SV_OK) {
      fprintf(stderr, "abi_from_c: call %d returned %s (%s)\n", i, sv_status_string(st[i]), sv_last_error());
      return 1;
    }
  if (dev_status != SV_OK || err_bits) return fail("device error word set");
  printf("gpu step ok\n");
  return 0;
}

int main(int argc, char** argv) {
  if (argc == 2 && !strcmp(argv[1], "host")) return host_checks();
  if (argc == 4 && !strcmp(argv[1], "gpu")) return gpu_step(argv[2], argv[3]);
  fprintf(stderr, "usage: abi_from_c host | abi_from_c gpu IN OUT\n");
  return 2;
}
