// One verify round of a dense quantized decoder, enqueued as a single call.
//
// mlx-dspark wiki page, "Architecture": the target runs [anchor] + m drafts
// through one forward and the accept step commits the longest accepted
// prefix.  The layer body is the plainest dense block (the pages give none):
//
//   a  = RMSNorm(h)                    fused into the preparation of qkv's input
//   qkv = a Wqkv^T                      q | k | v in one weight stream
//   h += q Wo^T                         q feeds o directly (no attention state)
//   a2 = RMSNorm(h)                    fused into the preparation of gate|up's input
//   gu = a2 Wgu^T                       gate | up in one weight stream
//   h += (silu(g) * u) Wdown^T          SwiGLU fused into the preparation of down's input
//
// then a = RMSNorm(h), the vocab head with its row statistics, and the accept
// step.  Every launch carries the programmatic-serialization attribute, so a
// projection's weight stream starts while the previous kernel drains; the
// whole sequence can be captured into one CUDA graph by the caller.
#include <algorithm>
#include <cstdio>
#include <cstring>

#include "sv_internal.h"
#include "sv_kernels.h"

namespace sv {

struct RoundLayout {
  size_t stats, qkv, gu, total;
};

static RoundLayout round_layout(const sv_model* md, int rows, bool& ok) {
  ok = false;
  RoundLayout L = {};
  const int K_h = md->hidden;
  const size_t qmm = std::max({qmm_bytes(rows, md->layers[0].qkv.N, K_h, false),
                               qmm_bytes(rows, md->hidden, md->q_dim, false),
                               qmm_bytes(rows, 2 * md->inter, K_h, false),
                               qmm_bytes(rows, md->hidden, md->inter, false),
                               qmm_bytes(rows, md->vocab, K_h, true)});
  if (qmm == 0) return L;
  const size_t acc = accept_bytes(rows, rows);
  size_t off = align256(std::max(qmm, acc));
  L.stats = off; off = align256(off + (size_t)rows * 12);
  L.qkv = off;   off = align256(off + (size_t)rows * md->layers[0].qkv.N * 2);
  L.gu = off;    off = align256(off + (size_t)rows * 2 * md->inter * 2);
  L.total = off;
  ok = true;
  return L;
}

static int check_proj(const sv_qweight& w, int N, int K, int bits, int M, const char* what, int layer) {
  int st = check_weight(w.wq, w.scales, w.biases, w.N, w.K, bits, 64, M);
  if (st) {
    char detail[256];
    snprintf(detail, sizeof(detail), "%s", sv_last_error());
    return fail(st, "layer %d %s: %s", layer, what, detail);
  }
  if ((N >= 0 && w.N != N) || w.K != K)
    return fail(SV_EINVAL, "layer %d %s: shape %dx%d, expected %dx%d", layer, what, w.N, w.K, N, K);
  return SV_OK;
}

static int check_model(const sv_model* md, int M) {
  if (!md || !md->layers) return fail(SV_EINVAL, "model and its layer array must be non-null");
  if (md->n_layers < 1) return fail(SV_EINVAL, "n_layers must be >= 1");
  if (md->bits != 4 && md->bits != 8) return fail(SV_EUNSUPPORTED, "bits must be 4 or 8");
  if (md->hidden < 1 || md->q_dim < 1 || md->inter < 1 || md->vocab < 2)
    return fail(SV_EINVAL, "model dimensions must be positive");
  if (!(md->rms_eps >= 0.f)) return fail(SV_EINVAL, "rms_eps must be >= 0");
  const int Nqkv = md->layers[0].qkv.N;
  if (Nqkv < md->q_dim) return fail(SV_EINVAL, "qkv must hold at least q_dim rows");
  for (int l = 0; l < md->n_layers; ++l) {
    const sv_layer& L = md->layers[l];
    int st;
    if ((st = check_proj(L.qkv, Nqkv, md->hidden, md->bits, M, "qkv", l))) return st;
    if ((st = check_proj(L.o, md->hidden, md->q_dim, md->bits, M, "o", l))) return st;
    if ((st = check_proj(L.gate_up, 2 * md->inter, md->hidden, md->bits, M, "gate_up", l))) return st;
    if ((st = check_proj(L.down, md->hidden, md->inter, md->bits, M, "down", l))) return st;
  }
  return check_proj(md->lm_head, md->vocab, md->hidden, md->bits, M, "lm_head", -1);
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t sv_round_workspace_bytes(const sv_model* model, int rows) {
  if (!model || !model->layers || model->n_layers < 1 || rows < 1 || rows > MAX_M) return 0;
  bool ok;
  RoundLayout L = round_layout(model, rows, ok);
  return ok ? L.total : 0;
}

int sv_verify_round(const sv_model* model, int B, const int32_t* row_offsets, uint16_t* hidden, int ldh,
                    float temperature, const float* q, int ldq, const int32_t* draft, const float* u, float* logits,
                    int ldl, int32_t* out_len, int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                    void* stream) {
  if (B < 1 || !row_offsets) return fail(SV_EINVAL, "B must be >= 1 with row offsets");
  const int M = row_offsets[B];
  if (M < 1 || M > MAX_M) return fail(M > MAX_M ? SV_EUNSUPPORTED : SV_EINVAL, "total rows %d not in [1, 32]", M);
  int st = check_model(model, M);
  if (st) return st;
  st = check_accept(B, row_offsets, logits, ldl, nullptr, nullptr, nullptr, q, ldq, draft, model->vocab, temperature,
                    u, out_len, out_tokens);
  if (st) return st;
  if (!hidden || ldh < model->hidden || !aligned(hidden, 2)) return fail(SV_EINVAL, "bad hidden-state buffer");
  if (!workspace || !aligned(workspace, 256)) return fail(SV_EINVAL, "workspace must be non-null, 256-byte aligned");
  bool ok;
  const RoundLayout L = round_layout(model, M, ok);
  if (!ok) return fail(SV_ECUDA, "no CUDA device");
  if (workspace_bytes < L.total) return fail(SV_EINVAL, "workspace too small: %zu < %zu", workspace_bytes, L.total);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint16_t* qkv = reinterpret_cast<uint16_t*>(base + L.qkv);
  uint16_t* gu = reinterpret_cast<uint16_t*>(base + L.gu);
  float* rmax = reinterpret_cast<float*>(base + L.stats);
  float* rsum = rmax + M;
  int32_t* rarg = reinterpret_cast<int32_t*>(rsum + M);
  const int H = model->hidden, Dq = model->q_dim, I = model->inter, bits = model->bits;
  const int Nqkv = model->layers[0].qkv.N;
  const float eps = model->rms_eps;
#define SV_TRY(x)            \
  do {                       \
    int st_ = (x);           \
    if (st_) return st_;     \
  } while (0)
  for (int l = 0; l < model->n_layers; ++l) {
    const sv_layer& W = model->layers[l];
    SV_TRY(qmm_prepare_internal(hidden, ldh, M, H, bits, PREP_RMSNORM, nullptr, 0, nullptr, eps, workspace, s));
    SV_TRY(qmm_run_internal(W.qkv.wq, W.qkv.scales, W.qkv.biases, Nqkv, H, bits, M, EPI_BF16, qkv, Nqkv, nullptr, 0,
                            nullptr, 0, 0.f, nullptr, nullptr, nullptr, workspace, s));
    SV_TRY(qmm_prepare_internal(qkv, Nqkv, M, Dq, bits, PREP_PLAIN, nullptr, 0, nullptr, 0.f, workspace, s));
    SV_TRY(qmm_run_internal(W.o.wq, W.o.scales, W.o.biases, H, Dq, bits, M, EPI_BF16_RESIDUAL, hidden, ldh, hidden,
                            ldh, nullptr, 0, 0.f, nullptr, nullptr, nullptr, workspace, s));
    SV_TRY(qmm_prepare_internal(hidden, ldh, M, H, bits, PREP_RMSNORM, nullptr, 0, nullptr, eps, workspace, s));
    SV_TRY(qmm_run_internal(W.gate_up.wq, W.gate_up.scales, W.gate_up.biases, 2 * I, H, bits, M, EPI_BF16, gu, 2 * I,
                            nullptr, 0, nullptr, 0, 0.f, nullptr, nullptr, nullptr, workspace, s));
    SV_TRY(qmm_prepare_internal(gu, 2 * I, M, I, bits, PREP_SWIGLU, gu + I, 2 * I, nullptr, 0.f, workspace, s));
    SV_TRY(qmm_run_internal(W.down.wq, W.down.scales, W.down.biases, H, I, bits, M, EPI_BF16_RESIDUAL, hidden, ldh,
                            hidden, ldh, nullptr, 0, 0.f, nullptr, nullptr, nullptr, workspace, s));
  }
  SV_TRY(qmm_prepare_internal(hidden, ldh, M, H, bits, PREP_RMSNORM, nullptr, 0, nullptr, eps, workspace, s));
  SV_TRY(qmm_run_internal(model->lm_head.wq, model->lm_head.scales, model->lm_head.biases, model->vocab, H, bits, M,
                          EPI_LOGITS, nullptr, 0, nullptr, 0, logits, ldl, temperature, rmax, rsum, rarg, workspace,
                          s));
  SV_TRY(accept_internal(B, row_offsets, logits, ldl, rmax, temperature > 0.f ? rsum : nullptr, rarg, q, ldq, draft,
                         model->vocab, temperature, u, out_len, out_tokens, workspace, s));
#undef SV_TRY
  return SV_OK;
}

}  // extern "C"
