// One verify round of a dense quantized decoder, enqueued as a single call.
//
// mlx-dspark wiki page, "Architecture": the target runs [anchor] + m drafts
// through one forward and the accept step commits the longest accepted
// prefix.  The layer body is the plainest dense block (the pages give none):
//
//   qkv = RMSNorm(h) Wqkv^T            q | k | v in one weight stream
//   h  += q Wo^T                        q feeds o directly (no attention state)
//   gu  = RMSNorm(h) Wgu^T              gate / up rows interleaved in 64-row blocks
//   h  += (silu(gate) * up) Wdown^T
//
// then logits = RMSNorm(h) Wlm^T with row statistics, and the accept step.
// All 4 * layers + 1 projections run as the phases of one persistent launch:
// each phase's epilogue prepares the next phase's input (the RMSNorm row scale
// is applied to the consuming projection's output), so nothing runs between
// projections but a grid-wide barrier, behind which the next weights already
// stream.  Launches: input preparation, the phases, the row-statistics merge,
// the accept step.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "sv_internal.h"
#include "sv_kernels.h"

namespace sv {

struct RoundLayout {
  Layout ws;
  size_t stats, qkv, gu, pair, total;
  int grid;
};

static bool round_layout(const sv_model* md, int rows, RoundLayout& R) {
  const int MP = 8 * ((rows + 7) / 8);
  R.grid = stream_max_grid(md->bits, MP);
  if (R.grid <= 0) return false;
  const int K_cap = std::max({md->hidden, md->q_dim, md->inter});
  const int vocab_tiles = (md->vocab + BN - 1) / BN;
  R.ws = workspace_layout(rows, K_cap, R.grid, vocab_tiles, 2);
  size_t off = align256(std::max(R.ws.total, accept_bytes(rows, rows)));
  R.stats = off; off = align256(off + (size_t)rows * 12);
  R.qkv = off;   off = align256(off + (size_t)rows * md->layers[0].qkv.N * 2);
  R.gu = off;    off = align256(off + (size_t)rows * 2 * md->inter * 2);
  R.pair = off;  off = align256(off + (size_t)((md->inter + BN - 1) / BN) * BN * MP * 4);
  R.total = off;
  return true;
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
  if (w.packed && !aligned(w.packed, 16)) return fail(SV_EINVAL, "layer %d %s: packed weight not 16-byte aligned", layer, what);
  return SV_OK;
}

static int check_model(const sv_model* md, int M) {
  if (!md || !md->layers) return fail(SV_EINVAL, "model and its layer array must be non-null");
  if (md->n_layers < 1) return fail(SV_EINVAL, "n_layers must be >= 1");
  if (4 * md->n_layers + 1 > MAX_PHASES) return fail(SV_EUNSUPPORTED, "at most %d layers", (MAX_PHASES - 1) / 4);
  if (!bits_supported(md->bits)) return fail(SV_EUNSUPPORTED, "bits must be 2, 4 or 8");
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

static void set_phase(Phase& ph, const sv_qweight& w, int kind, int in_buf, int out_buf) {
  memset(&ph, 0, sizeof(ph));
  ph.wq = reinterpret_cast<const uint8_t*>(w.wq);
  ph.packed = static_cast<const uint8_t*>(w.packed);
  ph.scales = w.scales;
  ph.biases = w.biases;
  ph.N = w.N;
  ph.K = w.K;
  ph.kind = kind;
  ph.in_buf = in_buf;
  ph.out_buf = out_buf;
}

// A plan holds the tensor maps (weights, scales, biases) of every projection
// of a model, in phase order, in device memory: the persistent kernel reads a
// phase's maps from there, so they are encoded once per model instead of once
// per round.  The host remembers which model each plan was built for.
static uint64_t mix(uint64_t h, uint64_t v) { return (h ^ v) * 0x100000001b3ull; }  // FNV-1a over 64-bit words
static uint64_t hash_qweight(uint64_t h, const sv_qweight& w) {
  h = mix(h, reinterpret_cast<uintptr_t>(w.wq));
  h = mix(h, reinterpret_cast<uintptr_t>(w.scales));
  h = mix(h, reinterpret_cast<uintptr_t>(w.biases));
  return mix(h, ((uint64_t)(uint32_t)w.N << 32) | (uint32_t)w.K);
}
static uint64_t model_fingerprint(const sv_model* md) {
  uint64_t h = 0xcbf29ce484222325ull;
  const int dims[6] = {md->n_layers, md->hidden, md->q_dim, md->inter, md->vocab, md->bits};
  for (int d : dims) h = mix(h, (uint32_t)d);
  for (int l = 0; l < md->n_layers; ++l) {
    const sv_layer& L = md->layers[l];
    h = hash_qweight(hash_qweight(hash_qweight(hash_qweight(h, L.qkv), L.o), L.gate_up), L.down);
  }
  return hash_qweight(h, md->lm_head);
}
static std::mutex g_plan_mu;
static std::unordered_map<const void*, uint64_t> g_plans;

static size_t plan_bytes_for(const sv_model* md) { return (size_t)(4 * md->n_layers + 1) * 3 * sizeof(CUtensorMap); }

}  // namespace sv

using namespace sv;

extern "C" {

size_t sv_round_workspace_bytes(const sv_model* model, int rows) {
  if (!model || !model->layers || model->n_layers < 1 || rows < 1 || rows > MAX_M) return 0;
  RoundLayout R;
  return round_layout(model, rows, R) ? R.total : 0;
}

size_t sv_round_plan_bytes(const sv_model* model) {
  if (!model || !model->layers || model->n_layers < 1 || 4 * model->n_layers + 1 > MAX_PHASES) return 0;
  return plan_bytes_for(model);
}

int sv_round_plan_init(const sv_model* model, void* plan, size_t plan_bytes) {
  int st = check_model(model, 1);
  if (st) return st;
  if (!plan || !aligned(plan, 256)) return fail(SV_EINVAL, "plan must be non-null and 256-byte aligned");
  const size_t need = plan_bytes_for(model);
  if (plan_bytes < need) return fail(SV_EINVAL, "plan too small: %zu < %zu", plan_bytes, need);
  std::vector<CUtensorMap> maps((size_t)(4 * model->n_layers + 1) * 3);
  size_t n = 0;
  auto add = [&](const sv_qweight& w) {
    CUtensorMap m3[3];
    int r = encode_weight_maps(m3, w.wq, w.scales, w.biases, w.N, w.K, model->bits);
    for (int i = 0; i < 3; ++i) maps[n++] = m3[i];
    return r;
  };
  for (int l = 0; l < model->n_layers; ++l) {
    const sv_layer& L = model->layers[l];
    if ((st = add(L.qkv)) || (st = add(L.o)) || (st = add(L.gate_up)) || (st = add(L.down))) return st;
  }
  if ((st = add(model->lm_head))) return st;
  cudaError_t e = cudaMemcpy(plan, maps.data(), need, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "copy plan to the device");
  std::lock_guard<std::mutex> lock(g_plan_mu);
  g_plans[plan] = model_fingerprint(model);
  return SV_OK;
}

int sv_verify_round(const sv_model* model, const void* plan, int B, const int32_t* row_offsets, uint16_t* hidden, int ldh,
                    float temperature, const float* q, int ldq, const int32_t* draft, const float* u, float* logits,
                    int ldl, int32_t* out_len, int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                    void* stream, void* event_start, void* event_stop, void* accept_wait_event) {
  if (B < 1 || !row_offsets) return fail(SV_EINVAL, "B must be >= 1 with row offsets");
  const int M = row_offsets[B];
  if (M < 1 || M > MAX_M) return fail(M > MAX_M ? SV_EUNSUPPORTED : SV_EINVAL, "total rows %d not in [1, 32]", M);
  int st = check_model(model, M);
  if (st) return st;
  st = check_accept(B, row_offsets, logits, ldl, nullptr, nullptr, nullptr, q, ldq, draft, model->vocab, temperature,
                    u, out_len, out_tokens);
  if (st) return st;
  if (!hidden || ldh < model->hidden || !aligned(hidden, 2)) return fail(SV_EINVAL, "bad hidden-state buffer");
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    auto it = g_plans.find(plan);
    if (!plan || it == g_plans.end() || it->second != model_fingerprint(model))
      return fail(SV_EINVAL, "plan was not built for this model (sv_round_plan_init)");
  }
  if (!workspace || !aligned(workspace, 256)) return fail(SV_EINVAL, "workspace must be non-null, 256-byte aligned");
  RoundLayout R;
  if (!round_layout(model, M, R)) return fail(SV_ECUDA, "no CUDA device");
  if (workspace_bytes < R.total) return fail(SV_EINVAL, "workspace too small: %zu < %zu", workspace_bytes, R.total);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* qkv = reinterpret_cast<__nv_bfloat16*>(base + R.qkv);
  __nv_bfloat16* gu = reinterpret_cast<__nv_bfloat16*>(base + R.gu);
  __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(hidden);
  float* rmax = reinterpret_cast<float*>(base + R.stats);
  float* rsum = rmax + M;
  int32_t* rarg = reinterpret_cast<int32_t*>(rsum + M);
  const int bits = model->bits, Nqkv = model->layers[0].qkv.N, I = model->inter;

  static thread_local StreamParams p;  // about 22 KB: kept off the stack
  stream_params_init(p, workspace, R.ws, M, R.grid, model->rms_eps);
  p.maps = static_cast<const CUtensorMap*>(plan);
  p.pair_words = reinterpret_cast<float*>(base + R.pair);
  int n = 0;
  for (int l = 0; l < model->n_layers; ++l) {
    const sv_layer& W = model->layers[l];
    Phase& a = p.ph[n++];
    set_phase(a, W.qkv, PH_STORE, 0, 1);
    a.y = qkv;
    a.ldy = Nqkv;
    a.prep_tiles = model->q_dim / BN;
    Phase& o = p.ph[n++];
    set_phase(o, W.o, PH_RESID, 1, 0);
    o.y = h;
    o.res = h;
    o.ldy = o.ldr = ldh;
    Phase& g = p.ph[n++];
    set_phase(g, W.gate_up, PH_GATEUP, 0, 1);
    g.y = gu;
    g.ldy = 2 * I;
    g.half = I;
    Phase& d = p.ph[n++];
    set_phase(d, W.down, PH_RESID, 1, 0);
    d.y = h;
    d.res = h;
    d.ldy = d.ldr = ldh;
  }
  set_phase(p.ph[n++], model->lm_head, PH_LOGITS, 0, -1);
  p.n_phases = n;
  p.logits = logits;
  p.ldl = ldl;
  p.inv_temp = temperature > 0.f ? 1.f / temperature : 0.f;

  st = prepare_into(hidden, ldh, M, model->hidden, bits, PREP_RMSNORM, nullptr, 0, nullptr, model->rms_eps, p.act[0],
                    s);
  if (st) return st;
  cudaError_t e;
  if (event_start && (e = cudaEventRecord(static_cast<cudaEvent_t>(event_start), s)) != cudaSuccess)
    return cuda_fail(e, "record event_start");
  e = launch_stream(bits, p, s);
  if (e != cudaSuccess) return cuda_fail(e, "verify-round launch");
  if (event_stop && (e = cudaEventRecord(static_cast<cudaEvent_t>(event_stop), s)) != cudaSuccess)
    return cuda_fail(e, "record event_stop");
  e = launch_lmhead_finalize(p.tile_stats, (model->vocab + BN - 1) / BN, p.MP, M, p.inv_temp, rmax, rsum, rarg, s);
  if (e != cudaSuccess) return cuda_fail(e, "lm_head finalize launch");
  if (accept_wait_event && (e = cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(accept_wait_event), 0)) != cudaSuccess)
    return cuda_fail(e, "wait for accept_wait_event");
  return accept_internal(B, row_offsets, logits, ldl, rmax, temperature > 0.f ? rsum : nullptr, rarg, q, ldq, draft,
                         model->vocab, temperature, u, out_len, out_tokens, workspace, s);
}

}  // extern "C"
