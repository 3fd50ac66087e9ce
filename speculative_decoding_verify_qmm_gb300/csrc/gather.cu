// Gather-qmm: the verify block's rows routed to mixture-of-experts weights.
//
// mlx-dspark PyPI page, "Results at a glance" (the MoE rows): on an MoE target
// every extra verify row pulls in a fresh set of experts, so the verify cost
// is the union of the experts the rows select.  Wiki page, "Key techniques":
// each weight group is dequantized once and reused across rows.  Here a pair
// p = (row r_p, expert e_p) asks for Y[p, :] = X[r_p, :] * W_{e_p}^T; the
// pairs are grouped by expert on the device, every selected expert's weight
// is streamed exactly once, and each of its tiles is applied to all the rows
// routed to it (up to 32), with the same factored group arithmetic as the
// verify matmul.
//
// Three launches: routing (group the pairs by expert, in expert order and
// pair order within an expert), the gathered activation preparation (one
// prepared block per selected expert), and a persistent kernel whose CTAs take
// contiguous ranges of (selected expert, 64-row tile) items, with a TMA-fed
// ring of stages, eight consumer warps and one producer warp.
#include "sv_internal.h"
#include "sv_ptx.cuh"
#include "sv_prep.cuh"
#include "stream_kernel.cuh"

namespace sv {

constexpr int GQ_THREADS = (NCW + 1) * 32;  // consumers + one producer warp

struct GatherRoute {
  const int32_t* pair_rows;
  const int32_t* pair_experts;
  int P, E, M, MP, A;
  int* n_active;    // [1]
  int* act_expert;  // [A]
  int* act_count;   // [A]
  int* act_pairs;   // [A][MP]
  int* abort_word;  // [1], cleared here
};

// Groups the pairs by expert: selected experts in increasing id, each with its
// pairs in increasing pair index.  One CTA; invalid pairs are skipped and
// flagged.
__global__ void __launch_bounds__(256) gather_route_kernel(const GatherRoute g) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int sm[];
  int* cnt = sm;                 // [E]
  int* slot = sm + g.E;          // [E]: selected index of an expert, or -1
  int* run = sm + 2 * g.E;       // [E]: pairs placed so far
  __shared__ int s_wsum[8];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int e = tid; e < g.E; e += 256) {
    cnt[e] = 0;
    run[e] = 0;
  }
  if (tid == 0) *g.abort_word = 0;
  __syncthreads();
  for (int p = tid; p < g.P; p += 256) {
    const int e = g.pair_experts[p], r = g.pair_rows[p];
    if (e >= 0 && e < g.E && r >= 0 && r < g.M)
      atomicAdd(&cnt[e], 1);
    else
      raise_error(ERR_BAD_INPUT);
  }
  __syncthreads();
  // selected index of every expert: an exclusive scan of (cnt > 0) in expert order
  const int per = (g.E + 255) / 256, e0 = min(g.E, tid * per), e1 = min(g.E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += cnt[e] > 0;
  int incl = local;
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_wsum[wid] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < wid; ++w) base += s_wsum[w];
  int idx = base + incl - local;
  for (int e = e0; e < e1; ++e) {
    if (cnt[e] > 0) {
      slot[e] = idx;
      if (idx < g.A) {
        g.act_expert[idx] = e;
        g.act_count[idx] = min(cnt[e], g.MP);
      }
      if (cnt[e] > g.MP) raise_error(ERR_BAD_INPUT);  // more pairs than rows for one expert
      ++idx;
    } else {
      slot[e] = -1;
    }
  }
  if (tid == 255) *g.n_active = min(idx, g.A);
  __syncthreads();
  // place the pairs in pair order: warp 0 walks 32 pairs at a time
  if (wid == 0) {
    for (int p0 = 0; p0 < g.P; p0 += 32) {
      const int p = p0 + lane;
      int e = -1;
      if (p < g.P) {
        const int ee = g.pair_experts[p], r = g.pair_rows[p];
        if (ee >= 0 && ee < g.E && r >= 0 && r < g.M) e = ee;
      }
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(same & ((1u << lane) - 1u));
      const int k = e >= 0 ? run[e] + rank : 0;
      if (e >= 0 && k < g.MP && slot[e] < g.A) g.act_pairs[slot[e] * g.MP + k] = p;
      __syncwarp();
      if (e >= 0 && rank == __popc(same) - 1) run[e] += __popc(same);  // the group's last lane advances it
      __syncwarp();
    }
  }
}

struct GatherPrep {
  const __nv_bfloat16* x;
  int ldx, K, MP;
  const int32_t* pair_rows;
  const int* n_active;
  const int* act_count;
  const int* act_pairs;
  ActBuf act0;             // the prepared block of selected expert 0
  size_t xp_stride, xs_stride, sq_stride;  // elements between selected experts' blocks
};

// Grid (K / 512, MP, A): one warp per group of one padded row of one selected expert.
template <int BITS>
__global__ void __launch_bounds__(256) gather_prep_kernel(const GatherPrep a) {
  pdl_trigger();
  pdl_wait();
  const int sel = blockIdx.z, m = blockIdx.y;
  if (sel >= *a.n_active) return;
  const int g = blockIdx.x * 8 + (threadIdx.x >> 5);
  const __nv_bfloat16* row = nullptr;
  if (m < a.act_count[sel]) row = a.x + (size_t)a.pair_rows[a.act_pairs[sel * a.MP + m]] * a.ldx;
  ActBuf out;
  out.xp = a.act0.xp + sel * a.xp_stride;
  out.xs = a.act0.xs + sel * a.xs_stride;
  out.sq = a.act0.sq + sel * a.sq_stride;
  prep_group<BITS, PREP_PLAIN>(row, nullptr, nullptr, 0.f, m, g, a.MP, a.K, out);
}

struct GatherParams {
  CUtensorMap tm[3];        // stacked expert weights [E * N, K]: codes, scales, biases
  int N, K, grid;
  const int* n_active;
  const int* act_expert;
  const int* act_count;
  const int* act_pairs;
  const __half* xp0;        // prepared activations of selected expert 0
  const float* xs0;
  size_t xp_stride, xs_stride;
  __nv_bfloat16* y;
  int ldy;
  int* abort_word;
};

template <int BITS, int NT>
__global__ void __launch_bounds__(GQ_THREADS, 1) gather_kernel(const __grid_constant__ GatherParams p) {
  using C = StreamCfg<BITS, NT>;
  constexpr int S = C::STAGES;
  constexpr int MP = C::MP;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[S], empty_bar[S];
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red = reinterpret_cast<float*>(smem + S * C::STAGE_BYTES);  // [4 quarters][16 * MP]
  volatile int* abort_v = &abort_flag;
  volatile int* abort_g = p.abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], NCW);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // the routing and the prepared activations come from the previous launches
  const int tiles = (p.N + BN - 1) / BN, upt = p.K / KC;
  const int items = *p.n_active * tiles;
  const int i0 = (int)((long long)blockIdx.x * items / p.grid), i1 = (int)((long long)(blockIdx.x + 1) * items / p.grid);

  if (warp == NCW) {
    // ============================================================ producer
    if (lane != 0) return;
    const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
    int n = 0;
    bool bad = false;
    for (int i = i0; i < i1 && !bad; ++i) {
      const int sel = i / tiles, tile = i % tiles;
      const int row0 = p.act_expert[sel] * p.N + tile * BN;
      const __half* xp = p.xp0 + sel * p.xp_stride;
      const float* xs = p.xs0 + sel * p.xs_stride;
      for (int kc = 0; kc < upt; ++kc, ++n) {
        const int sg = n % S;
        if (n >= S && !mbar_wait_bounded(&empty_bar[sg], ((n / S) - 1) & 1, abort_v)) {
          if (!*abort_v) raise_error(ERR_TIMEOUT_EMPTY);
          *abort_v = 1;
          *abort_g = 1;
          bad = true;
          break;
        }
        uint8_t* st = smem + sg * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full_bar[sg], C::UNIT_BYTES + C::X_BYTES + C::XS_BYTES);
        tma_load_3d(st, p.tm, &full_bar[sg], 0, row0, kc * C::ATOMS, pol_w);
        tma_load_2d(st + C::S_OFF, p.tm + 1, &full_bar[sg], kc * GPS, row0, pol_w);
        tma_load_2d(st + C::B_OFF, p.tm + 2, &full_bar[sg], kc * GPS, row0, pol_w);
        bulk_load(st + C::X_OFF, xp + (size_t)kc * (KC / 32) * MP * 32, C::X_BYTES, &full_bar[sg], pol_x);
        bulk_load(st + C::XS_OFF, xs + (size_t)kc * GPS * 2 * MP, C::XS_BYTES, &full_bar[sg], pol_x);
      }
    }
    // copies in flight land before the CTA may exit (bounded)
    if (!bad && !*abort_v) {
      for (int k = (n - S > 0 ? n - S : 0); k < n; ++k) mbar_wait_bounded(&full_bar[k % S], (k / S) & 1, abort_v);
    } else {
      const unsigned long long t0 = global_ns();
      while (global_ns() - t0 < 50000ull) __nanosleep(1000);
    }
    return;
  }

  // ================================================================ consumers
  const int q = warp >> 1, kh = warp & 1, gid = lane >> 2, t = lane & 3;
  int n = 0;
  for (int i = i0; i < i1; ++i) {
    const int sel = i / tiles, tile = i % tiles;
    float tot[NT][4];
    zero4<NT>(tot);
    for (int kc = 0; kc < upt; ++kc, ++n) {
      const int s = n % S;
      if (!(*abort_v)) {
        if (mbar_wait_bounded(&full_bar[s], (n / S) & 1, abort_v)) {
          consume_stage<BITS, NT>(smem + s * C::STAGE_BYTES, q, kh, lane, tot);
        } else {
          raise_error(ERR_TIMEOUT_FULL);
          *abort_v = 1;
          *abort_g = 1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    // the two k halves meet in shared memory (fixed order), then k-half 0 writes
    float* rb = red + q * 16 * MP;
    if (kh == 1) red_store<NT>(rb, tot, lane);
    named_bar_sync(1 + q, 64);
    if (kh == 0 && !(*abort_v)) {
      red_add<NT, false>(rb, tot, lane);
      const int cnt = p.act_count[sel];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = 8 * j + 2 * t + (e & 1);
          const int col = tile * BN + 16 * q + gid + 8 * (e >> 1);
          if (m < cnt && col < p.N) {
            const int pair = p.act_pairs[sel * MP + m];
            p.y[(size_t)pair * p.ldy + col] = __float2bfloat16_rn(tot[j][e]);
          }
        }
    }
    named_bar_sync(1 + q, 64);  // the slot is read before the next item overwrites it
  }
}

template <int BITS, int NT>
static cudaError_t launch_gather_t(const GatherParams& p, cudaStream_t s) {
  using C = StreamCfg<BITS, NT>;
  constexpr int SMEM = 1024 + C::STAGES * C::STAGE_BYTES + 4 * 16 * C::MP * 4;
  static_assert(SMEM + 1024 <= 227 * 1024, "shared memory budget");
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gather_kernel<BITS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.grid), dim3(GQ_THREADS), SMEM, s, attr);
  return cudaLaunchKernelEx(&cfg, gather_kernel<BITS, NT>, p);
}

template <int BITS>
static cudaError_t launch_gather_b(const GatherParams& p, int MP, cudaStream_t s) {
  switch (MP / 8) {
    case 1: return launch_gather_t<BITS, 1>(p, s);
    case 2: return launch_gather_t<BITS, 2>(p, s);
    case 3: return launch_gather_t<BITS, 3>(p, s);
    case 4: return launch_gather_t<BITS, 4>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

// Workspace: [abort word, n_active | pad to 256][act_expert][act_count][act_pairs][prepared blocks]
struct GatherLayout {
  size_t expert, count, pairs, act, xp_bytes, xs_bytes, sq_bytes, per_sel, total;
};
static GatherLayout gather_layout(int A, int MP, int K) {
  GatherLayout L;
  size_t off = 256;
  L.expert = off; off = align256(off + (size_t)A * 4);
  L.count = off;  off = align256(off + (size_t)A * 4);
  L.pairs = off;  off = align256(off + (size_t)A * MP * 4);
  L.xp_bytes = align256((size_t)K * MP * 2);
  L.xs_bytes = align256((size_t)(K / GROUP) * 2 * MP * 4);
  L.sq_bytes = align256((size_t)(K / GROUP + 1) * MP * 4);
  L.per_sel = L.xp_bytes + L.xs_bytes + L.sq_bytes;
  L.act = off;    off += (size_t)A * L.per_sel;
  L.total = off;
  return L;
}

constexpr int GQ_MAX_PAIRS = 1024;
constexpr int GQ_MAX_EXPERTS = 4096;

static int check_gather(int E, int N, int K, int bits, int group, int M, int P) {
  if (!bits_supported(bits)) return fail(SV_EUNSUPPORTED, "bits must be 2, 4 or 8 (got %d)", bits);
  if (group != GROUP) return fail(SV_EUNSUPPORTED, "group size must be 64 (got %d)", group);
  if (E < 1 || E > GQ_MAX_EXPERTS) return fail(SV_EINVAL, "E must be in [1, %d] (got %d)", GQ_MAX_EXPERTS, E);
  if (N < 1 || (long long)E * N > (long long)MAX_TILES * BN) return fail(SV_EINVAL, "E * N out of range");
  if (K < KC || K % KC || K > (1 << 20)) return fail(SV_EUNSUPPORTED, "K must be a positive multiple of 512");
  if (M < 1 || M > MAX_M) return fail(M > MAX_M ? SV_EUNSUPPORTED : SV_EINVAL, "M must be in [1, 32] (got %d)", M);
  if (P < 1 || P > GQ_MAX_PAIRS) return fail(SV_EINVAL, "P must be in [1, %d] (got %d)", GQ_MAX_PAIRS, P);
  return SV_OK;
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t sv_gather_qmm_workspace_bytes(int P, int M, int N, int K, int E, int bits) {
  if (check_gather(E, N, K, bits, GROUP, M, P)) return 0;
  const int MP = 8 * ((M + 7) / 8), A = P < E ? P : E;
  return gather_layout(A, MP, K).total;
}

int sv_gather_qmm(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int E, int N, int K, int bits,
                  int group, const uint16_t* x, int ldx, int M, const int32_t* pair_rows, const int32_t* pair_experts,
                  int P, uint16_t* y, int ldy, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_gather(E, N, K, bits, group, M, P);
  if (st) return st;
  if (!wq || !scales || !biases || !x || !pair_rows || !pair_experts || !y || !workspace)
    return fail(SV_EINVAL, "null pointer argument");
  if (!aligned(wq, 16) || !aligned(scales, 16) || !aligned(biases, 16))
    return fail(SV_EINVAL, "wq, scales and biases must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(SV_EINVAL, "workspace must be 256-byte aligned");
  if (ldx < K || ldy < N) return fail(SV_EINVAL, "ldx must be >= K and ldy >= N");
  const int MP = 8 * ((M + 7) / 8), A = P < E ? P : E;
  const GatherLayout L = gather_layout(A, MP, K);
  if (workspace_bytes < L.total) return fail(SV_EINVAL, "workspace too small: %zu < %zu", workspace_bytes, L.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  int* abort_word = reinterpret_cast<int*>(base);
  int* n_active = reinterpret_cast<int*>(base + 4);

  GatherRoute r;
  r.pair_rows = pair_rows;
  r.pair_experts = pair_experts;
  r.P = P;
  r.E = E;
  r.M = M;
  r.MP = MP;
  r.A = A;
  r.n_active = n_active;
  r.act_expert = reinterpret_cast<int*>(base + L.expert);
  r.act_count = reinterpret_cast<int*>(base + L.count);
  r.act_pairs = reinterpret_cast<int*>(base + L.pairs);
  r.abort_word = abort_word;
  {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(1), dim3(256), (size_t)3 * E * sizeof(int), s, attr);
    cudaError_t e = cudaFuncSetAttribute(gather_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         3 * GQ_MAX_EXPERTS * (int)sizeof(int));
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, gather_route_kernel, r);
    if (e != cudaSuccess) return cuda_fail(e, "gather routing launch");
  }
  GatherPrep gp;
  gp.x = reinterpret_cast<const __nv_bfloat16*>(x);
  gp.ldx = ldx;
  gp.K = K;
  gp.MP = MP;
  gp.pair_rows = pair_rows;
  gp.n_active = n_active;
  gp.act_count = r.act_count;
  gp.act_pairs = r.act_pairs;
  gp.act0.xp = reinterpret_cast<__half*>(base + L.act);
  gp.act0.xs = reinterpret_cast<float*>(base + L.act + L.xp_bytes);
  gp.act0.sq = reinterpret_cast<float*>(base + L.act + L.xp_bytes + L.xs_bytes);
  gp.xp_stride = L.per_sel / 2;
  gp.xs_stride = L.per_sel / 4;
  gp.sq_stride = L.per_sel / 4;
  {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(K / KC, MP, A), dim3(256), 0, s, attr);
    cudaError_t e = bits == 8 ? cudaLaunchKernelEx(&cfg, gather_prep_kernel<8>, gp)
                              : (bits == 4 ? cudaLaunchKernelEx(&cfg, gather_prep_kernel<4>, gp)
                                           : cudaLaunchKernelEx(&cfg, gather_prep_kernel<2>, gp));
    if (e != cudaSuccess) return cuda_fail(e, "gather preparation launch");
  }
  static thread_local GatherParams p;
  memset(static_cast<void*>(&p), 0, sizeof(p));
  st = encode_weight_maps(p.tm, wq, scales, biases, E * N, K, bits);
  if (st) return st;
  const int tiles = (N + BN - 1) / BN;
  const int sms = device_sm_count();
  if (sms <= 0) return fail(SV_ECUDA, "no CUDA device");
  p.N = N;
  p.K = K;
  p.grid = A * tiles < sms ? A * tiles : sms;
  p.n_active = n_active;
  p.act_expert = r.act_expert;
  p.act_count = r.act_count;
  p.act_pairs = r.act_pairs;
  p.xp0 = gp.act0.xp;
  p.xs0 = gp.act0.xs;
  p.xp_stride = gp.xp_stride;
  p.xs_stride = gp.xs_stride;
  p.y = reinterpret_cast<__nv_bfloat16*>(y);
  p.ldy = ldy;
  p.abort_word = abort_word;
  cudaError_t e = bits == 8 ? launch_gather_b<8>(p, MP, s)
                            : (bits == 4 ? launch_gather_b<4>(p, MP, s) : launch_gather_b<2>(p, MP, s));
  if (e != cudaSuccess) return cuda_fail(e, "gather matmul launch");
  return SV_OK;
}

}  // extern "C"
