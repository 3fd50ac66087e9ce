// Accept step of the verify round, row statistics of raw logits, and Philox.
//
// Greedy (T == 0): longest prefix of drafts equal to the target argmax, then
// the target's own token (mlx-dspark wiki page, "Architecture"; hysenlabs
// review, "The Problem").  Sampled (T > 0): accept draft d of row i iff
// u[i] < p_i[d] / q_i[d]; at the first rejection draw from the residual
// max(0, p - q), else draw the bonus token from p_m (mlx-dspark releases page,
// v0.0.2 "Highlights").
//
// One launch covers B requests x NB vocabulary chunks.  Every CTA recomputes
// the (at most 31) accept decisions of its request from fp64 ratios, then sums
// the draw weights of its chunk in fp64.  The last CTA of a request to finish
// (atomic counter, no spinning) turns the chunk sums into a prefix, finds the
// chunk holding u[m] * Z and scans it in index order.
#include "sv_internal.h"
#include "sv_ptx.cuh"
#include "sv_kernels.h"

namespace sv {

constexpr int ACC_THREADS = 256;

__global__ void __launch_bounds__(ACC_THREADS) accept_kernel(const AcceptParams p) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y, chunk = blockIdx.x, tid = threadIdx.x;
  const int r0 = p.offs[b];
  const int m = p.offs[b + 1] - r0 - 1;
  const int qd0 = r0 - b;  // first q / draft row of this request
  const int V = p.V;

  if (!(p.temperature > 0.f)) {
    if (chunk != 0 || tid != 0) return;
    int a = m;
    for (int i = 0; i < m; ++i)
      if (p.draft[qd0 + i] != p.row_argmax[r0 + i]) { a = i; break; }
    for (int i = 0; i < a; ++i) p.out_tokens[r0 + i] = p.draft[qd0 + i];
    p.out_tokens[r0 + a] = p.row_argmax[r0 + a];
    p.out_len[b] = a + 1;
    return;
  }

  __shared__ int s_j, s_last, s_cstar, s_flag;
  __shared__ double s_pre, s_theta;
  __shared__ double s_w[ACC_THREADS], s_p[ACC_THREADS];
  __shared__ int s_i[ACC_THREADS];

  // ---- accept decisions (fp64 ratio, one lane per draft)
  if (tid < 32) {
    bool rej = false;
    if (tid < m) {
      const int d = p.draft[qd0 + tid];
      if (d < 0 || d >= V) {
        rej = true;
        if (chunk == 0) raise_error(ERR_BAD_INPUT);
      } else {
        const double qd = p.q[(size_t)(qd0 + tid) * p.ldq + d];
        const double z = p.logits[(size_t)(r0 + tid) * p.ldl + d];
        const double pd = exp((z - (double)p.row_max[r0 + tid]) / (double)p.temperature) /
                          (double)p.row_sumexp[r0 + tid];
        const double r = qd == 0.0 ? INFINITY : pd / qd;
        rej = !((double)p.u[r0 + tid] < r);
      }
    }
    const unsigned mask = __ballot_sync(0xffffffffu, rej);
    if (tid == 0) s_j = mask ? __ffs(mask) - 1 : m;
  }
  __syncthreads();
  const int j = s_j;
  const bool resid = j < m;
  const int row = r0 + j;
  const float* z = p.logits + (size_t)row * p.ldl;
  const float* qr = resid ? p.q + (size_t)(qd0 + j) * p.ldq : nullptr;
  const float zmax = p.row_max[row], S = p.row_sumexp[row], T = p.temperature;
  auto weight = [&](int k, float& pk) -> float {
    pk = expf((z[k] - zmax) / T) / S;
    return resid ? fmaxf(0.f, pk - qr[k]) : pk;
  };

  // ---- chunk sums of the draw weights (and of p, for the zero-residual fallback)
  const int NB = p.nb;
  const int k0 = (int)((long long)chunk * V / NB), k1 = (int)((long long)(chunk + 1) * V / NB);
  double sw = 0.0, sp = 0.0;
  for (int k = k0 + tid; k < k1; k += ACC_THREADS) {
    float pk;
    const float wk = weight(k, pk);
    sw += wk;
    sp += pk;
  }
  s_w[tid] = sw;
  s_p[tid] = sp;
  __syncthreads();
  for (int w = ACC_THREADS / 2; w; w >>= 1) {
    if (tid < w) { s_w[tid] += s_w[tid + w]; s_p[tid] += s_p[tid + w]; }
    __syncthreads();
  }
  if (tid == 0) {
    double* cs = p.chunk_sums + ((size_t)b * NB + chunk) * 2;
    cs[0] = s_w[0];
    cs[1] = s_p[0];
    __threadfence();
    s_last = atomicAdd(p.counters + b, 1) == NB - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of the request: locate u[m] * Z
  __shared__ double s_cw[64], s_cp[64];
  if (tid < NB) {
    const double* cs = p.chunk_sums + ((size_t)b * NB + tid) * 2;
    s_cw[tid] = __ldcg(cs);
    s_cp[tid] = __ldcg(cs + 1);
  }
  __syncthreads();
  if (tid == 0) {
    double zw = 0.0, zp = 0.0;
    for (int c = 0; c < NB; ++c) { zw += s_cw[c]; zp += s_cp[c]; }
    const int use_p = resid && !(zw > 0.0);
    const double* sums = use_p ? s_cp : s_cw;
    const double Z = use_p ? zp : zw;
    const double theta = (double)p.u[r0 + m] * Z;
    double pre = 0.0;
    int cstar = -1;
    for (int c = 0; c < NB; ++c) {
      if (pre + sums[c] > theta) { cstar = c; break; }
      pre += sums[c];
    }
    int flag = use_p;  // bit 0: draw from p; bit 1: take the last positive weight
    if (cstar < 0) {   // rounding left theta at the total: last chunk with positive weight
      flag |= 2;
      for (int c = NB - 1; c >= 0; --c)
        if (sums[c] > 0.0) { cstar = c; break; }
      if (cstar < 0) cstar = NB - 1;
    }
    s_cstar = cstar;
    s_pre = pre;
    s_theta = theta;
    s_flag = flag;
    p.counters[b] = 0;
  }
  __syncthreads();
  const int cstar = s_cstar, flag = s_flag;
  const bool from_p = flag & 1;
  const int c0 = (int)((long long)cstar * V / NB), c1 = (int)((long long)(cstar + 1) * V / NB);
  const int len = c1 - c0, per = (len + ACC_THREADS - 1) / ACC_THREADS;
  const int a = c0 + tid * per, e = min(c1, a + per);
  double local = 0.0;
  int last_pos = -1;
  for (int k = a; k < e; ++k) {
    float pk;
    const float wk = weight(k, pk);
    const float wv = from_p ? pk : wk;
    local += wv;
    if (wv > 0.f) last_pos = k;
  }
  s_w[tid] = local;
  __syncthreads();
  if (tid == 0) {  // exclusive prefix over the threads' sub-ranges, in index order
    double run = s_pre;
    for (int i = 0; i < ACC_THREADS; ++i) { const double v = s_w[i]; s_w[i] = run; run += v; }
  }
  __syncthreads();
  int cand = 0x7fffffff;
  if (!(flag & 2)) {
    double run = s_w[tid];
    for (int k = a; k < e; ++k) {
      float pk;
      const float wk = weight(k, pk);
      run += from_p ? pk : wk;
      if (run > s_theta) { cand = k; break; }
    }
  }
  s_i[tid] = cand;
  __syncthreads();
  for (int w = ACC_THREADS / 2; w; w >>= 1) {
    if (tid < w) s_i[tid] = min(s_i[tid], s_i[tid + w]);
    __syncthreads();
  }
  int token = s_i[0];
  __syncthreads();
  if (token == 0x7fffffff) {  // no crossing inside the chunk: last positive weight
    s_i[tid] = last_pos;
    __syncthreads();
    for (int w = ACC_THREADS / 2; w; w >>= 1) {
      if (tid < w) s_i[tid] = max(s_i[tid], s_i[tid + w]);
      __syncthreads();
    }
    token = s_i[0] < 0 ? c1 - 1 : s_i[0];
  }
  if (tid == 0) {
    for (int i = 0; i < j; ++i) p.out_tokens[r0 + i] = p.draft[qd0 + i];
    p.out_tokens[r0 + j] = token;
    p.out_len[b] = j + 1;
  }
}

// Row max / lowest argmax / sum-exp of raw fp32 logits (for callers that do
// not pass the lm_head statistics).  One block per row.
__global__ void __launch_bounds__(1024) row_stats_kernel(const float* __restrict__ logits, int ldl, int V,
                                                         float temperature, float* row_max, float* row_sumexp,
                                                         int32_t* row_argmax) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, tid = threadIdx.x;
  const float* z = logits + (size_t)r * ldl;
  __shared__ float sb[1024];
  __shared__ int si[1024];
  __shared__ double sd[1024];
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int k = tid; k < V; k += 1024) {
    const float v = z[k];
    if (v > best) { best = v; bi = k; }  // ascending k per thread: first maximum kept
  }
  sb[tid] = best;
  si[tid] = bi;
  __syncthreads();
  for (int w = 512; w; w >>= 1) {
    if (tid < w) {
      const float ob = sb[tid + w];
      const int oi = si[tid + w];
      if (ob > sb[tid] || (ob == sb[tid] && oi < si[tid])) { sb[tid] = ob; si[tid] = oi; }
    }
    __syncthreads();
  }
  best = sb[0];
  bi = si[0];
  if (temperature > 0.f) {
    double acc = 0.0;
    for (int k = tid; k < V; k += 1024) acc += (double)expf((z[k] - best) / temperature);
    sd[tid] = acc;
    __syncthreads();
    for (int w = 512; w; w >>= 1) {
      if (tid < w) sd[tid] += sd[tid + w];
      __syncthreads();
    }
  }
  if (tid == 0) {
    row_max[r] = best;
    row_argmax[r] = bi;
    if (temperature > 0.f) row_sumexp[r] = (float)sd[0];
  }
}

// Philox-4x32-10 (Salmon et al., SC'11): multiply-xor rounds with a Weyl key schedule.
__global__ void __launch_bounds__(256) philox_kernel(uint64_t seed, uint64_t subseq, uint64_t offset, int n,
                                                     float* out) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint64_t idx = offset + (uint64_t)i, blk = idx >> 2;
  uint32_t c0 = (uint32_t)blk, c1 = (uint32_t)(blk >> 32), c2 = (uint32_t)subseq, c3 = (uint32_t)(subseq >> 32);
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  const uint32_t w = (idx & 3) == 0 ? c0 : (idx & 3) == 1 ? c1 : (idx & 3) == 2 ? c2 : c3;
  out[i] = (float)(w >> 8) * 5.9604644775390625e-08f;  // 2^-24
}

cudaError_t launch_accept(const AcceptParams& p, int B, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.temperature > 0.f ? p.nb : 1, B), dim3(ACC_THREADS), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, accept_kernel, p);
}

cudaError_t launch_row_stats(const float* logits, int ldl, int rows, int V, float temperature, float* row_max,
                             float* row_sumexp, int32_t* row_argmax, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(rows), dim3(1024), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, row_stats_kernel, logits, ldl, V, temperature, row_max, row_sumexp, row_argmax);
}

cudaError_t launch_philox(uint64_t seed, uint64_t subseq, uint64_t offset, int n, float* out, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3((n + 255) / 256), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, philox_kernel, seed, subseq, offset, n, out);
}

}  // namespace sv
