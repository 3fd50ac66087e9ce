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
// chunk holding u[m] * Z, and the one thread whose sub-range of that chunk
// holds the crossing scans it in index order.  Sums and prefixes are shuffle
// trees in a fixed order: fp64 is slow on this part, and serial fp64 chains
// dominated the step's time.
#include "sv_internal.h"
#include "sv_ptx.cuh"
#include "sv_kernels.h"

namespace sv {

constexpr int ACC_THREADS = 256;
constexpr int ACC_CACHE = 8192;  // vocabulary chunk held in shared memory by the drawing CTA
constexpr int ACC_BATCH = 10;    // vocabulary elements per thread whose loads are in flight together

// Warp reductions and scans in a fixed order (shuffle trees), so every run
// adds the same values in the same order.
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
__device__ __forceinline__ double warp_incl_scan(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}
__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__global__ void __launch_bounds__(ACC_THREADS) accept_kernel(const AcceptParams p) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y, chunk = blockIdx.x, tid = threadIdx.x;
  const int r0 = p.offs[b];
  const int m = p.offs[b + 1] - r0 - 1;
  const int qd0 = r0 - b;  // first q / draft row of this request
  const int V = p.V;

  if (!(p.temperature > 0.f)) {
    // greedy: one lane per draft (m <= 31); the first mismatch is the lowest set bit of a ballot
    if (chunk != 0 || tid >= 32) return;
    const int d = tid < m ? p.draft[qd0 + tid] : 0;
    const unsigned miss = __ballot_sync(0xffffffffu, tid < m && d != p.row_argmax[r0 + tid]);
    const int a = miss ? __ffs(miss) - 1 : m;
    if (tid < a) p.out_tokens[r0 + tid] = d;
    if (tid == 0) {
      p.out_tokens[r0 + a] = p.row_argmax[r0 + a];
      p.out_len[b] = a + 1;
    }
    return;
  }

  __shared__ int s_j, s_last, s_cstar, s_flag;
  __shared__ double s_pre, s_theta;
  __shared__ double s_w[ACC_THREADS / 32], s_p[ACC_THREADS / 32];
  __shared__ int s_i[2 * (ACC_THREADS / 32)];
  __shared__ float s_cache[ACC_CACHE];

  // ---- accept decisions (fp64 ratio, one lane per draft)
  if (tid < 32) {
    bool rej = false;
    if (tid < m) {
      const int d = p.draft[qd0 + tid];
      if (d < 0 || d >= V) {
        rej = true;
        if (chunk == 0) raise_error(ERR_BAD_INPUT);
      } else {
        // fp32 ratio (relative error a few 1e-7); fp64 only when u is near it
        const float qd = p.q[(size_t)(qd0 + tid) * p.ldq + d];
        const float z = p.logits[(size_t)(r0 + tid) * p.ldl + d];
        const float zmx = p.row_max[r0 + tid], ui = p.u[r0 + tid];
        const float se = p.tkey ? p.tnorm[r0 + tid] : p.row_sumexp[r0 + tid];
        bool kept = true;  // a token the truncated target never emits is rejected
        if (p.tkey) {
          const uint32_t kd = order_key(z), K = p.tkey[r0 + tid];
          kept = kd > K || (kd == K && d <= p.tidx[r0 + tid]);
        }
        const float r32 = !kept ? 0.f : (qd == 0.f ? INFINITY : expf((z - zmx) / p.temperature) / se / qd);
        if (!kept) {
          rej = true;
        } else if (fabsf(ui - r32) > 1e-5f * fmaxf(1.f, r32)) {
          rej = !(ui < r32);
        } else {
          const double pd = exp(((double)z - (double)zmx) / (double)p.temperature) / (double)se;
          rej = !((double)ui < pd / (double)qd);
        }
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
  const bool trunc = p.tkey != nullptr;
  const float zmax = p.row_max[row], S = trunc ? p.tnorm[row] : p.row_sumexp[row], T = p.temperature;
  const uint32_t tK = trunc ? p.tkey[row] : 0u;
  const int tI = trunc ? p.tidx[row] : V;
  // p_k = exp((z_k - zmax) / T) / S with the two divisions as products by
  // reciprocals taken once (a few fp32 ulps, far below the draw's 1e-6 Z
  // exemption) and vanishing terms set to 0: every element of the vocabulary
  // passes through here, and the IEEE forms took slow paths on most of them
  const float inv_t = 1.f / T, inv_s = 1.f / S;
  auto weight = [&](int k, float& pk) -> float {
    const float zk = z[k];
    bool kept = true;
    if (trunc) {
      const uint32_t key = order_key(zk);
      kept = key > tK || (key == tK && k <= tI);
    }
    pk = kept ? exp_term((zk - zmax) * inv_t) * inv_s : 0.f;
    return resid ? fmaxf(0.f, pk - qr[k]) : pk;
  };

  // ---- chunk sums of the draw weights (and of p, for the zero-residual fallback)
  const int NB = p.nb;
  const int k0 = (int)((long long)chunk * V / NB), k1 = (int)((long long)(chunk + 1) * V / NB);
  float sw = 0.f, sp = 0.f;  // at most a few dozen terms per thread: fp32 holds them to ~1e-7
  // ACC_BATCH elements per turn with their loads issued together (the loop
  // is latency-bound: every element is a load from L2)
  for (int k = k0 + tid; k < k1; k += ACC_BATCH * ACC_THREADS) {
    float wk[ACC_BATCH], pk[ACC_BATCH];
#pragma unroll
    for (int v = 0; v < ACC_BATCH; ++v) {
      const int kk = k + v * ACC_THREADS;
      wk[v] = pk[v] = 0.f;
      if (kk < k1) wk[v] = weight(kk, pk[v]);
    }
#pragma unroll
    for (int v = 0; v < ACC_BATCH; ++v) {
      sw += wk[v];
      sp += pk[v];
    }
  }
  const int lane = tid & 31, wid = tid >> 5;
  const double dsw = warp_sum((double)sw), dsp = warp_sum((double)sp);
  if (lane == 0) {
    s_w[wid] = dsw;
    s_p[wid] = dsp;
  }
  __syncthreads();
  if (tid == 0) {
    double tw = 0.0, tp = 0.0;
    for (int w = 0; w < ACC_THREADS / 32; ++w) { tw += s_w[w]; tp += s_p[w]; }  // fixed order
    double* cs = p.chunk_sums + ((size_t)b * NB + chunk) * 2;
    cs[0] = tw;
    cs[1] = tp;
    __threadfence();
    s_last = atomicAdd(p.counters + b, 1) == NB - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < j) p.out_tokens[r0 + tid] = p.draft[qd0 + tid];  // the accepted drafts (j <= 31), one thread each

  // ---- last CTA of the request: locate u[m] * Z among the chunks (warp 0:
  // lane l holds chunks l and l + 32; inclusive scans by shuffles)
  if (wid == 0) {
    const double* cs = p.chunk_sums + (size_t)b * NB * 2;
    double w0 = lane < NB ? __ldcg(cs + 2 * lane) : 0.0, w1 = lane + 32 < NB ? __ldcg(cs + 2 * (lane + 32)) : 0.0;
    double p0 = lane < NB ? __ldcg(cs + 2 * lane + 1) : 0.0, p1 = lane + 32 < NB ? __ldcg(cs + 2 * (lane + 32) + 1) : 0.0;
    const double zw = warp_sum(w0) + warp_sum(w1), zp = warp_sum(p0) + warp_sum(p1);
    const int use_p = resid && !(zw > 0.0);
    double a0 = use_p ? p0 : w0, a1 = use_p ? p1 : w1;
    const double Z = use_p ? zp : zw;
    const double theta = (double)p.u[r0 + m] * Z;
    const double i0 = warp_incl_scan(a0);
    const double i1 = warp_incl_scan(a1) + __shfl_sync(0xffffffffu, i0, 31);
    // first chunk whose inclusive prefix exceeds theta
    const unsigned c0m = __ballot_sync(0xffffffffu, lane < NB && i0 > theta);
    const unsigned c1m = __ballot_sync(0xffffffffu, lane + 32 < NB && i1 > theta);
    int cstar = c0m ? __ffs(c0m) - 1 : (c1m ? 32 + __ffs(c1m) - 1 : -1);
    int flag = use_p;  // bit 0: draw from p; bit 1: take the last positive weight
    if (cstar < 0) {   // rounding left theta at the total: last chunk with positive weight
      flag |= 2;
      const unsigned q0 = __ballot_sync(0xffffffffu, lane < NB && a0 > 0.0);
      const unsigned q1 = __ballot_sync(0xffffffffu, lane + 32 < NB && a1 > 0.0);
      cstar = q1 ? 63 - __clz(q1) : (q0 ? 31 - __clz(q0) : NB - 1);
    }
    // exclusive prefix of chunk cstar
    const double excl0 = i0 - a0, excl1 = i1 - a1;
    const double pre = cstar < 32 ? __shfl_sync(0xffffffffu, excl0, cstar & 31) : __shfl_sync(0xffffffffu, excl1, cstar & 31);
    if (lane == 0) {
      s_cstar = cstar;
      s_pre = pre;
      s_theta = theta;
      s_flag = flag;
      p.counters[b] = 0;
    }
  }
  __syncthreads();
  const int cstar = s_cstar, flag = s_flag;
  const bool from_p = flag & 1;
  const int c0 = (int)((long long)cstar * V / NB), c1 = (int)((long long)(cstar + 1) * V / NB);
  const int len = c1 - c0, per = (len + ACC_THREADS - 1) / ACC_THREADS;
  const int a = c0 + tid * per, e = min(c1, a + per);
  // the chunk's draw weights, filled with coalesced loads when they fit in
  // shared memory; each thread then sums its contiguous sub-range
  const bool cached = len <= ACC_CACHE;
  if (cached) {
    for (int k = c0 + tid; k < c1; k += ACC_BATCH * ACC_THREADS) {
      float wv[ACC_BATCH];
#pragma unroll
      for (int v = 0; v < ACC_BATCH; ++v) {
        const int kk = k + v * ACC_THREADS;
        float pk = 0.f, wk = 0.f;
        if (kk < c1) wk = weight(kk, pk);
        wv[v] = from_p ? pk : wk;
      }
#pragma unroll
      for (int v = 0; v < ACC_BATCH; ++v)
        if (k + v * ACC_THREADS < c1) s_cache[k + v * ACC_THREADS - c0] = wv[v];
    }
    __syncthreads();
  }
  auto draw_weight = [&](int k) -> float {
    if (cached) return s_cache[k - c0];
    float pk;
    const float wk = weight(k, pk);
    return from_p ? pk : wk;
  };
  float local32 = 0.f;
  int last_pos = -1;
  for (int k = a; k < e; ++k) {
    const float wv = draw_weight(k);
    local32 += wv;
    if (wv > 0.f) last_pos = k;
  }
  const double local = local32;
  const double incl = warp_incl_scan(local);
  if (lane == 31) s_w[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const double t = lane < ACC_THREADS / 32 ? s_w[lane] : 0.0;
    const double ti = warp_incl_scan(t);
    if (lane < ACC_THREADS / 32) s_p[lane] = ti - t;  // exclusive prefix of each warp
  }
  __syncthreads();
  const double start = s_pre + s_p[wid] + (incl - local);
  // only the thread whose sub-range holds the crossing scans it
  int cand = 0x7fffffff;
  if (!(flag & 2) && start <= s_theta && start + local > s_theta) {
    double run = start;
    for (int k = a; k < e; ++k) {
      run += draw_weight(k);
      if (run > s_theta) { cand = k; break; }
    }
    if (cand == 0x7fffffff) cand = last_pos >= 0 ? last_pos : e - 1;  // rounding inside the range
  }
  cand = warp_min(cand);
  if (lane == 0) s_i[wid] = cand;
  const int lp = warp_max(last_pos);
  __syncthreads();
  if (tid == 0) {
    int token = 0x7fffffff;
    for (int w = 0; w < ACC_THREADS / 32; ++w) token = min(token, s_i[w]);
    s_j = token;
  }
  if (lane == 0) s_i[ACC_THREADS / 32 + wid] = lp;
  __syncthreads();
  if (tid == 0) {
    int token = s_j;
    if (token == 0x7fffffff) {  // no crossing inside the chunk: last positive weight
      int lastp = -1;
      for (int w = 0; w < ACC_THREADS / 32; ++w) lastp = max(lastp, s_i[ACC_THREADS / 32 + w]);
      token = lastp < 0 ? c1 - 1 : lastp;
    }
    p.out_tokens[r0 + j] = token;
    p.out_len[b] = j + 1;
  }
}

// Row max / lowest argmax / sum-exp of raw fp32 logits (for callers that do
// not pass the lm_head statistics).  One thread-block cluster of up to 8 CTAs
// per row, each a slice of it; the slices' results meet in distributed
// shared memory (in slice order, so the lowest index of the maximum wins).
__global__ void __launch_bounds__(1024) row_stats_kernel(const float* __restrict__ logits, int ldl, int V,
                                                         float temperature, float* row_max, float* row_sumexp,
                                                         int32_t* row_argmax) {
  pdl_trigger();
  pdl_wait();
  const unsigned C = cluster_ctas(), rank = cluster_rank();
  const int r = blockIdx.x / C, tid = threadIdx.x;
  const int slice = (V + (int)C - 1) / (int)C;
  const int v0 = min(V, (int)rank * slice), v1 = min(V, v0 + slice);
  const float* z = logits + (size_t)r * ldl;
  __shared__ float sb[1024];
  __shared__ int si[1024];
  __shared__ u128 sd[32];
  __shared__ float cbest;
  __shared__ int cidx;
  __shared__ unsigned long long csum[2];
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int k = v0 + tid; k < v1; k += 1024) {
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
  if (tid == 0) {
    cbest = sb[0];
    cidx = si[0];
  }
  cluster_sync();
  best = -INFINITY;
  bi = 0x7fffffff;
  for (unsigned q = 0; q < C; ++q) {
    const float ob = __uint_as_float(ld_peer_u32(peer(&cbest, q)));
    const int oi = (int)ld_peer_u32(peer(&cidx, q));
    if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
  }
  double se = 0.0;
  if (temperature > 0.f) {  // the fp32 exp terms summed exactly (fixed point)
    u128 acc = 0;
    for (int k = v0 + tid; k < v1; k += 1024) acc += to_fixed(exp_term((z[k] - best) / temperature));
    acc = warp_sum_u128(acc);
    if ((tid & 31) == 0) sd[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
      u128 t = 0;
      for (int w = 0; w < 32; ++w) t += sd[w];
      csum[0] = (unsigned long long)t;
      csum[1] = (unsigned long long)(t >> 64);
    }
    cluster_sync();
    if (tid == 0) {
      u128 t = 0;
      for (unsigned q = 0; q < C; ++q)
        t += ((u128)ld_peer_u64(peer(&csum[1], q)) << 64) + ld_peer_u64(peer(&csum[0], q));
      se = fixed_to_double(t);
    }
  }
  if (rank == 0 && tid == 0) {
    row_max[r] = best;
    row_argmax[r] = bi;
    if (temperature > 0.f) row_sumexp[r] = (float)se;
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
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

// CTAs per row for row_stats_kernel: the largest cluster of up to 8 the device can place.
static int row_stats_cluster() {
  static int cached = 0;
  if (cached) return cached;
  int c = 8;
  for (; c > 1; c >>= 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c);
    cfg.blockDim = dim3(1024);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, row_stats_kernel, &cfg) == cudaSuccess && n > 0) break;
    cudaGetLastError();  // clear a refusal; try a smaller cluster
  }
  cached = c;
  return c;
}

cudaError_t launch_row_stats(const float* logits, int ldl, int rows, int V, float temperature, float* row_max,
                             float* row_sumexp, int32_t* row_argmax, cudaStream_t s) {
  const int c = row_stats_cluster();
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(rows * c), dim3(1024), 0, s, attr);
  attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
  attr[cfg.numAttrs].val.clusterDim.x = c;
  attr[cfg.numAttrs].val.clusterDim.y = 1;
  attr[cfg.numAttrs].val.clusterDim.z = 1;
  ++cfg.numAttrs;
  return cudaLaunchKernelEx(&cfg, row_stats_kernel, logits, ldl, V, temperature, row_max, row_sumexp, row_argmax);
}

cudaError_t launch_philox(uint64_t seed, uint64_t subseq, uint64_t offset, int n, float* out, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3((n + 255) / 256), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, philox_kernel, seed, subseq, offset, n, out);
}

}  // namespace sv
