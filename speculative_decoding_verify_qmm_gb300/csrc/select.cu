// Top-k / top-p truncation bounds of vocabulary rows, truncated probability
// rows, and per-token log-probabilities.
//
// mlx-dspark releases page, v0.1.0 "Highlights": lossless top-p / top-k
// sampling applies nucleus / top-k truncation to both the draft and the
// target, so the accepted output is an exact sample of the truncated target.
// A row is ordered by its own values, largest first, ties to the lower index
// (the target by its fp32 logits, a probability row by its values); top_k
// keeps the first top_k tokens, then top_p keeps the shortest prefix of those
// whose share of their mass reaches top_p.  Releases page, v0.2.0
// "Highlights": logprobs / top_logprobs, the chosen and the top target
// log-probabilities per token.
//
// One thread-block cluster per row (up to 8 CTAs, each a slice of the row).
// The kept set is always "key > K, or key == K and index <= I" for an
// order-preserving 32-bit key of the value: a radix select over the key's
// four bytes (most significant first) finds K - by counts for top_k, by mass
// for top_p - and one scan over the tied keys finds I.  Each CTA histograms
// its slice; the CTAs exchange their bin totals, maxima and sums through
// distributed shared memory, one cluster barrier per exchange, and every CTA
// takes the same decisions from the same totals.  Everything stays on chip,
// so these calls need no workspace.
//
// Masses are summed exactly: every weight (a probability, or an fp32 exp
// term, both at most 1 for valid rows) is a 64.64 fixed-point integer, exact
// for weights from 2^-40 up and truncated below, and integer sums do not
// depend on their order.  Each warp keeps private 256-bin histograms,
// updated with shared-memory atomics (a mass as a 64-bit add on its fraction
// word that carries into its integer word), so a hot bin is contended only
// within a warp (a probability row puts nearly every key in a handful of
// top-byte bins).
#include <climits>
#include <cmath>

#include "sv_internal.h"
#include "sv_ptx.cuh"
#include "sv_kernels.h"

namespace sv {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_MAX_CLUSTER = 8;  // CTAs per row (the portable cluster size)
// Elements a thread loads before it updates the histograms: the loads of a
// batch are independent and in flight together (loads interleaved with the
// shared-memory atomics went out one L2 round trip after another).
constexpr int SEL_BATCH = 4;

struct SelShared {
  int cnt[256];          // the cluster's bin totals of the current pass
  double mass[256];
  double wsum[SEL_WARPS];
  int wint[SEL_WARPS];
  int bin;
  double above;
  double total;
  // this CTA's values that the other CTAs of the cluster read (one slot per use)
  float cmax;
  unsigned long long csum[2][2];  // exact sums (kept mass, log-sum): fraction word, integer word
  int ccount[2];                  // tied keys in this slice, per tie search
  int cfound[2];                  // the tie index if it lies in this slice, else INT_MAX
  int n_top;
  uint32_t top_key[32];
  int top_idx[32];
};

// Per-warp histograms (dynamic shared memory): counts, and masses as 64.64
// fixed point split into the fraction word and the integer word.
struct SelHist {
  unsigned int cnt[SEL_WARPS][256];
  unsigned long long lo[SEL_WARPS][256];
  unsigned long long hi[SEL_WARPS][256];
  u128 part[SEL_WARPS];
  // this CTA's bin totals, read by the other CTAs; two buffers by pass parity,
  // so a pass's totals are never overwritten while another CTA reads them
  unsigned int tot_cnt[2][256];
  unsigned long long tot_lo[2][256];
  unsigned long long tot_hi[2][256];
};

// Exact block-wide sum of per-thread fixed-point values, as a double.
__device__ double block_sum_fixed(u128 v, SelHist& h, SelShared& sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_sum_u128(v);
  __syncthreads();
  if (lane == 0) h.part[wid] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    u128 t = 0;
    for (int w = 0; w < SEL_WARPS; ++w) t += h.part[w];
    sh.total = fixed_to_double(t);
  }
  __syncthreads();
  const double r = sh.total;
  __syncthreads();
  return r;
}

// One radix pass over a row, this CTA taking indices [v0, v1): among the
// elements whose key matches `prefix` under `pmask` and that `keep` admits,
// the count (and with WITH_MASS the exact weight sum) per value of the key's
// byte at `shift`, summed over the cluster's CTAs into sh.cnt / sh.mass; with
// WITH_MASS, sh.total is the mass of all of them.  `buf` alternates between
// consecutive passes.  Every thread of every CTA of the cluster calls it.
template <bool WITH_MASS, typename Keep, typename Weight>
__device__ void radix_pass(const float* x, int v0, int v1, int shift, uint32_t prefix, uint32_t pmask, Keep keep,
                           Weight weight, int buf, unsigned C, SelHist& h, SelShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int b = lane; b < 256; b += 32) {
    h.cnt[wid][b] = 0u;
    if (WITH_MASS) h.lo[wid][b] = h.hi[wid][b] = 0ull;
  }
  __syncwarp();
  for (int vb = v0 + tid; vb < v1; vb += SEL_BATCH * SEL_THREADS) {
    float xs[SEL_BATCH];
#pragma unroll
    for (int j = 0; j < SEL_BATCH; ++j) {
      const int v = vb + j * SEL_THREADS;
      xs[j] = v < v1 ? __ldg(x + v) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < SEL_BATCH; ++j) {
      const int v = vb + j * SEL_THREADS;
      const uint32_t key = order_key(xs[j]);
      if (v >= v1 || (key & pmask) != prefix || !keep(key, v)) continue;
      const int b = (key >> shift) & 255;
      atomicAdd(&h.cnt[wid][b], 1u);
      if (WITH_MASS) {
        const u128 wf = to_fixed(weight(xs[j]));
        const unsigned long long lo = (unsigned long long)wf, hi = (unsigned long long)(wf >> 64);
        const unsigned long long old = atomicAdd(&h.lo[wid][b], lo);
        const unsigned long long carry = old > ~lo ? 1ull : 0ull;  // this add wrapped the fraction word
        if (hi | carry) atomicAdd(&h.hi[wid][b], hi + carry);
      }
    }
  }
  __syncthreads();
  if (tid < 256) {  // this CTA's bin totals
    unsigned int c = 0u;
    u128 m = 0;
    for (int w = 0; w < SEL_WARPS; ++w) {
      c += h.cnt[w][tid];
      if (WITH_MASS) m += ((u128)h.hi[w][tid] << 64) + h.lo[w][tid];
    }
    h.tot_cnt[buf][tid] = c;
    if (WITH_MASS) {
      h.tot_lo[buf][tid] = (unsigned long long)m;
      h.tot_hi[buf][tid] = (unsigned long long)(m >> 64);
    }
  }
  cluster_sync();
  u128 m = 0;
  if (tid < 256) {  // the cluster's bin totals
    unsigned int c = 0u;
    for (unsigned r = 0; r < C; ++r) {
      c += ld_peer_u32(peer(&h.tot_cnt[buf][tid], r));
      if (WITH_MASS)
        m += ((u128)ld_peer_u64(peer(&h.tot_hi[buf][tid], r)) << 64) + ld_peer_u64(peer(&h.tot_lo[buf][tid], r));
    }
    sh.cnt[tid] = (int)c;
    if (WITH_MASS) sh.mass[tid] = fixed_to_double(m);
  }
  if (WITH_MASS) {
    block_sum_fixed(m, h, sh);  // sh.total: the exact mass of every admitted element
  } else {
    __syncthreads();
  }
}

// The cluster-wide exact sum of per-thread fixed-point values, through slot
// `slot` of sh.csum (each slot serves one sum per launch).
__device__ double cluster_sum_fixed(u128 v, int slot, unsigned C, SelHist& h, SelShared& sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_sum_u128(v);
  __syncthreads();
  if (lane == 0) h.part[wid] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    u128 t = 0;
    for (int w = 0; w < SEL_WARPS; ++w) t += h.part[w];
    sh.csum[slot][0] = (unsigned long long)t;
    sh.csum[slot][1] = (unsigned long long)(t >> 64);
  }
  cluster_sync();
  if (threadIdx.x == 0) {
    u128 t = 0;
    for (unsigned r = 0; r < C; ++r)
      t += ((u128)ld_peer_u64(peer(&sh.csum[slot][1], r)) << 64) + ld_peer_u64(peer(&sh.csum[slot][0], r));
    sh.total = fixed_to_double(t);
  }
  __syncthreads();
  const double res = sh.total;
  __syncthreads();
  return res;
}

// Sum over the lanes above this one (fixed shuffle order).
template <typename T>
__device__ __forceinline__ T suffix_above(T v, int lane) {
  T incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T o = __shfl_down_sync(0xffffffffu, incl, off);
    if (lane + off < 32) incl += o;
  }
  return incl - v;
}

// Run by warp 0.  Finds the highest bin b with (weight of bins above b) +
// hist[b] >= need - the bin holding the need-th unit of weight counted from
// the top - and stores b and the weight strictly above it in sh.bin /
// sh.above.  If rounding leaves need above the total, the lowest non-empty bin.
template <typename T>
__device__ void find_bin(const T* hist, T need, int lane, SelShared& sh) {
  T s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += hist[8 * lane + j];
  const T ab = suffix_above(s, lane);
  const unsigned here = __ballot_sync(0xffffffffu, ab < need && ab + s >= need);
  const unsigned nonempty = __ballot_sync(0xffffffffu, s > T(0));
  const bool lowest = here == 0u;
  const int src = !lowest ? 31 - __clz(here) : (nonempty ? __ffs(nonempty) - 1 : 0);
  if (lane == src) {
    T acc = ab;
    int b = -1, low = -1;
    for (int j = 7; j >= 0; --j) {
      const T h = hist[8 * lane + j];
      if (h > T(0)) low = j;
      if (!lowest && acc + h >= need) {
        b = j;
        break;
      }
      acc += h;
    }
    if (b < 0) {  // rounding: the lowest non-empty bin of this lane
      b = low < 0 ? 0 : low;
      acc = ab;
      for (int j = 7; j > b; --j) acc += hist[8 * lane + j];
    }
    sh.bin = 8 * lane + b;
    sh.above = (double)acc;
  }
}

__device__ float block_max(float v, SelShared& sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  __syncthreads();
  if (lane == 0) sh.wsum[wid] = v;
  __syncthreads();
  float t = -INFINITY;
  for (int w = 0; w < SEL_WARPS; ++w) t = fmaxf(t, (float)sh.wsum[w]);
  __syncthreads();
  return t;
}

// The r-th (1-based) lowest index v <= limit whose key equals K, this CTA
// scanning [v0, v1).  Each thread counts a contiguous index range; the CTAs'
// counts (through slot `slot`) and a block scan in index order find the range
// that holds it.  Every thread of every CTA of the cluster calls it.
__device__ int tie_index(const float* x, int v0, int v1, uint32_t K, int limit, int r, int slot, unsigned C,
                         unsigned rank, SelShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n = max(0, min(v1, limit + 1) - v0);
  const int per = (n + SEL_THREADS - 1) / SEL_THREADS;
  const int a = v0 + min(n, tid * per), e = v0 + min(n, tid * per + per);
  int c = 0;
  for (int vb = a; vb < e; vb += SEL_BATCH) {
    float xs[SEL_BATCH];
#pragma unroll
    for (int j = 0; j < SEL_BATCH; ++j) xs[j] = vb + j < e ? __ldg(x + vb + j) : 0.f;
#pragma unroll
    for (int j = 0; j < SEL_BATCH; ++j) c += vb + j < e && order_key(xs[j]) == K;
  }
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) sh.wint[wid] = incl;
  if (tid == 0) sh.cfound[slot] = INT_MAX;
  __syncthreads();
  int base = 0, cta_total = 0;
  for (int w = 0; w < SEL_WARPS; ++w) {
    if (w < wid) base += sh.wint[w];
    cta_total += sh.wint[w];
  }
  if (tid == 0) sh.ccount[slot] = cta_total;
  cluster_sync();
  for (unsigned q = 0; q < rank; ++q) base += (int)ld_peer_u32(peer(&sh.ccount[slot], q));  // ties in earlier CTAs
  const int excl = base + incl - c;
  if (c > 0 && excl < r && excl + c >= r) {
    int k = excl;
    for (int v = a; v < e; ++v)
      if (order_key(x[v]) == K && ++k == r) {
        sh.cfound[slot] = v;
        break;
      }
  }
  cluster_sync();
  int found = INT_MAX;
  for (unsigned q = 0; q < C; ++q) found = min(found, (int)ld_peer_u32(peer(&sh.cfound[slot], q)));
  return found == INT_MAX ? limit : found;  // not reached only through rounding: keep every tie
}

__global__ void __launch_bounds__(SEL_THREADS) select_kernel(const SelectArgs p) {
  pdl_trigger();
  pdl_wait();
  __shared__ SelShared sh;
  extern __shared__ __align__(16) uint8_t sel_dyn[];
  SelHist& h = *reinterpret_cast<SelHist*>(sel_dyn);
  const unsigned C = cluster_ctas(), rank = cluster_rank();
  const int row = blockIdx.x / C, tid = threadIdx.x, lane = tid & 31;
  const float* x = p.x + (size_t)row * p.ldx;
  const int V = p.V;
  const int slice = (V + (int)C - 1) / (int)C;
  const int v0 = min(V, (int)rank * slice), v1 = min(V, v0 + slice);
  const bool probs = p.mode == SEL_PROBS;
  const float T = (p.mode == SEL_TOPN && !(p.temperature > 0.f)) ? 1.f : p.temperature;
  float xmax = 0.f;
  if (!probs) {
    if (p.mode == SEL_LOGITS && p.row_max) {
      xmax = p.row_max[row];
    } else {
      float mx = -INFINITY;
      for (int v = v0 + tid; v < v1; v += SEL_THREADS) mx = fmaxf(mx, x[v]);
      mx = block_max(mx, sh);
      if (tid == 0) sh.cmax = mx;
      cluster_sync();
      xmax = -INFINITY;
      for (unsigned q = 0; q < C; ++q) xmax = fmaxf(xmax, __uint_as_float(ld_peer_u32(peer(&sh.cmax, q))));
    }
  }
  // a token's weight: exp((z - max) / T) exactly as the accept step computes it, or the probability
  auto weight = [&](float xv) -> float { return probs ? xv : exp_term((xv - xmax) / T); };
  auto all = [](uint32_t, int) { return true; };
  int pass = 0;  // alternates the bin-total buffers

  // ---- top-k: the k-th key in the order (by counts), then its tie index
  const int k_lim = p.mode == SEL_TOPN ? min(p.top_n, V) : p.top_k;
  uint32_t Kk = 0u;
  int Ik = V - 1;
  if (k_lim > 0 && k_lim < V) {
    uint32_t prefix = 0u, pmask = 0u;
    int need = k_lim;
    for (int shift = 24; shift >= 0; shift -= 8) {
      radix_pass<false>(x, v0, v1, shift, prefix, pmask, all, weight, (pass++) & 1, C, h, sh);
      if (tid < 32) find_bin<int>(sh.cnt, need, lane, sh);
      __syncthreads();
      prefix |= (uint32_t)sh.bin << shift;
      pmask |= 255u << shift;
      need -= (int)sh.above;
      __syncthreads();
    }
    Kk = prefix;
    Ik = tie_index(x, v0, v1, Kk, V - 1, need, 0, C, rank, sh);
  }
  auto kept_k = [&](uint32_t key, int v) { return key > Kk || (key == Kk && v <= Ik); };

  // ---- top-p over the top-k survivors: the key (by mass) where the mass
  // counted from the top reaches top_p of theirs, then the tie index
  uint32_t K = Kk;
  int I = Ik;
  double kept_mass = 0.0;
  if (p.mode != SEL_TOPN && p.top_p < 1.f) {
    uint32_t prefix = 0u, pmask = 0u;
    double above_total = 0.0, theta = 0.0;
    int ties = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
      radix_pass<true>(x, v0, v1, shift, prefix, pmask, kept_k, weight, (pass++) & 1, C, h, sh);
      if (shift == 24) theta = (double)p.top_p * sh.total;  // the first pass sees every survivor
      // at least the smallest positive weight: rounding never turns the search upside down
      if (tid < 32) find_bin<double>(sh.mass, fmax(theta - above_total, 4.9e-324), lane, sh);
      __syncthreads();
      prefix |= (uint32_t)sh.bin << shift;
      pmask |= 255u << shift;
      above_total += sh.above;
      ties = sh.cnt[sh.bin];
      __syncthreads();
    }
    K = prefix;
    // every tied token has the same value, hence the same weight; the tied
    // tokens to keep and the kept mass are the same scalars for every thread,
    // so one thread computes them (fp64, a divide) and shares them
    if (tid == 0) {
      const uint32_t u = (K & 0x80000000u) ? (K & 0x7fffffffu) : ~K;
      const double wt = fixed_to_double(to_fixed(weight(__uint_as_float(u))));
      int r = wt > 0.0 ? (int)ceil((theta - above_total) / wt) : ties;
      r = max(1, min(r, ties));
      sh.bin = r;
      sh.above = above_total + (double)r * wt;
    }
    __syncthreads();
    const int r = sh.bin;
    kept_mass = sh.above;
    __syncthreads();
    I = tie_index(x, v0, v1, K, K == Kk ? Ik : V - 1, r, 1, C, rank, sh);
  } else if (p.mode != SEL_TOPN) {
    u128 w = 0;
    for (int v = v0 + tid; v < v1; v += SEL_THREADS) {
      const float xv = x[v];
      if (kept_k(order_key(xv), v)) w += to_fixed(weight(xv));
    }
    kept_mass = cluster_sum_fixed(w, 0, C, h, sh);
  }

  if (p.mode == SEL_LOGITS) {
    if (rank == 0 && tid == 0) {
      p.out_key[row] = K;
      p.out_idx[row] = I;
      p.out_norm[row] = (float)kept_mass;
    }
  } else if (p.mode == SEL_PROBS) {
    float* y = p.y + (size_t)row * p.ldy;
    if (tid == 0) sh.total = 1.0 / kept_mass;  // one fp64 divide, shared
    __syncthreads();
    const double inv = sh.total;
    for (int v = v0 + tid; v < v1; v += SEL_THREADS) {
      const float xv = x[v];
      const uint32_t key = order_key(xv);
      y[v] = (key > K || (key == K && v <= I)) ? (float)((double)xv * inv) : 0.f;
    }
  } else {
    // ---- SEL_TOPN: log-probabilities of the chosen token and of the top_n tokens
    u128 sx = 0;
    for (int v = v0 + tid; v < v1; v += SEL_THREADS) sx += to_fixed(exp_term((x[v] - xmax) / T));
    const double s_sum = cluster_sum_fixed(sx, 1, C, h, sh);
    if (tid == 0) sh.above = log(s_sum);  // one fp64 log, shared
    __syncthreads();
    const double log_s = sh.above;
    if (p.top_n > 0) {
      // each CTA lists its slice's kept tokens (k_lim of them in the whole row, at most 32)
      if (tid == 0) sh.n_top = 0;
      __syncthreads();
      for (int v = v0 + tid; v < v1; v += SEL_THREADS) {
        const uint32_t key = order_key(x[v]);
        if (kept_k(key, v)) {
          const int slot = atomicAdd(&sh.n_top, 1);
          if (slot < 32) {
            sh.top_key[slot] = key;
            sh.top_idx[slot] = v;
          }
        }
      }
      cluster_sync();
      if (rank == 0 && tid < 32) {  // the first CTA gathers the lists and ranks them
        uint32_t kl = 0u;
        int il = -1, n = 0;
        for (unsigned q = 0; q < C; ++q) {
          const int nq = min((int)ld_peer_u32(peer(&sh.n_top, q)), 32);
          if (lane >= n && lane < n + nq) {
            kl = ld_peer_u32(peer(&sh.top_key[lane - n], q));
            il = (int)ld_peer_u32(peer(&sh.top_idx[lane - n], q));
          }
          n = min(32, n + nq);
        }
        int rk = 0;
        for (int j = 0; j < n; ++j) {
          const uint32_t kj = __shfl_sync(0xffffffffu, kl, j);
          const int ij = __shfl_sync(0xffffffffu, il, j);
          rk += lane < n && (kj > kl || (kj == kl && ij < il));
        }
        if (lane < n && rk < p.top_n) {
          p.top_ids[(size_t)row * p.top_n + rk] = il;
          p.top_lp[(size_t)row * p.top_n + rk] = (float)(((double)x[il] - (double)xmax) / (double)T - log_s);
        }
      }
    }
    if (rank == 0 && tid == 0 && p.chosen) {
      const int c = p.chosen[row];
      p.chosen_lp[row] = (c >= 0 && c < V) ? (float)(((double)x[c] - (double)xmax) / (double)T - log_s) : NAN;
    }
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
}

// CTAs per row: the largest cluster of up to 8 that the device can place.
static int select_cluster() {
  static int cached = 0;
  if (cached) return cached;
  int c = SEL_MAX_CLUSTER;
  for (; c > 1; c >>= 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c);
    cfg.blockDim = dim3(SEL_THREADS);
    cfg.dynamicSmemBytes = sizeof(SelHist);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, select_kernel, &cfg) == cudaSuccess && n > 0) break;
    cudaGetLastError();  // clear a refusal; try a smaller cluster
  }
  cached = c;
  return c;
}

cudaError_t launch_select(const SelectArgs& a, int rows, cudaStream_t s) {
  static bool attr_set = false;  // the attribute is per function
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SelHist));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int c = select_cluster();
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(rows * c), dim3(SEL_THREADS), sizeof(SelHist), s, attr);
  attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
  attr[cfg.numAttrs].val.clusterDim.x = c;
  attr[cfg.numAttrs].val.clusterDim.y = 1;
  attr[cfg.numAttrs].val.clusterDim.z = 1;
  ++cfg.numAttrs;
  return cudaLaunchKernelEx(&cfg, select_kernel, a);
}

}  // namespace sv
