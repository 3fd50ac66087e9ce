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
// One CTA per row.  The kept set is always "key > K, or key == K and index
// <= I" for an order-preserving 32-bit key of the value: a radix select over
// the key's four bytes (most significant first) finds K - by counts for
// top_k, by mass for top_p - and one scan over the tied keys finds I.
// Everything stays in the CTA, so these calls need no workspace.
//
// Masses are summed exactly: every weight (a probability, or an fp32 exp
// term, both at most 1 for valid rows) is a 64.64 fixed-point integer, exact
// for weights from 2^-40 up and truncated below, and integer sums do not
// depend on their order.  Each warp keeps private 256-bin histograms,
// updated with shared-memory atomics (a mass as a 64-bit add on its fraction
// word that carries into its integer word), so a hot bin is contended only
// within a warp (a probability row puts nearly every key in a handful of
// top-byte bins).
#include <cmath>

#include "sv_internal.h"
#include "sv_ptx.cuh"
#include "sv_kernels.h"

namespace sv {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;

struct SelShared {
  int cnt[256];
  double mass[256];
  double wsum[SEL_WARPS];
  int wint[SEL_WARPS];
  int bin;
  double above;
  double total;
  int ifound;
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

// One radix pass over a row: among the elements whose key matches `prefix`
// under `pmask` and that `keep` admits, the count (and with WITH_MASS the
// exact weight sum) per value of the key's byte at `shift`, into sh.cnt /
// sh.mass; with WITH_MASS, sh.total is the mass of all of them.  Every thread
// of the block calls it.
template <bool WITH_MASS, typename Keep, typename Weight>
__device__ void radix_pass(const float* x, int V, int shift, uint32_t prefix, uint32_t pmask, Keep keep, Weight weight,
                           SelHist& h, SelShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int b = lane; b < 256; b += 32) {
    h.cnt[wid][b] = 0u;
    if (WITH_MASS) h.lo[wid][b] = h.hi[wid][b] = 0ull;
  }
  __syncwarp();
  for (int v = tid; v < V; v += SEL_THREADS) {
    const float xv = x[v];
    const uint32_t key = order_key(xv);
    if ((key & pmask) != prefix || !keep(key, v)) continue;
    const int b = (key >> shift) & 255;
    atomicAdd(&h.cnt[wid][b], 1u);
    if (WITH_MASS) {
      const u128 wf = to_fixed(weight(xv));
      const unsigned long long lo = (unsigned long long)wf, hi = (unsigned long long)(wf >> 64);
      const unsigned long long old = atomicAdd(&h.lo[wid][b], lo);
      const unsigned long long carry = old > ~lo ? 1ull : 0ull;  // this add wrapped the fraction word
      if (hi | carry) atomicAdd(&h.hi[wid][b], hi + carry);
    }
  }
  __syncthreads();
  u128 m = 0;
  for (int b = tid; b < 256; b += SEL_THREADS) {
    unsigned int c = 0u;
    for (int w = 0; w < SEL_WARPS; ++w) {
      c += h.cnt[w][b];
      if (WITH_MASS) m += ((u128)h.hi[w][b] << 64) + h.lo[w][b];
    }
    sh.cnt[b] = (int)c;
    if (WITH_MASS) sh.mass[b] = fixed_to_double(m);
  }
  if (WITH_MASS) {
    block_sum_fixed(m, h, sh);  // sh.total: the exact mass of every admitted element
  } else {
    __syncthreads();
  }
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

__device__ double block_sum(double v, SelShared& sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if (lane == 0) sh.wsum[wid] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < SEL_WARPS; ++w) t += sh.wsum[w];  // fixed order
  __syncthreads();
  return t;
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

// The r-th (1-based) lowest index v <= limit whose key equals K.  Each thread
// counts its contiguous index range; a block scan in index order finds the
// range that holds it.
__device__ int tie_index(const float* x, int V, uint32_t K, int limit, int r, SelShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (V + SEL_THREADS - 1) / SEL_THREADS;
  const int a = min(V, tid * per), e = min(V, min(a + per, limit + 1));
  int c = 0;
  for (int v = a; v < e; ++v) c += order_key(x[v]) == K;
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) sh.wint[wid] = incl;
  if (tid == 0) sh.ifound = limit;  // not reached only through rounding: keep every tie
  __syncthreads();
  int base = 0;
  for (int w = 0; w < wid; ++w) base += sh.wint[w];
  const int excl = base + incl - c;
  if (c > 0 && excl < r && excl + c >= r) {
    int k = excl;
    for (int v = a; v < e; ++v)
      if (order_key(x[v]) == K && ++k == r) {
        sh.ifound = v;
        break;
      }
  }
  __syncthreads();
  const int found = sh.ifound;
  __syncthreads();
  return found;
}

__global__ void __launch_bounds__(SEL_THREADS) select_kernel(const SelectArgs p) {
  pdl_trigger();
  pdl_wait();
  __shared__ SelShared sh;
  extern __shared__ __align__(16) uint8_t sel_dyn[];
  SelHist& h = *reinterpret_cast<SelHist*>(sel_dyn);
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const float* x = p.x + (size_t)row * p.ldx;
  const int V = p.V;
  const bool probs = p.mode == SEL_PROBS;
  const float T = (p.mode == SEL_TOPN && !(p.temperature > 0.f)) ? 1.f : p.temperature;
  float xmax = 0.f;
  if (!probs) {
    if (p.mode == SEL_LOGITS && p.row_max) {
      xmax = p.row_max[row];
    } else {
      float mx = -INFINITY;
      for (int v = tid; v < V; v += SEL_THREADS) mx = fmaxf(mx, x[v]);
      xmax = block_max(mx, sh);
    }
  }
  // a token's weight: exp((z - max) / T) exactly as the accept step computes it, or the probability
  auto weight = [&](float xv) -> float { return probs ? xv : exp_term((xv - xmax) / T); };
  auto all = [](uint32_t, int) { return true; };

  // ---- top-k: the k-th key in the order (by counts), then its tie index
  const int k_lim = p.mode == SEL_TOPN ? min(p.top_n, V) : p.top_k;
  uint32_t Kk = 0u;
  int Ik = V - 1;
  if (k_lim > 0 && k_lim < V) {
    uint32_t prefix = 0u, pmask = 0u;
    int need = k_lim;
    for (int shift = 24; shift >= 0; shift -= 8) {
      radix_pass<false>(x, V, shift, prefix, pmask, all, weight, h, sh);
      if (tid < 32) find_bin<int>(sh.cnt, need, lane, sh);
      __syncthreads();
      prefix |= (uint32_t)sh.bin << shift;
      pmask |= 255u << shift;
      need -= (int)sh.above;
      __syncthreads();
    }
    Kk = prefix;
    Ik = tie_index(x, V, Kk, V - 1, need, sh);
  }
  auto kept_k = [&](uint32_t key, int v) { return key > Kk || (key == Kk && v <= Ik); };

  // ---- top-p over the top-k survivors: the key (by mass) where the mass
  // counted from the top reaches top_p of theirs, then the tie index
  uint32_t K = Kk;
  int I = Ik;
  double kept_mass;
  if (p.mode != SEL_TOPN && p.top_p < 1.f) {
    uint32_t prefix = 0u, pmask = 0u;
    double above_total = 0.0, theta = 0.0;
    int ties = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
      radix_pass<true>(x, V, shift, prefix, pmask, kept_k, weight, h, sh);
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
    // every tied token has the same value, hence the same weight
    float xk = 0.f;
    {
      const uint32_t u = (K & 0x80000000u) ? (K & 0x7fffffffu) : ~K;
      xk = __uint_as_float(u);
    }
    const double wt = fixed_to_double(to_fixed(weight(xk)));
    int r = wt > 0.0 ? (int)ceil((theta - above_total) / wt) : ties;
    r = max(1, min(r, ties));
    I = tie_index(x, V, K, K == Kk ? Ik : V - 1, r, sh);
    kept_mass = above_total + (double)r * wt;
  } else if (p.mode != SEL_TOPN) {
    u128 w = 0;
    for (int v = tid; v < V; v += SEL_THREADS) {
      const float xv = x[v];
      if (kept_k(order_key(xv), v)) w += to_fixed(weight(xv));
    }
    kept_mass = block_sum_fixed(w, h, sh);
  } else {
    kept_mass = 0.0;
  }

  if (p.mode == SEL_LOGITS) {
    if (tid == 0) {
      p.out_key[row] = K;
      p.out_idx[row] = I;
      p.out_norm[row] = (float)kept_mass;
    }
    return;
  }
  if (p.mode == SEL_PROBS) {
    float* y = p.y + (size_t)row * p.ldy;
    const double inv = 1.0 / kept_mass;
    for (int v = tid; v < V; v += SEL_THREADS) {
      const float xv = x[v];
      const uint32_t key = order_key(xv);
      y[v] = (key > K || (key == K && v <= I)) ? (float)((double)xv * inv) : 0.f;
    }
    return;
  }

  // ---- SEL_TOPN: log-probabilities of the chosen token and of the top_n tokens
  u128 s = 0;
  for (int v = tid; v < V; v += SEL_THREADS) s += to_fixed(exp_term((x[v] - xmax) / T));
  const double log_s = log(block_sum_fixed(s, h, sh));
  if (p.top_n == 0) {
    if (tid == 0 && p.chosen) {
      const int c = p.chosen[row];
      p.chosen_lp[row] = (c >= 0 && c < V) ? (float)(((double)x[c] - (double)xmax) / (double)T - log_s) : NAN;
    }
    return;
  }
  if (tid == 0) sh.n_top = 0;
  __syncthreads();
  for (int v = tid; v < V; v += SEL_THREADS) {
    const uint32_t key = order_key(x[v]);
    if (kept_k(key, v)) {
      const int slot = atomicAdd(&sh.n_top, 1);
      if (slot < 32) {
        sh.top_key[slot] = key;
        sh.top_idx[slot] = v;
      }
    }
  }
  __syncthreads();
  if (tid < 32) {
    const int n = min(sh.n_top, 32);
    if (lane < n) {
      const uint32_t kl = sh.top_key[lane];
      const int il = sh.top_idx[lane];
      int rank = 0;
      for (int j = 0; j < n; ++j) {
        const uint32_t kj = sh.top_key[j];
        rank += kj > kl || (kj == kl && sh.top_idx[j] < il);
      }
      if (rank < p.top_n) {
        p.top_ids[(size_t)row * p.top_n + rank] = il;
        p.top_lp[(size_t)row * p.top_n + rank] = (float)(((double)x[il] - (double)xmax) / (double)T - log_s);
      }
    }
    if (lane == 0 && p.chosen) {
      const int c = p.chosen[row];
      p.chosen_lp[row] = (c >= 0 && c < V) ? (float)(((double)x[c] - (double)xmax) / (double)T - log_s) : NAN;
    }
  }
}

cudaError_t launch_select(const SelectArgs& a, int rows, cudaStream_t s) {
  static bool attr_set = false;  // the attribute is per function
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SelHist));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(rows), dim3(SEL_THREADS), sizeof(SelHist), s, attr);
  return cudaLaunchKernelEx(&cfg, select_kernel, a);
}

}  // namespace sv
