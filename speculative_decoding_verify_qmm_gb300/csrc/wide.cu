// Wide-block quantized matmul on the 5th-generation tensor cores (33..512 rows).
//
// mlx-dspark PyPI page, "Prompt processing (prefill)": wide blocks (prompt
// chunks, long verify blocks) dequantize the weights once per block rather
// than once per output tile; wiki page, "Key techniques": one weight group is
// dequantized once and reused across every row.  Past 32 rows the contraction
// is dense enough for tcgen05.mma: a CTA owns 128 weight rows, eight warps
// dequantize each 64-wide k-step of them into fp16 in shared memory (the
// 128-byte-swizzled K-major layout the tensor cores read), one thread issues
// tcgen05.mma with the weights as the 128-row A operand and the block's rows
// as the N operand (up to 256 per instruction), accumulating in fp32 in tensor
// memory, and the dequantizing warps read the accumulators back (tcgen05.ld)
// for the epilogue.  A producer warp keeps a ring of stages filled by TMA: the
// stage's raw codes, scales and biases, and the matching 64-wide slice of the
// activations, prepared once as fp16 scaled by a power of two per row (exact
// for every bf16 value; the scale is undone in the epilogue).
//
// Arithmetic: w = fp16(scale * code + bias) - one fused fp16 multiply-add of
// the exact code, so within half an fp16 ulp (relative 2^-11) of the exact
// affine weight and of the oracle's fp32 weight - times the exact fp16
// activations, fp32 accumulation.  A 32-bit word of W = 32 / bits codes is
// dequantized as the pairs (c_j, c_j+W/2): each is one mask of the shifted word
// OR'ed into the mantissa of 1024 (fp16 1024 + c, exact), one subtraction of
// 1024 and one fused multiply-add, two weights per instruction.  The weight
// row's k order inside each word is then 0, W/2, 1, W/2+1, ...; the prepared
// activations are stored in the same order, so the contraction is unchanged.  When a projection has too few 128-row
// tiles to fill the GPU, k is split across CTAs and a second kernel adds the
// fp32 partials in split order.
#include <cstring>

#include "sv_internal.h"
#include "sv_ptx.cuh"
#include "sv_tc05.cuh"

namespace sv {

constexpr int WT = 128;            // weight rows per tile (the MMA's M)
constexpr int WK = 64;             // k per stage: one 128-byte fp16 row
constexpr int W_DQ = 8;            // dequantizing (then epilogue) warps: two threads per weight row
constexpr int W_PROD = W_DQ;       // the TMA producer warp
constexpr int W_MMA = W_DQ + 1;    // the MMA-issuing warp, which also owns the tensor memory
constexpr int W_THREADS = (W_DQ + 2) * 32;
constexpr int W_MAX_STAGES = 6;

struct WideParams {
  CUtensorMap tm_codes, tm_scales, tm_biases, tm_x;
  int N, K, M, Mpad, stages, splits, ks_total;
  int mchunks, chunk;                // the block's rows in mchunks CTAs of `chunk` rows (<= 256, one MMA operand)
  int stage_bytes, codes_bytes;      // codes_bytes: one stage's raw codes (128 rows)
  uint32_t tmem_cols;
  const float* inv_scale;            // [Mpad]: 2^-e of each activation row
  __nv_bfloat16* y; int ldy;         // splits == 1: the output
  const __nv_bfloat16* res; int ldr; // optional residual (splits == 1)
  float* partials;                   // splits > 1: [splits][M][N] fp32
};

// Stage layout (1024-aligned): [A fp16 128 x 64, swizzled][X fp16 rows x 64, swizzled][codes][scales][biases]
__host__ __device__ inline int wide_x_off() { return WT * 128; }
__host__ __device__ inline int wide_codes_off(int rows) { return WT * 128 + rows * 128; }

// The W / 2 weight pairs (c_j, c_j+W/2) of one code word, W = 32 / BITS,
// as fp16 s * c + b.
template <int BITS>
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, __half2 b2, uint32_t* out) {
  constexpr uint32_t MASK = BITS == 8 ? 0x00ff00ffu : (BITS == 4 ? 0x000f000fu : 0x00030003u);
  const __half2 k1024 = __half2half2(__ushort_as_half((unsigned short)0x6400));
#pragma unroll
  for (int j = 0; j < 16 / BITS; ++j) {
    const uint32_t biased = ((w >> (BITS * j)) & MASK) | 0x64006400u;  // fp16 1024 + c in each half
    const __half2 c2 = __hsub2(*reinterpret_cast<const __half2*>(&biased), k1024);
    const __half2 w2 = __hfma2(s2, c2, b2);
    out[j] = *reinterpret_cast<const uint32_t*>(&w2);
  }
}

template <int BITS>
__global__ void __launch_bounds__(W_THREADS, 2) wide_kernel(const __grid_constant__ WideParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[W_MAX_STAGES], deq_bar[W_MAX_STAGES], empty_bar[W_MAX_STAGES], acc_bar, fin_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort_v = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.stages;
  // CTAs of one weight tile are adjacent (its row chunks and k splits run together and share it in L2)
  const int per_tile = p.mchunks * p.splits;
  const int tile = blockIdx.x / per_tile, mc = (blockIdx.x % per_tile) / p.splits, split = blockIdx.x % p.splits;
  const int n0 = tile * WT, m0 = mc * p.chunk;
  const int ks0 = (int)((long long)split * p.ks_total / p.splits);
  const int ks1 = (int)((long long)(split + 1) * p.ks_total / p.splits);
  const int nk = ks1 - ks0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&deq_bar[s], W_DQ);  // one arrival per dequantizing warp
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&acc_bar, 1);
    mbar_init(&fin_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(&s_tmem, p.tmem_cols);
    tmem_relinquish();
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();  // the prepared activations come from the previous launch

  if (warp == W_PROD) {
    // ============================================================ producer
    if (lane == 0) {
      const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
      const uint32_t tx = (uint32_t)(p.codes_bytes + 2 * WT * 8 * 2 + p.chunk * 128);
      bool bad = false;
      int i = 0;
      for (; i < nk; ++i) {
        const int s = i % S, ks = ks0 + i;
        if (i >= S && !mbar_wait_bounded(&empty_bar[s], ((i / S) - 1) & 1, abort_v)) {
          if (!*abort_v) raise_error(ERR_TIMEOUT_EMPTY);
          *abort_v = 1;
          bad = true;
          break;
        }
        uint8_t* st = smem + s * p.stage_bytes;
        uint8_t* codes = st + wide_codes_off(p.chunk);
        mbar_arrive_expect_tx(&full_bar[s], tx);
        tma_load_2d(codes, &p.tm_codes, &full_bar[s], ks * WK * BITS / 8, n0, pol_w);
        tma_load_2d(codes + p.codes_bytes, &p.tm_scales, &full_bar[s], (ks / 8) * 8, n0, pol_w);
        tma_load_2d(codes + p.codes_bytes + WT * 16, &p.tm_biases, &full_bar[s], (ks / 8) * 8, n0, pol_w);
        tma_load_2d(st + wide_x_off(), &p.tm_x, &full_bar[s], ks * WK, m0, pol_x);
      }
      // copies in flight land before the CTA may finish (bounded)
      if (!bad && !*abort_v) {
        for (int k = (i - S > 0 ? i - S : 0); k < i; ++k) mbar_wait_bounded(&full_bar[k % S], (k / S) & 1, abort_v);
      } else {
        const unsigned long long t0 = global_ns();
        while (global_ns() - t0 < 50000ull) __nanosleep(1000);
      }
    }
  } else if (warp == W_MMA) {
    // ============================================================ MMA issue
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk && !*abort_v; ++i) {
        const int s = i % S;
        if (!mbar_wait_bounded(&full_bar[s], (i / S) & 1, abort_v) ||
            !mbar_wait_bounded(&deq_bar[s], (i / S) & 1, abort_v)) {
          if (!*abort_v) raise_error(ERR_TIMEOUT_FULL);
          *abort_v = 1;
          break;
        }
        tc05_fence_after();
        const uint32_t a_base = smem_u32(smem + s * p.stage_bytes);
        const uint32_t x_base = a_base + wide_x_off();
#pragma unroll
        for (int kk = 0; kk < WK / 16; ++kk) {
          const uint64_t a_desc = sw128_desc(a_base + kk * 32);
          tc05_mma_f16(tmem, a_desc, sw128_desc(x_base + kk * 32), f16_idesc(WT, p.chunk), i > 0 || kk > 0);
        }
        tc05_commit(&empty_bar[s]);  // the stage is free once these MMAs have read it
        ++issued;
      }
      tc05_commit(&acc_bar);   // the accumulators are final once every MMA has completed
      // no MMA may still be running when the tensor memory is freed: this wait
      // ignores the abort flag and ends only on completion or the time limit
      tc05_commit(&fin_bar);
      volatile int never = 0;
      mbar_wait_bounded(&fin_bar, 0, &never);
      (void)issued;
    }
  } else {
    // ================================================= dequant, then epilogue
    // thread t: weight row r = t % 128 of the tile, k half h = t / 128 (32 codes)
    const int r = threadIdx.x & (WT - 1), h = threadIdx.x / WT;
    constexpr int HB = WK * BITS / 16;  // code bytes of half a row's k-step
    constexpr int PW = 16 / BITS;       // weight pairs per code word
    for (int i = 0; i < nk; ++i) {
      const int s = i % S, ks = ks0 + i;
      // the warp decides together: its arrival below is one per warp
      bool ok = !*abort_v && mbar_wait_bounded(&full_bar[s], (i / S) & 1, abort_v);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (!*abort_v) raise_error(ERR_TIMEOUT_FULL);
        *abort_v = 1;
        break;
      }
      uint8_t* st = smem + s * p.stage_bytes;
      const uint8_t* codes = st + wide_codes_off(p.chunk) + r * (WK * BITS / 8) + h * HB;
      const __half* sc = reinterpret_cast<const __half*>(st + wide_codes_off(p.chunk) + p.codes_bytes);
      const __half* bi = sc + WT * 8;
      const __half2 s2 = __half2half2(sc[r * 8 + (ks & 7)]);
      const __half2 b2 = __half2half2(bi[r * 8 + (ks & 7)]);
      uint32_t words[BITS];  // the thread's 32 codes
      if constexpr (BITS >= 4) {
#pragma unroll
        for (int j = 0; j < BITS; j += 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(codes + 4 * j);
          words[j] = v.x; words[j + 1] = v.y; words[j + 2] = v.z; words[j + 3] = v.w;
        }
      } else {  // 2-bit: 8 bytes per half row
        const uint2 v = *reinterpret_cast<const uint2*>(codes);
        words[0] = v.x; words[1] = v.y;
      }
      uint32_t pairs[16];
#pragma unroll
      for (int j = 0; j < BITS; ++j) dequant_word<BITS>(words[j], s2, b2, pairs + PW * j);
      uint8_t* arow = st + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int c = 4 * h + cc;  // 16-byte chunk (8 fp16) of the row's 128 bytes
        *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) =
            make_uint4(pairs[4 * cc], pairs[4 * cc + 1], pairs[4 * cc + 2], pairs[4 * cc + 3]);
      }
      fence_proxy_async_smem();  // the tensor cores read these writes through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&deq_bar[s]);
    }
    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (weight rows), the
    // first half of the columns (block rows) for w < 4, the second for w >= 4
    bool ok = !*abort_v && mbar_wait_bounded(&acc_bar, 0, abort_v);
    ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective: the whole warp reads or none
    tc05_fence_after();
    const int lq = warp & 3;
    const int nb = n0 + 32 * lq;  // this warp's 32 weight rows (the lane's is nb + lane)
    const int split_col = (p.chunk / 32) * 16;  // a multiple of 16: the loads read 16 columns at a time
    const int col0 = (warp >> 2) ? split_col : 0, col1 = (warp >> 2) ? p.chunk : split_col;
    // Scratch in the stage ring, idle once the accumulators are final (every
    // copy has landed and every MMA has read its stage): per warp 4 KB, the
    // row scales of its columns, then one 16 x 32 chunk in output order.
    float* const s_inv = reinterpret_cast<float*>(smem + warp * 4096);
    uint8_t* const s_buf = smem + warp * 4096 + 512;
    const bool partial_out = p.splits > 1;
    // 16-byte stores along an output row need aligned rows (and residual rows)
    const bool vec = partial_out
                         ? (p.N % 4 == 0)
                         : (p.ldy % 8 == 0 && (reinterpret_cast<uintptr_t>(p.y) & 15) == 0 &&
                            (!p.res || (p.ldr % 8 == 0 && (reinterpret_cast<uintptr_t>(p.res) & 15) == 0)));
    if (ok) {
      for (int i = lane; i < col1 - col0; i += 32) {
        const int m = m0 + col0 + i;
        s_inv[i] = m < p.M ? p.inv_scale[m] : 0.f;
      }
      __syncwarp();
      for (int col = col0; col < col1; col += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(32 * lq) << 16) + (uint32_t)col, v);
        const int mc = m0 + col;  // block row of column j: mc + j
        if (partial_out) {
          float* buf = reinterpret_cast<float*>(s_buf);  // [16][32]
#pragma unroll
          for (int j = 0; j < 16; ++j) buf[j * 32 + lane] = v[j] * s_inv[col - col0 + j];
          __syncwarp();
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int q = lane + 32 * t, j = q >> 3, c = q & 7, m = mc + j, nn = nb + 4 * c;
            if (m >= p.M) continue;
            float* dst = p.partials + ((size_t)split * p.M + m) * p.N + nn;
            if (vec && nn + 4 <= p.N) {
              *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(buf + j * 32 + 4 * c);
            } else {
              for (int e = 0; e < 4 && nn + e < p.N; ++e) dst[e] = buf[j * 32 + 4 * c + e];
            }
          }
        } else {
          __nv_bfloat16* buf = reinterpret_cast<__nv_bfloat16*>(s_buf);  // [16][32]
#pragma unroll
          for (int j = 0; j < 16; ++j) buf[j * 32 + lane] = __float2bfloat16_rn(v[j] * s_inv[col - col0 + j]);
          __syncwarp();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int q = lane + 32 * t, j = q >> 2, c = q & 3, m = mc + j, nn = nb + 8 * c;
            if (m >= p.M) continue;
            const __nv_bfloat16* src = buf + j * 32 + 8 * c;
            __nv_bfloat16* dst = p.y + (size_t)m * p.ldy + nn;
            if (vec && nn + 8 <= p.N) {
              uint4 o = *reinterpret_cast<const uint4*>(src);
              if (p.res) {  // y = bf16(residual + bf16(product)), element by element
                const uint4 rr = *reinterpret_cast<const uint4*>(p.res + (size_t)m * p.ldr + nn);
                const __nv_bfloat16* rb = reinterpret_cast<const __nv_bfloat16*>(&rr);
                __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(&o);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  ob[e] = __float2bfloat16_rn(__bfloat162float(rb[e]) + __bfloat162float(ob[e]));
              }
              *reinterpret_cast<uint4*>(dst) = o;
            } else {
              for (int e = 0; e < 8 && nn + e < p.N; ++e) {
                float out = __bfloat162float(src[e]);
                if (p.res) out = __bfloat162float(p.res[(size_t)m * p.ldr + nn + e]) + out;
                dst[e] = __float2bfloat16_rn(out);
              }
            }
          }
        }
        __syncwarp();  // the chunk buffer is rewritten by the next chunk
      }
    } else if (!*abort_v) {
      raise_error(ERR_TIMEOUT_FULL);
    }
  }
  tc05_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc05_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// Activations for the wide kernel: fp16 x * 2^e per row (e = 15 - exponent of
// the row's max |x|), 2^-e per row; rows M .. Mpad-1 zero.  Inside each block of
// W = 32 / bits k (one code word) the values are stored in the dequantized
// weights' order: position q holds k = q / 2 + (q % 2) * W / 2.  One block per row.
__global__ void __launch_bounds__(256) wide_prep_kernel(const __nv_bfloat16* __restrict__ x, int ldx, int M, int K,
                                                        int bits, __half* __restrict__ x16, float* __restrict__ inv) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x, tid = threadIdx.x;
  __shared__ float s_max[8];
  float mx = 0.f;
  if (m < M)
    for (int k = tid; k < K; k += 256) mx = fmaxf(mx, fabsf(__bfloat162float(x[(size_t)m * ldx + k])));
  for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((tid & 31) == 0) s_max[tid >> 5] = mx;
  __syncthreads();
  mx = 0.f;
  for (int w = 0; w < 8; ++w) mx = fmaxf(mx, s_max[w]);
  const int e = scale_exponent(mx);
  const float sc = pow2_exact(e);
  const int W = 32 / bits;
  for (int q = tid; q < K; q += 256) {
    const int k = (q & ~(W - 1)) + ((q & (W - 1)) >> 1) + (q & 1) * (W / 2);
    x16[(size_t)m * K + q] = __float2half_rn(m < M ? __bfloat162float(x[(size_t)m * ldx + k]) * sc : 0.f);
  }
  if (tid == 0) inv[m] = pow2_exact(-e);
}

// Sum of the split partials in split order, then bf16 (with the optional residual).
__global__ void __launch_bounds__(256) wide_finish_kernel(const float* __restrict__ part, int splits, int M, int N,
                                                          const __nv_bfloat16* __restrict__ res, int ldr,
                                                          __nv_bfloat16* __restrict__ y, int ldy) {
  pdl_trigger();
  pdl_wait();
  const size_t total = (size_t)M * N;
  for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < total; i += (size_t)gridDim.x * 256) {
    float acc = 0.f;
    for (int j = 0; j < splits; ++j) acc += part[(size_t)j * total + i];
    const int m = (int)(i / N), n = (int)(i % N);
    float out = __bfloat162float(__float2bfloat16_rn(acc));
    if (res) out = __bfloat162float(res[(size_t)m * ldr + n]) + out;
    y[(size_t)m * ldy + n] = __float2bfloat16_rn(out);
  }
}

struct WidePlan {
  int Mpad, mchunks, chunk, stages, splits, tiles, ks_total, stage_bytes, smem;
  size_t x16, inv, partials, total;
};

static WidePlan wide_plan(int M, int N, int K, int bits, int sms) {
  WidePlan w;
  // an MMA takes at most 256 rows (a multiple of 16): wider blocks are two
  // equal row chunks, each its own CTA
  w.mchunks = M > 256 ? 2 : 1;
  w.Mpad = w.mchunks == 1 ? 16 * ((M + 15) / 16) : 32 * ((M + 31) / 32);
  w.chunk = w.Mpad / w.mchunks;
  const int codes = WT * WK * bits / 8;
  w.stage_bytes = (wide_codes_off(w.chunk) + codes + 2 * WT * 16 + 1023) / 1024 * 1024;
  w.tiles = (N + WT - 1) / WT;
  w.ks_total = K / WK;
  uint32_t cols = 32;  // tensor-memory columns of one CTA's accumulators
  while ((int)cols < w.chunk) cols <<= 1;
  // Time model of a plan (CTAs per SM, stages S, k splits s), in us: each
  // k-step of a CTA is a chain of a copy, barrier hops, the dequantizing and
  // the MMAs, and each wave of CTAs has a fixed part (pipeline fill,
  // tensor-memory set-up, epilogue):
  //   waves x (k-steps x (0.514 + 1.071 / S + per_sm x (0.000202 rows - 0.076))
  //            + 3.57 - 0.00706 rows)
  //   + for s > 1: 2.44e-6 x M x N x s (fp32 partials out and back) + 5.35.
  // Least-squares fit (relative error) to 256 forced plans (one or two CTAs
  // per SM, 1-16 splits; 8-bit gate|up, down and q and 4-bit gate|up and down
  // shapes at 33, 64, 128, 256 and 512 rows): median error 5 %, and the plan
  // it picks is the measured best or within 6 % of it for every shape and
  // width (the picks' times sum to 1252 us against 1248 for the best).  Two
  // CTAs per SM (half the stages each, when their tensor memory and shared
  // memory fit) win when they put the grid in fewer waves, e.g. the 192
  // gate|up tiles at 64 rows: 103 us in two waves of one CTA per SM, 72 in one
  // wave of two.
  const int items = w.tiles * w.mchunks;
  const int max_split = w.ks_total / 8 > 0 ? w.ks_total / 8 : 1;
  const int one_sm_budget = 226 * 1024 - 1024;  // one CTA per SM; 1 KB of it aligns the stages
  const int two_sm_budget = 228 * 1024 / 2 - 2048 - 1024;  // per CTA: system reserve and barriers, alignment
  int best_stages = one_sm_budget / w.stage_bytes, best_split = 1;
  if (best_stages > W_MAX_STAGES) best_stages = W_MAX_STAGES;
  if (sms > 0) {
    double best = 1e30;
    for (int per_sm = 1; per_sm <= 2; ++per_sm) {
      int st = (per_sm == 1 ? one_sm_budget : two_sm_budget) / w.stage_bytes;
      if (st > W_MAX_STAGES) st = W_MAX_STAGES;
      if (st < 2 || per_sm * cols > 512) continue;
      const long long slots = (long long)sms * per_sm;
      const double step_us = 0.514 + 1.071 / st + per_sm * (0.000202 * w.chunk - 0.076);
      const double wave_us = 3.57 - 0.00706 * w.chunk;
      for (int sp = 1; sp <= max_split && sp <= 16; ++sp) {
        const double waves = (double)((items * (long long)sp + slots - 1) / slots);
        const double ksteps = (double)((w.ks_total + sp - 1) / sp);
        const double partials_us = sp > 1 ? 2.44e-6 * M * (double)N * sp + 5.35 : 0.0;
        const double cost = waves * (ksteps * step_us + wave_us) + partials_us;
        if (cost < best * (1.0 - 1e-9)) {
          best = cost;
          best_stages = st;
          best_split = sp;
        }
      }
    }
  }
  w.stages = best_stages;
  w.splits = best_split;
  w.smem = 1024 + w.stages * w.stage_bytes;
  size_t off = COUNTER_BYTES;
  w.x16 = off;      off = align256(off + (size_t)w.Mpad * K * 2);
  w.inv = off;      off = align256(off + (size_t)w.Mpad * 4);
  w.partials = off; off = align256(off + (w.splits > 1 ? (size_t)w.splits * M * N * 4 : 0));
  w.total = off;
  return w;
}

template <int BITS>
static cudaError_t launch_wide_t(const WideParams& p, int grid, int smem, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    // every plan needs at most 226 KB of dynamic shared memory (the rest of
    // the 227 KB opt-in limit holds the kernel's barriers)
    cudaError_t e = cudaFuncSetAttribute(wide_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         226 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(W_THREADS), smem, s, attr);
  return cudaLaunchKernelEx(&cfg, wide_kernel<BITS>, p);
}

size_t wide_bytes(int M, int N, int K, int bits) { return wide_plan(M, N, K, bits, device_sm_count()).total; }

int wide_qmm(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
             const uint16_t* x, int ldx, int M, uint16_t* y, int ldy, const uint16_t* residual, int ldr, void* ws,
             cudaStream_t s) {
  const int sms = device_sm_count();
  if (sms <= 0) return fail(SV_ECUDA, "no CUDA device");
  const WidePlan w = wide_plan(M, N, K, bits, sms);
  if (w.stages < 2) return fail(SV_EUNSUPPORTED, "rows %d need more shared memory than a CTA has", M);
  uint8_t* base = static_cast<uint8_t*>(ws);
  __half* x16 = reinterpret_cast<__half*>(base + w.x16);
  float* inv = reinterpret_cast<float*>(base + w.inv);
  {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(w.Mpad), dim3(256), 0, s, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, wide_prep_kernel, reinterpret_cast<const __nv_bfloat16*>(x), ldx, M, K,
                                       bits, x16, inv);
    if (e != cudaSuccess) return cuda_fail(e, "wide preparation launch");
  }
  static thread_local WideParams p;
  memset(static_cast<void*>(&p), 0, sizeof(p));
  const uint64_t row_bytes = (uint64_t)K * bits / 8, G = (uint64_t)(K / GROUP);
  int st = encode_tiled_2d(&p.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, row_bytes, (uint64_t)N, row_bytes,
                         (uint32_t)(WK * bits / 8), WT, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!st) st = encode_tiled_2d(&p.tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, G, (uint64_t)N, G * 2, 8, WT,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!st) st = encode_tiled_2d(&p.tm_biases, CU_TENSOR_MAP_DATA_TYPE_UINT16, biases, G, (uint64_t)N, G * 2, 8, WT,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!st) st = encode_tiled_2d(&p.tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, (uint64_t)K, (uint64_t)w.Mpad,
                              (uint64_t)K * 2, WK, w.chunk, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st) return st;
  p.N = N;
  p.K = K;
  p.M = M;
  p.Mpad = w.Mpad;
  p.mchunks = w.mchunks;
  p.chunk = w.chunk;
  p.stages = w.stages;
  p.splits = w.splits;
  p.ks_total = w.ks_total;
  p.stage_bytes = w.stage_bytes;
  p.codes_bytes = WT * WK * bits / 8;
  uint32_t cols = 32;
  while ((int)cols < w.chunk) cols <<= 1;
  p.tmem_cols = cols;
  p.inv_scale = inv;
  p.y = reinterpret_cast<__nv_bfloat16*>(y);
  p.ldy = ldy;
  p.res = reinterpret_cast<const __nv_bfloat16*>(residual);
  p.ldr = ldr;
  p.partials = w.splits > 1 ? reinterpret_cast<float*>(base + w.partials) : nullptr;
  const int grid = w.tiles * w.mchunks * w.splits;
  cudaError_t e = bits == 8 ? launch_wide_t<8>(p, grid, w.smem, s)
                            : (bits == 4 ? launch_wide_t<4>(p, grid, w.smem, s) : launch_wide_t<2>(p, grid, w.smem, s));
  if (e != cudaSuccess) return cuda_fail(e, "wide matmul launch");
  if (w.splits > 1) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(4 * sms), dim3(256), 0, s, attr);
    e = cudaLaunchKernelEx(&cfg, wide_finish_kernel, (const float*)p.partials, w.splits, M, N, p.res, ldr, p.y, ldy);
    if (e != cudaSuccess) return cuda_fail(e, "wide finish launch");
  }
  return SV_OK;
}

}  // namespace sv
