// Skinny affine-group-quantized matmul for the verify round:
//
//     Y[m, n] = sum_k X[m, k] * (scale[n, k/64] * code[n, k] + bias[n, k/64]),  M <= 32 rows.
//
// mlx-dspark wiki page, "Key techniques": the verify kernel dequantizes each
// weight group once and reuses it across all rows.  Here that becomes a
// factored form evaluated per group g and row n,
//
//     Y[m, n] += scale[n,g] * sum_{k in g} X[m,k] * (code[n,k] - off)  +  (bias[n,g] + off*scale[n,g]) * sum_{k in g} X[m,k]
//
// where the inner sum runs on the tensor cores (codes are exact small integers
// in fp16, `off` = 128 or 8 centres them) and the two group terms are applied
// in fp32 registers, so no weight is ever rounded to a 16-bit float.  The
// activations arrive as fp16 scaled by 2^e per (row, 512-wide k chunk) (see
// prep.cu); the chunk's 2^-e is folded in once per stage.
//
// Structure (one persistent CTA per SM, stream-K over (64-row tile, 512-k chunk)
// units so every SM streams the same number of weight bytes):
//   * warp 8, one lane: TMA producer.  Per stage it loads the 64 x 512 code
//     tile (128-byte swizzled boxes), the 64 x 8 scale and bias boxes, and the
//     matching slice of the prepared activations (bulk copies), into a ring
//     of shared-memory stages guarded by full/empty mbarriers.  Weights stream
//     with an L2 evict-first hint; the small activation slices with evict-last.
//   * warps 0-7: consumers, two per scheduler.  Warp w owns rows
//     32*(w/4) .. +31 of the tile and groups 2*(w%4), 2*(w%4)+1 of each stage:
//     ldmatrix the codes, turn them into fp16 with byte-permute / LOP3 tricks,
//     mma.sync m16n8k16 against the activation fragments, fold each group into
//     fp32 sums.
//   * at the end of a tile the four warps of each 32-row half add their sums in
//     a fixed order; a tile split across CTAs is finished by whichever
//     contributor arrives last (atomic counter, no spinning), which adds the
//     partials in CTA order, so results are bitwise reproducible.
#pragma once

#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {

constexpr int RT = 2;  // m16 row tiles per consumer warp (32 rows)

template <int BITS, int NT>
struct QmmCfg {
  static constexpr int MP = 8 * NT;
  static constexpr int ROW_BYTES = KC * BITS / 8;  // code bytes per row per stage
  static constexpr int ATOMS = ROW_BYTES / 128;    // 128-byte swizzle atoms per row
  static constexpr int W_BYTES = BN * ROW_BYTES;
  static constexpr int X_BYTES = MP * KC * 2;
  static constexpr int XS_BYTES = (GPS + 1) * MP * 4;  // group sums, then the chunk's 2^-e
  static constexpr int SB_BYTES = BN * GPS * 2;
  static constexpr int X_OFF = W_BYTES;
  static constexpr int XS_OFF = X_OFF + X_BYTES;
  static constexpr int S_OFF = (XS_OFF + XS_BYTES + 127) / 128 * 128;
  static constexpr int B_OFF = S_OFF + SB_BYTES;
  static constexpr int TX_BYTES = W_BYTES + X_BYTES + XS_BYTES + 2 * SB_BYTES;
  static constexpr int STAGE_BYTES = (B_OFF + SB_BYTES + 1023) / 1024 * 1024;
  static constexpr int HALF_RED = 32 * MP * 4;     // one reduction buffer (32 rows)
  static constexpr int RED_BYTES = 4 * HALF_RED;   // two buffers per half
  static constexpr int BUDGET = 227 * 1024 - 2048 - RED_BYTES;
  static constexpr int STAGES_FIT = BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + RED_BYTES;
  static_assert(STAGES >= 2, "stage ring too small");
  static_assert(SMEM <= 227 * 1024 - 1024, "shared memory budget");
};

__device__ __forceinline__ int owner_of(long long u, const Schedule& s) {
  return static_cast<int>(((u + 1) * s.grid - 1) / s.total_units);
}
__device__ __forceinline__ int unit_begin(int c, const Schedule& s) {
  return static_cast<int>(static_cast<long long>(c) * s.total_units / s.grid);
}

// fp16 pair (1024 + c0, 1024 + c1) from two code bytes, then centred: (c0 - 128, c1 - 128).
__device__ __forceinline__ uint32_t cvt8(uint32_t codes, uint32_t sel) {
  uint32_t v = __byte_perm(codes, 0x64646464u, sel);
  __half2 h = __hadd2(*reinterpret_cast<__half2*>(&v), __half2half2(__ushort_as_half(0xE480)));  // -1152
  return *reinterpret_cast<uint32_t*>(&h);
}
// Four fp16 pairs (n - 8) from the eight 4-bit codes of one word; nibble j is element 8t + j.
// P0 = (n0, n4), P1 = (n1, n5), P2 = (n2, n6), P3 = (n3, n7).
__device__ __forceinline__ void cvt4(uint32_t w, uint32_t (&P)[4]) {
  const __half2 sub = __half2half2(__ushort_as_half(0xE408));        // -1032
  const __half2 sixteenth = __half2half2(__ushort_as_half(0x2C00));  // 1/16
  const __half2 sub_hi = __half2half2(__ushort_as_half(0xD480));     // -72
  uint32_t lo = (w & 0x000F000Fu) | 0x64006400u;
  uint32_t hi = (w & 0x00F000F0u) | 0x64006400u;
  uint32_t w8 = w >> 8;
  uint32_t lo2 = (w8 & 0x000F000Fu) | 0x64006400u;
  uint32_t hi2 = (w8 & 0x00F000F0u) | 0x64006400u;
  __half2 r0 = __hadd2(*reinterpret_cast<__half2*>(&lo), sub);
  __half2 r1 = __hfma2(*reinterpret_cast<__half2*>(&hi), sixteenth, sub_hi);
  __half2 r2 = __hadd2(*reinterpret_cast<__half2*>(&lo2), sub);
  __half2 r3 = __hfma2(*reinterpret_cast<__half2*>(&hi2), sixteenth, sub_hi);
  P[0] = *reinterpret_cast<uint32_t*>(&r0);
  P[1] = *reinterpret_cast<uint32_t*>(&r1);
  P[2] = *reinterpret_cast<uint32_t*>(&r2);
  P[3] = *reinterpret_cast<uint32_t*>(&r3);
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&a)[RT][NT][4]) {
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int j = 0; j < NT; ++j) a[r][j][0] = a[r][j][1] = a[r][j][2] = a[r][j][3] = 0.f;
}

// One consumer warp's share of one stage: groups 2kq, 2kq+1 for rows 32nh .. 32nh+31.
template <int BITS, int NT>
__device__ __forceinline__ void consume_stage(const uint8_t* st, int nh, int kq, int lane, float (&tot)[RT][NT][4]) {
  using C = QmmCfg<BITS, NT>;
  constexpr int MP = C::MP;
  constexpr float OFF = BITS == 8 ? 128.f : 8.f;
  const int gid = lane >> 2, t = lane & 3;
  const uint32_t w_base = smem_u32(st);
  const uint32_t x_base = smem_u32(st + C::X_OFF);
  const float* xs = reinterpret_cast<const float*>(st + C::XS_OFF);
  const uint32_t* sc = reinterpret_cast<const uint32_t*>(st + C::S_OFF);  // [64][4] half2 words
  const uint32_t* bi = reinterpret_cast<const uint32_t*>(st + C::B_OFF);
  // ldmatrix lane roles: matrix mi = lane/8 (row half = mi&1, chunk = mi>>1), row-in-matrix rr = lane%8
  const int mi = lane >> 3, rr = lane & 7;

  float sacc[RT][NT][4];
  zero_acc<NT>(sacc);
  // scale / bias pairs of this warp's two groups for its four rows per m-tile
  float s_v[RT][2][2], b_v[RT][2][2];  // [r][lo/hi][group]
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = 32 * nh + 16 * r + gid + 8 * h;
      const __half2 s2 = *reinterpret_cast<const __half2*>(sc + n * 4 + kq);
      const __half2 b2 = *reinterpret_cast<const __half2*>(bi + n * 4 + kq);
      s_v[r][h][0] = __low2float(s2);
      s_v[r][h][1] = __high2float(s2);
      b_v[r][h][0] = fmaf(OFF, s_v[r][h][0], __low2float(b2));
      b_v[r][h][1] = fmaf(OFF, s_v[r][h][1], __high2float(b2));
    }

#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const int gl = 2 * kq + gi;  // group index within the stage
    uint32_t bfr[2][NT][4];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk)
#pragma unroll
      for (int j = 0; j < NT; ++j)
        lds128(bfr[blk][j], x_base + ((((gl * 2 + blk) * MP + 8 * j + gid) * 32 + 8 * t) * 2));
    float2 xsv[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) xsv[j] = *reinterpret_cast<const float2*>(xs + gl * MP + 8 * j + 2 * t);

#pragma unroll
    for (int r = 0; r < RT; ++r) {
      float acc[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
      const int lrow = 32 * nh + 16 * r + (mi & 1) * 8 + rr;  // row this lane addresses for ldmatrix
      if constexpr (BITS == 8) {
        // atom kq holds groups 2kq, 2kq+1; group gi = 16-byte chunks 4gi .. 4gi+3 (one k16 step each)
        const uint32_t arow = w_base + kq * (BN * 128) + lrow * 128;
        uint32_t q[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int chunk = 4 * gi + 2 * h + (mi >> 1);
          ldsm_x4(q[h], arow + ((chunk ^ rr) << 4));
        }
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint32_t lo = q[s >> 1][(s & 1) * 2], hi = q[s >> 1][(s & 1) * 2 + 1];
          uint32_t a[4] = {cvt8(lo, 0x4140u), cvt8(hi, 0x4140u), cvt8(lo, 0x4342u), cvt8(hi, 0x4342u)};
#pragma unroll
          for (int j = 0; j < NT; ++j)
            mma_16816(acc[j], a, bfr[s >> 1][j][(s & 1) * 2], bfr[s >> 1][j][(s & 1) * 2 + 1]);
        }
      } else {
        // atom kq/2 holds groups 4(kq/2) .. +3; group gi = chunks (kq&1)*4 + 2gi + {0,1}
        const uint32_t arow = w_base + (kq >> 1) * (BN * 128) + lrow * 128;
        const int chunk = (kq & 1) * 4 + 2 * gi + (mi >> 1);
        uint32_t q[4];
        ldsm_x4(q, arow + ((chunk ^ rr) << 4));
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t Plo[4], Phi[4];
          cvt4(q[2 * c], Plo);
          cvt4(q[2 * c + 1], Phi);
          uint32_t a0[4] = {Plo[0], Phi[0], Plo[1], Phi[1]};
          uint32_t a1[4] = {Plo[2], Phi[2], Plo[3], Phi[3]};
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            mma_16816(acc[j], a0, bfr[c][j][0], bfr[c][j][1]);
            mma_16816(acc[j], a1, bfr[c][j][2], bfr[c][j][3]);
          }
        }
      }
      // fold the group: sacc += s * acc + (b + off*s) * xsum   (chunk-scaled domain)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        sacc[r][j][0] = fmaf(s_v[r][0][gi], acc[j][0], fmaf(b_v[r][0][gi], xsv[j].x, sacc[r][j][0]));
        sacc[r][j][1] = fmaf(s_v[r][0][gi], acc[j][1], fmaf(b_v[r][0][gi], xsv[j].y, sacc[r][j][1]));
        sacc[r][j][2] = fmaf(s_v[r][1][gi], acc[j][2], fmaf(b_v[r][1][gi], xsv[j].x, sacc[r][j][2]));
        sacc[r][j][3] = fmaf(s_v[r][1][gi], acc[j][3], fmaf(b_v[r][1][gi], xsv[j].y, sacc[r][j][3]));
      }
    }
  }
  // undo the chunk's activation scale: tot += 2^-e[m] * sacc
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float2 f = *reinterpret_cast<const float2*>(xs + GPS * MP + 8 * j + 2 * t);
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      tot[r][j][0] = fmaf(f.x, sacc[r][j][0], tot[r][j][0]);
      tot[r][j][1] = fmaf(f.y, sacc[r][j][1], tot[r][j][1]);
      tot[r][j][2] = fmaf(f.x, sacc[r][j][2], tot[r][j][2]);
      tot[r][j][3] = fmaf(f.y, sacc[r][j][3], tot[r][j][3]);
    }
  }
}

template <int NT>
__device__ __forceinline__ void red_store(float* buf, const float (&tot)[RT][NT][4], int lane) {
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) buf[((r * NT + j) * 4 + e) * 32 + lane] = tot[r][j][e];
}
template <int NT, bool GLOBAL>
__device__ __forceinline__ void red_add(const float* buf, float (&tot)[RT][NT][4], int lane) {
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float* a = buf + ((r * NT + j) * 4 + e) * 32 + lane;
        tot[r][j][e] += GLOBAL ? __ldcg(a) : *a;
      }
}

// Final epilogue of one 32-row half of a tile, run by one warp holding its whole sum.
template <int NT>
__device__ __forceinline__ void half_epilogue(const QmmParams& p, int tile, int nh, const float (&tot)[RT][NT][4],
                                              int lane) {
  const int gid = lane >> 2, t = lane & 3;
  const int n0 = tile * BN + 32 * nh;
  // per-column factor: the RMSNorm scale 1/sqrt(mean(x^2) + eps) of the activation
  // row when the input was prepared with RMSNorm, else 1
  const int chunks = p.sch.K / KC;
  float rf[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int m = 8 * j + 2 * t + c;
      const float eps = __ldcg(p.rms + (size_t)chunks * p.MP + m);
      float f = 1.f;
      if (eps >= 0.f) {
        float ss = 0.f;
        for (int q = 0; q < chunks; ++q) ss += __ldcg(p.rms + (size_t)q * p.MP + m);
        f = 1.f / sqrtf(ss / (float)p.sch.K + eps);
      }
      rf[j][c] = f;
    }
  if (p.mode != EPI_LOGITS) {
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = n0 + 16 * r + gid + (e >> 1) * 8;
          const int m = 8 * j + 2 * t + (e & 1);
          if (n < p.sch.N && m < p.M) {
            __nv_bfloat16 yb = __float2bfloat16_rn(tot[r][j][e] * rf[j][e & 1]);
            if (p.mode == EPI_BF16_RESIDUAL)
              yb = __float2bfloat16_rn(__bfloat162float(p.res[(size_t)m * p.ldres + n]) + __bfloat162float(yb));
            p.y[(size_t)m * p.ldy + n] = yb;
          }
        }
    return;
  }
  // logits + per-row stats of these 32 columns
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int m = 8 * j + 2 * t + c;
      float best = -INFINITY;
      int bidx = 0x7fffffff;
      float v[RT][2];
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = n0 + 16 * r + gid + 8 * h;
          v[r][h] = tot[r][j][2 * h + c] * rf[j][c];
          if (n < p.sch.N) {
            if (m < p.M) p.logits[(size_t)m * p.ldl + n] = v[r][h];
            if (v[r][h] > best) { best = v[r][h]; bidx = n; }  // ascending n: first maximum kept
          }
        }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, off);
        if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
      }
      float se = 0.f;
      if (p.inv_temp > 0.f) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (n0 + 16 * r + gid + 8 * h < p.sch.N) se += expf((v[r][h] - best) * p.inv_temp);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) se += __shfl_xor_sync(0xffffffffu, se, off);
      }
      if (gid == 0) {
        float* ts = p.tile_stats + ((size_t)(tile * 2 + nh) * p.MP + m) * 3;
        ts[0] = best;
        ts[1] = __int_as_float(bidx);
        ts[2] = se;
      }
    }
}

template <int BITS, int NT>
__global__ void __launch_bounds__(QMM_THREADS, 1)
qmm_stream_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                  const __grid_constant__ CUtensorMap tm_b, const QmmParams p) {
  using C = QmmCfg<BITS, NT>;
  constexpr int STAGES = C::STAGES;
  constexpr int HALF_FLOATS = C::HALF_RED / 4;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);  // [half][2][32*MP]
  volatile int* abort_v = &abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Schedule& sch = p.sch;
  const int upt = sch.units_per_tile;
  const int u_begin = unit_begin(blockIdx.x, sch);
  const int u_end = unit_begin(blockIdx.x + 1, sch);
  const int n_units = u_end - u_begin;
  const int first_tile = u_begin / upt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], NCW);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_w);
      prefetch_tensormap(&tm_s);
      prefetch_tensormap(&tm_b);
      const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
      const int pre = n_units < STAGES ? n_units : STAGES;
      auto load_weights = [&](int i) {
        const int u = u_begin + i, tile = u / upt, kc = u % upt, s = i % STAGES;
        uint8_t* st = smem + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full_bar[s], C::TX_BYTES);
#pragma unroll
        for (int a = 0; a < C::ATOMS; ++a)
          tma_load_2d(st + a * (BN * 128), &tm_w, &full_bar[s], kc * C::ROW_BYTES + a * 128, tile * BN, pol_w);
        tma_load_2d(st + C::S_OFF, &tm_s, &full_bar[s], kc * GPS, tile * BN, pol_w);
        tma_load_2d(st + C::B_OFF, &tm_b, &full_bar[s], kc * GPS, tile * BN, pol_w);
      };
      auto load_acts = [&](int i) {
        const int u = u_begin + i, kc = u % upt, s = i % STAGES;
        uint8_t* st = smem + s * C::STAGE_BYTES;
        bulk_load(st + C::X_OFF, p.xp + (size_t)kc * (KC / 32) * C::MP * 32, C::X_BYTES, &full_bar[s], pol_x);
        bulk_load(st + C::XS_OFF, p.xsum + (size_t)kc * (GPS + 1) * C::MP, C::XS_BYTES, &full_bar[s], pol_x);
      };
      // Weights never depend on earlier kernels: start streaming them before
      // waiting for the producer of the activations.
      for (int i = 0; i < pre; ++i) load_weights(i);
      pdl_wait();
      for (int i = 0; i < pre; ++i) load_acts(i);
      for (int i = pre; i < n_units; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait_bounded(&empty_bar[s], ((i / STAGES) - 1) & 1, abort_v)) {
          raise_error(ERR_TIMEOUT_EMPTY);
          *abort_v = 1;
          // drain: wait (bounded) for copies already issued into the ring
          for (int k = (i - STAGES > 0 ? i - STAGES : 0); k < i; ++k)
            mbar_wait_bounded(&full_bar[k % STAGES], (k / STAGES) & 1, abort_v);
          break;
        }
        load_weights(i);
        load_acts(i);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int nh = warp >> 2, kq = warp & 3;
  float* red0 = red + (nh * 2 + 0) * HALF_FLOATS;
  float* red1 = red + (nh * 2 + 1) * HALF_FLOATS;
  pdl_wait();
  float tot[RT][NT][4];
  zero_acc<NT>(tot);

  for (int i = 0; i < n_units; ++i) {
    const int u = u_begin + i, tile = u / upt, kc = u % upt, s = i % STAGES;
    if (!*abort_v) {
      if (mbar_wait_bounded(&full_bar[s], (i / STAGES) & 1, abort_v)) {
        consume_stage<BITS, NT>(smem + s * C::STAGE_BYTES, nh, kq, lane, tot);
      } else {
        raise_error(ERR_TIMEOUT_FULL);
        *abort_v = 1;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);

    if (kc == upt - 1 || i == n_units - 1) {
      // ---- fixed-order sum of the half's four warps: (k0 + k2) + (k1 + k3)
      const int bar = 1 + nh;
      named_bar_sync(bar, 128);
      if (kq == 2) red_store<NT>(red0, tot, lane);
      if (kq == 3) red_store<NT>(red1, tot, lane);
      named_bar_sync(bar, 128);
      if (kq == 0) red_add<NT, false>(red0, tot, lane);
      if (kq == 1) red_add<NT, false>(red1, tot, lane);
      named_bar_sync(bar, 128);
      if (kq == 1) red_store<NT>(red0, tot, lane);
      named_bar_sync(bar, 128);
      if (kq == 0) {
        red_add<NT, false>(red0, tot, lane);
        const int c_first = owner_of((long long)tile * upt, sch);
        const int c_last = owner_of((long long)tile * upt + upt - 1, sch);
        if (c_first == c_last) {
          half_epilogue<NT>(p, tile, nh, tot, lane);
        } else {
          const int slot = (tile == first_tile) ? 0 : 1;
          float* mine = p.partials + (((size_t)blockIdx.x * 2 + slot) * 2 + nh) * HALF_FLOATS;
          red_store<NT>(mine, tot, lane);
          __threadfence();
          __syncwarp();
          int last = 0;
          if (lane == 0) last = (atomicAdd(p.counters + tile * 2 + nh, 1) == c_last - c_first);
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) {
            __threadfence();
            zero_acc<NT>(tot);
            for (int c = c_first; c <= c_last; ++c) {
              const int cslot = (tile == unit_begin(c, sch) / upt) ? 0 : 1;
              red_add<NT, true>(p.partials + (((size_t)c * 2 + cslot) * 2 + nh) * HALF_FLOATS, tot, lane);
            }
            half_epilogue<NT>(p, tile, nh, tot, lane);
            if (lane == 0) p.counters[tile * 2 + nh] = 0;
          }
        }
      }
      zero_acc<NT>(tot);
    }
  }
}

}  // namespace sv
