// Persistent multi-phase verify matmul.
//
// One launch runs a sequence of "phases"; each phase is one skinny
// affine-group-quantized matmul of the verify round (a q|k|v, o, gate|up, down
// or vocab-head projection):
//
//     Y[m, n] = sum_k X[m, k] * (scale[n, k/64] * code[n, k] + bias[n, k/64]),  M <= 32 rows.
//
// mlx-dspark wiki page, "Key techniques": the verify kernel dequantizes each
// weight group once and reuses it across all rows.  Here that is a factored
// form evaluated per group g and weight row n,
//
//     Y[m, n] += scale[n,g] * sum_{k in g} X[m,k] * (code[n,k] - off)  +  (bias[n,g] + off*scale[n,g]) * sum_{k in g} X[m,k]
//
// with the inner sums on the tensor cores (codes are exact small integers in
// fp16: 8-bit codes enter as 1024 + c, off = -1024, straight from one byte
// permute; 4-bit codes are centred, off = 8) and the two group terms in fp32,
// so no weight is ever rounded to a 16-bit float.  Activations arrive as fp16 scaled
// by 2^e per (row, group) so that every bf16 value keeps all its bits.
//
// Work and data flow (one CTA per SM; stream-K over (64-row tile, 512-k chunk)
// units, so every SM streams the same number of weight bytes):
//   * warps 8 and 13 (producers) fill a ring of shared-memory stages with TMA
//     copies, warp 8 the weights and warp 13 the activations (each step of a
//     producer's loop waits behind the consumers' shared-memory traffic, so
//     the copies are few, large, and split over two warps): from unit-packed
//     weights one bulk copy per stage, otherwise the tile's codes as one 3D
//     box of 128-byte pieces x 64 rows with the 128-byte swizzle (ldmatrix
//     then reads them without bank conflicts), one 64 x 8 box each of scales
//     and biases, and the matching slice of the prepared activations as plain
//     bulk copies.  The weights run ahead into the next phase while the
//     current phase drains (by one or two units while the CTA is still
//     finishing the phase: more copies in flight slow the transition
//     itself; without a limit once it has arrived at the barrier); only the
//     activation copies wait for the grid-wide phase barrier.
//   * warps 0-7 (consumers) are 4 row quarters x 2 k halves: ldmatrix the codes,
//     turn them into fp16 with byte-permute / LOP3, mma.sync m16n8k16 against
//     the activation fragments, fold each group into fp32 sums.  At a tile's
//     end the two k halves are added (fixed order) into one of two result
//     slots in shared memory, and the consumers go straight on to the next
//     unit: nothing that waits on global memory runs on them.
//   * warps 9-12 (epilogue, one per row quarter) finish each tile from its
//     result slot.  A tile split across CTAs is finished by the CTA whose
//     range holds its first unit; the others reach the tile first and publish
//     their partial sums as self-announcing words, which the finisher polls
//     and adds in CTA order, so results are bitwise reproducible.  The
//     finishing epilogue writes the phase output and prepares it as the next
//     phase's input (fp16 scaling, group sums, RMSNorm statistics, SwiGLU of
//     gate/up block pairs).
//   * between phases the last epilogue warp of every CTA to finish the phase
//     arrives on a grid counter; the producer issues the next phase's
//     activation copies once all CTAs have arrived.  Every wait is bounded
//     (about 2 s) and ends in an error flag, never in a hang.
#pragma once

#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {

#ifndef RUN_AHEAD_M8
#define RUN_AHEAD_M8 2
#endif

template <int BITS, int NT>
struct StreamCfg {
  static constexpr int MP = 8 * NT;
  static constexpr int ROW_BYTES = KC * BITS / 8;  // code bytes per weight row per stage
  static constexpr int ATOMS = ROW_BYTES / 128;    // 128-byte swizzled boxes per stage
  static constexpr int W_BYTES = BN * ROW_BYTES;
  static constexpr int X_BYTES = MP * KC * 2;
  static constexpr int XS_BYTES = GPS * 2 * MP * 4;  // per group: scaled sums, then 2^-e
  static constexpr int SB_BYTES = BN * GPS * 2;
  // stage: [codes][scales][biases] (one packed unit, or three TMA boxes) then [activations][group sums]
  static constexpr int S_OFF = W_BYTES;
  static constexpr int B_OFF = S_OFF + SB_BYTES;
  static constexpr int UNIT_BYTES = B_OFF + SB_BYTES;  // one unit of a packed weight
  static constexpr int X_OFF = UNIT_BYTES;
  static constexpr int XS_OFF = X_OFF + X_BYTES;
  static constexpr int STAGE_BYTES = (XS_OFF + XS_BYTES + 1023) / 1024 * 1024;  // swizzle atoms 1024-aligned
  static constexpr int RED_FLOATS = 16 * MP;        // one quarter's 16 rows
  static constexpr int RED_BYTES = 2 * 4 * RED_FLOATS * 4;  // result slot x quarter
  static constexpr int EPI_BYTES = 5 * 4 * MP * 4 + 256;    // cross-quarter scratch
  static constexpr int BUDGET = 227 * 1024 - 1024 - 2048 - RED_BYTES - EPI_BYTES;
  static constexpr int STAGES_FIT = BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + RED_BYTES + EPI_BYTES;
  // units of a phase whose grid barrier has not opened that the weight warp
  // may copy ahead while this CTA is still finishing the previous phase:
  // more copies in flight then slow the transition's chain of L2 round trips
  // (split-tile fixup, barrier, first activation copy) by more than they
  // save.  Once the CTA has arrived at the barrier the ring fills without a
  // limit (measured best: 2 units at M <= 8, 1 above).
  static constexpr int RUN_AHEAD = NT == 1 ? RUN_AHEAD_M8 : 1;
  static_assert(STAGES >= 2, "stage ring too small");
  static_assert(SMEM + 2048 <= 227 * 1024, "shared memory budget");
  static_assert(W_BYTES % 1024 == 0 && X_OFF % 16 == 0 && XS_OFF % 16 == 0 && S_OFF % 128 == 0 &&
                    B_OFF % 128 == 0, "copy destination alignment");
};

// ------------------------------------------------------------ schedule math
__device__ __forceinline__ int ph_units(const Phase& ph) { return ((ph.N + BN - 1) / BN) * (ph.K / KC); }
// Units of a phase are split over `grid` CTAs in contiguous ranges (stream-K).
__device__ __forceinline__ int unit_start(int c, int total, int grid) {
  return static_cast<int>(static_cast<long long>(c) * total / grid);
}
__device__ __forceinline__ int unit_owner(long long u, int total, int grid) {
  return static_cast<int>(((u + 1) * grid - 1) / total);
}

// Walks this CTA's units phase by phase, in the order both producer and
// consumers process them.
struct UnitIter {
  int phase, u, u_end, total;
  __device__ __forceinline__ void start(const StreamParams& p, int ph_from) {
    phase = ph_from - 1;
    u = u_end = 0;
    advance_phase(p);
  }
  __device__ __forceinline__ void advance_phase(const StreamParams& p) {
    do {
      ++phase;
      if (phase >= p.n_phases) return;
      total = ph_units(p.ph[phase]);
      const int g = p.grid;
      u = unit_start(blockIdx.x, total, g);
      u_end = unit_start(blockIdx.x + 1, total, g);
    } while (u >= u_end);
  }
  __device__ __forceinline__ bool done(const StreamParams& p) const { return phase >= p.n_phases; }
  __device__ __forceinline__ void next(const StreamParams& p) {
    if (++u >= u_end) advance_phase(p);
  }
};

// ---------------------------------------------------------- code conversion
// fp16 pair (1024 + c0, 1024 + c1) from two code bytes: one byte permute
// against the exponent byte 0x64 (1024 is exact, and so is 1024 + c for any
// byte c).  The 1024 is taken back out in fp32 with the group's bias term.
__device__ __forceinline__ uint32_t cvt8(uint32_t codes, uint32_t sel) { return __byte_perm(codes, 0x64646464u, sel); }
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

// Eight fp16 pairs (c - 2) from the sixteen 2-bit codes of one word; pair j =
// (c_j, c_{8+j}).  Field j of both 16-bit halves is masked in place and OR'ed
// into the mantissa of 1024, giving the exact fp16 value 1024 + c * 4^j' (j'
// its position after an optional shift by 10: c * 4^j' stays below 1024 for
// j' <= 4); one fp16 FMA by 4^-j' minus 1024 * 4^-j' + 2 leaves c - 2 exactly.
__device__ __forceinline__ void cvt2(uint32_t w, uint32_t (&P)[8]) {
  const uint32_t w10 = w >> 10;  // fields 5..7 of each half move to 0..2 (the high half's bits land above the masks)
  const uint32_t src[8] = {w, w, w, w, w, w10, w10, w10};
  const int pos[8] = {0, 1, 2, 3, 4, 0, 1, 2};
  const unsigned short scale[5] = {0x3C00, 0x3400, 0x2C00, 0x2400, 0x1C00};  // 1, 1/4, 1/16, 1/64, 1/256
  const unsigned short sub[5] = {0xE402, 0xDC08, 0xD420, 0xCC80, 0xC600};    // -1026, -258, -66, -18, -6
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t mask = 0x00030003u << (2 * pos[j]);
    uint32_t x = (src[j] & mask) | 0x64006400u;
    const __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), __half2half2(__ushort_as_half(scale[pos[j]])),
                              __half2half2(__ushort_as_half(sub[pos[j]])));
    P[j] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// Slot of the element at physical offset p (0..31) of a 32-element activation
// block, in the order the MMA fragments read the codes.
template <int BITS>
__device__ __forceinline__ int slot_of_phys(int p) {
  if (BITS == 8) {  // slot 8t + i holds element 4t + i (i < 4) or 16 + 4t + (i - 4)
    const int hi = p >> 4, q = p & 15;
    return 8 * (q >> 2) + 4 * hi + (q & 3);
  }
  const int j = p & 7;  // 4-bit: slot 8t + i holds nibble (0, 4, 1, 5, 2, 6, 3, 7)[i] of block 8t
  return (p & ~7) + (j < 4 ? 2 * j : 2 * (j - 4) + 1);
}
// Position (block * 32 + slot) within a group's two 32-element activation
// blocks of the group's element e (0..63).  8- and 4-bit codes keep every
// MMA k-step inside one 32-element half of the group.  A 2-bit word holds 16
// consecutive codes, so every step spans the whole group: thread t's word is
// codes 16t .. 16t + 15, its pair j = (c_j, c_{8+j}) feeds step j / 2 (slots
// 2t, 2t + 1 for even j, 2t + 8, 2t + 9 for odd j), and the steps 2b, 2b + 1
// form block b.
template <int BITS>
__device__ __forceinline__ int act_pos(int e) {
  if (BITS == 2) {
    const int t = e >> 4, j = e & 7, hi = (e >> 3) & 1;
    return (j >> 2) * 32 + 8 * t + ((j >> 1) & 1) * 4 + (j & 1) * 2 + hi;
  }
  return (e & 32) | slot_of_phys<BITS>(e & 31);
}

template <int NT>
__device__ __forceinline__ void zero4(float (&a)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) a[j][0] = a[j][1] = a[j][2] = a[j][3] = 0.f;
}

// One consumer warp's share of one stage: groups 4kh .. 4kh+3 for rows 16q .. 16q+15.
template <int BITS, int NT>
__device__ __forceinline__ void consume_stage(const uint8_t* st, int q, int kh, int lane, float (&tot)[NT][4]) {
  using C = StreamCfg<BITS, NT>;
  constexpr int MP = C::MP;
  // the tensor cores see code - OFF: 8-bit codes as 1024 + c, 4-bit ones centred as n - 8
  constexpr float OFF = BITS == 8 ? -1024.f : (BITS == 4 ? 8.f : 2.f);
  const int gid = lane >> 2, t = lane & 3;
  const uint32_t w_base = smem_u32(st);
  const uint32_t x_base = smem_u32(st + C::X_OFF);
  const float* xs = reinterpret_cast<const float*>(st + C::XS_OFF);
  const __half* sc = reinterpret_cast<const __half*>(st + C::S_OFF);  // [64][8]
  const __half* bi = reinterpret_cast<const __half*>(st + C::B_OFF);
  const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix mi (row half mi&1, chunk +mi>>1), row rr
  const int lrow = 16 * q + (mi & 1) * 8 + rr;
  // row lrow of a 128-byte swizzled box: 16-byte chunk c sits at c ^ (lrow & 7) = c ^ rr
  const uint32_t arow = w_base + lrow * 128;
  // this warp's four groups of scales / biases for its rows gid and gid + 8
  float s_v[2][4], b_v[2][4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int n = 16 * q + gid + 8 * h;
    const uint2 s4 = *reinterpret_cast<const uint2*>(sc + n * GPS + 4 * kh);
    const uint2 b4 = *reinterpret_cast<const uint2*>(bi + n * GPS + 4 * kh);
    const __half2 s01 = *reinterpret_cast<const __half2*>(&s4.x), s23 = *reinterpret_cast<const __half2*>(&s4.y);
    const __half2 b01 = *reinterpret_cast<const __half2*>(&b4.x), b23 = *reinterpret_cast<const __half2*>(&b4.y);
    s_v[h][0] = __low2float(s01);
    s_v[h][1] = __high2float(s01);
    s_v[h][2] = __low2float(s23);
    s_v[h][3] = __high2float(s23);
    b_v[h][0] = fmaf(OFF, s_v[h][0], __low2float(b01));
    b_v[h][1] = fmaf(OFF, s_v[h][1], __high2float(b01));
    b_v[h][2] = fmaf(OFF, s_v[h][2], __low2float(b23));
    b_v[h][3] = fmaf(OFF, s_v[h][3], __high2float(b23));
  }
  uint32_t q2[4];  // 2-bit: codes of two groups, loaded at even gi
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    const int gl = 4 * kh + gi;  // group index within the stage
    uint32_t bfr[2][NT][4];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk)
#pragma unroll
      for (int j = 0; j < NT; ++j)
        lds128(bfr[blk][j], x_base + ((((gl * 2 + blk) * MP + 8 * j + gid) * 32 + 8 * t) * 2));
    float acc[NT][4];
    zero4<NT>(acc);
    if constexpr (BITS == 8) {
      // box gl/2 holds groups 2(gl/2), 2(gl/2)+1; a group is 4 chunks (one k16 step each)
      uint32_t qd[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h)
        ldsm_x4(qd[h], arow + (gl >> 1) * (BN * 128) + (((4 * (gl & 1) + 2 * h + (mi >> 1)) ^ rr) << 4));
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint32_t lo = qd[s >> 1][(s & 1) * 2], hi = qd[s >> 1][(s & 1) * 2 + 1];
        uint32_t a[4] = {cvt8(lo, 0x4140u), cvt8(hi, 0x4140u), cvt8(lo, 0x4342u), cvt8(hi, 0x4342u)};
#pragma unroll
        for (int j = 0; j < NT; ++j)
          mma_16816(acc[j], a, bfr[s >> 1][j][(s & 1) * 2], bfr[s >> 1][j][(s & 1) * 2 + 1]);
      }
    } else if constexpr (BITS == 2) {
      // the stage's one 128-byte box holds all 8 groups, a group per 16-byte
      // chunk: one ldmatrix brings groups gl and gl + 1 for rows gid, gid + 8
      if ((gi & 1) == 0) ldsm_x4(q2, arow + (((gl + (mi >> 1)) ^ rr) << 4));
      uint32_t L[8], H[8];
      cvt2(q2[2 * (gi & 1)], L);
      cvt2(q2[2 * (gi & 1) + 1], H);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint32_t a[4] = {L[2 * s], H[2 * s], L[2 * s + 1], H[2 * s + 1]};
#pragma unroll
        for (int j = 0; j < NT; ++j)
          mma_16816(acc[j], a, bfr[s >> 1][j][(s & 1) * 2], bfr[s >> 1][j][(s & 1) * 2 + 1]);
      }
    } else {
      // box gl/4 holds groups 4(gl/4) .. +3; a group is 2 chunks
      uint32_t qd[4];
      ldsm_x4(qd, arow + (gl >> 2) * (BN * 128) + (((2 * (gl & 3) + (mi >> 1)) ^ rr) << 4));
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t Plo[4], Phi[4];
        cvt4(qd[2 * c], Plo);
        cvt4(qd[2 * c + 1], Phi);
        uint32_t a0[4] = {Plo[0], Phi[0], Plo[1], Phi[1]};
        uint32_t a1[4] = {Plo[2], Phi[2], Plo[3], Phi[3]};
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          mma_16816(acc[j], a0, bfr[c][j][0], bfr[c][j][1]);
          mma_16816(acc[j], a1, bfr[c][j][2], bfr[c][j][3]);
        }
      }
    }
    // tot += 2^-e * (s * acc + (b + off*s) * xsum)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float2 xsv = *reinterpret_cast<const float2*>(xs + (gl * 2) * MP + 8 * j + 2 * t);
      const float2 fv = *reinterpret_cast<const float2*>(xs + (gl * 2 + 1) * MP + 8 * j + 2 * t);
      tot[j][0] = fmaf(fv.x, fmaf(s_v[0][gi], acc[j][0], b_v[0][gi] * xsv.x), tot[j][0]);
      tot[j][1] = fmaf(fv.y, fmaf(s_v[0][gi], acc[j][1], b_v[0][gi] * xsv.y), tot[j][1]);
      tot[j][2] = fmaf(fv.x, fmaf(s_v[1][gi], acc[j][2], b_v[1][gi] * xsv.x), tot[j][2]);
      tot[j][3] = fmaf(fv.y, fmaf(s_v[1][gi], acc[j][3], b_v[1][gi] * xsv.y), tot[j][3]);
    }
  }
}

template <int NT>
__device__ __forceinline__ void red_store(float* buf, const float (&v)[NT][4], int lane) {
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) buf[(j * 4 + e) * 32 + lane] = v[j][e];
}
template <int NT, bool GLOBAL>
__device__ __forceinline__ void red_add(const float* buf, float (&v)[NT][4], int lane) {
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float* a = buf + (j * 4 + e) * 32 + lane;
      v[j][e] += GLOBAL ? __ldcg(a) : *a;
    }
}

// Split-tile partial sums travel through global memory as self-announcing
// words: a contributor stores each fp32 partial with all bits inverted, and
// the finisher polls the words themselves (zero = not yet written), adds them
// and zeroes them again for the next use.  No partial is ever the all-ones
// pattern (arithmetic yields only the canonical NaN), so no written word
// reads as zero; each 32-bit word is written and read whole, and the slot is
// next written only after a grid barrier that follows the zeroing.
template <int NT>
__device__ __forceinline__ void partial_store(float* buf, const float (&v)[NT][4], int lane) {
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      __stcg(reinterpret_cast<unsigned*>(buf) + (j * 4 + e) * 32 + lane, ~__float_as_uint(v[j][e]));
}
// Adds one contributor's partials (bounded wait; false on abort or timeout).
template <int NT>
__device__ __forceinline__ bool partial_take(float* buf, float (&v)[NT][4], int lane, volatile int* abort_v,
                                             volatile int* abort_g) {
  unsigned* w = reinterpret_cast<unsigned*>(buf);
  unsigned got[NT][4];
  const unsigned long long t0 = global_ns();
  for (unsigned it = 0;; ++it) {
    bool all = true;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        got[j][e] = __ldcv(w + (j * 4 + e) * 32 + lane);
        all &= got[j][e] != 0u;
      }
    if (all) break;
    if ((it & 15u) == 15u) {
      if (*abort_v) return false;
      const unsigned long long dt = global_ns() - t0;
      if (dt > 20000ull && *abort_g) return false;
      if (dt > WAIT_LIMIT_NS) {
        raise_error(ERR_TIMEOUT_FULL);
        *abort_v = 1;
        *abort_g = 1;
        return false;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[j][e] += __uint_as_float(~got[j][e]);
      __stcg(w + (j * 4 + e) * 32 + lane, 0u);
    }
  return true;
}

// Adds the partials of contributors c_first .. c_last (those with a non-empty
// unit range) in CTA order, fetching up to B of them at once: their loads are
// issued together and the wait is one L2 round trip, not one per contributor.
// Each contributor's words are read, added and zeroed as a whole, in CTA
// order, so the sum is bitwise reproducible.
template <int NT>
__device__ __forceinline__ bool partial_take_many(float* partials, int q, int c_first, int c_last, int total,
                                                  int grid, float (&v)[NT][4], int lane, volatile int* abort_v,
                                                  volatile int* abort_g) {
  constexpr int B = 2;                 // contributors fetched together (registers: B x NT x 4 per lane)
  constexpr int RF = 16 * 8 * NT;      // one quarter's floats
  unsigned* const w0 = reinterpret_cast<unsigned*>(partials) + (size_t)q * RF + lane;
  for (int c0 = c_first; c0 <= c_last; c0 += B) {
    bool need[B], have[B];
    unsigned got[B][NT][4];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int c = c0 + b;
      need[b] = c <= c_last && unit_start(c + 1, total, grid) > unit_start(c, total, grid);
      have[b] = !need[b];
    }
    // contributor c's words for this quarter and lane: w0 + c * (2 * 4 * RF) + (j * 4 + e) * 32
    auto word = [&](int b, int j, int e) { return w0 + (size_t)(c0 + b) * (8 * RF) + (j * 4 + e) * 32; };
    const unsigned long long t0 = global_ns();
    for (unsigned it = 0;; ++it) {
      bool all = true;
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (have[b]) continue;
        bool ok = true;
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            got[b][j][e] = __ldcv(word(b, j, e));
            ok &= got[b][j][e] != 0u;
          }
        have[b] = ok;
        all &= ok;
      }
      if (all) break;
      if ((it & 15u) == 15u) {
        if (*abort_v) return false;
        const unsigned long long dt = global_ns() - t0;
        if (dt > 20000ull && *abort_g) return false;
        if (dt > WAIT_LIMIT_NS) {
          raise_error(ERR_TIMEOUT_FULL);
          *abort_v = 1;
          *abort_g = 1;
          return false;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (!need[b]) continue;
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[j][e] += __uint_as_float(~got[b][j][e]);
          __stcg(word(b, j, e), 0u);
        }
    }
  }
  return true;
}

constexpr int EPI_BAR = 5;       // the four epilogue warps
constexpr int EPI_THREADS = 128;

// Epilogue scratch in shared memory.
struct EpiScratch {
  float* a;    // [4][MP]
  float* b;    // [4][MP]
  float* c;    // [4][MP]
  int* ia;     // [4][MP] (aliases c for the argmax)
  float* r;    // [4][MP]: RMSNorm sums of squares, one part per epilogue warp
};

// Turns this tile's 64 output columns (row values yv, already final) into group
// `grp` of the next phase's prepared activations: per row m, e = 15 - exponent
// of max|v|, fp16(v * 2^e) in MMA order, the group sum of v * 2^e, 2^-e, and
// (for a RMSNorm input) the group sum of v^2.  Run by the four epilogue warps.
template <int BITS, int NT>
__device__ void prepare_group(const StreamParams& p, const ActBuf& out, int grp, int Kn, int q, int lane,
                              const float (&yv)[NT][4], bool with_sq, float flag_value, EpiScratch& es) {
  constexpr int MP = 8 * NT;
  const int gid = lane >> 2, t = lane & 3;
  // 1. per column: max |v| and sum v^2 over this warp's 16 rows
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float mx = fmaxf(fabsf(yv[j][c]), fabsf(yv[j][2 + c]));
      float ss = yv[j][c] * yv[j][c] + yv[j][2 + c] * yv[j][2 + c];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
      }
      if (gid == 0) {
        es.a[q * MP + 8 * j + 2 * t + c] = mx;
        es.b[q * MP + 8 * j + 2 * t + c] = ss;
      }
    }
  named_bar_sync(EPI_BAR, EPI_THREADS);
  // 2. exponent per column, scaled fp16 values, partial group sums
  float sc[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int m = 8 * j + 2 * t + c;
      const int e = scale_exponent(fmaxf(fmaxf(es.a[m], es.a[MP + m]), fmaxf(es.a[2 * MP + m], es.a[3 * MP + m])));
      sc[j][c] = pow2_exact(e);
    }
  const int n_lo = 16 * q + gid, n_hi = n_lo + 8;
  __half* xp = out.xp;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int m = 8 * j + 2 * t + c;
      const float v0 = yv[j][c] * sc[j][c], v1 = yv[j][2 + c] * sc[j][c];
      const int p_lo = act_pos<BITS>(n_lo), p_hi = act_pos<BITS>(n_hi);
      xp[((size_t)(2 * grp + (p_lo >> 5)) * MP + m) * 32 + (p_lo & 31)] = __float2half_rn(v0);
      xp[((size_t)(2 * grp + (p_hi >> 5)) * MP + m) * 32 + (p_hi & 31)] = __float2half_rn(v1);
      float s = v0 + v1;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (gid == 0) es.c[q * MP + m] = s;
    }
  named_bar_sync(EPI_BAR, EPI_THREADS);
  // 3. one warp writes the group's sums (fixed quarter order)
  if (q == 0) {
    for (int m = lane; m < MP; m += 32) {
      const int e = scale_exponent(fmaxf(fmaxf(es.a[m], es.a[MP + m]), fmaxf(es.a[2 * MP + m], es.a[3 * MP + m])));
      float* xs = out.xs + (size_t)grp * 2 * MP;
      xs[m] = ((es.c[m] + es.c[MP + m]) + es.c[2 * MP + m]) + es.c[3 * MP + m];
      xs[MP + m] = pow2_exact(-e);
      if (with_sq) out.sq[(size_t)grp * MP + m] = ((es.b[m] + es.b[MP + m]) + es.b[2 * MP + m]) + es.b[3 * MP + m];
      if (grp == 0) out.sq[(size_t)(Kn / GROUP) * MP + m] = flag_value;
    }
  }
  named_bar_sync(EPI_BAR, EPI_THREADS);
}

// Loads the bf16 values this epilogue thread finishes for 64 output columns
// starting at `col0` (rows m = 8j + 2t + c, columns col0 + 16q + gid + 8h),
// zero where m >= M.  Read through L2: the values were written by other CTAs.
template <int NT>
__device__ __forceinline__ void load_tile_bf16(float (&v)[NT][4], const __nv_bfloat16* base, int ld, int col0, int M,
                                               int q, int lane) {
  const int gid = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = 8 * j + 2 * t + (e & 1);
      v[j][e] = m < M ? __bfloat162float(__ldcg(base + (size_t)m * ld + col0 + 16 * q + gid + 8 * (e >> 1))) : 0.f;
    }
}

// Who finishes what.  Tile `tile` of a phase covers units [tile*upt, (tile+1)*upt);
// it is finished by the owner of its first unit.  When that CTA's range ends
// inside the tile, the tile is the last one it works on in the phase, while
// every other contributor meets the tile first (its range starts inside it):
// contributors publish early, the finisher reads late.
__device__ __forceinline__ int tile_finisher(int tile, int upt, int total, int grid) {
  return unit_owner((long long)tile * upt, total, grid);
}

// Finishes one tile (all four epilogue warps, each holding 16 rows; values are
// the full sums, before the RMSNorm row factor).  `pre` holds what was fetched
// before the tile's sums arrived: the hidden-state rows of a PH_RESID tile or
// the partner up values of a gate tile whose up half another CTA finished,
// or the gate values of an up tile whose gate half this CTA finished.
// `g_keep` carries a gate tile's values to its up tile when one CTA finishes
// both (`pair_here`; they are copied to `pre` before the up tile's sums
// arrive, so that a register spill of `g_keep` is not reloaded in the tail);
// otherwise the up tile's finisher publishes its values and the gate tile's
// finisher, which meets its tile later, combines the two.
template <int BITS, int NT>
__device__ void finish_tile(const StreamParams& p, const Phase& ph, const ActBuf& out, int tile, int pair_here, int q, int lane,
                            float (&tot)[NT][4], const float (&rf)[NT][2], const float (&pre)[NT][4],
                            float (&g_keep)[NT][4], EpiScratch& es) {
  constexpr int MP = 8 * NT;
  const int gid = lane >> 2, t = lane & 3;
  const int n_lo = tile * BN + 16 * q + gid;  // rows n_lo and n_lo + 8
  float yv[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) yv[j][e] = tot[j][e] * rf[j][e & 1];

  if (ph.kind == PH_LOGITS) {
    // logits and per-row (max, lowest argmax, sum-exp) of these 64 columns
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int m = 8 * j + 2 * t + c;
        float best = -INFINITY;
        int bidx = 0x7fffffff;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = n_lo + 8 * h;
          if (n < ph.N) {
            if (m < p.M) p.logits[(size_t)m * p.ldl + n] = yv[j][2 * h + c];
            if (yv[j][2 * h + c] > best) { best = yv[j][2 * h + c]; bidx = n; }
          }
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          const float ob = __shfl_xor_sync(0xffffffffu, best, off);
          const int oi = __shfl_xor_sync(0xffffffffu, bidx, off);
          if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
        }
        if (gid == 0) {
          es.a[q * MP + m] = best;
          es.ia[q * MP + m] = bidx;
        }
      }
    named_bar_sync(EPI_BAR, EPI_THREADS);
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int m = 8 * j + 2 * t + c;
        float best = es.a[m];
        int bidx = es.ia[m];
#pragma unroll
        for (int qq = 1; qq < 4; ++qq) {
          const float ob = es.a[qq * MP + m];
          const int oi = es.ia[qq * MP + m];
          if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
        }
        float se = 0.f;
        if (p.inv_temp > 0.f) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (n_lo + 8 * h < ph.N) se += exp_term((yv[j][2 * h + c] - best) * p.inv_temp);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) se += __shfl_xor_sync(0xffffffffu, se, off);
        }
        if (gid == 0) es.b[q * MP + m] = se;
      }
    named_bar_sync(EPI_BAR, EPI_THREADS);
    if (q == 0)
      for (int m = lane; m < MP; m += 32) {
        float best = es.a[m];
        int bidx = es.ia[m];
        for (int qq = 1; qq < 4; ++qq) {
          const float ob = es.a[qq * MP + m];
          const int oi = es.ia[qq * MP + m];
          if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
        }
        float* ts = p.tile_stats + ((size_t)tile * MP + m) * 3;
        ts[0] = best;
        ts[1] = __int_as_float(bidx);
        ts[2] = ((es.b[m] + es.b[MP + m]) + es.b[2 * MP + m]) + es.b[3 * MP + m];
      }
    named_bar_sync(EPI_BAR, EPI_THREADS);
    return;
  }

  if (ph.kind == PH_GATEUP) {
    // interleaved 64-row blocks: tile 2j = gate rows of block j, tile 2j + 1 = up rows
    const int blk = tile >> 1, is_up = tile & 1;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = 8 * j + 2 * t + (e & 1);
        const int col = is_up * ph.half + blk * BN + 16 * q + gid + 8 * (e >> 1);
        const __nv_bfloat16 v = __float2bfloat16_rn(yv[j][e]);
        yv[j][e] = m < p.M ? __bfloat162float(v) : 0.f;
        if (m < p.M) ph.y[(size_t)m * ph.ldy + col] = v;
      }
    if (!is_up && pair_here) {  // this CTA finishes the up tile next: keep the gate values
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) g_keep[j][e] = yv[j][e];
      return;
    }
    if (is_up && !pair_here) {  // the gate tile's finisher (another CTA) combines the pair
      partial_store<NT>(p.pair_words + ((size_t)blk * 4 + q) * (16 * MP), yv, lane);
      return;
    }
    // s = bf16(silu(g) * u)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = 8 * j + 2 * t + (e & 1);
        const float g = is_up ? pre[j][e] : yv[j][e];  // an up tile's pre holds its gate values
        const float u = is_up ? yv[j][e] : pre[j][e];
        yv[j][e] = m < p.M ? __bfloat162float(__float2bfloat16_rn(silu_f32(g) * u)) : 0.f;
      }
    prepare_group<BITS, NT>(p, out, blk, ph.half, q, lane, yv, false, -1.f, es);
    return;
  }

  if (ph.kind == PH_RESID) {
    // h = bf16(res + bf16(y)) (res may be y itself); h is the next phase's RMSNorm input
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = 8 * j + 2 * t + (e & 1);
        const int n = n_lo + 8 * (e >> 1);
        float v = 0.f;
        if (m < p.M) {
          const __nv_bfloat16 nb = __float2bfloat16_rn(pre[j][e] + __bfloat162float(__float2bfloat16_rn(yv[j][e])));
          ph.y[(size_t)m * ph.ldy + n] = nb;
          v = __bfloat162float(nb);
        }
        yv[j][e] = v;
      }
    if (ph.out_buf >= 0) prepare_group<BITS, NT>(p, out, tile, ph.N, q, lane, yv, true, p.rms_eps, es);
    return;
  }

  // PH_STORE: bf16 output; the first prep_tiles tiles also feed the next phase
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = 8 * j + 2 * t + (e & 1);
      const int n = n_lo + 8 * (e >> 1);
      const __nv_bfloat16 v = __float2bfloat16_rn(yv[j][e]);
      if (m < p.M && n < ph.N) ph.y[(size_t)m * ph.ldy + n] = v;
      yv[j][e] = m < p.M ? __bfloat162float(v) : 0.f;
    }
  if (tile < ph.prep_tiles)
    prepare_group<BITS, NT>(p, out, tile, ph.prep_tiles * BN, q, lane, yv, false, -1.f, es);
}

// RMSNorm row factors 1/sqrt(mean(x^2) + eps) of the phase input for this
// thread's columns, or 1 when the input is not an RMSNorm input.  The four
// epilogue warps split the groups into four contiguous ranges; in each, LPC
// lanes per column sum every LPC-th group with eight loads in flight, a fixed
// shuffle tree adds the lanes, and the four parts are added in warp order
// through shared memory (all four warps call this together).
template <int NT>
__device__ __forceinline__ void rms_factors(const ActBuf& a, int K, int q, int lane, float (&rf)[NT][2], float* part_sums) {
  constexpr int MP = 8 * NT;
  constexpr int LPC = MP == 8 ? 4 : (MP == 16 ? 2 : 1);  // MP = 24: lanes 24..31 idle
  const int G = K / GROUP;
  const float eps = __ldcg(a.sq + (size_t)G * MP);
  if (!(eps >= 0.f)) {  // the same word for every warp: all take this branch or none
#pragma unroll
    for (int j = 0; j < NT; ++j) rf[j][0] = rf[j][1] = 1.f;
    return;
  }
  const int m = lane % MP, part = lane / MP;
  const int g0 = q * G / 4, g1 = (q + 1) * G / 4;
  float ss = 0.f;
  if (part < LPC) {
    int g = g0 + part;
    for (; g + 7 * LPC < g1; g += 8 * LPC) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __ldcg(a.sq + (size_t)(g + i * LPC) * MP + m);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += v[i];
    }
    for (; g < g1; g += LPC) ss += __ldcg(a.sq + (size_t)g * MP + m);
  }
#pragma unroll
  for (int off = MP; off < MP * LPC; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if (lane < MP) part_sums[q * MP + lane] = ss;
  named_bar_sync(EPI_BAR, EPI_THREADS);
  const float tot = ((part_sums[m] + part_sums[MP + m]) + part_sums[2 * MP + m]) + part_sums[3 * MP + m];
  const float r_mine = 1.f / sqrtf(tot / (float)K + eps);
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int c = 0; c < 2; ++c) rf[j][c] = __shfl_sync(0xffffffffu, r_mine, 8 * j + 2 * (lane & 3) + c);
}

template <int BITS, int NT>
__global__ void __launch_bounds__(QMM_THREADS, 1) stream_kernel(const __grid_constant__ StreamParams p) {
  using C = StreamCfg<BITS, NT>;
  constexpr int S = C::STAGES;
  constexpr int MP = C::MP;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[S], empty_bar[S], res_full[2], res_empty[2];
  __shared__ int abort_flag;
  __shared__ int ready_ph;             // highest phase whose grid barrier the producer passed
  __shared__ int arrived_ph;           // highest phase this CTA's epilogue has finished (arrived for)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red = reinterpret_cast<float*>(smem + S * C::STAGE_BYTES);  // result slots [2][4][16*MP]
  float* epi = red + 2 * 4 * C::RED_FLOATS;
  EpiScratch es;
  es.a = epi;
  es.b = epi + 4 * MP;
  es.c = epi + 8 * MP;
  es.ia = reinterpret_cast<int*>(epi + 12 * MP);
  es.r = epi + 16 * MP;
  volatile int* abort_v = &abort_flag;
  volatile int* abort_g = p.abort_all;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 2);  // the weight warp and the activation warp
      mbar_init(&empty_bar[s], NCW);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&res_full[r], 4 * 32);   // the k-half-0 consumer threads
      mbar_init(&res_empty[r], NEW * 32);  // the epilogue threads
    }
    abort_flag = 0;
    ready_ph = 0;
    arrived_ph = -1;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();

  if (warp == NCW || warp == XPW) {
    // ============================================================ producers
    // Warp NCW copies each stage's weights (codes, scales, biases); warp XPW
    // copies its activations once the stage's phase is open.  Two issuing
    // warps: one lane completes only a few copy instructions per
    // microsecond.  Each arrives once per stage use on the stage's full
    // barrier (count 2) with its own byte count.
    // one lane issues: the others leave at once, so no per-unit step of the
    // loop needs a shuffle or a warp barrier (each of those queues behind the
    // consumers' shared-memory traffic)
    if (lane != 0) return;
    const bool is_x = warp == XPW;
    const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
    UnitIter it;
    it.start(p, 0);
    int n = 0;                 // units issued so far by this warp
    int ahead_ph = -1, ahead_n = 0;  // (weight warp) units issued of the newest phase not yet open
    int ready = 0;             // (activation warp) highest phase whose activations may be loaded
    int mapped = -1;           // (weight warp) last phase whose tensor maps were prefetched
    bool pdl_done = !is_x;     // the weight warp never reads what the previous kernel wrote
    unsigned long long t_wait = 0;
    bool bad = false;
    // per-unit work reads only registers: the phase table lives in the
    // kernel's parameter block, whose reads can miss the constant cache
    struct {
      int phase = -1, upt = 1;
      const uint8_t* packed = nullptr;
      const __half* xp = nullptr;
      const float* xs = nullptr;
    } cur;
    auto maps_of = [&](int phase) -> const CUtensorMap* { return p.maps ? p.maps + 3 * phase : p.tm; };
    while (!it.done(p)) {
      bool go = false;
      // the stage must be free: its previous unit consumed
      bool free_slot = n < S || mbar_test_wait(&empty_bar[n % S], ((n / S) - 1) & 1);
      if (free_slot && !is_x && it.phase > ld_acquire_cta(&ready_ph) &&
          it.phase > ld_acquire_cta(&arrived_ph) + 1) {
        if (ahead_ph != it.phase) {
          ahead_ph = it.phase;
          ahead_n = 0;
        }
        free_slot = ahead_n < C::RUN_AHEAD;
        ahead_n += free_slot;
      }
      if (free_slot) {
        if (!is_x) {
          go = true;
        } else if (!pdl_done) {  // the first phase's activations come from the previous kernel
          pdl_wait();
          pdl_done = true;
          continue;
        } else if (it.phase <= ready) {
          go = true;
        } else if (ld_acquire(p.grid_bar + it.phase) >= (unsigned)p.grid) {
          // grid barrier of this unit's phase: one counter per transition, so
          // CTAs that skip ahead through phases in which they have no units
          // cannot stand in for CTAs still working
          fence_proxy_async();
          ready = it.phase;
          st_release_cta(&ready_ph, ready);
          go = true;
        }
      }
      if (go) {
        if (it.phase != cur.phase) {  // the phase's fields, read from the parameter block once per phase
          const Phase& ph = p.ph[it.phase];
          cur.phase = it.phase;
          cur.upt = ph.K / KC;
          cur.packed = ph.packed;
          cur.xp = p.act[ph.in_buf].xp;
          cur.xs = p.act[ph.in_buf].xs;
        }
        const int upt = cur.upt, kc = it.u % upt, sg = n % S;
        uint8_t* st = smem + sg * C::STAGE_BYTES;
        if (!is_x) {
          const int tile = it.u / upt;
          const CUtensorMap* tm = maps_of(it.phase);
          if (it.phase != mapped) {  // warm the descriptor cache for this phase and the next
            if (it.phase + 1 < p.n_phases && p.maps)
              for (int k = 0; k < 3; ++k) prefetch_tensormap(maps_of(it.phase + 1) + k);
            mapped = it.phase;
          }
          mbar_arrive_expect_tx(&full_bar[sg], C::UNIT_BYTES);
          if (cur.packed) {  // one contiguous unit: codes already swizzled, then scales, biases
            bulk_load(st, cur.packed + (size_t)it.u * C::UNIT_BYTES, C::UNIT_BYTES, &full_bar[sg], pol_w);
          } else {
            tma_load_3d(st, tm, &full_bar[sg], 0, tile * BN, kc * C::ATOMS, pol_w);  // all pieces of the stage
            tma_load_2d(st + C::S_OFF, tm + 1, &full_bar[sg], kc * GPS, tile * BN, pol_w);
            tma_load_2d(st + C::B_OFF, tm + 2, &full_bar[sg], kc * GPS, tile * BN, pol_w);
          }
        } else {
          mbar_arrive_expect_tx(&full_bar[sg], C::X_BYTES + C::XS_BYTES);
          bulk_load(st + C::X_OFF, cur.xp + (size_t)kc * (KC / 32) * MP * 32, C::X_BYTES, &full_bar[sg], pol_x);
          bulk_load(st + C::XS_OFF, cur.xs + (size_t)kc * GPS * 2 * MP, C::XS_BYTES, &full_bar[sg], pol_x);
        }
        it.next(p);
        ++n;
        t_wait = 0;
        continue;
      }
      // nothing to do: back off briefly, bounded overall.  The abort flags are
      // looked at only once a wait has lasted 20 us, so an idle turn costs no
      // global-memory round trip.
      __nanosleep(32);
      const unsigned long long now = global_ns();
      if (!t_wait) t_wait = now;
      if (now - t_wait > 20000ull && ((*abort_v | *abort_g) || now - t_wait > WAIT_LIMIT_NS)) {
        if (!(*abort_v | *abort_g)) raise_error(ERR_TIMEOUT_EMPTY);
        *abort_v = 1;
        *abort_g = 1;
        bad = true;
        break;
      }
    }
    // drain copies already issued into the ring before the CTA may exit; after
    // an abort a stage may never complete, so give its copies a fixed 50 us
    // to land instead
    if (!bad && !*abort_v) {
      for (int k = (n - S > 0 ? n - S : 0); k < n; ++k)
        mbar_wait_bounded(&full_bar[k % S], (k / S) & 1, abort_v);
    } else {
      const unsigned long long t0 = global_ns();
      while (global_ns() - t0 < 50000ull) __nanosleep(1000);
    }
    return;
  }

  // ================================================================== consumers
  if (warp < NCW) {
    const int q = warp >> 1, kh = warp & 1;
    float tot[NT][4];
    zero4<NT>(tot);
    int i = 0, n_te = 0;  // units consumed, tile ends handed over
    for (int ph_i = 0; ph_i < p.n_phases; ++ph_i) {
      const Phase ph = p.ph[ph_i];
      const int upt = ph.K / KC, total = ph_units(ph);
      const int pg = p.grid;
      const int u0 = unit_start(blockIdx.x, total, pg), u1 = unit_start(blockIdx.x + 1, total, pg);
      for (int u = u0; u < u1; ++u, ++i) {
        const int kc = u % upt, s = i % S;
        if (!(*abort_v)) {
          if (mbar_wait_bounded(&full_bar[s], (i / S) & 1, abort_v)) {
            consume_stage<BITS, NT>(smem + s * C::STAGE_BYTES, q, kh, lane, tot);
          } else {
            raise_error(ERR_TIMEOUT_FULL);
            *abort_v = 1;
            *abort_g = 1;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        if (kc != upt - 1 && u != u1 - 1) continue;
        // ---- tile end: the two k halves meet in result slot n_te % 2 (fixed
        // order: half 1 stores, half 0 adds) and the epilogue warps take it
        const int slot = n_te & 1;
        if (n_te >= 2 && !(*abort_v) && !mbar_wait_bounded(&res_empty[slot], ((n_te >> 1) - 1) & 1, abort_v)) {
          raise_error(ERR_TIMEOUT_EMPTY);
          *abort_v = 1;
          *abort_g = 1;
        }
        float* rb = red + (slot * 4 + q) * C::RED_FLOATS;
        if (kh == 1) red_store<NT>(rb, tot, lane);
        named_bar_sync(1 + q, 64);
        if (kh == 0) {
          red_add<NT, false>(rb, tot, lane);
          red_store<NT>(rb, tot, lane);
          mbar_arrive(&res_full[slot]);
        }
        zero4<NT>(tot);
        ++n_te;
      }
    }
    return;
  }

  // ================================================================== epilogue
  // Warps NCW + 1 .. NCW + 4, one per row quarter.  They walk the same tile
  // ends as the consumers and finish each tile: split-tile fixup, output, the
  // next phase's prepared input.  Everything a tile's finish needs from other
  // CTAs (split partials, hidden-state rows, partner up values) is fetched
  // before the tile's own sums arrive, so the tail of a phase is short.
  const int q = warp - (NCW + 1);
  pdl_wait();
  float rf[NT][2];
  float g_keep[NT][4];
  zero4<NT>(g_keep);
  int n_te = 0;
  for (int ph_i = 0; ph_i < p.n_phases; ++ph_i) {
    // the phase's fields and buffers, read from the parameter block once per
    // phase (before its barrier opens) instead of at every use in the tail
    const Phase ph = p.ph[ph_i];
    const ActBuf in_a = p.act[ph.in_buf];
    ActBuf out_a = {};
    if (ph.out_buf >= 0) out_a = p.act[ph.out_buf];
    const int upt = ph.K / KC, total = ph_units(ph);
    const int pg = p.grid;
    const int u0 = unit_start(blockIdx.x, total, pg), u1 = unit_start(blockIdx.x + 1, total, pg);
    if (u0 < u1) {
      // this phase's inputs are complete once the producer passed its grid barrier
      if (ph_i > 0) {
        const unsigned long long t0 = global_ns();
        while (ld_acquire_cta(&ready_ph) < ph_i) {
          if ((*abort_v | *abort_g) || global_ns() - t0 > WAIT_LIMIT_NS) break;
          __nanosleep(32);
        }
      }
      rms_factors<NT>(in_a, ph.K, q, lane, rf, es.r);
      const int first_tile = u0 / upt, last_tile = (u1 - 1) / upt;
      // the hidden-state rows of the last residual tile this CTA finishes are
      // fetched now (h was last written two phases ago): that tile's finish
      // is at the end of the phase, on its critical path, and would
      // otherwise wait one L2 round trip for them.  They are held in g_keep,
      // which carries values only between the two tiles of a gate/up block.
      int pre_tile = -1;
      if (ph.kind == PH_RESID) {
        for (int t = last_tile; t >= first_tile; --t)
          if (tile_finisher(t, upt, total, pg) == (int)blockIdx.x) {
            pre_tile = t;
            break;
          }
        if (pre_tile >= 0) load_tile_bf16<NT>(g_keep, ph.res, ph.ldr, pre_tile * BN, p.M, q, lane);
      }
      for (int tile = first_tile; tile <= last_tile; ++tile) {
        const int fin = tile_finisher(tile, upt, total, pg);
        const int c_last = unit_owner((long long)tile * upt + upt - 1, total, pg);
        const bool finisher = fin == (int)blockIdx.x;
        float pre[NT][4], part[NT][4];
        zero4<NT>(pre);
        zero4<NT>(part);
        int pair_here = 0;  // gate/up: one CTA finishes both tiles of the block
        if (finisher) {
          // ---- fetch ahead: contributors' partials (they met this tile first)
          if (c_last != fin) {
            if constexpr (NT <= 3) {  // contributors fetched two at a time
              partial_take_many<NT>(p.partials, q, fin + 1, c_last, total, pg, part, lane, abort_v, abort_g);
            } else {                  // 32 rows: one at a time (the batched form's registers would spill)
              for (int c = fin + 1; c <= c_last; ++c)
                if (unit_start(c + 1, total, pg) > unit_start(c, total, pg) &&
                    !partial_take<NT>(p.partials + (((size_t)c * 2) * 4 + q) * C::RED_FLOATS, part, lane, abort_v,
                                      abort_g))
                  break;
            }
          }
          // ... the hidden-state rows of a residual tile, the partner of a gate tile
          if (ph.kind == PH_RESID) {
            if (tile == pre_tile) {
#pragma unroll
              for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) pre[j][e] = g_keep[j][e];
            } else {
              load_tile_bf16<NT>(pre, ph.res, ph.ldr, tile * BN, p.M, q, lane);
            }
          } else if (ph.kind == PH_GATEUP) {
            const int blk = tile >> 1;
            pair_here = tile_finisher(2 * blk, upt, total, pg) == tile_finisher(2 * blk + 1, upt, total, pg);
            if (!(tile & 1) && !pair_here)  // the up values, published by their finisher as self-announcing words
              partial_take<NT>(p.pair_words + ((size_t)blk * 4 + q) * C::RED_FLOATS, pre, lane, abort_v, abort_g);
            if ((tile & 1) && pair_here) {  // the gate values this CTA kept, read back before the sums arrive
#pragma unroll
              for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) pre[j][e] = g_keep[j][e];
            }
          }
        }
        // ---- the tile's own sums from the consumers
        const int slot = n_te & 1;
        float tot[NT][4];
        zero4<NT>(tot);
        const bool ok = !(*abort_v) && mbar_wait_bounded(&res_full[slot], (n_te >> 1) & 1, abort_v);
        if (ok) {
          red_add<NT, false>(red + (slot * 4 + q) * C::RED_FLOATS, tot, lane);
        } else if (!(*abort_v)) {
          raise_error(ERR_TIMEOUT_FULL);
          *abort_v = 1;
          *abort_g = 1;
        }
        mbar_arrive(&res_empty[slot]);
        ++n_te;
        if (!finisher) {
          // contributor: publish the partial sums (the finisher polls them)
          partial_store<NT>(p.partials + (((size_t)blockIdx.x * 2) * 4 + q) * C::RED_FLOATS, tot, lane);
          continue;
        }
        if (c_last != fin) {  // own sums first, then the contributors' in CTA order
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) tot[j][e] += part[j][e];
        }
        finish_tile<BITS, NT>(p, ph, out_a, tile, pair_here, q, lane, tot, rf, pre, g_keep, es);
      }
    }
    // phase done: the epilogue warps' writes (which other CTAs read through
    // the generic proxy and through bulk copies) are published by one release
    // after a barrier over the four warps
    fence_proxy_async();
    named_bar_sync(EPI_BAR, EPI_THREADS);
    if (q == 0 && lane == 0 && ph_i + 1 < p.n_phases) red_release_add(p.grid_bar + ph_i + 1, 1u);
    if (q == 0 && lane == 0) st_release_cta(&arrived_ph, ph_i);  // the weights may now fill the ring
  }
  named_bar_sync(6, NEW * 32);  // every arrival of this CTA is made
  // the last CTA to finish resets the grid counters (the workspace's counters
  // are zero between calls): every CTA has made all its arrivals by then
  if (q == 0 && lane == 0) {
    __threadfence();
    if (atomicAdd(p.exit_counter, 1) == p.grid - 1) {
      for (int t = 1; t < p.n_phases; ++t) p.grid_bar[t] = 0;
      *p.exit_counter = 0;
      __threadfence();
    }
  }
}

}  // namespace sv
