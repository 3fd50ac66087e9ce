// Unit-packed weights: a one-time relayout of a quantized weight (same bytes,
// plus zero rows up to a multiple of 64) so that each (64-row tile, 512-wide
// k chunk) unit of the verify matmul is one contiguous block:
//
//   [codes: 128-byte pieces x 64 rows, each row's 16-byte chunk c stored at
//    c ^ (row & 7) (the 128-byte swizzle the consumers read)]
//   [scales: 64 rows x 8 groups fp16] [biases: 64 rows x 8 groups fp16]
//
// units in tile-major, chunk-minor order.  A stage of the weight stream is
// then one bulk copy instead of a strided 3D box and two 16-byte-wide boxes.
#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {

size_t packed_bytes(int N, int K, int bits) {
  const size_t tiles = (size_t)(N + BN - 1) / BN, units = tiles * (size_t)(K / KC);
  const size_t unit = (size_t)BN * KC * bits / 8 + 2 * (size_t)BN * GPS * 2;
  return units * unit;
}

template <int BITS>
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t* __restrict__ wq, const uint16_t* __restrict__ scales,
                                                   const uint16_t* __restrict__ biases, int N, int K,
                                                   uint8_t* __restrict__ out) {
  constexpr int ROW_BYTES = KC * BITS / 8, W_BYTES = BN * ROW_BYTES, SB_BYTES = BN * GPS * 2;
  constexpr int UNIT = W_BYTES + 2 * SB_BYTES, CHUNKS = ROW_BYTES / 16;
  const int upt = K / KC, u = blockIdx.x, tile = u / upt, kc = u % upt;
  const size_t row_total = (size_t)K * BITS / 8, G = (size_t)K / GROUP;
  uint8_t* dst = out + (size_t)u * UNIT;
  for (int i = threadIdx.x; i < BN * CHUNKS; i += blockDim.x) {
    const int r = i / CHUNKS, j = i % CHUNKS, n = tile * BN + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < N) v = *reinterpret_cast<const uint4*>(wq + (size_t)n * row_total + (size_t)kc * ROW_BYTES + (size_t)j * 16);
    const int piece = j / 8, c = j % 8;
    *reinterpret_cast<uint4*>(dst + piece * (BN * 128) + r * 128 + ((c ^ (r & 7)) << 4)) = v;
  }
  for (int r = threadIdx.x; r < 2 * BN; r += blockDim.x) {
    const int row = r % BN, n = tile * BN + row;
    const uint16_t* src = r < BN ? scales : biases;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < N) v = *reinterpret_cast<const uint4*>(src + (size_t)n * G + (size_t)kc * GPS);
    *reinterpret_cast<uint4*>(dst + W_BYTES + (r < BN ? 0 : SB_BYTES) + row * GPS * 2) = v;
  }
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t sv_qmm_pack_bytes(int N, int K, int bits) {
  if (N < 1 || N > MAX_TILES * BN || K < KC || K % KC || K > (1 << 20) || !bits_supported(bits)) return 0;
  return packed_bytes(N, K, bits);
}

int sv_qmm_pack(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits, int group,
                void* packed, size_t packed_size, void* stream) {
  int st = check_weight(wq, scales, biases, N, K, bits, group, 1);
  if (st) return st;
  if (!packed || !aligned(packed, 16)) return fail(SV_EINVAL, "packed must be non-null and 16-byte aligned");
  const size_t need = packed_bytes(N, K, bits);
  if (packed_size < need) return fail(SV_EINVAL, "packed buffer too small: %zu < %zu", packed_size, need);
  const unsigned units = (unsigned)(((size_t)N + BN - 1) / BN * (size_t)(K / KC));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* w = reinterpret_cast<const uint8_t*>(wq);
  uint8_t* out = static_cast<uint8_t*>(packed);
  if (bits == 8)
    pack_kernel<8><<<units, 256, 0, s>>>(w, scales, biases, N, K, out);
  else if (bits == 4)
    pack_kernel<4><<<units, 256, 0, s>>>(w, scales, biases, N, K, out);
  else
    pack_kernel<2><<<units, 256, 0, s>>>(w, scales, biases, N, K, out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "pack launch");
  return SV_OK;
}

}  // extern "C"
