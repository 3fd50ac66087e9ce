// Allocation-free form of the verify matmul.
//
// Some callers cannot hand the library a workspace: code that runs where
// cudaMalloc is off limits - a plugin inside a host application that owns
// every byte of device memory, a runtime that forbids allocation after
// start-up because cudaMalloc can synchronize the device and stall other
// work, or a real-time loop with a fixed memory budget.  For them
// sv_qmm_verify_noalloc keeps its scratch (the counter block, the prepared
// activations and the split-K partials) in one file-scope device array of
// fixed size.  Every GPU that loads this library holds that array until the
// process exits.
#include "sv_internal.h"

namespace sv {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(4) << 20;  // 4 MiB

static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up on
// every call, with the calling thread's current device: once the module is
// loaded this is a cheap table lookup, and it stays right if the context was
// torn down and rebuilt (cudaDeviceReset) since the previous call.
static int noalloc_scratch(void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
  *out = p;
  return SV_OK;
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t sv_qmm_noalloc_scratch_bytes(void) { return NOALLOC_SCRATCH_BYTES; }

int sv_qmm_verify_noalloc(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int N, int K, int bits,
                          int group, const uint16_t* x, int ldx, int M, uint16_t* y, int ldy,
                          const uint16_t* residual, int ldr, void* stream) {
  int st = check_weight(wq, scales, biases, N, K, bits, group, M);
  if (st) return st;
  if (!x || !y) return fail(SV_EINVAL, "x and y must be non-null");
  if (ldx < K || ldy < N || (residual && ldr < N)) return fail(SV_EINVAL, "ldx must be >= K, ldy and ldr >= N");
  if (!aligned(x, 2) || !aligned(y, 2) || (residual && !aligned(residual, 2)))
    return fail(SV_EINVAL, "x, y, residual must be 2-byte aligned");
  const size_t need = qmm_bytes(M, N, K, bits, false);
  if (need == 0) return fail(SV_ECUDA, "no CUDA device");
  if (need > NOALLOC_SCRATCH_BYTES)
    return fail(SV_EUNSUPPORTED,
                "this call needs %zu bytes of scratch but the built-in array holds %zu; "
                "use sv_qmm_verify with a caller-provided workspace",
                need, NOALLOC_SCRATCH_BYTES);
  void* ws = nullptr;
  st = noalloc_scratch(&ws);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the last call left; the exit and abort words and
  // the split-tile partials must start at zero, so clear them (a failed
  // earlier call may have left them set).  No allocation: memsets of the
  // array itself.
  size_t part_off = 0, part_bytes = 0;
  qmm_partials_region(M, N, K, bits, &part_off, &part_bytes);
  cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(ws) + EXIT_CTR_OFF, 0, 8, s);  // exit, abort
  if (e == cudaSuccess) e = cudaMemsetAsync(static_cast<uint8_t*>(ws) + part_off, 0, part_bytes, s);
  if (e != cudaSuccess) return cuda_fail(e, "clear scratch counters");
  st = qmm_prepare_internal(x, ldx, M, K, bits, PREP_PLAIN, nullptr, 0, nullptr, 0.f, ws, s);
  if (st) return st;
  return qmm_run_internal(wq, scales, biases, N, K, bits, M, residual ? 1 : 0, y, ldy,
                          residual, ldr, nullptr, 0, 0.f, nullptr, nullptr, nullptr, ws, s);
}

}  // extern "C"
