// Instantiations of the persistent verify matmul for 2-bit codes (one
// translation unit per code width so they compile in parallel).
#include "stream_kernel.cuh"

namespace sv {

template <int NT>
static cudaError_t launch_one(const StreamParams& p, cudaStream_t s) {
  using C = StreamCfg<2, NT>;
  static bool attr_set = false;  // the attribute is per function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(stream_kernel<2, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.grid), dim3(QMM_THREADS), C::SMEM, s, attr);
  if (p.n_phases > 1) {  // grid barriers between phases need every CTA resident
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, stream_kernel<2, NT>, p);
}

cudaError_t launch_stream_b2(const StreamParams& p, cudaStream_t s) {
  switch (p.MP / 8) {
    case 1: return launch_one<1>(p, s);
    case 2: return launch_one<2>(p, s);
    case 3: return launch_one<3>(p, s);
    case 4: return launch_one<4>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

// CTAs of this kernel that fit on the device at once (cooperative launch limit).
int stream_max_grid_b2(int MP) {
  int per_sm = 0, dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = cudaErrorInvalidValue;
  switch (MP / 8) {
#define SV_OCC(NT)                                                                                           \
  case NT:                                                                                                   \
    cudaFuncSetAttribute(stream_kernel<2, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,              \
                         StreamCfg<2, NT>::SMEM);                                                          \
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_kernel<2, NT>, QMM_THREADS,         \
                                                      StreamCfg<2, NT>::SMEM);                             \
    break;
    SV_OCC(1) SV_OCC(2) SV_OCC(3) SV_OCC(4)
#undef SV_OCC
    default: break;
  }
  if (e != cudaSuccess) return 0;
  return per_sm * sms;
}

}  // namespace sv
