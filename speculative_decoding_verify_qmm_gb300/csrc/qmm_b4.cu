// Instantiations of the verify-matmul kernel for 4-bit codes (one translation
// unit per code width so the two compile in parallel).
#include "qmm_kernel.cuh"

namespace sv {

template <int NT>
static cudaError_t launch_one(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tb,
                              const QmmParams& p, cudaStream_t s) {
  using C = QmmCfg<4, NT>;
  static bool attr_set = false;  // per process; the attribute is per function, not per device
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(qmm_stream_kernel<4, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.sch.grid), dim3(QMM_THREADS), C::SMEM, s, attr);
  return cudaLaunchKernelEx(&cfg, qmm_stream_kernel<4, NT>, tw, ts, tb, p);
}

cudaError_t launch_qmm_b4(int NT, const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tb,
                             const QmmParams& p, cudaStream_t s) {
  switch (NT) {
    case 1: return launch_one<1>(tw, ts, tb, p, s);
    case 2: return launch_one<2>(tw, ts, tb, p, s);
    case 3: return launch_one<3>(tw, ts, tb, p, s);
    case 4: return launch_one<4>(tw, ts, tb, p, s);
    default: return cudaErrorInvalidValue;
  }
}

int qmm_smem_b4(int NT) {
  switch (NT) {
    case 1: return QmmCfg<4, 1>::SMEM;
    case 2: return QmmCfg<4, 2>::SMEM;
    case 3: return QmmCfg<4, 3>::SMEM;
    case 4: return QmmCfg<4, 4>::SMEM;
    default: return 0;
  }
}

}  // namespace sv
