// Launcher and instantiations of the MXFP8 CTA-pair grouped GEMM (STORE epilogue).
#include "gemm_mx2.cuh"
#include "kernels.h"

namespace moe {

template <int SCHED>
static cudaError_t launch_mxp_t(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                                const CUtensorMap& sfb, const CUtensorMap& c, const GemmParams& p,
                                cudaStream_t stream) {
  auto kern = grouped_gemm_mx_pair_kernel<SCHED>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MXP_SMEM_BYTES);
  if (err != cudaSuccess) return err;
  static const int grid = pair_grid(reinterpret_cast<const void*>(kern), MXP_THREADS, MXP_SMEM_BYTES);
  kern<<<grid, MXP_THREADS, MXP_SMEM_BYTES, stream>>>(a, b, sfa, sfb, c, p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gemm_mx_pair(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                                const CUtensorMap& sfb, const CUtensorMap& c, const GemmParams& p,
                                cudaStream_t stream) {
  switch (kind) {
    case GEMM_ROWS_STORE: return launch_mxp_t<SCHED_ROWS>(a, b, sfa, sfb, c, p, stream);
    case GEMM_KGROUP_STORE: return launch_mxp_t<SCHED_KGROUP>(a, b, sfa, sfb, c, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
