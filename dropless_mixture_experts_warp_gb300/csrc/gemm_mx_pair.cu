// CTA-pair instantiations of the MXFP8 grouped GEMM.
#include "gemm_mx2.cuh"
#include "kernels.h"

namespace moe {

template <int SCHED, int EPI>
static cudaError_t launch_mxp_t(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                                const CUtensorMap& sfb, const CUtensorMap& c, const GemmParams& p,
                                cudaStream_t stream) {
  auto kern = grouped_gemm_mx_pair_kernel<SCHED, EPI>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mxp_smem_bytes(EPI));
  if (err != cudaSuccess) return err;
  static const int grid = pair_grid(reinterpret_cast<const void*>(kern), gemm_threads(EPI), mxp_smem_bytes(EPI));
  kern<<<grid, gemm_threads(EPI), mxp_smem_bytes(EPI), stream>>>(a, b, sfa, sfb, c, p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gemm_mx_pair(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                                const CUtensorMap& sfb, const CUtensorMap& c, const GemmParams& p,
                                cudaStream_t stream) {
  switch (kind) {
    case GEMM_ROWS_STORE: return launch_mxp_t<SCHED_ROWS, EPI_STORE>(a, b, sfa, sfb, c, p, stream);
    case GEMM_KGROUP_STORE: return launch_mxp_t<SCHED_KGROUP, EPI_STORE>(a, b, sfa, sfb, c, p, stream);
    case GEMM_ROWS_SWIGLU_FWD_MXQ: return launch_mxp_t<SCHED_ROWS, EPI_SWIGLU_FWD_MX>(a, b, sfa, sfb, c, p, stream);
    case GEMM_ROWS_SWIGLU_BWD_MXQ: return launch_mxp_t<SCHED_ROWS, EPI_SWIGLU_BWD_MX>(a, b, sfa, sfb, c, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
