// Instantiations of the CTA-pair grouped GEMM.
#include "kernels.h"

namespace moe {

cudaError_t launch_gemm_pair(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                             cudaStream_t stream) {
  switch (kind) {
    case GEMM_ROWS_SWIGLU_FWD:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_SWIGLU_FWD, false, false>(a, b, p, stream);
    case GEMM_ROWS_STORE:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_STORE, false, false>(a, b, p, stream);
    case GEMM_ROWS_STORE_BMN:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_STORE, false, true>(a, b, p, stream);
    case GEMM_ROWS_SWIGLU_BWD:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_SWIGLU_BWD, false, true>(a, b, p, stream);
    case GEMM_KGROUP_STORE:
      return launch_gemm_pair_t<SCHED_KGROUP, EPI_STORE, true, true>(a, b, p, stream);
    case GEMM_DENSE_AMN_BK:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_STORE, true, false>(a, b, p, stream);
    case GEMM_DENSE_AMN_BMN:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_STORE, true, true>(a, b, p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
