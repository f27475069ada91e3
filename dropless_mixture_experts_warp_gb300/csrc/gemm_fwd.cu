// Instantiations of the grouped GEMM used by the forward pass (and the dense test
// hook with an MN-major A operand).
#include "kernels.h"

namespace moe {

cudaError_t launch_gemm_fwd(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, cudaStream_t stream) {
  switch (kind) {
    case GEMM_ROWS_SWIGLU_FWD:
      return launch_gemm_t<SCHED_ROWS, EPI_SWIGLU_FWD, false, false>(a, b, p, stream);
    case GEMM_ROWS_STORE:
      return launch_gemm_t<SCHED_ROWS, EPI_STORE, false, false>(a, b, p, stream);
    case GEMM_DENSE_AMN_BK:
      return launch_gemm_t<SCHED_ROWS, EPI_STORE, true, false>(a, b, p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
