// Instantiations of the MXFP8 grouped GEMM.
#include "gemm_mx.cuh"
#include "kernels.h"

namespace moe {

template <int SCHED, int EPI>
static cudaError_t launch_mx_t(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                               cudaStream_t stream) {
  // the STORE epilogue writes through a tensor map of the output
  CUtensorMap c = a;
  if (EPI == EPI_STORE) {
    if (!p.out || p.ldo % 8 != 0 || (reinterpret_cast<uintptr_t>(p.out) & 15u)) return cudaErrorInvalidValue;
    const uint64_t rows = SCHED == SCHED_KGROUP ? static_cast<uint64_t>(p.E) * p.M : static_cast<uint64_t>(p.row_limit);
    if (!make_tensor_map_store(&c, p.out, p.N, p.ldo, rows)) return cudaErrorInvalidValue;
  }
  auto kern = grouped_gemm_mx_kernel<SCHED, EPI>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mx_smem_bytes(EPI));
  if (err != cudaSuccess) return err;
  kern<<<num_sms(), gemm_threads(EPI), mx_smem_bytes(EPI), stream>>>(a, b, c, p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gemm_mx(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                           cudaStream_t stream) {
  switch (kind) {
    case GEMM_ROWS_SWIGLU_FWD: return launch_mx_t<SCHED_ROWS, EPI_SWIGLU_FWD>(a, b, p, stream);
    case GEMM_ROWS_STORE: return launch_mx_t<SCHED_ROWS, EPI_STORE>(a, b, p, stream);
    case GEMM_ROWS_SWIGLU_BWD: return launch_mx_t<SCHED_ROWS, EPI_SWIGLU_BWD>(a, b, p, stream);
    case GEMM_KGROUP_STORE: return launch_mx_t<SCHED_KGROUP, EPI_STORE>(a, b, p, stream);
    case GEMM_ROWS_SWIGLU_FWD_MXQ: return launch_mx_t<SCHED_ROWS, EPI_SWIGLU_FWD_MX>(a, b, p, stream);
    case GEMM_ROWS_SWIGLU_BWD_MXQ: return launch_mx_t<SCHED_ROWS, EPI_SWIGLU_BWD_MX>(a, b, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
