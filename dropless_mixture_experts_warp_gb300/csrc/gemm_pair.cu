// Instantiations of the CTA-pair grouped GEMM.
#include "kernels.h"

namespace moe {

cudaError_t launch_gemm_pair(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                             cudaStream_t stream) {
  CUtensorMap c = a, dd = a;
  if (kind == GEMM_ROWS_SWIGLU_FWD) {  // maps of G|U [rows][2f] and h [rows][f]
    const uintptr_t al = reinterpret_cast<uintptr_t>(p.gu_out) | reinterpret_cast<uintptr_t>(p.h_out);
    if (!p.gu_out || !p.h_out || (al & 15u) || p.f % 8 != 0) return cudaErrorInvalidValue;
    const uint64_t rows = static_cast<uint64_t>(p.row_limit);
    if (!make_tensor_map_store(&c, p.gu_out, 2ull * p.f, 2ull * p.f, rows) ||
        !make_tensor_map_store(&dd, p.h_out, static_cast<uint64_t>(p.f), static_cast<uint64_t>(p.f), rows))
      return cudaErrorInvalidValue;
  } else if (kind == GEMM_ROWS_SWIGLU_BWD) {  // maps of dG|dU and of the saved G|U, both [rows][2f]
    const uintptr_t al = reinterpret_cast<uintptr_t>(p.dgu_out) | reinterpret_cast<uintptr_t>(p.gu_in);
    if (!p.dgu_out || !p.gu_in || (al & 15u) || p.f % 32 != 0) return cudaErrorInvalidValue;
    const uint64_t rows = static_cast<uint64_t>(p.row_limit);
    if (!make_tensor_map_store(&c, p.dgu_out, 2ull * p.f, 2ull * p.f, rows) ||
        !make_tensor_map_store(&dd, p.gu_in, 2ull * p.f, 2ull * p.f, rows))
      return cudaErrorInvalidValue;
  } else {  // STORE: a map of the output
    if (!p.out || p.ldo % 8 != 0 || (reinterpret_cast<uintptr_t>(p.out) & 15u)) return cudaErrorInvalidValue;
    const uint64_t rows = kind == GEMM_KGROUP_STORE ? static_cast<uint64_t>(p.E) * p.M
                                                    : static_cast<uint64_t>(p.row_limit);
    if (!make_tensor_map_store(&c, p.out, p.N, p.ldo, rows)) return cudaErrorInvalidValue;
  }
  switch (kind) {
    case GEMM_ROWS_SWIGLU_FWD:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_SWIGLU_FWD, false, false>(a, b, c, dd, p, stream);
    case GEMM_ROWS_STORE:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_STORE, false, false>(a, b, c, dd, p, stream);
    case GEMM_ROWS_STORE_BMN:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_STORE, false, true>(a, b, c, dd, p, stream);
    case GEMM_ROWS_SWIGLU_BWD:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_SWIGLU_BWD, false, true>(a, b, c, dd, p, stream);
    case GEMM_KGROUP_STORE:
      return launch_gemm_pair_t<SCHED_KGROUP, EPI_STORE, true, true>(a, b, c, dd, p, stream);
    case GEMM_DENSE_AMN_BK:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_STORE, true, false>(a, b, c, dd, p, stream);
    case GEMM_DENSE_AMN_BMN:
      return launch_gemm_pair_t<SCHED_ROWS, EPI_STORE, true, true>(a, b, c, dd, p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
