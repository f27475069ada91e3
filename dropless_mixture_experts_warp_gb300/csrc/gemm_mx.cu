// Launcher and instantiations of the MXFP8 grouped GEMM.
#include "gemm_mx.cuh"
#include "kernels.h"

namespace moe {

template <int SCHED, int EPI>
static cudaError_t launch_mx_t(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, const GemmParams& p,
                               cudaStream_t stream) {
  auto kern = grouped_gemm_mx_kernel<SCHED, EPI>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mx_smem_bytes(EPI));
  if (err != cudaSuccess) return err;
  kern<<<num_sms(), mx_threads(EPI), mx_smem_bytes(EPI), stream>>>(a, b, c, p);
  count_launch();
  return cudaGetLastError();
}

// The weight gradients (ragged K, plain bf16 output) run on CTA pairs (gemm_mx2.cuh) where
// their output rows come in 256-row pairs: DeepSeek-V3 shape down wgrad 1640 -> 1700 TF/s,
// uniform 1024-row experts 2142 -> 2382.  The row-scheduled products stay on single CTAs:
// on pairs an expert with an odd number of 128-row tiles wastes half of its last pair tile
// (1.28x the rows instead of 1.12x at the DeepSeek-V3 shape) and they measured 5-7 % slower.

cudaError_t launch_gemm_mx(GemmKind kind, const MxMat& a, const MxMat& b, GemmParams p, cudaStream_t stream) {
  const bool split = kind == GEMM_ROWS_SWIGLU_FWD_MXQ;
  const bool kgroup = kind == GEMM_KGROUP_STORE;
  const bool store = kind == GEMM_ROWS_STORE || kgroup;
  if (!store && kind != GEMM_ROWS_SWIGLU_FWD_MXQ && kind != GEMM_ROWS_SWIGLU_BWD_MXQ) return cudaErrorInvalidValue;
  if (p.BN != 128 && p.BN != 256) return cudaErrorInvalidValue;
  if (split && p.BN != 256) return cudaErrorInvalidValue;  // gate and up halves are whole 128-row SF tiles
  p.sfa = a.sf;
  p.sfb = b.sf;
  const bool pair = kgroup && p.M % 256 == 0 && num_sms() >= 2;
  // B box: this CTA's half of the BN rows on pairs, the gate (or up) half for the split
  // epilogue, else BN
  const int b_box = (split || pair) ? p.BN / 2 : p.BN;
  CUtensorMap ta, tb, tc;
  if (a.fp4 || !make_tensor_map_u8(&ta, a.codes, a.inner, a.outer, 128, BM)) return cudaErrorInvalidValue;
  if (b.fp4) {  // E2M1 weights: 4-bit codes, MMA B format E2M1
    if (!make_tensor_map_fp4(&tb, b.codes, b.inner, b.outer, b_box)) return cudaErrorInvalidValue;
    p.b_fmt = MX_FMT_E2M1;
  } else {
    if (!make_tensor_map_u8(&tb, b.codes, b.inner, b.outer, 128, b_box)) return cudaErrorInvalidValue;
    p.b_fmt = MX_FMT_E4M3;
  }
  tc = ta;
  if (kind == GEMM_ROWS_SWIGLU_BWD_MXQ && p.BN == 256) {  // the SwiGLU' epilogue reads G|U by tensor loads
    if (!p.gu_in || (reinterpret_cast<uintptr_t>(p.gu_in) & 15u) || p.f % 32 != 0) return cudaErrorInvalidValue;
    if (!make_tensor_map_store(&tc, p.gu_in, 2ull * p.f, 2ull * p.f, static_cast<uint64_t>(p.row_limit)))
      return cudaErrorInvalidValue;
  }
  if (store) {  // the STORE epilogue writes through a tensor map of the output
    if (!p.out || p.ldo % 8 != 0 || (reinterpret_cast<uintptr_t>(p.out) & 15u)) return cudaErrorInvalidValue;
    const uint64_t rows = kgroup ? static_cast<uint64_t>(p.E) * p.M : static_cast<uint64_t>(p.row_limit);
    if (!make_tensor_map_store(&tc, p.out, p.N, p.ldo, rows)) return cudaErrorInvalidValue;
  }
  if (pair) {
    // B's SF tiles in the replicated form where the caller has them (one 2 KB tensor load a
    // tile, one tensor-pipe copy for both tiles of a 256-row B tile)
    p.sfb_rep = (b.sf_rep && p.BN == 256) ? 1 : 0;
    CUtensorMap tsa, tsb;
    const bool sfb_ok = p.sfb_rep ? make_tensor_map_sf(&tsb, b.sf_rep, 4 * b.inner * b.outer / 32, 8)
                                  : make_tensor_map_sf(&tsb, b.sf, b.inner * b.outer / 32);
    if (!make_tensor_map_sf(&tsa, a.sf, a.inner * a.outer / 32) || !sfb_ok) return cudaErrorInvalidValue;
    return launch_gemm_mx_pair(kind, ta, tb, tsa, tsb, tc, p, stream);
  }
  switch (kind) {
    case GEMM_ROWS_STORE: return launch_mx_t<SCHED_ROWS, EPI_STORE>(ta, tb, tc, p, stream);
    case GEMM_KGROUP_STORE: return launch_mx_t<SCHED_KGROUP, EPI_STORE>(ta, tb, tc, p, stream);
    case GEMM_ROWS_SWIGLU_FWD_MXQ: return launch_mx_t<SCHED_ROWS, EPI_SWIGLU_FWD_MX>(ta, tb, tc, p, stream);
    case GEMM_ROWS_SWIGLU_BWD_MXQ: return launch_mx_t<SCHED_ROWS, EPI_SWIGLU_BWD_MX>(ta, tb, tc, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
