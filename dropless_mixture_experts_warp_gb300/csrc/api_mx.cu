// C-ABI entry points of the MXFP8 path.
#include <cstring>

#include "kernels.h"

namespace moe {
static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static moe_status cuda_st(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_mx_quantize_rows(const moe_bf16* src, int64_t rows, int32_t C, int64_t ld,
                                const int32_t* nrows_dev, uint8_t* codes, uint8_t* scales, void* stream) {
  if (rows < 0 || C <= 0 || ld < C) return MOE_ERR_INVALID_ARG;
  if (C % 128 || ld % 8) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (!src || !codes || !scales) return MOE_ERR_INVALID_ARG;
  if (!al16(src) || !al16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u)) return MOE_ERR_ALIGNMENT;
  return cuda_st(launch_quant_rows(src, rows, C, ld, nrows_dev, codes, scales, static_cast<cudaStream_t>(stream)));
}

moe_status moe_mx_quantize_cols(const moe_bf16* src, int32_t batch, int64_t rows, int32_t C,
                                const int32_t* nrows_dev, uint8_t* codes_t, uint8_t* scales, void* stream) {
  if (batch < 0 || rows < 0 || C <= 0) return MOE_ERR_INVALID_ARG;
  if (rows % 128 || C % 128) return MOE_ERR_UNSUPPORTED;
  if (rows == 0 || batch == 0) return MOE_OK;
  if (!src || !codes_t || !scales) return MOE_ERR_INVALID_ARG;
  if (!al16(src) || !al16(codes_t)) return MOE_ERR_ALIGNMENT;
  return cuda_st(launch_quant_cols_t(src, batch, rows, C, nrows_dev, codes_t, scales,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_mxfp8(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b, const uint8_t* b_sf,
                          moe_bf16* c, int32_t M, int32_t N, int32_t K, int32_t* dev_status, void* stream) {
  if (!a || !a_sf || !b || !b_sf || !c || !dev_status) return MOE_ERR_INVALID_ARG;
  if (M < 128 || N < 128 || K < 128 || M % 128 || N % 128 || K % 128) return MOE_ERR_UNSUPPORTED;
  if (!al16(a) || !al16(b) || !al16(c) || !al16(a_sf) || !al16(b_sf)) return MOE_ERR_ALIGNMENT;
  const int bn = N % 256 == 0 ? 256 : 128;
  CUtensorMap ta, tb;
  if (!make_tensor_map_u8(&ta, a, K, M, 128, BM) || !make_tensor_map_u8(&tb, b, K, N, 128, bn))
    return MOE_ERR_CUDA;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.BN = bn; p.N = N; p.K = K; p.M = M; p.E = 1; p.row_offsets = nullptr; p.m_fastest = 1;
  p.out = c; p.ldo = N; p.row_limit = M; p.status = dev_status;
  p.sfa = a_sf; p.sfb = b_sf; p.a_sf_ktiles = K / 128; p.b_sf_ktiles = K / 128;
  return cuda_st(launch_gemm_mx(GEMM_ROWS_STORE, ta, tb, p, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
