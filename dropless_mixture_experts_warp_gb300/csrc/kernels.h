// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include "common.cuh"
#include "gemm.cuh"
#include "gemm2.cuh"

namespace moe {

constexpr int ROUTE_TOKENS = 128;  // tokens per routing block (16 per warp)
constexpr int ROW_ALIGN = MOE_ROW_ALIGN;

inline int route_blocks(int T) { return T > 0 ? (T + ROUTE_TOKENS - 1) / ROUTE_TOKENS : 1; }

// Scratch of moe_route_topk that moe_permute reads back.
struct RouteScratch {
  int32_t* counter;     // 1 int, reset by the call
  int32_t* block_hist;  // [blocks][E] tokens of each routing block per expert
  int32_t* block_base;  // [blocks][E] rows of expert e taken by earlier blocks
  int32_t* local_rank;  // [T][k] rank of (t, j) among the block's tokens of its expert
};

void count_launch();
int num_sms();

// Options of the group-limited sigmoid router (see route_topk_kernel).
struct GroupedRoute {
  const float* bias;  // [E] selection bias or NULL
  int n_group, topk_group;
  float scale;        // routed scaling factor of the weights
};
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int score, int32_t* topk_idx,
                              float* topk_w, int32_t* split_sizes, int32_t* offsets,
                              int32_t* row_offsets, const RouteScratch& ws, int32_t* status,
                              cudaStream_t stream, const GroupedRoute* grouped = nullptr);
cudaError_t launch_permute(const void* x, int T, int d, int E, int k, const int32_t* topk_idx,
                           const float* topk_w, const int32_t* split_sizes, const int32_t* row_offsets,
                           const RouteScratch& ws, void* xp, int32_t* row_to_token,
                           int32_t* token_to_row, float* w_rows, int rows_cap, int32_t* status,
                           cudaStream_t stream);
cudaError_t launch_combine_bwd(const void* dy, int T, int d, int E, int k, const int32_t* token_to_row,
                               const int32_t* split_sizes, const int32_t* row_offsets, void* dy_rows,
                               int rows_cap, cudaStream_t stream);
cudaError_t launch_combine(const void* rows, int T, int d, int k, const int32_t* token_to_row,
                           const void* shared, void* out, int rows_cap, cudaStream_t stream);
cudaError_t launch_dw_reduce(const float* part, int stride, const int32_t* row_offsets, int E,
                             float* dw_rows, int max_rows, cudaStream_t stream);
cudaError_t launch_route_bwd(const float* logits, int T, int E, int k, int score,
                             const int32_t* topk_idx, const float* topk_w, const float* dw_rows,
                             const int32_t* token_to_row, float* d_logits, int rows_cap,
                             cudaStream_t stream, float scale = 1.0f);

cudaError_t launch_wait_timeout(int32_t* status, long long limit, cudaStream_t stream);

// Grouped-GEMM variants (scheduling, epilogue, A/B majorness).
enum GemmKind {
  GEMM_ROWS_SWIGLU_FWD = 0,  // ragged rows, K-major A and B, SwiGLU*w epilogue
  GEMM_ROWS_STORE = 1,       // ragged rows (or dense), K-major A and B
  GEMM_ROWS_STORE_BMN = 2,   // ragged rows (or dense), K-major A, MN-major B
  GEMM_ROWS_SWIGLU_BWD = 3,  // ragged rows, K-major A, MN-major B, SwiGLU' epilogue
  GEMM_KGROUP_STORE = 4,     // ragged K (weight gradients), MN-major A and B
  GEMM_DENSE_AMN_BK = 5,     // dense, MN-major A, K-major B (test hook)
  GEMM_DENSE_AMN_BMN = 6,    // dense, MN-major A and B (test hook)
  GEMM_ROWS_SWIGLU_FWD_MXQ = 7,  // MXFP8 only: gate/up epilogue writing quantised h
  GEMM_ROWS_SWIGLU_BWD_MXQ = 8   // MXFP8 only: SwiGLU' epilogue writing quantised dG|dU
};

cudaError_t launch_gemm_fwd(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, cudaStream_t stream);
cudaError_t launch_gemm_bwd(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, cudaStream_t stream);
// The same products on CTA pairs (M = 256 per MMA; K-major B tensor maps with boxes of
// BN/2 rows; BN 128 or 256; SCHED_KGROUP needs p.M % 256 == 0).
cudaError_t launch_gemm_pair(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                             const GemmParams& p, cudaStream_t stream);

// The CTA-pair kernel where the product allows it (tiles at least 128 columns wide;
// weight gradients in 256-row pairs), else the single-CTA kernel (bwd selects the
// translation unit holding the backward instantiations).
cudaError_t launch_best(GemmKind kind, bool bwd, const CUtensorMap& a, const CUtensorMap& b,
                        const GemmParams& p, cudaStream_t stream);

// Grid of a persistent CTA-pair kernel: as many pairs as can be resident at once
// (an SM whose TPC neighbour is unavailable cannot host half of a pair), at most
// one per two SMs.
int pair_grid(const void* kern, int threads, int smem_bytes);

// c: tensor map of the bf16 output for the STORE epilogue, of G|U for the SwiGLU one,
// of dG|dU for the SwiGLU' one; dd: of h for the SwiGLU epilogue, of the saved G|U
// (read) for the SwiGLU' one (unused otherwise)
template <int SCHED, int EPI, bool A_MN, bool B_MN>
cudaError_t launch_gemm_pair_t(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                               const CUtensorMap& dd, const GemmParams& p, cudaStream_t stream) {
  auto kern = grouped_gemm_pair_kernel<SCHED, EPI, A_MN, B_MN>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p_smem_bytes(EPI));
  if (err != cudaSuccess) return err;
  static const int grid = pair_grid(reinterpret_cast<const void*>(kern), pair_threads(EPI), p_smem_bytes(EPI));
  kern<<<grid, pair_threads(EPI), p_smem_bytes(EPI), stream>>>(a, b, c, dd, p);
  count_launch();
  return cudaGetLastError();
}

// One MXFP8 operand, K-major: E4M3 codes [outer][inner] (inner = K) and their SF tiles;
// fp4 (B operands only): E2M1 codes packed two a byte ([outer][inner / 2] bytes).
struct MxMat {
  const uint8_t* codes;
  const uint8_t* sf;
  uint64_t inner, outer;
  bool fp4;
  const uint8_t* sf_rep = nullptr;  // the SF tiles each four times over (SF_REP_TILE_BYTES), or NULL
};
// MXFP8 grouped GEMM; kind is one of GEMM_ROWS_STORE, GEMM_KGROUP_STORE,
// GEMM_ROWS_SWIGLU_FWD_MXQ, GEMM_ROWS_SWIGLU_BWD_MXQ.  p.sfa/p.sfb are taken from a
// and b.
cudaError_t launch_gemm_mx(GemmKind kind, const MxMat& a, const MxMat& b, GemmParams p, cudaStream_t stream);
// The CTA-pair form for GEMM_ROWS_STORE and GEMM_KGROUP_STORE (BN = 256 or 128, B boxes
// of BN / 2 rows, SF maps from make_tensor_map_sf; SCHED_KGROUP needs p.M % 256 == 0).
cudaError_t launch_gemm_mx_pair(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                                const CUtensorMap& sfb, const CUtensorMap& c, const GemmParams& p,
                                cudaStream_t stream);
cudaError_t launch_route_maps(int T, int E, int k, const int32_t* topk_idx, const float* topk_w,
                              const int32_t* split_sizes, const int32_t* row_offsets, const RouteScratch& ws,
                              int32_t* row_to_token, int32_t* token_to_row, float* w_rows, int rows_cap,
                              int32_t* status, cudaStream_t stream);
cudaError_t launch_quant_rows(const void* src, long long rows, int C, long long ld, const int32_t* nrows_dev,
                              uint8_t* codes, uint8_t* sf, cudaStream_t stream);
cudaError_t launch_quant_cols_t(const void* src, int batch, long long rows, int C, const int32_t* nrows_dev,
                                uint8_t* codes, uint8_t* sf, cudaStream_t stream, const int32_t* row_map = nullptr,
                                uint8_t* codes_rows = nullptr, uint8_t* sf_rows = nullptr, bool fp4 = false,
                                uint8_t* sf_rep = nullptr);
RouteScratch route_scratch(const moe_dims& d, void* ws);
float* workspace_dw_part(const moe_dims& d, void* ws);
bool make_tensor_map_sf(CUtensorMap* m, const void* base, uint64_t bytes, uint32_t box_rows = 2);
bool make_tensor_map_store(CUtensorMap* m, const void* base, uint64_t cols, uint64_t ld, uint64_t rows);
bool make_tensor_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                          uint32_t box_inner, uint32_t box_outer);
bool make_tensor_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer);
// Packed 4-bit codes [outer][inner / 2] bytes loaded as 16-element groups padded to 16
// bytes in shared memory (the layout the block-scaled MMA reads for E2M1 under
// kind::mxf8f6f4), 128B swizzle; box_inner must be 128 elements.
bool make_tensor_map_fp4(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer);

template <int SCHED, int EPI, bool A_MN, bool B_MN>
cudaError_t launch_gemm_t(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                          cudaStream_t stream) {
  auto kern = grouped_gemm_kernel<SCHED, EPI, A_MN, B_MN>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES);
  if (err != cudaSuccess) return err;
  kern<<<num_sms(), gemm_threads(EPI), GEMM_SMEM_BYTES, stream>>>(a, b, p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
