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
  const MxMat ma{a, a_sf, static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const MxMat mb{b, b_sf, static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.BN = bn; p.N = N; p.K = K; p.M = M; p.E = 1; p.row_offsets = nullptr; p.m_fastest = 1;
  p.out = c; p.ldo = N; p.row_limit = M; p.status = dev_status;
  p.a_sf_ktiles = K / 128; p.b_sf_ktiles = K / 128;
  return cuda_st(launch_gemm_mx(GEMM_ROWS_STORE, ma, mb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_mxf8f4(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b4, const uint8_t* b_sf,
                           moe_bf16* c, int32_t M, int32_t N, int32_t K, int32_t* dev_status, void* stream) {
  if (!a || !a_sf || !b4 || !b_sf || !c || !dev_status) return MOE_ERR_INVALID_ARG;
  if (M < 128 || N < 128 || K < 128 || M % 128 || N % 128 || K % 128) return MOE_ERR_UNSUPPORTED;
  if (!al16(a) || !al16(c) || !al16(a_sf) || !al16(b_sf)) return MOE_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(b4) & 31u) return MOE_ERR_ALIGNMENT;   // 4-bit tensor loads want 32 bytes
  const int bn = N % 256 == 0 ? 256 : 128;
  const MxMat ma{a, a_sf, static_cast<uint64_t>(K), static_cast<uint64_t>(M), false};
  const MxMat mb{b4, b_sf, static_cast<uint64_t>(K), static_cast<uint64_t>(N), true};
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.BN = bn; p.N = N; p.K = K; p.M = M; p.E = 1; p.row_offsets = nullptr; p.m_fastest = 1;
  p.out = c; p.ldo = N; p.row_limit = M; p.status = dev_status;
  p.a_sf_ktiles = K / 128; p.b_sf_ktiles = K / 128;
  return cuda_st(launch_gemm_mx(GEMM_ROWS_STORE, ma, mb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_mx4_quantize_cols(const moe_bf16* src, int32_t batch, int64_t rows, int32_t C, uint8_t* codes_t,
                                 uint8_t* scales_t, uint8_t* codes, uint8_t* scales, void* stream) {
  if (batch < 0 || rows < 0 || C <= 0) return MOE_ERR_INVALID_ARG;
  if (rows % 128 || C % 128) return MOE_ERR_UNSUPPORTED;
  if (rows == 0 || batch == 0) return MOE_OK;
  if (!src || !codes_t || !scales_t || !codes || !scales) return MOE_ERR_INVALID_ARG;
  if (!al16(src) || !al16(codes_t) || !al16(codes) || !al16(scales_t) || !al16(scales)) return MOE_ERR_ALIGNMENT;
  return cuda_st(launch_quant_cols_t(src, batch, rows, C, nullptr, codes_t, scales_t,
                                     static_cast<cudaStream_t>(stream), nullptr, codes, scales, true));
}

}  // extern "C"

// ============================================================================ layer path

namespace moe {

static inline size_t a256(size_t x) { return (x + 255) / 256 * 256; }
static int bn_mx(int n) { return n % 256 == 0 ? 256 : 128; }

// One MXFP8 operand: codes and their SF tiles.
struct MxOp {
  uint8_t* codes;
  uint8_t* sf;
};

static size_t op_bytes(size_t elems, bool fp4 = false) { return a256(fp4 ? elems / 2 : elems) + a256(elems / 32); }

static MxOp carve_op(uint8_t*& p, size_t elems, bool fp4 = false) {
  MxOp o;
  o.codes = p;
  p += a256(fp4 ? elems / 2 : elems);
  o.sf = p;
  p += a256(elems / 32);
  return o;
}

// FP8 x FP4 experts: the weights are E2M1 codes (MXFP4), the activations stay E4M3.
static bool w4(const moe_dims& d) { return d.prec == MOE_PREC_MXFP8_W4; }
// Quantised weights are read by 4-bit tensor loads (FP4) that want 32-byte alignment.
static bool wq_aligned(const moe_dims& d, const void* wq) {
  return (reinterpret_cast<uintptr_t>(wq) & (w4(d) ? 31u : 15u)) == 0;
}

// Quantised weights: W_gu along d ([E*2f][d]), W_gu along 2f ([E][d][2f]),
// W_d along f ([E*d][f]), W_d along d ([E][f][d]); E2M1 codes packed two a byte when
// the weights are FP4.
struct MxWeights {
  MxOp gu_rows, gu_cols, d_rows, d_cols;
};

static MxWeights carve_weights(const moe_dims& d, void* base) {
  uint8_t* p = static_cast<uint8_t*>(base);
  const size_t n = static_cast<size_t>(d.E) * 2 * d.f * d.d;
  const size_t m = static_cast<size_t>(d.E) * d.f * d.d;
  const bool f4 = w4(d);
  MxWeights w;
  w.gu_rows = carve_op(p, n, f4);
  w.gu_cols = carve_op(p, n, f4);
  w.d_rows = carve_op(p, m, f4);
  w.d_cols = carve_op(p, m, f4);
  return w;
}

// Quantised activations of one step, each along the contraction axis of its GEMM; after
// them, the SF tiles of x's and h's column-wise codes again in the replicated form
// (SF_REP_TILE_BYTES a tile) that the CTA-pair weight gradients read for their B operand.
struct MxActs {
  MxOp xp_rows, xp_cols, h_rows, h_cols, dy_rows, dy_cols, dgu_rows, dgu_cols;
  uint8_t* xp_cols_sf_rep;
  uint8_t* h_cols_sf_rep;
};
static size_t sf_rep_bytes(size_t elems) { return a256(elems / 32 * 4); }

static MxActs carve_acts(const moe_dims& d, int64_t R_cap, void* base) {
  uint8_t* p = static_cast<uint8_t*>(base);
  const size_t rd = static_cast<size_t>(R_cap) * d.d, rf = static_cast<size_t>(R_cap) * d.f;
  MxActs a;
  a.xp_rows = carve_op(p, rd);
  a.xp_cols = carve_op(p, rd);
  a.h_rows = carve_op(p, rf);
  a.h_cols = carve_op(p, rf);
  a.dy_rows = carve_op(p, rd);
  a.dy_cols = carve_op(p, rd);
  a.dgu_rows = carve_op(p, 2 * rf);
  a.dgu_cols = carve_op(p, 2 * rf);
  a.xp_cols_sf_rep = p;
  p += sf_rep_bytes(rd);
  a.h_cols_sf_rep = p;
  p += sf_rep_bytes(rf);
  return a;
}

static MxMat mat(const MxOp& o, int64_t inner, int64_t outer, bool fp4 = false) {
  return MxMat{o.codes, o.sf, static_cast<uint64_t>(inner), static_cast<uint64_t>(outer), fp4};
}

static moe_status mx_common(const moe_dims* dims) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->f % 128 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static GemmParams mx_params() {
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.band_krows = BAND_KROWS_E4M3;
  return p;
}

}  // namespace moe

extern "C" {

size_t moe_mx_weights_size(const moe_dims* dims) {
  if (mx_common(dims) != MOE_OK) return 0;
  const size_t n = static_cast<size_t>(dims->E) * 2 * dims->f * dims->d;
  const size_t m = static_cast<size_t>(dims->E) * dims->f * dims->d;
  return 2 * op_bytes(n, w4(*dims)) + 2 * op_bytes(m, w4(*dims));
}

size_t moe_mx_workspace_size(const moe_dims* dims) {
  if (mx_common(dims) != MOE_OK) return 0;
  const size_t R = static_cast<size_t>(moe_row_capacity(dims));
  const size_t rd = R * dims->d, rf = R * dims->f;
  return 4 * op_bytes(rd) + 2 * op_bytes(rf) + 2 * op_bytes(2 * rf) + sf_rep_bytes(rd) + sf_rep_bytes(rf);
}

moe_status moe_mx_quantize_weights(const moe_dims* dims, const moe_bf16* w_gu, const moe_bf16* w_d, void* wq,
                                   void* stream) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!w_gu || !w_d || !wq) return MOE_ERR_INVALID_ARG;
  if (!al16(w_gu) || !al16(w_d) || !wq_aligned(d, wq)) return MOE_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MxWeights w = carve_weights(d, wq);
  // one read of each weight: column-wise codes per expert and row-wise codes of the same tiles
  if (launch_quant_cols_t(w_gu, d.E, 2ll * d.f, d.d, nullptr, w.gu_cols.codes, w.gu_cols.sf, s, nullptr,
                          w.gu_rows.codes, w.gu_rows.sf, w4(d)) != cudaSuccess ||
      launch_quant_cols_t(w_d, d.E, d.d, d.f, nullptr, w.d_cols.codes, w.d_cols.sf, s, nullptr, w.d_rows.codes,
                          w.d_rows.sf, w4(d)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_permute_mx(const moe_dims* dims, const moe_bf16* x, const int32_t* topk_idx, const float* topk_w,
                          const int32_t* split_sizes, const int32_t* row_offsets, const void* workspace,
                          void* mx_ws, int32_t* row_to_token, int32_t* token_to_row, float* w_rows,
                          int32_t* dev_status, void* stream) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!split_sizes || !row_offsets || !mx_ws || !row_to_token || !w_rows || !dev_status) return MOE_ERR_INVALID_ARG;
  if (d.T > 0 && (!x || !topk_idx || !topk_w || !token_to_row)) return MOE_ERR_INVALID_ARG;
  if (!workspace) return MOE_ERR_WORKSPACE;
  if (!al16(x) || !al16(mx_ws)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = moe_row_capacity(dims);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MxActs a = carve_acts(d, R_cap, mx_ws);
  RouteScratch rs = route_scratch(d, const_cast<void*>(workspace));
  // the maps, then one gathered pass over x for the row-wise (gate/up GEMM) and the
  // column-wise (gate/up weight gradient) codes of the permuted rows
  if (launch_route_maps(d.T, d.E, d.k, topk_idx, topk_w, split_sizes, row_offsets, rs, row_to_token, token_to_row,
                        w_rows, static_cast<int>(R_cap), dev_status, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (d.T == 0) return MOE_OK;
  return cuda_st(launch_quant_cols_t(x, 1, R_cap, d.d, row_offsets + d.E, a.xp_cols.codes, a.xp_cols.sf, s,
                                     row_to_token, a.xp_rows.codes, a.xp_rows.sf, false, a.xp_cols_sf_rep));
}

moe_status moe_combine_bwd_mx(const moe_dims* dims, const moe_bf16* dy, const int32_t* row_to_token,
                              const int32_t* split_sizes, const int32_t* row_offsets, void* mx_ws, void* stream) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!split_sizes || !row_offsets || !mx_ws || !row_to_token) return MOE_ERR_INVALID_ARG;
  if (d.T > 0 && !dy) return MOE_ERR_INVALID_ARG;
  if (!al16(dy) || !al16(mx_ws)) return MOE_ERR_ALIGNMENT;
  if (d.T == 0) return MOE_OK;
  const int64_t R_cap = moe_row_capacity(dims);
  MxActs a = carve_acts(d, R_cap, mx_ws);
  // one gathered pass over dY: row-wise codes (down dgrad) and column-wise codes (down wgrad)
  return cuda_st(launch_quant_cols_t(dy, 1, R_cap, d.d, row_offsets + d.E, a.dy_cols.codes, a.dy_cols.sf,
                                     static_cast<cudaStream_t>(stream), row_to_token, a.dy_rows.codes,
                                     a.dy_rows.sf));
}

moe_status moe_gemm_gate_up_mx(const moe_dims* dims, const int32_t* row_offsets, const float* w_rows,
                               const void* wq, void* mx_ws, moe_bf16* gu, int32_t* dev_status, void* stream) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!row_offsets || !w_rows || !wq || !mx_ws || !gu || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!wq_aligned(d, wq) || !al16(mx_ws) || !al16(gu)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = moe_row_capacity(dims), R = static_cast<int64_t>(d.T) * d.k;
  MxWeights w = carve_weights(d, const_cast<void*>(wq));
  MxActs a = carve_acts(d, R_cap, mx_ws);
  MxMat ma = mat(a.xp_rows, d.d, R_cap);
  MxMat mb = mat(w.gu_rows, d.d, 2ll * d.f * d.E, w4(d));
  GemmParams p = mx_params();
  p.BN = 256; p.N = d.f; p.K = d.d; p.E = d.E; p.row_offsets = row_offsets; p.b_rows_per_expert = 2 * d.f;
  p.m_fastest = ORDER_PER_GROUP; p.f = d.f; p.row_limit = R_cap; p.w_rows = w_rows;
  p.gu_out = gu; p.status = dev_status;
  p.a_sf_ktiles = d.d / 128; p.b_sf_ktiles = d.d / 128;
  p.q_rows = a.h_rows.codes; p.q_rows_sf = a.h_rows.sf; p.q_cols = a.h_cols.codes; p.q_cols_sf = a.h_cols.sf;
  p.q_cols_sf_rep = a.h_cols_sf_rep;
  p.q_cols_ld = R_cap; p.q_cols_ktiles = static_cast<int>(R_cap / 128);
  return cuda_st(launch_gemm_mx(GEMM_ROWS_SWIGLU_FWD_MXQ, ma, mb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_down_mx(const moe_dims* dims, const int32_t* row_offsets, const void* wq, void* mx_ws,
                            moe_bf16* y_rows, int32_t* dev_status, void* stream) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!row_offsets || !wq || !mx_ws || !y_rows || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!wq_aligned(d, wq) || !al16(mx_ws) || !al16(y_rows)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = moe_row_capacity(dims), R = static_cast<int64_t>(d.T) * d.k;
  MxWeights w = carve_weights(d, const_cast<void*>(wq));
  MxActs a = carve_acts(d, R_cap, mx_ws);
  const int bn = bn_mx(d.d);
  MxMat ma = mat(a.h_rows, d.f, R_cap);
  MxMat mb = mat(w.d_rows, d.f, static_cast<uint64_t>(d.d) * d.E, w4(d));
  GemmParams p = mx_params();
  p.BN = bn; p.N = d.d; p.K = d.f; p.E = d.E; p.row_offsets = row_offsets; p.b_rows_per_expert = d.d;
  p.m_fastest = ORDER_PER_GROUP; p.out = y_rows; p.ldo = d.d; p.row_limit = R_cap; p.status = dev_status;
  p.a_sf_ktiles = d.f / 128; p.b_sf_ktiles = d.f / 128;
  return cuda_st(launch_gemm_mx(GEMM_ROWS_STORE, ma, mb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_down_dgrad_mx(const moe_dims* dims, const int32_t* row_offsets, const float* w_rows,
                                  const void* wq, void* mx_ws, const moe_bf16* gu, float* dw_rows, void* workspace,
                                  int32_t* dev_status, void* stream) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!row_offsets || !w_rows || !wq || !mx_ws || !gu || !dw_rows || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!workspace) return MOE_ERR_WORKSPACE;
  if (!wq_aligned(d, wq) || !al16(mx_ws) || !al16(gu)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = moe_row_capacity(dims), R = static_cast<int64_t>(d.T) * d.k;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MxWeights w = carve_weights(d, const_cast<void*>(wq));
  MxActs a = carve_acts(d, R_cap, mx_ws);
  float* dw_part = workspace_dw_part(d, workspace);
  const int bn = bn_mx(d.f);
  MxMat ma = mat(a.dy_rows, d.d, R_cap);
  MxMat mb = mat(w.d_cols, d.d, static_cast<uint64_t>(d.f) * d.E, w4(d));
  GemmParams p = mx_params();
  p.BN = bn; p.N = d.f; p.K = d.d; p.E = d.E; p.row_offsets = row_offsets; p.b_rows_per_expert = d.f;
  p.m_fastest = ORDER_PER_GROUP; p.f = d.f; p.row_limit = R_cap; p.w_rows = w_rows; p.gu_in = gu;
  p.dw_part = dw_part; p.dw_stride = d.f / bn; p.status = dev_status;
  p.a_sf_ktiles = d.d / 128; p.b_sf_ktiles = d.d / 128;
  p.q_rows = a.dgu_rows.codes; p.q_rows_sf = a.dgu_rows.sf; p.q_cols = a.dgu_cols.codes;
  p.q_cols_sf = a.dgu_cols.sf; p.q_cols_ld = R_cap; p.q_cols_ktiles = static_cast<int>(R_cap / 128);
  if (launch_gemm_mx(GEMM_ROWS_SWIGLU_BWD_MXQ, ma, mb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_st(launch_dw_reduce(dw_part, d.f / bn, row_offsets, d.E, dw_rows, static_cast<int>(R_cap), s));
}

moe_status moe_gemm_down_wgrad_mx(const moe_dims* dims, const int32_t* row_offsets, void* mx_ws, moe_bf16* dw_d,
                                  int32_t* dev_status, void* stream) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!row_offsets || !mx_ws || !dw_d || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!al16(mx_ws) || !al16(dw_d)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = moe_row_capacity(dims);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MxActs a = carve_acts(d, R_cap, mx_ws);
  const int bn = bn_mx(d.f);
  MxMat ma = mat(a.dy_cols, R_cap, d.d);
  MxMat mb = mat(a.h_cols, R_cap, d.f);
  mb.sf_rep = a.h_cols_sf_rep;
  GemmParams p = mx_params();
  p.BN = bn; p.N = d.f; p.M = d.d; p.E = d.E; p.row_offsets = row_offsets; p.m_fastest = (d.d <= d.f) ? 1 : 0;
  p.out = dw_d; p.ldo = d.f; p.row_limit = d.d; p.status = dev_status;
  p.a_sf_ktiles = static_cast<int>(R_cap / 128);
  p.b_sf_ktiles = static_cast<int>(R_cap / 128);
  return cuda_st(launch_gemm_mx(GEMM_KGROUP_STORE, ma, mb, p, s));
}

moe_status moe_gemm_gate_up_dgrad_mx(const moe_dims* dims, const int32_t* row_offsets, const void* wq,
                                     void* mx_ws, moe_bf16* dxp, int32_t* dev_status, void* stream) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!row_offsets || !wq || !mx_ws || !dxp || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!wq_aligned(d, wq) || !al16(mx_ws) || !al16(dxp)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = moe_row_capacity(dims), R = static_cast<int64_t>(d.T) * d.k;
  MxWeights w = carve_weights(d, const_cast<void*>(wq));
  MxActs a = carve_acts(d, R_cap, mx_ws);
  const int bn = bn_mx(d.d);
  MxMat ma = mat(a.dgu_rows, 2ll * d.f, R_cap);
  MxMat mb = mat(w.gu_cols, 2ll * d.f, static_cast<uint64_t>(d.d) * d.E, w4(d));
  GemmParams p = mx_params();
  p.BN = bn; p.N = d.d; p.K = 2 * d.f; p.E = d.E; p.row_offsets = row_offsets; p.b_rows_per_expert = d.d;
  p.m_fastest = ORDER_PER_GROUP; p.out = dxp; p.ldo = d.d; p.row_limit = R_cap; p.status = dev_status;
  p.a_sf_ktiles = 2 * d.f / 128; p.b_sf_ktiles = 2 * d.f / 128;
  return cuda_st(launch_gemm_mx(GEMM_ROWS_STORE, ma, mb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_gate_up_wgrad_mx(const moe_dims* dims, const int32_t* row_offsets, void* mx_ws,
                                     moe_bf16* dw_gu, int32_t* dev_status, void* stream) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!row_offsets || !mx_ws || !dw_gu || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!al16(mx_ws) || !al16(dw_gu)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = moe_row_capacity(dims);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MxActs a = carve_acts(d, R_cap, mx_ws);
  const int bn = bn_mx(d.d);
  MxMat ma = mat(a.dgu_cols, R_cap, 2ll * d.f);
  MxMat mb = mat(a.xp_cols, R_cap, d.d);
  mb.sf_rep = a.xp_cols_sf_rep;
  GemmParams p = mx_params();
  p.BN = bn; p.N = d.d; p.M = 2 * d.f; p.E = d.E; p.row_offsets = row_offsets;
  p.m_fastest = (2 * d.f <= d.d) ? 1 : 0; p.out = dw_gu; p.ldo = d.d; p.row_limit = 2 * d.f;
  p.status = dev_status;
  p.a_sf_ktiles = static_cast<int>(R_cap / 128);
  p.b_sf_ktiles = static_cast<int>(R_cap / 128);
  return cuda_st(launch_gemm_mx(GEMM_KGROUP_STORE, ma, mb, p, s));
}

// Steps 3-5 and their backward as one call each, MXFP8 operands: the per-GEMM calls above
// in order (the composites of moe_grouped_mlp_fwd / moe_grouped_mlp_bwd).
moe_status moe_grouped_mlp_fwd_mx(const moe_dims* dims, const int32_t* row_offsets, const float* w_rows,
                                  const void* wq, void* mx_ws, moe_bf16* gu, moe_bf16* y_rows, int32_t* dev_status,
                                  void* stream) {
  if (!y_rows) return MOE_ERR_INVALID_ARG;   // checked before anything is enqueued
  if (!al16(y_rows)) return MOE_ERR_ALIGNMENT;
  moe_status st = moe_gemm_gate_up_mx(dims, row_offsets, w_rows, wq, mx_ws, gu, dev_status, stream);
  if (st != MOE_OK) return st;
  return moe_gemm_down_mx(dims, row_offsets, wq, mx_ws, y_rows, dev_status, stream);
}

moe_status moe_grouped_mlp_bwd_mx(const moe_dims* dims, const int32_t* row_offsets, const float* w_rows,
                                  const void* wq, void* mx_ws, const moe_bf16* gu, moe_bf16* dxp, moe_bf16* dw_gu,
                                  moe_bf16* dw_d, float* dw_rows, void* workspace, int32_t* dev_status,
                                  void* stream) {
  if (!dxp || !dw_gu || !dw_d) return MOE_ERR_INVALID_ARG;   // checked before anything is enqueued
  if (!al16(dxp) || !al16(dw_gu) || !al16(dw_d)) return MOE_ERR_ALIGNMENT;
  moe_status st = moe_gemm_down_dgrad_mx(dims, row_offsets, w_rows, wq, mx_ws, gu, dw_rows, workspace, dev_status,
                                         stream);
  if (st != MOE_OK) return st;
  st = moe_gemm_down_wgrad_mx(dims, row_offsets, mx_ws, dw_d, dev_status, stream);
  if (st != MOE_OK) return st;
  st = moe_gemm_gate_up_dgrad_mx(dims, row_offsets, wq, mx_ws, dxp, dev_status, stream);
  if (st != MOE_OK) return st;
  return moe_gemm_gate_up_wgrad_mx(dims, row_offsets, mx_ws, dw_gu, dev_status, stream);
}

}  // extern "C"

// ============================================================================ shared expert

namespace moe {

// Quantised shared-expert weights: W_gu_s along d ([2fs][d]) and along 2fs ([d][2fs]),
// W_d_s along fs ([d][fs]) and along d ([fs][d]).
static MxWeights carve_shared_weights(const moe_dims& d, void* base) {
  uint8_t* p = static_cast<uint8_t*>(base);
  const size_t n = 2ull * d.f_shared * d.d, m = static_cast<size_t>(d.f_shared) * d.d;
  const bool f4 = w4(d);
  MxWeights w;
  w.gu_rows = carve_op(p, n, f4);
  w.gu_cols = carve_op(p, n, f4);
  w.d_rows = carve_op(p, m, f4);
  w.d_cols = carve_op(p, m, f4);
  return w;
}

// Quantised shared-expert activations over the T tokens.
static MxActs carve_shared_acts(const moe_dims& d, void* base) {
  uint8_t* p = static_cast<uint8_t*>(base);
  const size_t td = static_cast<size_t>(d.T) * d.d, tf = static_cast<size_t>(d.T) * d.f_shared;
  MxActs a;
  a.xp_rows = carve_op(p, td);
  a.xp_cols = carve_op(p, td);
  a.h_rows = carve_op(p, tf);
  a.h_cols = carve_op(p, tf);
  a.dy_rows = carve_op(p, td);
  a.dy_cols = carve_op(p, td);
  a.dgu_rows = carve_op(p, 2 * tf);
  a.dgu_cols = carve_op(p, 2 * tf);
  a.xp_cols_sf_rep = p;
  p += sf_rep_bytes(td);
  a.h_cols_sf_rep = p;
  p += sf_rep_bytes(tf);
  return a;
}

static moe_status mx_shared_common(const moe_dims* dims) {
  moe_status st = mx_common(dims);
  if (st != MOE_OK) return st;
  if (dims->f_shared <= 0) return MOE_ERR_INVALID_ARG;
  if (dims->f_shared % 128 != 0 || dims->T % 128 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace moe

extern "C" {

size_t moe_mx_shared_weights_size(const moe_dims* dims) {
  if (mx_shared_common(dims) != MOE_OK) return 0;
  const size_t n = 2ull * dims->f_shared * dims->d, m = static_cast<size_t>(dims->f_shared) * dims->d;
  return 2 * op_bytes(n, w4(*dims)) + 2 * op_bytes(m, w4(*dims));
}

size_t moe_mx_shared_workspace_size(const moe_dims* dims) {
  if (mx_shared_common(dims) != MOE_OK) return 0;
  const size_t td = static_cast<size_t>(dims->T) * dims->d, tf = static_cast<size_t>(dims->T) * dims->f_shared;
  return 4 * op_bytes(td) + 2 * op_bytes(tf) + 2 * op_bytes(2 * tf) + sf_rep_bytes(td) + sf_rep_bytes(tf);
}

moe_status moe_mx_quantize_shared_weights(const moe_dims* dims, const moe_bf16* w_gu_s, const moe_bf16* w_d_s,
                                          void* wq_s, void* stream) {
  moe_status st = mx_shared_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!w_gu_s || !w_d_s || !wq_s) return MOE_ERR_INVALID_ARG;
  if (!al16(w_gu_s) || !al16(w_d_s) || !wq_aligned(d, wq_s)) return MOE_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MxWeights w = carve_shared_weights(d, wq_s);
  const int fs = d.f_shared;
  if (launch_quant_cols_t(w_gu_s, 1, 2ll * fs, d.d, nullptr, w.gu_cols.codes, w.gu_cols.sf, s, nullptr,
                          w.gu_rows.codes, w.gu_rows.sf, w4(d)) != cudaSuccess ||
      launch_quant_cols_t(w_d_s, 1, d.d, fs, nullptr, w.d_cols.codes, w.d_cols.sf, s, nullptr, w.d_rows.codes,
                          w.d_rows.sf, w4(d)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_shared_mlp_fwd_mx(const moe_dims* dims, const moe_bf16* x, const void* wq_s, void* mx_ws_s,
                                 moe_bf16* gu_s, moe_bf16* y_s, int32_t* dev_status, void* stream) {
  moe_status st = mx_shared_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (d.T == 0) return MOE_OK;
  if (!x || !wq_s || !mx_ws_s || !gu_s || !y_s || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !wq_aligned(d, wq_s) || !al16(mx_ws_s) || !al16(gu_s) || !al16(y_s)) return MOE_ERR_ALIGNMENT;
  const int fs = d.f_shared, T = d.T;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MxWeights w = carve_shared_weights(d, const_cast<void*>(wq_s));
  MxActs a = carve_shared_acts(d, mx_ws_s);
  MxMat ma, mb;
  GemmParams p;
  // x along d (gate/up GEMM) and along T (its weight gradient, in the backward pass)
  if (launch_quant_cols_t(x, 1, T, d.d, nullptr, a.xp_cols.codes, a.xp_cols.sf, s, nullptr, a.xp_rows.codes,
                          a.xp_rows.sf, false, a.xp_cols_sf_rep) != cudaSuccess)
    return MOE_ERR_CUDA;
  ma = mat(a.xp_rows, d.d, T);
  mb = mat(w.gu_rows, d.d, 2ll * fs, w4(d));
  p = mx_params();
  p.BN = 256; p.N = fs; p.K = d.d; p.M = T; p.E = 1; p.b_rows_per_expert = 2 * fs;
  p.m_fastest = ORDER_PER_GROUP; p.f = fs;
  p.row_limit = T; p.gu_out = gu_s; p.status = dev_status;
  p.a_sf_ktiles = d.d / 128; p.b_sf_ktiles = d.d / 128;
  p.q_rows = a.h_rows.codes; p.q_rows_sf = a.h_rows.sf; p.q_cols = a.h_cols.codes; p.q_cols_sf = a.h_cols.sf;
  p.q_cols_sf_rep = a.h_cols_sf_rep;
  p.q_cols_ld = T; p.q_cols_ktiles = T / 128;
  if (launch_gemm_mx(GEMM_ROWS_SWIGLU_FWD_MXQ, ma, mb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  const int bn = bn_mx(d.d);
  ma = mat(a.h_rows, fs, T);
  mb = mat(w.d_rows, fs, d.d, w4(d));
  p = mx_params();
  p.BN = bn; p.N = d.d; p.K = fs; p.M = T; p.E = 1; p.b_rows_per_expert = d.d; p.m_fastest = ORDER_PER_GROUP;
  p.out = y_s; p.ldo = d.d; p.row_limit = T; p.status = dev_status;
  p.a_sf_ktiles = fs / 128; p.b_sf_ktiles = fs / 128;
  return cuda_st(launch_gemm_mx(GEMM_ROWS_STORE, ma, mb, p, s));
}

moe_status moe_shared_mlp_bwd_mx(const moe_dims* dims, const void* wq_s, void* mx_ws_s, const moe_bf16* gu_s,
                                 const moe_bf16* dy, moe_bf16* dx_s, moe_bf16* dw_gu_s, moe_bf16* dw_d_s,
                                 int32_t* dev_status, void* stream) {
  moe_status st = mx_shared_common(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const int fs = d.f_shared, T = d.T;
  if (!wq_s || !dw_gu_s || !dw_d_s || !dev_status) return MOE_ERR_INVALID_ARG;
  if (T == 0) {  // no token: the shared weights get zero gradients
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(dw_gu_s, 0, 2ull * fs * d.d * 2, s) != cudaSuccess ||
        cudaMemsetAsync(dw_d_s, 0, static_cast<size_t>(fs) * d.d * 2, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (!mx_ws_s || !gu_s || !dy || !dx_s) return MOE_ERR_INVALID_ARG;
  if (!wq_aligned(d, wq_s) || !al16(mx_ws_s) || !al16(gu_s) || !al16(dy) || !al16(dx_s) || !al16(dw_gu_s) ||
      !al16(dw_d_s))
    return MOE_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MxWeights w = carve_shared_weights(d, const_cast<void*>(wq_s));
  MxActs a = carve_shared_acts(d, mx_ws_s);
  MxMat ma, mb;
  GemmParams p;
  // dH = dy W_d_s, SwiGLU' epilogue (weight 1, no dw) writing quantised dG|dU
  if (launch_quant_cols_t(dy, 1, T, d.d, nullptr, a.dy_cols.codes, a.dy_cols.sf, s, nullptr, a.dy_rows.codes,
                          a.dy_rows.sf) != cudaSuccess)
    return MOE_ERR_CUDA;
  int bn = bn_mx(fs);
  ma = mat(a.dy_rows, d.d, T);
  mb = mat(w.d_cols, d.d, fs, w4(d));
  p = mx_params();
  p.BN = bn; p.N = fs; p.K = d.d; p.M = T; p.E = 1; p.b_rows_per_expert = fs; p.m_fastest = ORDER_PER_GROUP; p.f = fs;
  p.row_limit = T; p.gu_in = gu_s; p.status = dev_status;
  p.a_sf_ktiles = d.d / 128; p.b_sf_ktiles = d.d / 128;
  p.q_rows = a.dgu_rows.codes; p.q_rows_sf = a.dgu_rows.sf; p.q_cols = a.dgu_cols.codes;
  p.q_cols_sf = a.dgu_cols.sf; p.q_cols_ld = T; p.q_cols_ktiles = T / 128;
  if (launch_gemm_mx(GEMM_ROWS_SWIGLU_BWD_MXQ, ma, mb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  // dW_d_s = dy^T h_s (K = T): dy column codes, h_s column codes from the forward
  ma = mat(a.dy_cols, T, d.d);
  mb = mat(a.h_cols, T, fs);
  mb.sf_rep = a.h_cols_sf_rep;
  p = mx_params();
  p.BN = bn; p.N = fs; p.M = d.d; p.K = T; p.E = 1; p.m_fastest = (d.d <= fs) ? 1 : 0;
  p.out = dw_d_s; p.ldo = fs; p.row_limit = d.d; p.status = dev_status;
  p.a_sf_ktiles = T / 128; p.b_sf_ktiles = T / 128;
  if (launch_gemm_mx(GEMM_KGROUP_STORE, ma, mb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  // dx_s = dgu_s W_gu_s (K = 2fs)
  bn = bn_mx(d.d);
  ma = mat(a.dgu_rows, 2ll * fs, T);
  mb = mat(w.gu_cols, 2ll * fs, d.d, w4(d));
  p = mx_params();
  p.BN = bn; p.N = d.d; p.K = 2 * fs; p.M = T; p.E = 1; p.b_rows_per_expert = d.d; p.m_fastest = ORDER_PER_GROUP;
  p.out = dx_s; p.ldo = d.d; p.row_limit = T; p.status = dev_status;
  p.a_sf_ktiles = 2 * fs / 128; p.b_sf_ktiles = 2 * fs / 128;
  if (launch_gemm_mx(GEMM_ROWS_STORE, ma, mb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  // dW_gu_s = dgu_s^T x (K = T)
  ma = mat(a.dgu_cols, T, 2ll * fs);
  mb = mat(a.xp_cols, T, d.d);
  mb.sf_rep = a.xp_cols_sf_rep;
  p = mx_params();
  p.BN = bn; p.N = d.d; p.M = 2 * fs; p.K = T; p.E = 1; p.m_fastest = (2 * fs <= d.d) ? 1 : 0;
  p.out = dw_gu_s; p.ldo = d.d; p.row_limit = 2 * fs; p.status = dev_status;
  p.a_sf_ktiles = T / 128; p.b_sf_ktiles = T / 128;
  return cuda_st(launch_gemm_mx(GEMM_KGROUP_STORE, ma, mb, p, s));
}

}  // extern "C"
