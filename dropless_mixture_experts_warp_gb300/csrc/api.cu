// C-ABI entry points of libmoe.so: argument checks, workspace carving, TMA tensor
// maps, kernel launches.  No entry point allocates device memory or synchronises,
// except moe_check_status.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "kernels.h"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

int pair_grid(const void* kern, int threads, int smem_bytes) {
  const int all = num_sms() & ~1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(all), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    return all;
  }
  return 2 * n < all ? 2 * n : all;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor [outer][inner] row-major, box [box_outer][box_inner], 128B swizzle,
// zero fill outside the tensor.
static bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint8 tensor (E4M3 codes) [outer][inner], 128B swizzle, zero fill.
bool make_tensor_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed E2M1 codes [outer][inner / 2] bytes (inner in elements): every 16 codes (8 bytes)
// land in 16 bytes of shared memory, so a 128-element row of the box fills 128 bytes laid
// out as an E4M3 row; 128B swizzle, box 128 elements x box_outer rows.
bool make_tensor_map_fp4(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner / 2};
  cuuint32_t box[2] = {128, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// SF tiles viewed as [bytes / 256][256] bytes, box of two rows: one 512-byte tile per load
// (the MXFP8 pair kernel fetches scale tiles by tensor loads so that both CTAs' bytes
// count on the leader's barrier).
bool make_tensor_map_sf(CUtensorMap* m, const void* base, uint64_t bytes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || bytes % (256 * box_rows) != 0 || bytes == 0) return false;
  cuuint64_t dims[2] = {256, bytes / 256};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same encoder, for the other translation units of the library.
bool make_tensor_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                          uint32_t box_inner, uint32_t box_outer) {
  return make_map(m, base, inner, outer, box_inner, box_outer);
}

// 2-D bf16 output [rows][ld] (cols <= ld used) for the tensor store of the GEMM
// epilogue: box 32 x 32, 64-byte swizzle; rows beyond `rows` are not written.
bool make_tensor_map_store(CUtensorMap* m, const void* base, uint64_t cols, uint64_t ld, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int64_t row_capacity(const moe_dims& d) {
  const int64_t R = static_cast<int64_t>(d.T) * d.k;
  return (R + ROW_ALIGN - 1) / ROW_ALIGN * ROW_ALIGN + static_cast<int64_t>(ROW_ALIGN) * d.E;
}

struct Carve {
  RouteScratch route;
  float* dw_part;
};

static size_t route_scratch_bytes(const moe_dims& d) {
  const size_t nb = route_blocks(d.T);
  return align256(sizeof(int32_t)) + 2 * align256(nb * d.E * sizeof(int32_t)) +
         align256(static_cast<size_t>(d.T) * d.k * sizeof(int32_t));
}

static int bn_for(int n) { return n % 256 == 0 ? 256 : (n % 128 == 0 ? 128 : 64); }

static size_t dw_part_bytes(const moe_dims& d) {
  return align256(static_cast<size_t>(row_capacity(d)) * (d.f / 64) * sizeof(float));
}

static Carve carve(const moe_dims& d, void* ws) {
  Carve c;
  uint8_t* p = static_cast<uint8_t*>(ws);
  const size_t nb = route_blocks(d.T);
  c.route.counter = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t));
  c.route.block_hist = reinterpret_cast<int32_t*>(p);
  p += align256(nb * d.E * sizeof(int32_t));
  c.route.block_base = reinterpret_cast<int32_t*>(p);
  p += align256(nb * d.E * sizeof(int32_t));
  c.route.local_rank = reinterpret_cast<int32_t*>(p);
  p += align256(static_cast<size_t>(d.T) * d.k * sizeof(int32_t));
  c.dw_part = reinterpret_cast<float*>(p);
  return c;
}

RouteScratch route_scratch(const moe_dims& d, void* ws) { return carve(d, ws).route; }

// The dw-partials region of a caller workspace (shared by the bf16 and MXFP8 calls).
float* workspace_dw_part(const moe_dims& d, void* ws) { return carve(d, ws).dw_part; }

static moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// The CTA-pair kernel serves every product whose tile is at least 128 columns wide
// (and, for the weight gradients, whose output rows come in 256-row pairs).
static bool pair_ok(GemmKind kind, const GemmParams& p) {
  if (p.BN < 128) return false;
  if (kind == GEMM_KGROUP_STORE && p.M % 256 != 0) return false;
  return true;
}

cudaError_t launch_best(GemmKind kind, bool bwd, const CUtensorMap& a, const CUtensorMap& b,
                        const GemmParams& p, cudaStream_t s) {
  if (pair_ok(kind, p)) return launch_gemm_pair(kind, a, b, p, s);
  return bwd ? launch_gemm_bwd(kind, a, b, p, s) : launch_gemm_fwd(kind, a, b, p, s);
}

static GemmParams gemm_params() {
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.band_krows = BAND_KROWS_BF16;
  return p;
}

}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_abi_version(void) { return 1; }

const char* moe_status_string(int32_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or option";
    case MOE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace missing";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_INVARIANT: return "routing counts do not sum to T*k";
    case MOE_ERR_SCRATCH_LIMIT: return "problem too large for the static scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

moe_status moe_check_dims(const moe_dims* dims) {
  if (!dims) return MOE_ERR_INVALID_ARG;
  const moe_dims& d = *dims;
  if (d.T < 0 || d.d <= 0 || d.f <= 0 || d.E <= 0 || d.k <= 0 || d.f_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (d.k > d.E || d.k > 32) return MOE_ERR_INVALID_ARG;
  if (d.score != MOE_SCORE_SOFTMAX && d.score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (d.prec != MOE_PREC_BF16 && d.prec != MOE_PREC_MXFP8 && d.prec != MOE_PREC_MXFP8_W4) return MOE_ERR_INVALID_ARG;
  if (d.prec != MOE_PREC_BF16 && (d.f % 128 != 0 || d.f_shared % 128 != 0)) return MOE_ERR_UNSUPPORTED;
  if (d.E > MAX_EXPERTS) return MOE_ERR_UNSUPPORTED;
  if (d.d % 128 != 0 || d.f % 64 != 0 || d.f_shared % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (row_capacity(d) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int64_t moe_row_capacity(const moe_dims* dims) {
  if (moe_check_dims(dims) != MOE_OK) return -1;
  return row_capacity(*dims);
}

size_t moe_workspace_size(const moe_dims* dims) {
  if (moe_check_dims(dims) != MOE_OK) return 0;
  return route_scratch_bytes(*dims) + dw_part_bytes(*dims);
}

uint64_t moe_launch_count(void) { return g_launches.load(); }

moe_status moe_route_topk(const moe_dims* dims, const float* logits, int32_t* topk_idx,
                          float* topk_w, int32_t* split_sizes, int32_t* offsets,
                          int32_t* row_offsets, void* workspace, int32_t* dev_status,
                          void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!split_sizes || !offsets || !row_offsets || !dev_status) return MOE_ERR_INVALID_ARG;
  if (d.T > 0 && (!logits || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (!workspace) return MOE_ERR_WORKSPACE;
  Carve c = carve(d, workspace);
  return cuda_status(launch_route_topk(logits, d.T, d.E, d.k, d.score, topk_idx, topk_w, split_sizes,
                                       offsets, row_offsets, c.route, dev_status,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_route_topk_grouped(const moe_dims* dims, const float* logits, const float* bias, int32_t n_group,
                                  int32_t topk_group, float routed_scale, int32_t* topk_idx, float* topk_w,
                                  int32_t* split_sizes, int32_t* offsets, int32_t* row_offsets, void* workspace,
                                  int32_t* dev_status, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (d.score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (n_group < 1 || n_group > 32 || d.E % n_group != 0 || d.E / n_group < 2) return MOE_ERR_INVALID_ARG;
  if (topk_group < 1 || topk_group > n_group || d.k > topk_group * (d.E / n_group)) return MOE_ERR_INVALID_ARG;
  if (!(routed_scale > 0.0f)) return MOE_ERR_INVALID_ARG;
  if (!split_sizes || !offsets || !row_offsets || !dev_status) return MOE_ERR_INVALID_ARG;
  if (d.T > 0 && (!logits || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (!workspace) return MOE_ERR_WORKSPACE;
  Carve c = carve(d, workspace);
  const GroupedRoute gr{bias, n_group, topk_group, routed_scale};
  return cuda_status(launch_route_topk(logits, d.T, d.E, d.k, d.score, topk_idx, topk_w, split_sizes, offsets,
                                       row_offsets, c.route, dev_status, static_cast<cudaStream_t>(stream), &gr));
}

moe_status moe_permute(const moe_dims* dims, const moe_bf16* x, const int32_t* topk_idx,
                       const float* topk_w, const int32_t* split_sizes,
                       const int32_t* row_offsets, const void* workspace, moe_bf16* xp,
                       int32_t* row_to_token, int32_t* token_to_row, float* w_rows,
                       int32_t* dev_status, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!split_sizes || !row_offsets || !xp || !row_to_token || !w_rows || !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (d.T > 0 && (!x || !topk_idx || !topk_w || !token_to_row)) return MOE_ERR_INVALID_ARG;
  if (!workspace) return MOE_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(xp)) return MOE_ERR_ALIGNMENT;
  Carve c = carve(d, const_cast<void*>(workspace));
  return cuda_status(launch_permute(x, d.T, d.d, d.E, d.k, topk_idx, topk_w, split_sizes, row_offsets,
                                    c.route, xp, row_to_token, token_to_row, w_rows,
                                    static_cast<int>(row_capacity(d)), dev_status,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_gate_up(const moe_dims* dims, const moe_bf16* xp,
                            const int32_t* row_offsets, const float* w_rows,
                            const moe_bf16* w_gu, moe_bf16* gu, moe_bf16* h,
                            int32_t* dev_status, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!xp || !row_offsets || !w_rows || !w_gu || !gu || !h || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xp) || !aligned16(w_gu) || !aligned16(gu) || !aligned16(h)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = row_capacity(d);
  const int64_t R = static_cast<int64_t>(d.T) * d.k;
  const int bn = (d.f % 128 == 0) ? 256 : 128;  // gate half + up half
  CUtensorMap ta, tb;
  if (!make_map(&ta, xp, d.d, R_cap, 64, BM) || !make_map(&tb, w_gu, d.d, 2ll * d.f * d.E, 64, bn / 2))
    return MOE_ERR_CUDA;
  GemmParams p = gemm_params();
  p.BN = bn; p.N = d.f; p.K = d.d; p.E = d.E; p.row_offsets = row_offsets;
  p.b_rows_per_expert = 2 * d.f; p.m_fastest = ORDER_PER_GROUP; p.f = d.f;
  p.row_limit = R_cap; p.w_rows = w_rows; p.gu_out = gu; p.h_out = h; p.status = dev_status;
  return cuda_status(launch_best(GEMM_ROWS_SWIGLU_FWD, false, ta, tb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_down(const moe_dims* dims, const moe_bf16* h, const int32_t* row_offsets,
                         const moe_bf16* w_d, moe_bf16* y_rows, int32_t* dev_status, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!h || !row_offsets || !w_d || !y_rows || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w_d) || !aligned16(y_rows)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = row_capacity(d);
  const int64_t R = static_cast<int64_t>(d.T) * d.k;
  const int bn = bn_for(d.d) == 64 ? 128 : bn_for(d.d);
  CUtensorMap ta, tb;
  if (!make_map(&ta, h, d.f, R_cap, 64, BM) ||
      !make_map(&tb, w_d, d.f, static_cast<uint64_t>(d.d) * d.E, 64, bn / 2))   // CTA-pair boxes
    return MOE_ERR_CUDA;
  GemmParams p = gemm_params();
  p.BN = bn; p.N = d.d; p.K = d.f; p.E = d.E; p.row_offsets = row_offsets;
  p.b_rows_per_expert = d.d; p.m_fastest = ORDER_PER_GROUP;
  p.out = y_rows; p.ldo = d.d; p.row_limit = R_cap; p.status = dev_status;
  return cuda_status(launch_gemm_pair(GEMM_ROWS_STORE, ta, tb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_mlp_fwd(const moe_dims* dims, const moe_bf16* xp,
                               const int32_t* row_offsets, const float* w_rows,
                               const moe_bf16* w_gu, const moe_bf16* w_d, moe_bf16* gu,
                               moe_bf16* h, moe_bf16* y_rows, int32_t* dev_status,
                               void* stream) {
  moe_status st = moe_gemm_gate_up(dims, xp, row_offsets, w_rows, w_gu, gu, h, dev_status, stream);
  if (st != MOE_OK) return st;
  return moe_gemm_down(dims, h, row_offsets, w_d, y_rows, dev_status, stream);
}

moe_status moe_combine_fwd(const moe_dims* dims, const moe_bf16* rows,
                           const int32_t* token_to_row, const moe_bf16* shared,
                           moe_bf16* out, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (d.T > 0 && (!rows || !token_to_row || !out)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(rows) || !aligned16(shared) || !aligned16(out)) return MOE_ERR_ALIGNMENT;
  return cuda_status(launch_combine(rows, d.T, d.d, d.k, token_to_row, shared, out,
                                    static_cast<int>(row_capacity(d)),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_bwd(const moe_dims* dims, const moe_bf16* dy,
                           const int32_t* token_to_row, const int32_t* split_sizes,
                           const int32_t* row_offsets, moe_bf16* dy_rows, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!split_sizes || !row_offsets || !dy_rows) return MOE_ERR_INVALID_ARG;
  if (d.T > 0 && (!dy || !token_to_row)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(dy_rows)) return MOE_ERR_ALIGNMENT;
  return cuda_status(launch_combine_bwd(dy, d.T, d.d, d.E, d.k, token_to_row, split_sizes, row_offsets,
                                        dy_rows, static_cast<int>(row_capacity(d)),
                                        static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_down_dgrad(const moe_dims* dims, const moe_bf16* dy_rows,
                               const int32_t* row_offsets, const float* w_rows,
                               const moe_bf16* w_d, const moe_bf16* gu, moe_bf16* dgu,
                               float* dw_rows, void* workspace, int32_t* dev_status,
                               void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!dy_rows || !row_offsets || !w_rows || !w_d || !gu || !dgu || !dw_rows || !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (!workspace) return MOE_ERR_WORKSPACE;
  if (!aligned16(dy_rows) || !aligned16(w_d) || !aligned16(gu) || !aligned16(dgu))
    return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = row_capacity(d);
  const int64_t R = static_cast<int64_t>(d.T) * d.k;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Carve c = carve(d, workspace);
  const int bn = bn_for(d.f);
  // dH = dy_rows W_d[e]: B = W_d[e] stored [K=d][N=f], an MN-major operand
  CUtensorMap ta, tb;
  if (!make_map(&ta, dy_rows, d.d, R_cap, 64, BM) ||
      !make_map(&tb, w_d, d.f, static_cast<uint64_t>(d.d) * d.E, 64, 64))
    return MOE_ERR_CUDA;
  GemmParams p = gemm_params();
  p.BN = bn; p.N = d.f; p.K = d.d; p.E = d.E; p.row_offsets = row_offsets;
  p.b_k_per_expert = d.d; p.m_fastest = ORDER_PER_GROUP; p.f = d.f;
  p.row_limit = R_cap; p.w_rows = w_rows; p.gu_in = gu; p.dgu_out = dgu; p.dw_part = c.dw_part;
  p.dw_stride = d.f / bn; p.status = dev_status;
  if (launch_best(GEMM_ROWS_SWIGLU_BWD, true, ta, tb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_dw_reduce(c.dw_part, d.f / bn, row_offsets, d.E, dw_rows,
                                      static_cast<int>(R_cap), s));
}

moe_status moe_gemm_down_wgrad(const moe_dims* dims, const moe_bf16* dy_rows, const moe_bf16* h,
                               const int32_t* row_offsets, moe_bf16* dw_d, int32_t* dev_status,
                               void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!dy_rows || !h || !row_offsets || !dw_d || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy_rows) || !aligned16(h) || !aligned16(dw_d)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = row_capacity(d);
  // dW_d[e] = dy_rows_e^T h_e: [d, f], contraction over the rows of e
  CUtensorMap ta, tb;
  if (!make_map(&ta, dy_rows, d.d, R_cap, 64, 64) || !make_map(&tb, h, d.f, R_cap, 64, 64))
    return MOE_ERR_CUDA;
  GemmParams p = gemm_params();
  p.BN = bn_for(d.f); p.N = d.f; p.M = d.d; p.E = d.E; p.row_offsets = row_offsets;
  p.m_fastest = (d.d <= d.f) ? 1 : 0; p.out = dw_d; p.ldo = d.f; p.row_limit = d.d;
  p.status = dev_status;
  return cuda_status(launch_best(GEMM_KGROUP_STORE, true, ta, tb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_gate_up_dgrad(const moe_dims* dims, const moe_bf16* dgu,
                                  const int32_t* row_offsets, const moe_bf16* w_gu, moe_bf16* dxp,
                                  int32_t* dev_status, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!dgu || !row_offsets || !w_gu || !dxp || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dgu) || !aligned16(w_gu) || !aligned16(dxp)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = row_capacity(d);
  const int64_t R = static_cast<int64_t>(d.T) * d.k;
  const int bn = bn_for(d.d) == 64 ? 128 : bn_for(d.d);
  // dxp = dgu W_gu[e]: B = W_gu[e] stored [K=2f][N=d], an MN-major operand
  CUtensorMap ta, tb;
  if (!make_map(&ta, dgu, 2ll * d.f, R_cap, 64, BM) || !make_map(&tb, w_gu, d.d, 2ll * d.f * d.E, 64, 64))
    return MOE_ERR_CUDA;
  GemmParams p = gemm_params();
  p.BN = bn; p.N = d.d; p.K = 2 * d.f; p.E = d.E; p.row_offsets = row_offsets;
  p.b_k_per_expert = 2 * d.f; p.m_fastest = ORDER_PER_GROUP;
  p.out = dxp; p.ldo = d.d; p.row_limit = R_cap; p.status = dev_status;
  return cuda_status(launch_best(GEMM_ROWS_STORE_BMN, true, ta, tb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_gate_up_wgrad(const moe_dims* dims, const moe_bf16* dgu, const moe_bf16* xp,
                                  const int32_t* row_offsets, moe_bf16* dw_gu, int32_t* dev_status,
                                  void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!dgu || !xp || !row_offsets || !dw_gu || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dgu) || !aligned16(xp) || !aligned16(dw_gu)) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = row_capacity(d);
  // dW_gu[e] = dgu_e^T xp_e: [2f, d], contraction over the rows of e
  CUtensorMap ta, tb;
  if (!make_map(&ta, dgu, 2ll * d.f, R_cap, 64, 64) || !make_map(&tb, xp, d.d, R_cap, 64, 64))
    return MOE_ERR_CUDA;
  GemmParams p = gemm_params();
  p.BN = bn_for(d.d) == 64 ? 128 : bn_for(d.d); p.N = d.d; p.M = 2 * d.f; p.E = d.E;
  p.row_offsets = row_offsets; p.m_fastest = (2 * d.f <= d.d) ? 1 : 0; p.out = dw_gu; p.ldo = d.d;
  p.row_limit = 2 * d.f; p.status = dev_status;
  return cuda_status(launch_best(GEMM_KGROUP_STORE, true, ta, tb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_mlp_bwd(const moe_dims* dims, const moe_bf16* xp,
                               const int32_t* row_offsets, const float* w_rows,
                               const moe_bf16* w_gu, const moe_bf16* w_d,
                               const moe_bf16* gu, const moe_bf16* h,
                               const moe_bf16* dy_rows, moe_bf16* dgu, moe_bf16* dxp,
                               moe_bf16* dw_gu, moe_bf16* dw_d, float* dw_rows,
                               void* workspace, int32_t* dev_status, void* stream) {
  if (!xp || !h || !w_gu || !dxp || !dw_gu || !dw_d) return MOE_ERR_INVALID_ARG;
  moe_status st = moe_gemm_down_dgrad(dims, dy_rows, row_offsets, w_rows, w_d, gu, dgu, dw_rows,
                                      workspace, dev_status, stream);
  if (st != MOE_OK) return st;
  if ((st = moe_gemm_down_wgrad(dims, dy_rows, h, row_offsets, dw_d, dev_status, stream)) != MOE_OK)
    return st;
  if ((st = moe_gemm_gate_up_dgrad(dims, dgu, row_offsets, w_gu, dxp, dev_status, stream)) != MOE_OK)
    return st;
  return moe_gemm_gate_up_wgrad(dims, dgu, xp, row_offsets, dw_gu, dev_status, stream);
}

moe_status moe_shared_mlp_fwd(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_gu_s,
                              const moe_bf16* w_d_s, moe_bf16* gu_s, moe_bf16* h_s, moe_bf16* y_s,
                              int32_t* dev_status, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (d.f_shared <= 0) return MOE_ERR_INVALID_ARG;
  if (d.T == 0) return MOE_OK;
  if (!x || !w_gu_s || !w_d_s || !gu_s || !h_s || !y_s || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gu_s) || !aligned16(w_d_s) || !aligned16(gu_s) || !aligned16(h_s) ||
      !aligned16(y_s))
    return MOE_ERR_ALIGNMENT;
  const int fs = d.f_shared;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap ta, tb;
  // gate/up over all T tokens (one dense group), SwiGLU epilogue with weight 1
  const int bn1 = (fs % 128 == 0) ? 256 : 128;
  if (!make_map(&ta, x, d.d, d.T, 64, BM) || !make_map(&tb, w_gu_s, d.d, 2ll * fs, 64, bn1 / 2))
    return MOE_ERR_CUDA;
  GemmParams p = gemm_params();
  p.BN = bn1; p.N = fs; p.K = d.d; p.M = d.T; p.E = 1; p.b_rows_per_expert = 2 * fs; p.m_fastest = ORDER_PER_GROUP;
  p.f = fs; p.row_limit = d.T; p.gu_out = gu_s; p.h_out = h_s; p.status = dev_status;
  if (launch_best(GEMM_ROWS_SWIGLU_FWD, false, ta, tb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  // down
  const int bn2 = bn_for(d.d) == 64 ? 128 : bn_for(d.d);
  if (!make_map(&ta, h_s, fs, d.T, 64, BM) || !make_map(&tb, w_d_s, fs, d.d, 64, bn2 / 2)) return MOE_ERR_CUDA;
  p = gemm_params();
  p.BN = bn2; p.N = d.d; p.K = fs; p.M = d.T; p.E = 1; p.b_rows_per_expert = d.d; p.m_fastest = ORDER_PER_GROUP;
  p.out = y_s; p.ldo = d.d; p.row_limit = d.T; p.status = dev_status;
  return cuda_status(launch_gemm_pair(GEMM_ROWS_STORE, ta, tb, p, s));
}

moe_status moe_shared_mlp_bwd(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_gu_s,
                              const moe_bf16* w_d_s, const moe_bf16* gu_s, const moe_bf16* h_s,
                              const moe_bf16* dy, moe_bf16* dgu_s, moe_bf16* dx_s,
                              moe_bf16* dw_gu_s, moe_bf16* dw_d_s, int32_t* dev_status,
                              void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (d.f_shared <= 0) return MOE_ERR_INVALID_ARG;
  if (!w_gu_s || !w_d_s || !dw_gu_s || !dw_d_s || !dev_status) return MOE_ERR_INVALID_ARG;
  if (d.T > 0 && (!x || !gu_s || !h_s || !dy || !dgu_s || !dx_s)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gu_s) || !aligned16(w_d_s) || !aligned16(gu_s) || !aligned16(h_s) ||
      !aligned16(dy) || !aligned16(dgu_s) || !aligned16(dx_s) || !aligned16(dw_gu_s) || !aligned16(dw_d_s))
    return MOE_ERR_ALIGNMENT;
  const int fs = d.f_shared;
  const int T = d.T;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap ta, tb;
  GemmParams p;
  // With T = 0 only the (zero) weight gradients remain; their maps then point at a
  // weight tensor (never read: the contraction is empty) because a map needs a
  // non-empty tensor.
  const uint64_t rows = T > 0 ? static_cast<uint64_t>(T) : 1;
  const moe_bf16* dy_ = T > 0 ? dy : w_d_s;
  const moe_bf16* h_ = T > 0 ? h_s : w_d_s;
  const moe_bf16* x_ = T > 0 ? x : w_gu_s;
  const moe_bf16* dgu_ = T > 0 ? dgu_s : w_gu_s;
  if (T > 0) {
    // dH = dy W_d_s (MN-major B) with the SwiGLU' epilogue, weight 1, no dw
    if (!make_map(&ta, dy, d.d, T, 64, BM) || !make_map(&tb, w_d_s, fs, d.d, 64, 64)) return MOE_ERR_CUDA;
    p = gemm_params();
    p.BN = bn_for(fs); p.N = fs; p.K = d.d; p.M = T; p.E = 1; p.b_k_per_expert = d.d; p.m_fastest = ORDER_PER_GROUP;
    p.f = fs; p.row_limit = T; p.gu_in = gu_s; p.dgu_out = dgu_s; p.status = dev_status;
    if (launch_best(GEMM_ROWS_SWIGLU_BWD, true, ta, tb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  // dW_d_s = dy^T h_s  ([d, fs], K = T tokens)
  if (!make_map(&ta, dy_, d.d, rows, 64, 64) || !make_map(&tb, h_, fs, rows, 64, 64)) return MOE_ERR_CUDA;
  p = gemm_params();
  p.BN = bn_for(fs); p.N = fs; p.M = d.d; p.K = T; p.E = 1; p.m_fastest = (d.d <= fs) ? 1 : 0;
  p.out = dw_d_s; p.ldo = fs; p.row_limit = d.d; p.status = dev_status;
  if (launch_best(GEMM_KGROUP_STORE, true, ta, tb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (T > 0) {
    // dx_s = dgu_s W_gu_s (MN-major B)
    const int bnd = bn_for(d.d) == 64 ? 128 : bn_for(d.d);
    if (!make_map(&ta, dgu_s, 2ll * fs, T, 64, BM) || !make_map(&tb, w_gu_s, d.d, 2ll * fs, 64, 64))
      return MOE_ERR_CUDA;
    p = gemm_params();
    p.BN = bnd; p.N = d.d; p.K = 2 * fs; p.M = T; p.E = 1; p.b_k_per_expert = 2 * fs; p.m_fastest = ORDER_PER_GROUP;
    p.out = dx_s; p.ldo = d.d; p.row_limit = T; p.status = dev_status;
    if (launch_best(GEMM_ROWS_STORE_BMN, true, ta, tb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  // dW_gu_s = dgu_s^T x  ([2fs, d], K = T tokens)
  if (!make_map(&ta, dgu_, 2ll * fs, rows, 64, 64) || !make_map(&tb, x_, d.d, rows, 64, 64))
    return MOE_ERR_CUDA;
  p = gemm_params();
  p.BN = bn_for(d.d) == 64 ? 128 : bn_for(d.d); p.N = d.d; p.M = 2 * fs; p.K = T; p.E = 1;
  p.m_fastest = (2 * fs <= d.d) ? 1 : 0; p.out = dw_gu_s; p.ldo = d.d; p.row_limit = 2 * fs;
  p.status = dev_status;
  return cuda_status(launch_best(GEMM_KGROUP_STORE, true, ta, tb, p, s));
}

moe_status moe_route_topk_bwd(const moe_dims* dims, const float* logits,
                              const int32_t* topk_idx, const float* topk_w,
                              const float* dw_rows, const int32_t* token_to_row,
                              float* d_logits, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (d.T > 0 && (!logits || !topk_idx || !topk_w || !dw_rows || !token_to_row || !d_logits))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_route_bwd(logits, d.T, d.E, d.k, d.score, topk_idx, topk_w, dw_rows,
                                      token_to_row, d_logits, static_cast<int>(row_capacity(d)),
                                      static_cast<cudaStream_t>(stream)));
}

moe_status moe_route_topk_bwd_scaled(const moe_dims* dims, const float* logits, const int32_t* topk_idx,
                                     const float* topk_w, float routed_scale, const float* dw_rows,
                                     const int32_t* token_to_row, float* d_logits, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (d.score != MOE_SCORE_SIGMOID || !(routed_scale > 0.0f)) return MOE_ERR_INVALID_ARG;
  if (d.T > 0 && (!logits || !topk_idx || !topk_w || !dw_rows || !token_to_row || !d_logits))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_route_bwd(logits, d.T, d.E, d.k, d.score, topk_idx, topk_w, dw_rows, token_to_row,
                                      d_logits, static_cast<int>(row_capacity(d)),
                                      static_cast<cudaStream_t>(stream), routed_scale));
}

moe_status moe_check_status(const int32_t* dev_status, void* stream) {
  if (!dev_status) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return static_cast<moe_status>(v);
}

moe_status moe_gemm_bf16_pair(const moe_bf16* A, const moe_bf16* B, moe_bf16* C, int32_t M, int32_t N,
                              int32_t K, int32_t a_layout, int32_t b_layout, int32_t* dev_status, void* stream) {
  if (!A || !B || !C || !dev_status) return MOE_ERR_INVALID_ARG;
  if (M < 1 || N < 128 || K < 64 || N % 128 || K % 64) return MOE_ERR_UNSUPPORTED;
  if ((a_layout != 0 && a_layout != 1) || (b_layout != 0 && b_layout != 1)) return MOE_ERR_INVALID_ARG;
  if (a_layout == 1 && M % 8) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return MOE_ERR_ALIGNMENT;
  const int bn = N % 256 == 0 ? 256 : 128;
  CUtensorMap ta, tb;
  bool ok = a_layout == 0 ? make_map(&ta, A, K, M, 64, BM) : make_map(&ta, A, M, K, 64, 64);
  ok = ok && (b_layout == 0 ? make_map(&tb, B, K, N, 64, bn / 2) : make_map(&tb, B, N, K, 64, 64));
  if (!ok) return MOE_ERR_CUDA;
  GemmParams p = gemm_params();
  p.BN = bn; p.N = N; p.K = K; p.M = M; p.E = 1; p.row_offsets = nullptr;
  p.m_fastest = 1; p.out = C; p.ldo = N; p.row_limit = M; p.status = dev_status;
  GemmKind kind = a_layout == 0 ? (b_layout == 0 ? GEMM_ROWS_STORE : GEMM_ROWS_STORE_BMN)
                                : (b_layout == 0 ? GEMM_DENSE_AMN_BK : GEMM_DENSE_AMN_BMN);
  return cuda_status(launch_gemm_pair(kind, ta, tb, p, static_cast<cudaStream_t>(stream)));
}

moe_status moe_test_wait_timeout(int32_t* dev_status, int64_t limit_cycles, void* stream) {
  if (!dev_status || limit_cycles < 1 || limit_cycles > (1ll << 32)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_wait_timeout(dev_status, limit_cycles, static_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_bf16(const moe_bf16* A, const moe_bf16* B, moe_bf16* C, int32_t M,
                         int32_t N, int32_t K, int32_t a_layout, int32_t b_layout,
                         int32_t* dev_status, void* stream) {
  if (!A || !B || !C || !dev_status) return MOE_ERR_INVALID_ARG;
  if (M < 1 || N < 64 || K < 64 || N % 64 || K % 64) return MOE_ERR_UNSUPPORTED;
  if ((a_layout != 0 && a_layout != 1) || (b_layout != 0 && b_layout != 1)) return MOE_ERR_INVALID_ARG;
  if (a_layout == 1 && M % 8) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return MOE_ERR_ALIGNMENT;
  const int bn = bn_for(N);
  CUtensorMap ta, tb;
  bool ok = a_layout == 0 ? make_map(&ta, A, K, M, 64, BM) : make_map(&ta, A, M, K, 64, 64);
  ok = ok && (b_layout == 0 ? make_map(&tb, B, K, N, 64, bn) : make_map(&tb, B, N, K, 64, 64));
  if (!ok) return MOE_ERR_CUDA;
  GemmParams p = gemm_params();
  p.BN = bn; p.N = N; p.K = K; p.M = M; p.E = 1; p.row_offsets = nullptr;
  p.m_fastest = 1; p.out = C; p.ldo = N; p.row_limit = M; p.status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaSuccess;
  if (a_layout == 0 && b_layout == 0) err = launch_gemm_fwd(GEMM_ROWS_STORE, ta, tb, p, s);
  else if (a_layout == 0) err = launch_gemm_bwd(GEMM_ROWS_STORE_BMN, ta, tb, p, s);
  else if (b_layout == 0) err = launch_gemm_fwd(GEMM_DENSE_AMN_BK, ta, tb, p, s);
  else err = launch_gemm_bwd(GEMM_DENSE_AMN_BMN, ta, tb, p, s);
  return cuda_status(err);
}

}  // extern "C"
