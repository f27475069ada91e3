// A variant of moe_gemm_down_dgrad for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code embedded in a host program that owns all
// device memory through its own pool and hands its plugins no allocator, or a
// latency-critical loop where an allocation (and the device-wide synchronisation
// cudaMalloc/cudaFree may bring) is not allowed after start-up.  They can still pass
// their inputs and outputs, but not the workspace moe_gemm_down_dgrad wants for the
// per-tile partial sums of dw.  This variant keeps those partials in a file-scope
// device array instead, so it allocates nothing.
//
// The array is a module global: every GPU that loads the library holds its
// NOALLOC_DW_PART_BYTES until the process exits, and every call shares it, so two
// calls that overlap on the GPU (different streams, or different host threads) race
// on it.  Nothing in it needs to start at zero: each partial the reduction reads is
// written earlier by the same call.
#include <cstring>
#include <mutex>

#include "kernels.h"

namespace moe {

constexpr size_t NOALLOC_DW_PART_FLOATS = size_t(2) << 20;  // 8 MiB of fp32 partials
static __device__ __align__(256) float g_dw_part_scratch[NOALLOC_DW_PART_FLOATS];

// Device address of the array on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is looked up once per device
// (with that device current) and cached.
static cudaError_t scratch_address(float** out) {
  static std::mutex mu;
  static float* cached[64] = {nullptr};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == nullptr) {
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_dw_part_scratch);
    if (err != cudaSuccess) return err;
    cached[dev] = static_cast<float*>(ptr);
  }
  *out = cached[dev];
  return cudaSuccess;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_noalloc_scratch_bytes(void) { return NOALLOC_DW_PART_FLOATS * sizeof(float); }

extern "C" moe_status moe_gemm_down_dgrad_noalloc(const moe_dims* dims, const moe_bf16* dy_rows,
                                                  const int32_t* row_offsets, const float* w_rows,
                                                  const moe_bf16* w_d, const moe_bf16* gu,
                                                  moe_bf16* dgu, float* dw_rows,
                                                  int32_t* dev_status, void* stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!dy_rows || !row_offsets || !w_rows || !w_d || !gu || !dgu || !dw_rows || !dev_status)
    return MOE_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(dy_rows) | reinterpret_cast<uintptr_t>(w_d) |
                        reinterpret_cast<uintptr_t>(gu) | reinterpret_cast<uintptr_t>(dgu);
  if (mis & 15u) return MOE_ERR_ALIGNMENT;
  const int64_t R_cap = moe_row_capacity(dims);
  const int64_t R = static_cast<int64_t>(d.T) * d.k;
  const int bn = d.f % 256 == 0 ? 256 : (d.f % 128 == 0 ? 128 : 64);
  const int n_tiles = d.f / bn;
  if (static_cast<uint64_t>(R_cap) * static_cast<uint64_t>(n_tiles) > NOALLOC_DW_PART_FLOATS)
    return MOE_ERR_SCRATCH_LIMIT;  // rows x N tiles of partials must fit the static array
  float* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap ta, tb;
  if (!make_tensor_map_bf16(&ta, dy_rows, d.d, R_cap, 64, BM) ||
      !make_tensor_map_bf16(&tb, w_d, d.f, static_cast<uint64_t>(d.d) * d.E, 64, 64))
    return MOE_ERR_CUDA;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.BN = bn; p.N = d.f; p.K = d.d; p.E = d.E; p.row_offsets = row_offsets;
  p.b_k_per_expert = d.d; p.m_fastest = ORDER_PER_GROUP; p.band_krows = BAND_KROWS_BF16; p.f = d.f;
  p.row_limit = R_cap; p.w_rows = w_rows; p.gu_in = gu; p.dgu_out = dgu; p.dw_part = scratch;
  p.dw_stride = n_tiles; p.status = dev_status;
  // the same kernel choice as moe_gemm_down_dgrad, so both give the same bits
  if (launch_best(GEMM_ROWS_SWIGLU_BWD, true, ta, tb, p, s) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_dw_reduce(scratch, n_tiles, row_offsets, d.E, dw_rows, static_cast<int>(R_cap), s) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
