// MXFP8 quantisation: E4M3 codes with one E8M0 scale per 32 consecutive elements
// along the contraction axis of the GEMM that consumes them.
//
// Scale rule (OCP MX): e = floor(log2(amax)) - 8, clamped to [-127, 127], byte e + 127;
// codes = E4M3(x * 2^-e), round to nearest even, saturating at +-448 (hardware cvt).
// An all-zero block gets byte 0.
//
// Scale layout ("SF tiles"): for an operand with R rows (M or N) and K columns, the
// scales are stored as 512-byte tiles, tile (r/128, k/128) at (r/128 * K/128 + k/128)
// * 512; inside a tile the 32-bit word (r%32)*4 + (r%128)/32 holds, byte by byte, the
// scales of the four 32-element blocks of row r in that 128-wide K range.  A tile is
// exactly what one tcgen05.cp 32x128b.warpx4 moves into tensor memory for the
// block-scaled MMA.
#include "kernels.h"

namespace moe {

__device__ __forceinline__ size_t sf_byte_offset(long long r, long long k, long long k_tiles) {
  const long long tile = (r >> 7) * k_tiles + (k >> 7);
  const int word = static_cast<int>((r & 31) * 4 + ((r & 127) >> 5));
  return static_cast<size_t>(tile) * 512 + word * 4 + static_cast<int>((k & 127) >> 5);
}

// floor(log2(a)) - 8 clamped to [-127, 127] for a finite a >= 0 (-127 for a = 0).
__device__ __forceinline__ int mx_scale_exp(float a) {
  const uint32_t b = __float_as_uint(a);
  const int ef = static_cast<int>((b >> 23) & 0xFF);
  int fl;
  if (ef > 0) {
    fl = ef - 127;
  } else {
    const uint32_t m = b & 0x7FFFFF;
    if (m == 0) return -127;
    fl = (31 - __clz(m)) - 149;
  }
  return max(-127, min(127, fl - 8));
}

// 2^-e as an fp32 for e in [-127, 127] (2^-127 .. 2^127; 2^-127 is subnormal).
__device__ __forceinline__ float exp2_neg(int e) {
  const int f = 127 - e;  // biased exponent of 2^-e
  return f > 0 ? __uint_as_float(static_cast<uint32_t>(f) << 23) : __uint_as_float(0x00400000u);
}

// Two fp32 -> two E4M3 bytes (lo from `lo`, hi from `hi`), RNE, saturating.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantise 32 fp32 values (one block) into 8 words of codes; returns the scale byte.
__device__ __forceinline__ uint32_t quant_block32(const float (&v)[32], uint32_t (&codes)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = mx_scale_exp(amax);
  const float s = exp2_neg(e);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t a = cvt_e4m3x2(v[4 * w + 0] * s, v[4 * w + 1] * s);
    const uint32_t b = cvt_e4m3x2(v[4 * w + 2] * s, v[4 * w + 3] * s);
    codes[w] = a | (b << 16);
  }
  return static_cast<uint32_t>(e + 127);
}

// Row-wise: src bf16 [rows][C] (row stride ld elements) -> codes [rows][C], SF tiles
// with C/128 K tiles.  One warp per row, a lane per 128-column block.  Rows at or
// beyond *nrows_dev (if given) are skipped.
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t* __restrict__ src, long long rows,
                                                         int C, long long ld,
                                                         const int32_t* __restrict__ nrows_dev,
                                                         uint8_t* __restrict__ codes,
                                                         uint8_t* __restrict__ sf) {
  const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  long long limit = rows;
  if (nrows_dev) limit = min(limit, static_cast<long long>(*nrows_dev));
  if (r >= limit) return;
  const int kt = C / 128;
  for (int cb = lane; cb < kt; cb += 32) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + r * ld + cb * 128);
    uint4* d4 = reinterpret_cast<uint4*>(codes + r * C + cb * 128);
    uint32_t word = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = s4[g * 4 + q];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[q * 8 + 2 * i] = bf16_lo(w[i]);
          v[q * 8 + 2 * i + 1] = bf16_hi(w[i]);
        }
      }
      uint32_t c[8];
      word |= quant_block32(v, c) << (8 * g);
      d4[2 * g] = make_uint4(c[0], c[1], c[2], c[3]);
      d4[2 * g + 1] = make_uint4(c[4], c[5], c[6], c[7]);
    }
    const size_t off = sf_byte_offset(r, static_cast<long long>(cb) * 128, kt);
    *reinterpret_cast<uint32_t*>(sf + off) = word;  // the four bytes of this row and K tile
  }
}

// Column-wise, transposed: src bf16 [batch][rows][C] -> codes [batch][C][rows] and SF
// tiles (per batch) for an operand with C rows and a K of `rows`.  A block takes a
// 128 x 128 tile; a thread one column and two 32-row blocks.  Rows at or beyond
// *nrows_dev (if given) are skipped in whole 128-row tiles (the row space is padded
// to 128 per group, so a tile is either fully inside or fully outside).
__global__ void __launch_bounds__(256) quant_cols_t_kernel(const uint16_t* __restrict__ src, long long rows,
                                                           int C, const int32_t* __restrict__ nrows_dev,
                                                           uint8_t* __restrict__ codes,
                                                           uint8_t* __restrict__ sf) {
  __shared__ uint16_t tile[128][128 + 8];
  const long long b = blockIdx.z;
  const long long r0 = static_cast<long long>(blockIdx.y) * 128;
  const int c0 = blockIdx.x * 128;
  long long limit = rows;
  if (nrows_dev) limit = min(limit, static_cast<long long>(*nrows_dev));
  if (r0 >= limit) return;
  const uint16_t* s = src + b * rows * C;
  for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {  // 16 uint4 per 128-col row
    const int rr = i >> 4, q = i & 15;
    const uint4 u = (r0 + rr < rows)
                        ? *reinterpret_cast<const uint4*>(s + (r0 + rr) * C + c0 + q * 8)
                        : make_uint4(0u, 0u, 0u, 0u);
    uint32_t* t = reinterpret_cast<uint32_t*>(&tile[rr][q * 8]);
    t[0] = u.x; t[1] = u.y; t[2] = u.z; t[3] = u.w;
  }
  __syncthreads();
  const int c = threadIdx.x & 127;
  const int gpair = threadIdx.x >> 7;  // 0: row blocks 0,1; 1: row blocks 2,3
  const long long k_tiles = rows / 128;
  uint8_t* cb = codes + b * static_cast<long long>(C) * rows + static_cast<long long>(c0 + c) * rows;
  uint8_t* sfb = sf + b * (static_cast<long long>(C) * rows / 32);
#pragma unroll
  for (int gg = 0; gg < 2; ++gg) {
    const int g = gpair * 2 + gg;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(static_cast<uint32_t>(tile[g * 32 + i][c]) << 16);
    uint32_t w[8];
    const uint32_t sb = quant_block32(v, w);
    uint4* d4 = reinterpret_cast<uint4*>(cb + r0 + g * 32);
    d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    sfb[sf_byte_offset(c0 + c, r0 + g * 32, k_tiles)] = static_cast<uint8_t>(sb);
  }
}

cudaError_t launch_quant_rows(const void* src, long long rows, int C, long long ld, const int32_t* nrows_dev,
                              uint8_t* codes, uint8_t* sf, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const long long grid = (rows + 7) / 8;
  quant_rows_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(static_cast<const uint16_t*>(src), rows, C,
                                                                     ld, nrows_dev, codes, sf);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_quant_cols_t(const void* src, int batch, long long rows, int C, const int32_t* nrows_dev,
                                uint8_t* codes, uint8_t* sf, cudaStream_t stream) {
  if (rows == 0 || batch == 0) return cudaSuccess;
  dim3 grid(C / 128, static_cast<unsigned>(rows / 128), batch);
  quant_cols_t_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(src), rows, C, nrows_dev, codes,
                                                sf);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
