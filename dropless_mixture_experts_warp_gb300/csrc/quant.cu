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
// tiles (per batch) for an operand with C rows and a K of `rows`.  The work is
// 128 x 128 tiles; a thread takes two columns of one 32-row block of a tile.  Rows
// at or beyond *nrows_dev (if given) are skipped in whole 128-row tiles (the row
// space is padded to 128 per group, so a tile is either fully inside or fully
// outside).  Optional: row_map (batch 1) reads row r from src row row_map[r] (a
// negative entry reads zeros) -- the column-wise codes of a permuted matrix straight
// from its source; codes_rows/sf_rows also write the row-wise codes of the same tile
// ([batch*rows][C], K = C), so a source is read once for both orientations.
// Persistent blocks walk the tiles with the next tile's rows in flight (cp.async
// into the second of two input buffers) while the current one is quantised; the
// codes of a tile and its scales (exactly one 512-byte SF tile per orientation) are
// assembled in shared memory and leave as whole 128-byte lines.  Column blocks are
// read two columns at a time (32-bit shared loads), row blocks 16 bytes at a time.
// FP4 = true writes E2M1 codes instead (MXFP4 weights of FP8 x FP4 experts): two codes
// a byte, the lower element in the lower four bits, lines of 64 bytes, the scale rule
// with E2M1's largest exponent; the SF tiles are laid out as for E4M3.
constexpr int QC_IN_LD = 128 + 8;  // padded bf16 input rows
constexpr int QC_LD = 128 + 16;    // padded code rows (bytes)
constexpr int QC_IN_BYTES = 128 * QC_IN_LD * 2;
constexpr int QC_SMEM = 2 * QC_IN_BYTES + 2 * 128 * QC_LD + 2 * 512;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <bool FP4>
__global__ void __launch_bounds__(256) quant_cols_t_kernel(const uint16_t* __restrict__ src, int batch,
                                                           long long rows, int C,
                                                           const int32_t* __restrict__ nrows_dev,
                                                           uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                           const int32_t* __restrict__ row_map,
                                                           uint8_t* __restrict__ codes_rows,
                                                           uint8_t* __restrict__ sf_rows,
                                                           uint8_t* __restrict__ sf_rep) {
  extern __shared__ __align__(16) uint8_t qsm[];
  uint8_t* ct = qsm + 2 * QC_IN_BYTES;  // column-wise codes [128 cols][QC_LD]
  uint8_t* rt = ct + 128 * QC_LD;       // row-wise codes [128 rows][QC_LD]
  uint8_t* sft = rt + 128 * QC_LD;      // the two SF tiles
  long long limit = rows;
  if (nrows_dev) limit = min(limit, static_cast<long long>(*nrows_dev));
  const int ctiles = C / 128;
  const long long rtiles = (limit + 127) / 128;  // row tiles that hold rows
  const long long total = static_cast<long long>(batch) * rtiles * ctiles;
  const long long k_tiles = rows / 128;
  // tile t -> (batch, row tile, column tile) in 32-bit unsigned arithmetic (the launcher
  // keeps the tile count below 2^31): a 64-bit division is a long software sequence, and
  // three of them per tile and thread were a third of this kernel's instructions
  const unsigned u_ct = static_cast<unsigned>(ctiles), u_rt = static_cast<unsigned>(rtiles);
  struct Coord {
    unsigned b, rti, cti;
  };
  auto coord = [&](long long t) {
    const unsigned q = static_cast<unsigned>(t) / u_ct;
    return Coord{q / u_rt, q % u_rt, static_cast<unsigned>(t) - q * u_ct};
  };

  // the source rows of this thread's eight rows of tile t (-1: a zero row); with a row
  // map these are global loads, issued one tile ahead of the copies that use them
  auto rows_of = [&](long long t, int (&sr)[8]) {
    const long long rti = t < total ? coord(t).rti : 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const long long r = rti * 128 + (threadIdx.x >> 4) + 16 * j;
      sr[j] = (t >= total || r >= rows) ? -1 : (row_map ? row_map[r] : static_cast<int>(r));
    }
  };
  // issue the loads of tile t into input buffer `buf`
  auto fetch = [&](long long t, int buf, const int (&sr)[8]) {
    if (t < total) {
      const Coord tc = coord(t);
      const int cti = static_cast<int>(tc.cti);
      const long long b = tc.b;
      const uint16_t* s = src + (row_map ? 0 : b * rows * C);
      uint16_t(*tile)[QC_IN_LD] = reinterpret_cast<uint16_t(*)[QC_IN_LD]>(qsm + buf * QC_IN_BYTES);
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // 16 x 16 bytes per 128-column row, 8 per thread
        const int i = threadIdx.x + 256 * j;
        const int rr = i >> 4, q = i & 15;
        const bool ok = sr[j] >= 0;
        cp_async16(&tile[rr][q * 8], s + (ok ? static_cast<long long>(sr[j]) * C + cti * 128 + q * 8 : 0), ok);
      }
    }
    cp_async_commit();  // possibly empty: keeps one group per tile
  };

  const long long gs = gridDim.x;
  long long t = blockIdx.x;
  int sr_next[8];
  rows_of(t, sr_next);
  fetch(t, 0, sr_next);
  rows_of(t + gs, sr_next);
  for (int it = 0; t < total; ++it, t += gs) {
    const int buf = it & 1;
    fetch(t + gs, buf ^ 1, sr_next);
    rows_of(t + 2 * gs, sr_next);  // in flight while this tile is quantised
    cp_async_wait_prev();  // this tile's group has landed
    __syncthreads();
    const uint16_t(*tile)[QC_IN_LD] = reinterpret_cast<const uint16_t(*)[QC_IN_LD]>(qsm + buf * QC_IN_BYTES);
    const Coord tc = coord(t);
    const int cti = static_cast<int>(tc.cti);
    const long long rti = tc.rti;
    const long long b = tc.b;
    const long long r0 = rti * 128;
    const int c0 = cti * 128;
    {
      // column-wise: thread t takes columns 2 (t & 63), +1 and the 32-row block t >> 6;
      // one 32-bit shared load brings both columns of a row
      const int cp = threadIdx.x & 63, g = threadIdx.x >> 6;
      float v0[32], v1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(&tile[g * 32 + i][2 * cp]);
        v0[i] = bf16_lo(w);
        v1[i] = bf16_hi(w);
      }
      // ct line cp holds column 2 cp, line 64 + cp column 2 cp + 1 (no bank conflicts)
      if constexpr (FP4) {
        uint32_t w[4];
        uint32_t sb = quant_block32_e2m1(v0, w);
        *reinterpret_cast<uint4*>(ct + cp * QC_LD + g * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        sft[sf_byte_offset(2 * cp, g * 32, 1)] = static_cast<uint8_t>(sb);
        sb = quant_block32_e2m1(v1, w);
        *reinterpret_cast<uint4*>(ct + (64 + cp) * QC_LD + g * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        sft[sf_byte_offset(2 * cp + 1, g * 32, 1)] = static_cast<uint8_t>(sb);
      } else {
        uint32_t w[8];
        uint32_t sb = quant_block32(v0, w);
        uint4* d4 = reinterpret_cast<uint4*>(ct + cp * QC_LD + g * 32);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        sft[sf_byte_offset(2 * cp, g * 32, 1)] = static_cast<uint8_t>(sb);
        sb = quant_block32(v1, w);
        d4 = reinterpret_cast<uint4*>(ct + (64 + cp) * QC_LD + g * 32);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        sft[sf_byte_offset(2 * cp + 1, g * 32, 1)] = static_cast<uint8_t>(sb);
      }
    }
    if (codes_rows) {
      // row-wise codes of the same tile: thread t takes row t % 128, columns 64 (t / 128)
      // onwards (16-byte loads; the eight lanes of a load phase read eight consecutive
      // rows, which the padded row pitch puts on distinct banks)
      const int rr = threadIdx.x & 127;
      const int cc = (threadIdx.x >> 7) * 64;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        float v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 u = *reinterpret_cast<const uint4*>(&tile[rr][cc + blk * 32 + q * 8]);
          const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[q * 8 + 2 * i] = bf16_lo(ww[i]);
            v[q * 8 + 2 * i + 1] = bf16_hi(ww[i]);
          }
        }
        if constexpr (FP4) {
          uint32_t w[4];
          const uint32_t sb = quant_block32_e2m1(v, w);
          *reinterpret_cast<uint4*>(rt + rr * QC_LD + (cc + blk * 32) / 2) = make_uint4(w[0], w[1], w[2], w[3]);
          sft[512 + sf_byte_offset(rr, cc + blk * 32, 1)] = static_cast<uint8_t>(sb);
        } else {
          uint32_t w[8];
          const uint32_t sb = quant_block32(v, w);
          uint4* d4 = reinterpret_cast<uint4*>(rt + rr * QC_LD + cc + blk * 32);
          d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
          d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
          sft[512 + sf_byte_offset(rr, cc + blk * 32, 1)] = static_cast<uint8_t>(sb);
        }
      }
    }
    __syncthreads();
    // column-wise codes: 128 lines of 128 (FP4: 64) bytes at codes + ((c0 + column) * rows + r0) / EPB
    constexpr int EPB = FP4 ? 2 : 1;      // elements per code byte
    constexpr int QPL = 8 / EPB;          // 16-byte pieces per line
    uint8_t* cb = codes + b * static_cast<long long>(C) * rows / EPB;
#pragma unroll
    for (int j = 0; j < 4 / EPB; ++j) {
      const int i = threadIdx.x + 256 * j;
      const int line = i / QPL, q = i % QPL;
      const int col = line < 64 ? 2 * line : 2 * (line - 64) + 1;
      *reinterpret_cast<uint4*>(cb + (static_cast<long long>(c0 + col) * rows + r0) / EPB + q * 16) =
          *reinterpret_cast<const uint4*>(ct + line * QC_LD + q * 16);
    }
    if (threadIdx.x < 32) {
      const long long tile_sf = b * (static_cast<long long>(C) * rows / 32 / 512) + (c0 / 128) * k_tiles + r0 / 128;
      const uint4 v = reinterpret_cast<const uint4*>(sft)[threadIdx.x];
      reinterpret_cast<uint4*>(sf + tile_sf * 512)[threadIdx.x] = v;
      if (sf_rep)  // the same tile four times over (the CTA-pair weight gradients' B form)
#pragma unroll
        for (int r = 0; r < 4; ++r) reinterpret_cast<uint4*>(sf_rep + tile_sf * 2048 + r * 512)[threadIdx.x] = v;
    }
    if (codes_rows) {
      const long long grow0 = b * rows + r0;
#pragma unroll
      for (int j = 0; j < 4 / EPB; ++j) {
        const int i = threadIdx.x + 256 * j;
        const int line = i / QPL, q = i % QPL;
        *reinterpret_cast<uint4*>(codes_rows + ((grow0 + line) * C + c0) / EPB + q * 16) =
            *reinterpret_cast<const uint4*>(rt + line * QC_LD + q * 16);
      }
      if (threadIdx.x >= 32 && threadIdx.x < 64) {
        uint8_t* sfr = sf_rows + ((grow0 / 128) * (C / 128) + c0 / 128) * 512;
        reinterpret_cast<uint4*>(sfr)[threadIdx.x - 32] = reinterpret_cast<const uint4*>(sft + 512)[threadIdx.x - 32];
      }
    }
    __syncthreads();  // the input buffer, ct, rt and sft are reused
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Routing maps of the dispatch, without moving data: for every selection (t, j) its
// row in the padded row space (expert segment start + block base + stable rank
// within the block), both directions, and the routing weight of each row; blocks
// past the selection blocks mark one expert's padding rows (token -1, weight 0).
__global__ void __launch_bounds__(256) route_maps_kernel(int T, int E, int k, const int32_t* __restrict__ topk_idx,
                                                         const float* __restrict__ topk_w,
                                                         const int32_t* __restrict__ split_sizes,
                                                         const int32_t* __restrict__ row_offsets,
                                                         const int32_t* __restrict__ block_base,
                                                         const int32_t* __restrict__ local_rank,
                                                         int32_t* __restrict__ row_to_token,
                                                         int32_t* __restrict__ token_to_row, float* __restrict__ w_rows,
                                                         int sel_blocks, int rows_cap, int32_t* __restrict__ status) {
  if (static_cast<int>(blockIdx.x) < sel_blocks) {
    const long long gi = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
    if (gi >= static_cast<long long>(T) * k) return;
    const int t = static_cast<int>(gi / k);
    const int e = topk_idx[gi];
    int r = -1;
    if (e >= 0 && e < E)
      r = row_offsets[e] + block_base[static_cast<long long>(t / ROUTE_TOKENS) * E + e] + local_rank[gi];
    if (r < 0 || r >= rows_cap) {  // an out-of-range expert index or stale routing scratch
      set_status(status, MOE_ERR_INVARIANT);
      r = -1;
    } else {
      row_to_token[r] = t;
      w_rows[r] = topk_w[gi];
    }
    token_to_row[gi] = r;
  } else {
    const int e = blockIdx.x - sel_blocks;
    const int r0 = max(0, row_offsets[e] + split_sizes[e]);
    const int r1 = min(rows_cap, row_offsets[e + 1]);
    for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
      row_to_token[r] = -1;
      w_rows[r] = 0.0f;
    }
  }
}

cudaError_t launch_route_maps(int T, int E, int k, const int32_t* topk_idx, const float* topk_w,
                              const int32_t* split_sizes, const int32_t* row_offsets, const RouteScratch& ws,
                              int32_t* row_to_token, int32_t* token_to_row, float* w_rows, int rows_cap,
                              int32_t* status, cudaStream_t stream) {
  const long long sel = static_cast<long long>(T) * k;
  const int sel_blocks = static_cast<int>((sel + 255) / 256);
  route_maps_kernel<<<sel_blocks + E, 256, 0, stream>>>(T, E, k, topk_idx, topk_w, split_sizes, row_offsets,
                                                        ws.block_base, ws.local_rank, row_to_token, token_to_row,
                                                        w_rows, sel_blocks, rows_cap, status);
  count_launch();
  return cudaGetLastError();
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
                                uint8_t* codes, uint8_t* sf, cudaStream_t stream, const int32_t* row_map,
                                uint8_t* codes_rows, uint8_t* sf_rows, bool fp4, uint8_t* sf_rep) {
  if (rows == 0 || batch == 0) return cudaSuccess;  // callers pass rows % 128 == 0, C % 128 == 0
  auto kern = fp4 ? quant_cols_t_kernel<true> : quant_cols_t_kernel<false>;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, QC_SMEM);
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(batch) * (rows / 128) * (C / 128);
  if (tiles >= (1ll << 31)) return cudaErrorInvalidValue;  // the kernel indexes tiles in 32 bits
  const int grid = static_cast<int>(tiles < 2ll * num_sms() ? tiles : 2ll * num_sms());  // two blocks per SM
  kern<<<grid, 256, QC_SMEM, stream>>>(static_cast<const uint16_t*>(src), batch, rows, C, nrows_dev, codes, sf,
                                       row_map, codes_rows, sf_rows, sf_rep);
  count_launch();
  return cudaGetLastError();
}


}  // namespace moe
