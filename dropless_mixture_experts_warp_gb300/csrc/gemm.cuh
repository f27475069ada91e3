// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One CTA per SM, 6 warps:
//   warp 0      TMA producer: 128B-swizzled tiles of A and B into a 4-stage ring
//   warp 1      MMA issuer: tcgen05.mma (M=128, N=BN, K=16) into a TMEM accumulator;
//               owns the TMEM allocation (two accumulators of 256 fp32 columns)
//   warps 2..    epilogue (4 warps, 8 for the SwiGLU' epilogue): tcgen05.ld of the
//               accumulator, fused SwiGLU / SwiGLU' arithmetic, bf16 stores.  Warp w
//               reads TMEM lanes 32*(w%4)..+31; with 8 warps, w and w+4 split the columns.
// The two accumulators let the epilogue of one tile overlap the mainloop of the
// next.  Work tiles come from a device-side schedule derived from row_offsets, so
// the host never waits for the per-expert counts.
//
// Scheduling modes
//   SCHED_ROWS    ragged M: expert e owns output rows [row_offsets[e], row_offsets[e+1]),
//                 a multiple of 128, and multiplies them by its own weight B[e]
//                 (grouped GEMM of the forward and of the data-gradient backward).
//   SCHED_KGROUP  ragged K: out[e] = A_e^T B_e summed over the rows of expert e
//                 (weight gradients); an expert without rows gets zeros.
// Operand majorness: K-major tiles come straight from row-major [rows][K] tensors;
// MN-major tiles (A or B stored [K][MN]) use the transpose bits of the instruction
// descriptor, so no operand is ever transposed in memory.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_STAGE_BYTES_MAX = 256 * BK * 2;     // 32 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES_MAX;
constexpr int GEMM_SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
constexpr int TMEM_COLS = 512;
constexpr int ACC_STRIDE = 256;
// Epilogue warps: 8 for the SwiGLU' epilogues and the quantising SwiGLU epilogue (two
// per TMEM lane quarter, splitting the columns), 4 otherwise.  Block = producer warp +
// MMA warp + epilogue warps.
__host__ __device__ constexpr int epi_warps(int epi) { return (epi == 2 || epi == 3 || epi == 4) ? 8 : 4; }
__host__ __device__ constexpr int gemm_threads(int epi) { return 64 + 32 * epi_warps(epi); }
constexpr int MAX_EXPERTS = 1024;
constexpr long long WAIT_LIMIT_CYCLES = 1ll << 31;  // about one second

enum Epi {
  EPI_STORE = 0,
  EPI_SWIGLU_FWD = 1,     // G|U (bf16, saved) and h (bf16)
  EPI_SWIGLU_BWD = 2,     // dG|dU (bf16) and dw partials
  EPI_SWIGLU_FWD_MX = 3,  // G|U (bf16, saved) and h quantised row- and column-wise (MXFP8)
  EPI_SWIGLU_BWD_MX = 4   // dG|dU quantised row- and column-wise, and dw partials
};
enum Sched { SCHED_ROWS = 0, SCHED_KGROUP = 1 };
// Epilogues whose accumulator holds gate columns then up columns (B = gate rows, up rows)
__host__ __device__ constexpr bool gu_split(int epi) { return epi == EPI_SWIGLU_FWD || epi == EPI_SWIGLU_FWD_MX; }

struct GemmParams {
  int BN;                       // accumulator width: 64, 128 or 256
  int N;                        // output columns (SWIGLU_FWD: h columns = f)
  int K;                        // contraction length (SCHED_ROWS; dense SCHED_KGROUP)
  int M;                        // SCHED_KGROUP: output rows per expert; dense mode: rows
  int E;                        // groups
  const int32_t* row_offsets;   // [E+1] padded row offsets; NULL = one group of M rows
  int b_rows_per_expert;        // B K-major: rows of the B tensor per expert
  int b_k_per_expert;           // B MN-major (SCHED_ROWS): K rows per expert
  int m_fastest;                // tile order inside a group: 0 = N fastest, 1 = M fastest,
                                // ORDER_PER_GROUP (SCHED_ROWS): chosen per group, see rows_m_fastest
  int band_krows;               // SCHED_ROWS, > 0: the fast side in bands of band_krows / K tiles (banded)
  int f;                        // SwiGLU epilogues: intermediate width (offset of U)
  moe_bf16* out;                // EPI_STORE output
  long long ldo;                // its leading dimension (elements)
  long long row_limit;          // rows >= row_limit are not stored
  const float* w_rows;          // routing weight per row (SwiGLU epilogues); NULL = 1
  moe_bf16* gu_out;             // SWIGLU_FWD: saved G|U [rows][2f]
  moe_bf16* h_out;              // SWIGLU_FWD: h [rows][f]
  const moe_bf16* gu_in;        // SWIGLU_BWD: saved G|U
  moe_bf16* dgu_out;            // SWIGLU_BWD: dG|dU [rows][2f]
  float* dw_part;               // SWIGLU_BWD: per-row partial of dw, one per N tile (or NULL)
  int dw_stride;                // its row stride (= number of N tiles)
  int32_t* status;              // device status word
  // block-scaled (MXFP8) operands only: SF tiles and their number of K tiles per 128 rows
  const uint8_t* sfa;
  const uint8_t* sfb;
  int a_sf_ktiles;
  int b_sf_ktiles;
  int b_fmt;                    // B element format: MX_FMT_E4M3 (0) or MX_FMT_E2M1 (FP4 weights)
  // fused MXFP8 outputs of the *_MX epilogues: row-wise codes [rows][width] with SF
  // tiles (K = width), and column-wise codes [width][q_cols_ld] with SF tiles
  // (K = rows, q_cols_ktiles = q_cols_ld / 128); width = f (h) or 2f (dG|dU)
  uint8_t* q_rows;
  uint8_t* q_rows_sf;
  uint8_t* q_cols;
  uint8_t* q_cols_sf;
  long long q_cols_ld;
  int q_cols_ktiles;
  // the column-wise SF tiles again, each written four times over (SF_REP_TILE_BYTES per tile):
  // the operand form the CTA-pair weight-gradient kernel reads for B (NULL: not written)
  uint8_t* q_cols_sf_rep;
  int sfb_rep;                  // CTA-pair MXFP8 kernel: B's SF tiles are in that replicated form
};

// A replicated SF tile: the 512-byte tile four times, so that one 128x256b tensor-pipe copy of
// two of them fills the four TMEM lane quarters with both (see gemm_mx2.cuh).
constexpr int SF_REP_TILE_BYTES = 4 * 512;
__device__ __forceinline__ void store_sf_rep(uint8_t* rep, size_t off, uint8_t v) {
  uint8_t* t = rep + (off >> 9) * SF_REP_TILE_BYTES + (off & 511);
#pragma unroll
  for (int r = 0; r < 4; ++r) t[r * 512] = v;
}

struct TileCoord {
  int e, m, n, kblocks;
  int a_m, a_k;       // A: first row (K-major) / first column (MN-major), first K index
  int b_n, b_k;       // B: first N index (row for K-major, column for MN-major), first K index
  long long out_row;  // first output row of the tile
  int out_col;        // first output column
  long long out_base; // element offset of the group's output (SCHED_KGROUP)
};

// Ragged-K schedule (SCHED_KGROUP, the weight gradients): a tile's cost is its
// expert's row count, which routing skew spreads over an order of magnitude.  When
// one tile is a sizeable share of a worker's mean load (the longest above 5 %: few
// tiles per expert, a few experts holding most rows), plain round robin leaves some
// workers with the long end of every round, so the experts are visited in decreasing
// row count (ties: lower index first) and the workers deal the tiles in a snake:
// round r gives worker w tile r * W + w (r even) or r * W + W - 1 - w (r odd).
// Otherwise the experts keep their index order and the deal stays round robin (with
// many tiles per expert the sorted order measured slower: every worker then starts on
// the hottest expert at once).  order[rank] = expert; per: tiles per expert; W:
// workers.  Every thread of the block calls it once the row offsets are in shared
// memory; all get the same answer (true: sorted snake).
__device__ __forceinline__ bool kgroup_order(const int* s_ro, int E, int per, int W, int* order) {
  int longest = 0;
  for (int j = 0; j < E; ++j) longest = max(longest, s_ro[j + 1] - s_ro[j]);
  const long long mean_load = static_cast<long long>(s_ro[E] - s_ro[0]) * per / W;  // rows per worker
  const bool lpt = 20ll * longest > mean_load;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int n = s_ro[e + 1] - s_ro[e];
    int rank = e;
    if (lpt) {
      rank = 0;
      for (int j = 0; j < E; ++j) {
        const int m = s_ro[j + 1] - s_ro[j];
        rank += (m > n || (m == n && j < e)) ? 1 : 0;
      }
    }
    order[rank] = e;
  }
  return lpt;
}

// The tile worker w of W takes in its round r (see kgroup_order).
__device__ __forceinline__ int sched_tile(int r, int w, int W, bool snake) {
  return r * W + ((snake && (r & 1)) ? W - 1 - w : w);
}

// Tile order of one group of SCHED_ROWS.  Each group sweeps its shorter side fastest: the
// panels along that side (all of them) are revisited at every step along the longer side
// and stay in L2, while each panel of the longer side is read once, by the workers on it at
// the same time.  For a cold expert that is M (its few activation panels); for a hot expert
// with more row tiles than column tiles it is N (its weight panels) -- sweeping M first
// there streams its large block of activations from DRAM once per column of tiles.
constexpr int ORDER_PER_GROUP = 2;
__device__ __forceinline__ bool rows_m_fastest(int mode, int m_tiles, int n_tiles) {
  return mode == ORDER_PER_GROUP ? m_tiles <= n_tiles : mode != 0;
}

// SCHED_ROWS: when the panels along the fast side of a large group (K elements deep each)
// are more than L2 keeps beside the other side's stream, how much of them survives a sweep
// depends on the timing of every other worker (the same bf16 schedule read 1.2x to 1.6x its
// operand bytes from box to box).  So the fast side goes in bands: a band of b tiles of the
// fast side is swept fastest against the whole slow side, then the next band; b =
// band_krows / K keeps a band's panels within a fixed budget, and the slow side is streamed
// once per band.  (The ragged-K weight gradients keep one sweep: banding them by each
// expert's K measured 3-4 % slower.)
// band_krows for a 32 MB band of 256-row panels: bf16 and E4M3 operands
constexpr int BAND_KROWS_BF16 = (32 << 20) / (256 * 2);
constexpr int BAND_KROWS_E4M3 = (32 << 20) / 256;
__device__ __forceinline__ int band_of(const GemmParams& p, int K) {
  return p.band_krows > 0 ? max(1, p.band_krows / max(K, 1)) : (1 << 30);
}
// local tile -> (m, n) inside an mt x nt group; m_fast: M is the fast side
__device__ __forceinline__ void banded(int local, int mt, int nt, bool m_fast, int band, int& m, int& n) {
  const int r = m_fast ? mt : nt, l = m_fast ? nt : mt;
  const int b = band < r ? band : r;
  const int k = local / (b * l);
  const int rem = local - k * (b * l);
  const int w = min(b, r - k * b);  // the last band may be narrower
  const int fast = k * b + rem % w, slow = rem / w;
  m = m_fast ? fast : slow;
  n = m_fast ? slow : fast;
}

// order: the experts in their visiting order (SCHED_KGROUP, kgroup_order; unused for
// SCHED_ROWS)
template <int SCHED, int EPI, bool B_MN, int KB = BK>
__device__ __forceinline__ TileCoord tile_coord(const GemmParams& p, const int* s_ro, const int* order, int E,
                                                int n_tiles, int tile) {
  TileCoord c;
  if (SCHED == SCHED_ROWS) {
    int lo = 0, hi = E - 1;  // last expert whose first tile is <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((s_ro[mid] / BM) * n_tiles <= tile) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int local = tile - (s_ro[e] / BM) * n_tiles;
    const int mt = (s_ro[e + 1] - s_ro[e]) / BM;
    banded(local, mt, n_tiles, rows_m_fastest(p.m_fastest, mt, n_tiles), band_of(p, p.K), c.m, c.n);
    c.e = e;
    c.kblocks = p.K / KB;
    c.a_m = s_ro[e] + c.m * BM;
    c.a_k = 0;
    c.out_col = gu_split(EPI) ? c.n * (p.BN / 2) : c.n * p.BN;
    c.b_n = B_MN ? c.out_col : e * p.b_rows_per_expert + c.out_col;
    c.b_k = B_MN ? e * p.b_k_per_expert : 0;
    c.out_row = c.a_m;
    c.out_base = 0;
  } else {
    const int mt = p.M / BM;
    const int per = mt * n_tiles;
    const int e = order[tile / per];
    const int local = tile - (tile / per) * per;
    if (p.m_fastest) { c.m = local % mt; c.n = local / mt; }
    else { c.n = local % n_tiles; c.m = local / n_tiles; }
    c.e = e;
    c.kblocks = (s_ro[e + 1] - s_ro[e]) / KB;
    c.a_m = c.m * BM;
    c.a_k = s_ro[e];
    c.b_n = c.n * p.BN;
    c.b_k = s_ro[e];
    c.out_row = c.m * BM;
    c.out_col = c.n * p.BN;
    c.out_base = static_cast<long long>(e) * p.M * p.N;
  }
  return c;
}

// Two fp32 lanes for the packed Blackwell fp32 pipe (mul/fma .rn.f32x2: each lane
// rounds as the scalar instruction would).
struct F2 {
  float x, y;
};
__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
  F2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
  F2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float tanh_approx(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(x));
  return t;
}

// The logistic sigmoid in every SwiGLU epilogue goes through the identity
// sigmoid(g) = (1 + tanh(g / 2)) / 2 on the hardware tanh approximation: one
// special-function operation instead of an exponential and a reciprocal (absolute
// error about 2^-12, below bf16 resolution), computed as fma(0.5, tanh(0.5 g), 0.5).
// h = w silu(g) u = (w (g sigmoid(g))) u for two neighbouring columns.
__device__ __forceinline__ F2 swiglu_pair(F2 g, F2 u, F2 w2) {
  const F2 half{0.5f, 0.5f};
  const F2 hg = mul2(half, g);
  const F2 sg = fma2(half, F2{tanh_approx(hg.x), tanh_approx(hg.y)}, half);
  return mul2(mul2(w2, mul2(g, sg)), u);
}

// Shared state of the epilogue warps: the hand-off of the dw partials between the
// two epilogue warps of a TMEM lane quarter (second half -> first half, through
// mbarriers so every wait is bounded) and, for the *_MX epilogues, this warp's
// 32 x 17 fp32 transpose buffer.
struct DwHandoff {
  float* s_dw;             // [BM] partials of the second half
  uint64_t* full;          // [4] second half has written s_dw
  uint64_t* empty;         // [4] first half has read it
  uint32_t* phase;         // this thread's phase bit
  volatile int* abort_flag;
  float* xbuf = nullptr;   // [32][17] per warp (MX epilogues)
};

constexpr int XBUF_FLOATS = 32 * 17;

// Column-wise MXFP8 codes of a 32-row x 32-column fp32 chunk held one row per lane
// (v[i] = row `lane`, column col0 + i).  The warp's 32 rows are one 32-row block of
// every column: the block scale comes from the column's maximum over them.  The
// chunk goes through shared memory in two 16-column halves; then lane l holds rows
// (l >> 4) * 16 .. +16 of column l & 15, so the maximum needs one shuffle and the
// 16 codes leave as one 16-byte store.  codes: [cols][ld] (K = rows), scales: SF tiles.
__device__ __forceinline__ void quant_cols_chunk32(const float (&v)[32], float* xb, int lane, uint8_t* codes,
                                                   uint8_t* scales, long long ld, int ktiles, int col0,
                                                   long long rblk, bool ok, uint8_t* scales_rep = nullptr) {
  const int cc = lane & 15, hh = lane >> 4;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 16; ++j) xb[lane * 17 + j] = v[16 * s + j];
    __syncwarp();
    float cv[16], m[6];
#pragma unroll
    for (int i = 0; i < 16; ++i) cv[i] = xb[(hh * 16 + i) * 17 + cc];
#pragma unroll
    for (int j = 0; j < 5; ++j) m[j] = absmax3(cv[3 * j], cv[3 * j + 1], cv[3 * j + 2]);
    m[5] = absmax3(cv[15], cv[15], cv[15]);
    float a = absmax3(absmax3(m[0], m[1], m[2]), m[3], absmax3(m[4], m[5], m[5]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
    const int e = mx_scale_exp(a);
    const uint32_t sb = __float_as_uint(exp2_neg(e));
    const uint64_t ss = (static_cast<uint64_t>(sb) << 32) | sb;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float x0 = cv[4 * q], x1 = cv[4 * q + 1], x2 = cv[4 * q + 2], x3 = cv[4 * q + 3];
      mul_f32x2(x0, x1, ss);
      mul_f32x2(x2, x3, ss);
      w[q] = cvt_e4m3x4(x0, x1, x2, x3);
    }
    const int col = col0 + 16 * s + cc;
    if (ok) {
      *reinterpret_cast<uint4*>(codes + static_cast<long long>(col) * ld + rblk + hh * 16) =
          make_uint4(w[0], w[1], w[2], w[3]);
      if (hh == 0) {
        const size_t off = sf_byte_offset(col, rblk, ktiles);
        scales[off] = static_cast<uint8_t>(e + 127);
        if (scales_rep) store_sf_rep(scales_rep, off, static_cast<uint8_t>(e + 127));
      }
    }
  }
}

// STORE epilogue with early release.  Part 1: the warp's nc (<= 4) chunks of 32
// accumulator columns from col0 into registers (zeros for a tile without K blocks);
// the caller then hands the accumulator back to the MMA warp.
__device__ __forceinline__ void acc_load_chunks(uint32_t tbase, int col0, int nc, bool have, uint32_t (&r)[4][32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i < nc) {
      if (have) {
        tmem_ld32(tbase + col0 + 32 * i, r[i]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[i][j] = 0u;
      }
    }
  }
  tmem_wait_ld();
}

// A 32 x 32 bf16 box (row `lane`, 32 fp32 values) into a 2 KB staging buffer in the
// layout of a 64-byte-swizzled tensor store (16-byte chunk j of row r at j ^ ((r >> 1) & 3)).
__device__ __forceinline__ void stage_row_bf16(uint8_t* buf, int lane, const float (&v)[32]) {
  const uint32_t row_addr = smem_u32(buf) + lane * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_v4(row_addr + ((j ^ sw) << 4), pack_bf16(v[8 * j + 0], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                 pack_bf16(v[8 * j + 4], v[8 * j + 5]), pack_bf16(v[8 * j + 6], v[8 * j + 7]));
}

// Part 2: the chunks (columns x0 .. x0 + 32 nc of output rows y0 .. y0 + 31) leave as
// bf16 through the warp's 2 KB staging buffer (64-byte swizzle: 16-byte chunk j of row r
// at chunk j ^ ((r >> 1) & 3), free of bank conflicts)
// and one tensor store each, while the next tile accumulates.
__device__ __forceinline__ void store_chunks_tma(const CUtensorMap* tmC, const uint32_t (&r)[4][32], int nc, int x0,
                                                 int y0, int lane, uint8_t* stg) {
  const uint32_t row_addr = smem_u32(stg) + lane * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i < nc) {
      if (lane == 0) bulk_wait_read<0>();  // the previous store has read the buffer
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_shared_v4(row_addr + ((j ^ sw) << 4),
                     pack_bf16(__uint_as_float(r[i][8 * j + 0]), __uint_as_float(r[i][8 * j + 1])),
                     pack_bf16(__uint_as_float(r[i][8 * j + 2]), __uint_as_float(r[i][8 * j + 3])),
                     pack_bf16(__uint_as_float(r[i][8 * j + 4]), __uint_as_float(r[i][8 * j + 5])),
                     pack_bf16(__uint_as_float(r[i][8 * j + 6]), __uint_as_float(r[i][8 * j + 7])));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmC, stg, x0 + 32 * i, y0);
        bulk_commit();
      }
    }
  }
}

// Quantising SwiGLU epilogue (EPI_SWIGLU_FWD_MX) pieces, one 32-column chunk of a row
// at a time (h column col; G and U read from the accumulator): h = w silu(G) U in fp32,
// G and U rounded to bf16 pairs.
struct FwdMxChunk {
  float h[32];
  uint32_t g[16], u[16];  // bf16 pairs
};

__device__ __forceinline__ void fwd_mx_chunk(const uint32_t (&g)[32], const uint32_t (&u)[32], float w,
                                             FwdMxChunk& f) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const F2 h = swiglu_pair(F2{__uint_as_float(g[j]), __uint_as_float(g[j + 1])},
                             F2{__uint_as_float(u[j]), __uint_as_float(u[j + 1])}, F2{w, w});
    f.h[j] = h.x;
    f.h[j + 1] = h.y;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    f.g[j] = pack_bf16(__uint_as_float(g[2 * j]), __uint_as_float(g[2 * j + 1]));
    f.u[j] = pack_bf16(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1]));
  }
}

// G|U (bf16, saved for the backward pass), the row-wise codes of h (one 32-column
// block) and its column-wise codes (the warp's 32 rows, first row rblk, are one 32-row
// block of every column).
__device__ __forceinline__ void fwd_mx_store_chunk(const GemmParams& p, long long row, bool row_ok, bool blk_ok,
                                                   long long rblk, int col, int lane, float* xbuf,
                                                   const FwdMxChunk& f) {
  if (row_ok) {
    const long long ld2 = 2ll * p.f;
    uint4* gdst = reinterpret_cast<uint4*>(p.gu_out + row * ld2 + col);
    uint4* udst = reinterpret_cast<uint4*>(p.gu_out + row * ld2 + p.f + col);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      gdst[v] = make_uint4(f.g[4 * v], f.g[4 * v + 1], f.g[4 * v + 2], f.g[4 * v + 3]);
      udst[v] = make_uint4(f.u[4 * v], f.u[4 * v + 1], f.u[4 * v + 2], f.u[4 * v + 3]);
    }
    uint32_t q[8];
    const uint32_t sb = quant_block32(f.h, q);
    uint4* qd = reinterpret_cast<uint4*>(p.q_rows + row * p.f + col);
    qd[0] = make_uint4(q[0], q[1], q[2], q[3]);
    qd[1] = make_uint4(q[4], q[5], q[6], q[7]);
    p.q_rows_sf[sf_byte_offset(row, col, p.f / 128)] = static_cast<uint8_t>(sb);
  }
  quant_cols_chunk32(f.h, xbuf, lane, p.q_cols, p.q_cols_sf, p.q_cols_ld, p.q_cols_ktiles, col, rblk, blk_ok,
                     p.q_cols_sf_rep);
}

// Quantising SwiGLU' epilogue (EPI_SWIGLU_BWD_MX) pieces.  The saved G and U of one
// row's 32 h columns (bf16, 64 bytes each).
struct GuChunk {
  uint4 g[4], u[4];
};

__device__ __forceinline__ void load_gu_chunk(const GemmParams& p, long long row, bool row_ok, int col, GuChunk& x) {
  if (row_ok) {
    const long long ld2 = 2ll * p.f;
    const uint4* gsrc = reinterpret_cast<const uint4*>(p.gu_in + row * ld2 + col);
    const uint4* usrc = reinterpret_cast<const uint4*>(p.gu_in + row * ld2 + p.f + col);
#pragma unroll
    for (int v = 0; v < 4; ++v) { x.g[v] = __ldg(gsrc + v); x.u[v] = __ldg(usrc + v); }
  } else {
#pragma unroll
    for (int v = 0; v < 4; ++v) { x.g[v] = make_uint4(0u, 0u, 0u, 0u); x.u[v] = x.g[v]; }
  }
}

// SwiGLU' of one 32-column chunk: dH (fp32 accumulator columns) and the saved G, U
// (bf16) -> dG = w dH U silu'(G), dU = w dH silu(G), with sigmoid as in swiglu_pair and
// silu'(g) = sigmoid(g) (1 + g (1 - sigmoid(g))); returns the chunk's share of the
// row's sum of silu(G) U dH (eight fixed-order partial sums).  Neighbouring columns
// go through the packed fp32 pipe together.
__device__ __forceinline__ float swiglu_bwd_values(const uint32_t (&r)[32], const GuChunk& gu, float w,
                                                   float (&dg)[32], float (&du)[32]) {
  const F2 half{0.5f, 0.5f}, one{1.0f, 1.0f}, mone{-1.0f, -1.0f}, w2{w, w};
  F2 part[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint32_t gw[4] = {gu.g[v].x, gu.g[v].y, gu.g[v].z, gu.g[v].w};
    const uint32_t uw[4] = {gu.u[v].x, gu.u[v].y, gu.u[v].z, gu.u[v].w};
    part[v] = F2{0.0f, 0.0f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = 8 * v + 2 * q;
      const F2 g{bf16_lo(gw[q]), bf16_hi(gw[q])};
      const F2 u{bf16_lo(uw[q]), bf16_hi(uw[q])};
      const F2 dh{__uint_as_float(r[i]), __uint_as_float(r[i + 1])};
      const F2 hg = mul2(half, g);
      const F2 sg = fma2(half, F2{tanh_approx(hg.x), tanh_approx(hg.y)}, half);
      const F2 silu = mul2(g, sg);
      const F2 da = mul2(w2, dh);
      part[v] = fma2(mul2(silu, u), dh, part[v]);
      const F2 d = mul2(mul2(mul2(da, u), sg), fma2(g, fma2(sg, mone, one), one));
      const F2 e = mul2(da, silu);
      dg[i] = d.x;
      dg[i + 1] = d.y;
      du[i] = e.x;
      du[i + 1] = e.y;
    }
  }
  return ((part[0].x + part[0].y) + (part[1].x + part[1].y)) + ((part[2].x + part[2].y) + (part[3].x + part[3].y));
}

// One 32-column chunk: dH (fp32, accumulator columns of h columns col .. col + 31)
// and the saved G, U -> dG, dU as above, quantised along the row (dG at column col,
// dU at f + col of dG|dU) and down the columns (the warp's 32 rows form one block);
// dwp gathers the row's sum of silu(G) U dH.
__device__ __forceinline__ void bwd_mx_chunk(const GemmParams& p, long long row, bool row_ok, bool blk_ok, float w,
                                             int col, const uint32_t (&r)[32], const GuChunk& gu, float& dwp,
                                             float* xbuf, int lane, long long rblk) {
  const long long ld2 = 2ll * p.f;
  float dg[32], du[32];
  dwp += swiglu_bwd_values(r, gu, w, dg, du);
  if (row_ok) {
    uint32_t q[8];
    uint32_t sb = quant_block32(dg, q);
    uint4* qd = reinterpret_cast<uint4*>(p.q_rows + row * ld2 + col);
    qd[0] = make_uint4(q[0], q[1], q[2], q[3]);
    qd[1] = make_uint4(q[4], q[5], q[6], q[7]);
    p.q_rows_sf[sf_byte_offset(row, col, ld2 / 128)] = static_cast<uint8_t>(sb);
    sb = quant_block32(du, q);
    qd = reinterpret_cast<uint4*>(p.q_rows + row * ld2 + p.f + col);
    qd[0] = make_uint4(q[0], q[1], q[2], q[3]);
    qd[1] = make_uint4(q[4], q[5], q[6], q[7]);
    p.q_rows_sf[sf_byte_offset(row, p.f + col, ld2 / 128)] = static_cast<uint8_t>(sb);
  }
  quant_cols_chunk32(dg, xbuf, lane, p.q_cols, p.q_cols_sf, p.q_cols_ld, p.q_cols_ktiles, col, rblk, blk_ok);
  quant_cols_chunk32(du, xbuf, lane, p.q_cols, p.q_cols_sf, p.q_cols_ld, p.q_cols_ktiles, p.f + col, rblk, blk_ok);
}

// The row's dw partial of this N tile: with two warps per lane quarter the second
// half's sum goes through shared memory and the first half adds it (a fixed order).
template <int NH>
__device__ __forceinline__ bool dw_combine(const GemmParams& p, const TileCoord& c, long long row, bool row_ok,
                                           int half, int quarter, int row_in_tile, const DwHandoff& hand, float dwp) {
  const int lane = row_in_tile & 31;
  if (NH == 1) {
    if (row_ok && p.dw_part) p.dw_part[row * p.dw_stride + c.n] = dwp;
  } else if (p.dw_part) {
    const uint32_t ph = *hand.phase;
    *hand.phase ^= 1u;
    if (half == 1) {
      if (!mbar_wait_bounded(&hand.empty[quarter], ph ^ 1, hand.abort_flag, p.status, WAIT_LIMIT_CYCLES))
        return false;
      hand.s_dw[row_in_tile] = dwp;
      __syncwarp();
      if (lane == 0) mbar_arrive(&hand.full[quarter]);
    } else {
      if (!mbar_wait_bounded(&hand.full[quarter], ph, hand.abort_flag, p.status, WAIT_LIMIT_CYCLES))
        return false;
      if (row_ok) p.dw_part[row * p.dw_stride + c.n] = dwp + hand.s_dw[row_in_tile];
      __syncwarp();
      if (lane == 0) mbar_arrive(&hand.empty[quarter]);
    }
  }
  return true;
}

// Epilogue of one tile for one thread (one accumulator row, half of the columns):
// reads fp32 accumulator columns from TMEM (32 at a time) and applies the fused EPI
// step.  The two epilogue warps of a TMEM lane quarter split the tile's columns
// (`half` 0 or 1).  Every lane of both warps must call it (tcgen05.ld and the named
// barrier are collective).
template <int EPI, int NH = epi_warps(EPI) / 4>
__device__ __forceinline__ bool tile_epilogue(const GemmParams& p, const TileCoord& c, uint32_t tbase,
                                              long long row, bool row_ok, int BN, int half, int quarter,
                                              int row_in_tile, const DwHandoff& hand) {
  if (EPI == EPI_STORE) {
    const int cb = half * (BN / NH);
    for (int c0 = cb; c0 < cb + BN / NH; c0 += 32) {
      uint32_t r[32];
      if (c.kblocks > 0) {
        tmem_ld32(tbase + c0, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
      }
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + c.out_base + row * p.ldo + c.out_col + c0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 o;
          o.x = pack_bf16(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
          o.y = pack_bf16(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
          o.z = pack_bf16(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
          o.w = pack_bf16(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
          dst[v] = o;
        }
      }
    }
  } else if (EPI == EPI_SWIGLU_FWD) {
    // columns [0, BN/2) hold G, [BN/2, BN) hold U for h columns out_col .. +BN/2;
    // this half takes h columns [half*BN/4, (half+1)*BN/4)
    const int hw = BN / 2;
    const float w = !row_ok ? 0.0f : (p.w_rows ? p.w_rows[row] : 1.0f);
    const long long ld2 = 2ll * p.f;
    const int cb = half * (hw / NH);
    for (int c0 = cb; c0 < cb + hw / NH; c0 += 32) {
      uint32_t g[32], u[32];
      tmem_ld32(tbase + c0, g);
      tmem_ld32(tbase + hw + c0, u);
      tmem_wait_ld();
      if (row_ok) {
        uint4* gdst = reinterpret_cast<uint4*>(p.gu_out + row * ld2 + c.out_col + c0);
        uint4* udst = reinterpret_cast<uint4*>(p.gu_out + row * ld2 + p.f + c.out_col + c0);
        uint4* hdst = reinterpret_cast<uint4*>(p.h_out + row * p.f + c.out_col + c0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float hv[8], gv[8], uv[8];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            gv[i] = __uint_as_float(g[8 * v + i]);
            gv[i + 1] = __uint_as_float(g[8 * v + i + 1]);
            uv[i] = __uint_as_float(u[8 * v + i]);
            uv[i + 1] = __uint_as_float(u[8 * v + i + 1]);
            const F2 h = swiglu_pair(F2{gv[i], gv[i + 1]}, F2{uv[i], uv[i + 1]}, F2{w, w});
            hv[i] = h.x;
            hv[i + 1] = h.y;
          }
          gdst[v] = make_uint4(pack_bf16(gv[0], gv[1]), pack_bf16(gv[2], gv[3]),
                               pack_bf16(gv[4], gv[5]), pack_bf16(gv[6], gv[7]));
          udst[v] = make_uint4(pack_bf16(uv[0], uv[1]), pack_bf16(uv[2], uv[3]),
                               pack_bf16(uv[4], uv[5]), pack_bf16(uv[6], uv[7]));
          hdst[v] = make_uint4(pack_bf16(hv[0], hv[1]), pack_bf16(hv[2], hv[3]),
                               pack_bf16(hv[4], hv[5]), pack_bf16(hv[6], hv[7]));
        }
      }
    }
  } else if (EPI == EPI_SWIGLU_BWD_MX) {
    // as EPI_SWIGLU_BWD, but dG|dU are quantised from fp32 along their row (blocks of
    // 32 columns of 2f) and down their columns (the warp's 32 rows)
    const float w = !row_ok ? 0.0f : (p.w_rows ? p.w_rows[row] : 1.0f);
    const int lane = row_in_tile & 31;
    const long long rblk = row - lane;
    const bool blk_ok = __all_sync(0xffffffffu, row_ok);  // the warp's 32 rows are one block
    float dwp = 0.0f;
    const int cb = half * (BN / NH);
    // the saved G and U of the next chunk are fetched while this one is processed
    GuChunk nx;
    load_gu_chunk(p, row, row_ok, c.out_col + cb, nx);
    for (int c0 = cb; c0 < cb + BN / NH; c0 += 32) {
      const GuChunk cur = nx;
      if (c0 + 32 < cb + BN / NH) load_gu_chunk(p, row, row_ok, c.out_col + c0 + 32, nx);
      uint32_t r[32];
      tmem_ld32(tbase + c0, r);
      tmem_wait_ld();
      bwd_mx_chunk(p, row, row_ok, blk_ok, w, c.out_col + c0, r, cur, dwp, hand.xbuf, lane, rblk);
    }
    if (!dw_combine<NH>(p, c, row, row_ok, half, quarter, row_in_tile, hand, dwp)) return false;
  } else {  // EPI_SWIGLU_BWD: accumulator = dH for h columns out_col .. +BN; this half: BN/2 of them
    const float w = !row_ok ? 0.0f : (p.w_rows ? p.w_rows[row] : 1.0f);
    const long long ld2 = 2ll * p.f;
    float dwp = 0.0f;
    const int cb = half * (BN / NH);
    // the saved G and U of the next chunk are fetched while this one is processed
    GuChunk nx;
    load_gu_chunk(p, row, row_ok, c.out_col + cb, nx);
    for (int c0 = cb; c0 < cb + BN / NH; c0 += 32) {
      const GuChunk cur = nx;
      if (c0 + 32 < cb + BN / NH) load_gu_chunk(p, row, row_ok, c.out_col + c0 + 32, nx);
      uint32_t r[32];
      tmem_ld32(tbase + c0, r);
      tmem_wait_ld();
      float dg[32], du[32];
      dwp += swiglu_bwd_values(r, cur, w, dg, du);
      if (row_ok) {
        uint4* gdst = reinterpret_cast<uint4*>(p.dgu_out + row * ld2 + c.out_col + c0);
        uint4* udst = reinterpret_cast<uint4*>(p.dgu_out + row * ld2 + p.f + c.out_col + c0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          gdst[v] = make_uint4(pack_bf16(dg[8 * v], dg[8 * v + 1]), pack_bf16(dg[8 * v + 2], dg[8 * v + 3]),
                               pack_bf16(dg[8 * v + 4], dg[8 * v + 5]), pack_bf16(dg[8 * v + 6], dg[8 * v + 7]));
          udst[v] = make_uint4(pack_bf16(du[8 * v], du[8 * v + 1]), pack_bf16(du[8 * v + 2], du[8 * v + 3]),
                               pack_bf16(du[8 * v + 4], du[8 * v + 5]), pack_bf16(du[8 * v + 6], du[8 * v + 7]));
        }
      }
    }
    if (NH == 1) {
      if (row_ok && p.dw_part) p.dw_part[row * p.dw_stride + c.n] = dwp;
    } else if (p.dw_part) {
      // the two halves' partials, combined in a fixed order: first half + second half
      const int lane = row_in_tile & 31;
      const uint32_t ph = *hand.phase;
      *hand.phase ^= 1u;
      if (half == 1) {
        if (!mbar_wait_bounded(&hand.empty[quarter], ph ^ 1, hand.abort_flag, p.status, WAIT_LIMIT_CYCLES))
          return false;
        hand.s_dw[row_in_tile] = dwp;
        __syncwarp();
        if (lane == 0) mbar_arrive(&hand.full[quarter]);
      } else {
        if (!mbar_wait_bounded(&hand.full[quarter], ph, hand.abort_flag, p.status, WAIT_LIMIT_CYCLES))
          return false;
        if (row_ok) p.dw_part[row * p.dw_stride + c.n] = dwp + hand.s_dw[row_in_tile];
        __syncwarp();
        if (lane == 0) mbar_arrive(&hand.empty[quarter]);
      }
    }
  }
  return true;
}

template <int SCHED, int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(gemm_threads(EPI), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t dw_full_bar[4];
  __shared__ __align__(8) uint64_t dw_empty_bar[4];
  __shared__ float s_dw[BM];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_ro[MAX_EXPERTS + 1];
  __shared__ int s_order[SCHED == SCHED_KGROUP ? MAX_EXPERTS : 1];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~static_cast<uintptr_t>(1023));

  // Without row_offsets the problem is one dense group: M rows (SCHED_ROWS) or a
  // K of p.K rows (SCHED_KGROUP, rows past the tensor's end read as zeros).
  const int E = p.row_offsets ? p.E : 1;
  const int dense_rows = (SCHED == SCHED_KGROUP) ? (p.K + BK - 1) / BK * BK : (p.M + BM - 1) / BM * BM;
  for (int i = threadIdx.x; i <= E; i += blockDim.x)
    s_ro[i] = p.row_offsets ? p.row_offsets[i] : (i == 0 ? 0 : dense_rows);
  bool snake = false;
  if (SCHED == SCHED_KGROUP) {
    __syncthreads();
    const int per = (p.M / BM) * (p.N / p.BN);
    snake = kgroup_order(s_ro, E, per, gridDim.x, s_order);  // complete at the barrier below
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull_bar[a], 1); mbar_init(&tempty_bar[a], epi_warps(EPI)); }
    mbar_init(&drain_bar, 1);
    for (int q = 0; q < 4; ++q) { mbar_init(&dw_full_bar[q], 1); mbar_init(&dw_empty_bar[q], 1); }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) { tma_prefetch_desc(&tmA); tma_prefetch_desc(&tmB); }
  if (warp == 1) { tmem_alloc(&s_tmem_base, TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;

  const int BN = p.BN;
  const int n_tiles = gu_split(EPI) ? p.N / (BN / 2) : p.N / BN;
  const int total = (SCHED == SCHED_ROWS) ? (s_ro[E] / BM) * n_tiles : E * (p.M / BM) * n_tiles;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t stage_tx = A_STAGE_BYTES + BN * BK * 2;
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int rnd = 0, tile = sched_tile(0, blockIdx.x, gridDim.x, snake); ok && tile < total;
           tile = sched_tile(++rnd, blockIdx.x, gridDim.x, snake)) {
        const TileCoord c = tile_coord<SCHED, EPI, B_MN>(p, s_ro, s_order, E, n_tiles, tile);
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_STAGE_BYTES;
          uint64_t* bar = &full_bar[stage];
          mbar_arrive_expect_tx(bar, stage_tx);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          const int k0 = kb * BK;
          if (!A_MN) {
            tma_load_2d(sa, &tmA, bar, c.a_k + k0, c.a_m);
          } else {
            tma_load_2d(sa, &tmA, bar, c.a_m, c.a_k + k0);
            tma_load_2d(sa + 8192, &tmA, bar, c.a_m + 64, c.a_k + k0);
          }
          if (!B_MN) {
            if (gu_split(EPI)) {
              tma_load_2d(sb, &tmB, bar, k0, c.b_n);
              tma_load_2d(sb + (BN / 2) * 128, &tmB, bar, k0, c.b_n + p.f);
            } else {
              tma_load_2d(sb, &tmB, bar, c.b_k + k0, c.b_n);
            }
          } else {
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(sb + i * 8192, &tmB, bar, c.b_n + 64 * i, c.b_k + k0);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // No bulk copy may still be writing shared memory when the CTA exits.
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u) mbar_drain(&full_bar[s], (armed_parity >> s) & 1u, WAIT_LIMIT_CYCLES);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, BN, A_MN ? 1 : 0, B_MN ? 1 : 0);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int rnd = 0, tile = sched_tile(0, blockIdx.x, gridDim.x, snake); ok && tile < total;
           tile = sched_tile(++rnd, blockIdx.x, gridDim.x, snake)) {
        const TileCoord c = tile_coord<SCHED, EPI, B_MN>(p, s_ro, s_order, E, n_tiles, tile);
        if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1, abort_flag, p.status,
                               WAIT_LIMIT_CYCLES)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_STRIDE;
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // K-major: the next 16 elements are 32 bytes further along the swizzled row.
            // MN-major: the next 16 K rows are 16 * 128 bytes further; MN atoms of 64
            // elements repeat every 8 KB (one TMA box), 8-row K groups every 1 KB.
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_f16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&empty_bar[stage]);  // frees the stage once these MMAs have read it
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&tfull_bar[acc]);      // accumulator ready for the epilogue
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      // Every MMA must be finished before TMEM is released.
      tc_commit(&drain_bar);
      mbar_drain(&drain_bar, 0, WAIT_LIMIT_CYCLES);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0, dw_phase = 0;
    const DwHandoff hand{s_dw, dw_full_bar, dw_empty_bar, &dw_phase, abort_flag};
    for (int rnd = 0, tile = sched_tile(0, blockIdx.x, gridDim.x, snake); tile < total;
         tile = sched_tile(++rnd, blockIdx.x, gridDim.x, snake)) {
      const TileCoord c = tile_coord<SCHED, EPI, B_MN>(p, s_ro, s_order, E, n_tiles, tile);
      if (!mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, p.status, WAIT_LIMIT_CYCLES))
        break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_STRIDE;
      const long long row = c.out_row + row_in_tile;
      const bool row_ok = row < p.row_limit;

      if (!tile_epilogue<EPI>(p, c, tbase, row, row_ok, BN, (warp - 2) >> 2, q, row_in_tile, hand)) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace moe
