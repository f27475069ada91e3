// Persistent grouped GEMM with MXFP8 operands on tcgen05 (kind::mxf8f6f4.block_scale).
//
// Same roles and schedule as the bf16 kernel (gemm.cuh): warp 0 loads, warp 1 issues,
// the warps after them run the shared epilogue.  Differences:
//   * operands are E4M3 codes, both K-major, 128 codes (128 bytes) per stage row; B may
//     instead hold E2M1 codes (FP4 weights), packed two a byte in memory and spread by
//     the tensor load to the same 128 bytes a row in shared memory;
//   * each stage also has the E8M0 scale tiles of its A rows (512 B) and B rows
//     (512 B per 128 rows), fetched with contiguous bulk copies into a region after
//     the code stages; the MMA warp moves
//     them into TMEM with tcgen05.cp (32x128b, replicated to the four lane quarters)
//     and every MMA (K = 32) selects its byte of the scale words with the
//     scale-factor id of the instruction descriptor;
//   * TMEM holds one 256-column accumulator (BN = 256) or two of 128 (BN = 128) in
//     columns 0..255 and the scale factors of each stage from column 256 on.
#pragma once

#include "gemm.cuh"

namespace moe {

constexpr int MX_BK = 128;                                  // K elements (= bytes) per stage
constexpr int MX_A_BYTES = BM * MX_BK;                      // 16 KB
constexpr int MX_B_BYTES_MAX = 256 * MX_BK;                 // 32 KB
// The code stages share 192 KB: four of 48 KB for BN = 256, six of 32 KB for BN =
// 128 -- as many bytes in flight either way, which is what hides the load latency.
constexpr int MX_CODE_BYTES = 4 * (MX_A_BYTES + MX_B_BYTES_MAX);
constexpr int MX_MAX_STAGES = 6;
// scale tiles of stage s: SFA at MX_SF_OFF + s * MX_SF_STAGE, SFB (up to 2 tiles) 512 B after
constexpr int MX_SF_OFF = MX_CODE_BYTES;
constexpr int MX_SF_STAGE = 1536;
constexpr int MX_XBUF_OFF = MX_SF_OFF + MX_MAX_STAGES * MX_SF_STAGE;  // buffers of the epilogue warps
__host__ __device__ constexpr bool epi_quantises(int epi) { return epi == 3 || epi == 4; }
// Eight epilogue warps for every MX epilogue (two per TMEM lane quarter, splitting
// the columns); STORE reads its accumulator columns at once and releases them early.
__host__ __device__ constexpr int mx_epi_warps(int) { return 8; }
__host__ __device__ constexpr int mx_threads(int epi) { return 64 + 32 * mx_epi_warps(epi); }
// per epilogue warp: a transpose buffer (quantising epilogues) or a 2 KB staging
// buffer of the tensor store (EPI_STORE)
__host__ __device__ constexpr int mx_smem_bytes(int epi) {
  return MX_XBUF_OFF + (epi_quantises(epi) ? mx_epi_warps(epi) * XBUF_FLOATS * 4 : 0) +
         (epi == 0 ? mx_epi_warps(epi) * 2048 : 0) + 1024;
}
// Bytes a TMA load of one 128-element E2M1 row counts on its mbarrier: the 64 bytes of
// packed codes it moves, although the row spans 128 bytes of shared memory (each 8 bytes
// of codes followed by an 8-byte gap that the load leaves unwritten).
constexpr int MX_W4_TX_ROW_BYTES = 64;
constexpr int MX_SF_TMEM_COL = 256;                         // first scale-factor column
constexpr int MX_SF_COLS_PER_STAGE = 16;                    // 4 for A, up to 8 for B
// BN = 256 (four stages): the TMEM columns after the scale factors hold accumulator
// columns the SwiGLU epilogues have yet to process once they have released the
// accumulator (96 per epilogue warp of a lane quarter for SwiGLU', 64 for SwiGLU)
constexpr int MX_SPARE_COL = MX_SF_TMEM_COL + 4 * MX_SF_COLS_PER_STAGE;

template <int SCHED, int EPI>
__global__ void __launch_bounds__(mx_threads(EPI), 1)
    grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full_bar[MX_MAX_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[MX_MAX_STAGES];
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
  __shared__ __align__(8) uint64_t gu_bar[EPI == EPI_SWIGLU_BWD_MX ? 8 : 1];  // per epilogue warp

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~static_cast<uintptr_t>(1023));

  const int E = p.row_offsets ? p.E : 1;
  const int dense_rows =
      (SCHED == SCHED_KGROUP) ? (p.K + MX_BK - 1) / MX_BK * MX_BK : (p.M + BM - 1) / BM * BM;
  for (int i = threadIdx.x; i <= E; i += blockDim.x)
    s_ro[i] = p.row_offsets ? p.row_offsets[i] : (i == 0 ? 0 : dense_rows);
  bool snake = false;
  if (SCHED == SCHED_KGROUP) {
    __syncthreads();
    const int per = (p.M / BM) * (p.N / p.BN);
    snake = kgroup_order(s_ro, E, per, gridDim.x, s_order);  // complete at the barrier below
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < MX_MAX_STAGES; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    if (EPI == EPI_SWIGLU_BWD_MX)
      for (int w = 0; w < 8; ++w) mbar_init(&gu_bar[w], 1);
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull_bar[a], 1); mbar_init(&tempty_bar[a], mx_epi_warps(EPI)); }
    mbar_init(&drain_bar, 1);
    for (int q = 0; q < 4; ++q) { mbar_init(&dw_full_bar[q], 1); mbar_init(&dw_empty_bar[q], 1); }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (EPI == EPI_STORE || EPI == EPI_SWIGLU_BWD_MX) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) { tmem_alloc(&s_tmem_base, TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;

  const int BN = p.BN;                       // 128 or 256
  const int num_acc = BN <= 128 ? 2 : 1;
  const int stage_bytes = MX_A_BYTES + BN * MX_BK;
  // 4 or 6 operand stages; the SwiGLU' GEMM at BN = 256 keeps 3 and holds its warps'
  // G/U boxes in the fourth stage's memory
  const bool gu_boxes = EPI == EPI_SWIGLU_BWD_MX && BN == 256;
  const int stages = gu_boxes ? 3 : MX_CODE_BYTES / stage_bytes;
  const int n_tiles = gu_split(EPI) ? p.N / (BN / 2) : p.N / BN;
  const int total = (SCHED == SCHED_ROWS) ? (s_ro[E] / BM) * n_tiles : E * (p.M / BM) * n_tiles;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t b_row_tx = p.b_fmt == MX_FMT_E2M1 ? MX_W4_TX_ROW_BYTES : MX_BK;
      const uint32_t stage_tx = MX_A_BYTES + BN * b_row_tx + 512 + (BN / 128) * 512;
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int rnd = 0, tile = sched_tile(0, blockIdx.x, gridDim.x, snake); ok && tile < total;
           tile = sched_tile(++rnd, blockIdx.x, gridDim.x, snake)) {
        const TileCoord c = tile_coord<SCHED, EPI, false, MX_BK>(p, s_ro, s_order, E, n_tiles, tile);
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          uint8_t* sa = smem + stage * stage_bytes;
          uint8_t* sb = sa + MX_A_BYTES;
          uint8_t* sf = smem + MX_SF_OFF + stage * MX_SF_STAGE;
          uint64_t* bar = &full_bar[stage];
          mbar_arrive_expect_tx(bar, stage_tx);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          const int ka = c.a_k + kb * MX_BK;     // K index of A (and of B: b_k == a_k here)
          const int kbt = ka / MX_BK;
          tma_load_2d(sa, &tmA, bar, ka, c.a_m);
          bulk_load(sf,
                    p.sfa + (static_cast<size_t>(c.a_m / 128) * p.a_sf_ktiles + kbt) * 512, 512, bar);
          const int kbb = c.b_k + kb * MX_BK;
          const int kbtb = kbb / MX_BK;
          if (gu_split(EPI)) {                    // gate rows then up rows, 128 each
            tma_load_2d(sb, &tmB, bar, kbb, c.b_n);
            tma_load_2d(sb + (BN / 2) * MX_BK, &tmB, bar, kbb, c.b_n + p.f);
            bulk_load(sf + 512,
                      p.sfb + (static_cast<size_t>(c.b_n / 128) * p.b_sf_ktiles + kbtb) * 512, 512, bar);
            bulk_load(sf + 1024,
                      p.sfb + (static_cast<size_t>((c.b_n + p.f) / 128) * p.b_sf_ktiles + kbtb) * 512, 512,
                      bar);
          } else {
            tma_load_2d(sb, &tmB, bar, kbb, c.b_n);
            for (int i = 0; i < BN / 128; ++i)
              bulk_load(sf + 512 + 512 * i,
                        p.sfb + (static_cast<size_t>(c.b_n / 128 + i) * p.b_sf_ktiles + kbtb) * 512, 512, bar);
          }
          if (++stage == stages) { stage = 0; phase ^= 1; }
        }
      }
      for (int s = 0; s < stages; ++s)
        if ((armed >> s) & 1u) mbar_drain(&full_bar[s], (armed_parity >> s) & 1u, WAIT_LIMIT_CYCLES);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int rnd = 0, tile = sched_tile(0, blockIdx.x, gridDim.x, snake); ok && tile < total;
           tile = sched_tile(++rnd, blockIdx.x, gridDim.x, snake)) {
        const TileCoord c = tile_coord<SCHED, EPI, false, MX_BK>(p, s_ro, s_order, E, n_tiles, tile);
        if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1, abort_flag, p.status,
                               WAIT_LIMIT_CYCLES)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * stage_bytes);
          const uint32_t sb = sa + MX_A_BYTES;
          const uint32_t sf = smem_u32(smem + MX_SF_OFF + stage * MX_SF_STAGE);
          const uint32_t sfa_t = tmem_base + MX_SF_TMEM_COL + stage * MX_SF_COLS_PER_STAGE;
          const uint32_t sfb_t = sfa_t + 4;
          // scale tiles: 32 rows x 16 B each, 8-row core matrices 128 B apart
          tc_cp_32x128b_x4(sfa_t, smem_desc_plain(sf, 0, 128));
          for (int i = 0; i < BN / 128; ++i)
            tc_cp_32x128b_x4(sfb_t + 4 * i, smem_desc_plain(sf + 512 + 512 * i, 0, 128));
#pragma unroll
          for (int kk = 0; kk < MX_BK / 32; ++kk) {
            const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_mxf8(d_tmem, ad, bd, idesc_mxf8(BM, BN, kk, p.b_fmt), sfa_t, sfb_t, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == stages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&tfull_bar[acc]);
        if (++acc == num_acc) { acc = 0; acc_phase ^= 1; }
      }
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
    float* xbuf = reinterpret_cast<float*>(smem + MX_XBUF_OFF) + (warp - 2) * XBUF_FLOATS;
    uint8_t* stg = smem + MX_XBUF_OFF + (warp - 2) * 2048;
    const DwHandoff hand{s_dw, dw_full_bar, dw_empty_bar, &dw_phase, abort_flag, xbuf};
    uint32_t gu_phase = 0;
    bool gu_inflight = false;  // a G/U box load not yet waited for
    for (int rnd = 0, tile = sched_tile(0, blockIdx.x, gridDim.x, snake); tile < total;
         tile = sched_tile(++rnd, blockIdx.x, gridDim.x, snake)) {
      const TileCoord c = tile_coord<SCHED, EPI, false, MX_BK>(p, s_ro, s_order, E, n_tiles, tile);
      if (!mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, p.status, WAIT_LIMIT_CYCLES)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      const long long row = c.out_row + row_in_tile;
      if (EPI == EPI_STORE) {
        // this warp's half of the columns: read, release the accumulator, then store
        const int col0 = ((warp - 2) >> 2) * (BN / 2);
        uint32_t r[4][32];
        acc_load_chunks(tbase, col0, BN / 64, c.kblocks > 0, r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[acc]);
        if (++acc == num_acc) { acc = 0; acc_phase ^= 1; }
        // output rows: the padded row space (SCHED_ROWS) or expert e's block of M rows
        const long long y0 = (SCHED == SCHED_KGROUP ? static_cast<long long>(c.e) * p.M : 0ll) + c.out_row + q * 32;
        store_chunks_tma(&tmC, r, BN / 64, c.out_col + col0, static_cast<int>(y0), lane, stg);
        continue;
      }
      if (EPI == EPI_SWIGLU_FWD_MX) {
        // this warp's quarter of the h columns (BN / 4 = 64, two chunks; BN is 256 here):
        // the second chunk's G and U go to spare TMEM columns, the first chunk's stay in
        // registers, the accumulator is released, then the chunks are processed
        const bool row_ok = row < p.row_limit;
        const float w = !row_ok ? 0.0f : (p.w_rows ? p.w_rows[row] : 1.0f);
        const int half = (warp - 2) >> 2;
        const int cb = half * (BN / 4);
        const uint32_t sp = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + MX_SPARE_COL + half * 64;
        {
          uint32_t g1[32], u1[32];
          tmem_ld32(tbase + cb + 32, g1);
          tmem_ld32(tbase + BN / 2 + cb + 32, u1);
          tmem_wait_ld();
          tmem_st32(sp, g1);
          tmem_st32(sp + 32, u1);
        }
        uint32_t g0[32], u0[32];
        tmem_ld32(tbase + cb, g0);
        tmem_ld32(tbase + BN / 2 + cb, u0);
        tmem_wait_ld();
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[acc]);
        if (++acc == num_acc) { acc = 0; acc_phase ^= 1; }
        const long long rblk = row - lane;
        const bool blk_ok = __all_sync(0xffffffffu, row_ok);
        {
          FwdMxChunk f;
          fwd_mx_chunk(g0, u0, w, f);
          fwd_mx_store_chunk(p, row, row_ok, blk_ok, rblk, c.out_col + cb, lane, xbuf, f);
        }
        {
          uint32_t g1[32], u1[32];
          tmem_ld32(sp, g1);
          tmem_ld32(sp + 32, u1);
          tmem_wait_ld();
          FwdMxChunk f;
          fwd_mx_chunk(g1, u1, w, f);
          fwd_mx_store_chunk(p, row, row_ok, blk_ok, rblk, c.out_col + cb + 32, lane, xbuf, f);
        }
        continue;
      }
      if (EPI == EPI_SWIGLU_BWD_MX && BN == 256) {
        // this warp's 128 dH columns: three chunks go to spare TMEM columns, one stays in
        // registers, the accumulator is released, then the chunks are processed; the
        // saved G and U of each chunk arrive one chunk ahead by tensor loads (tmC, a map
        // of G|U) in the warp's 4 KB G/U box, which keeps the row-by-row reads off the
        // L1 path
        const int half = (warp - 2) >> 2;
        const int cb = half * 128;
        const bool row_ok = row < p.row_limit;
        const float w = !row_ok ? 0.0f : (p.w_rows ? p.w_rows[row] : 1.0f);
        const long long rblk = row - lane;
        const bool blk_ok = __all_sync(0xffffffffu, row_ok);
        const uint32_t spare = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + MX_SPARE_COL + half * 96;
        uint64_t* gbar = &gu_bar[warp - 2];
        uint8_t* gub = smem + 3 * stage_bytes + (warp - 2) * 4096;
        const uint32_t grow = smem_u32(gub) + lane * 64;  // this lane's row of the G box
        const int sw = (lane >> 1) & 3;                     // 64-byte swizzle of the box
        const int y0 = static_cast<int>(c.out_row + q * 32);
        auto gu_issue = [&](int col) {
          if (lane == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(gbar, 4096);
            tma_load_2d(gub, &tmC, gbar, col, y0);
            tma_load_2d(gub + 2048, &tmC, gbar, p.f + col, y0);
          }
          gu_inflight = true;
        };
        auto gu_take = [&](GuChunk& x) -> bool {
          if (!mbar_wait_bounded(gbar, gu_phase, abort_flag, p.status, WAIT_LIMIT_CYCLES)) return false;
          gu_phase ^= 1u;
          gu_inflight = false;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            x.g[v] = ld_shared_v4(grow + ((v ^ sw) << 4));
            x.u[v] = ld_shared_v4(grow + 2048 + ((v ^ sw) << 4));
          }
          __syncwarp();  // every lane has its rows: the box may be refilled
          return true;
        };
        gu_issue(c.out_col + cb + 96);  // the kept chunk's G and U, processed first
        uint32_t keep[32];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          uint32_t r[32];
          tmem_ld32(tbase + cb + 32 * i, r);
          tmem_wait_ld();
          tmem_st32(spare + 32 * i, r);
        }
        tmem_ld32(tbase + cb + 96, keep);
        tmem_wait_ld();
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[acc]);
        if (++acc == num_acc) { acc = 0; acc_phase ^= 1; }
        float dwp = 0.0f;
        bool ok;
        {
          GuChunk cur;
          ok = gu_take(cur);
          if (ok) {
            gu_issue(c.out_col + cb);
            bwd_mx_chunk(p, row, row_ok, blk_ok, w, c.out_col + cb + 96, keep, cur, dwp, xbuf, lane, rblk);
          }
        }
#pragma unroll 1
        for (int i = 0; ok && i < 3; ++i) {
          GuChunk cur;
          if (!gu_take(cur)) { ok = false; break; }
          if (i < 2) gu_issue(c.out_col + cb + 32 * (i + 1));
          uint32_t r[32];
          tmem_ld32(spare + 32 * i, r);
          tmem_wait_ld();
          bwd_mx_chunk(p, row, row_ok, blk_ok, w, c.out_col + cb + 32 * i, r, cur, dwp, xbuf, lane, rblk);
        }
        if (!ok) break;
        if (!dw_combine<2>(p, c, row, row_ok, half, q, row_in_tile, hand, dwp)) break;
        continue;
      }
      if (!tile_epilogue<EPI>(p, c, tbase, row, row < p.row_limit, BN, (warp - 2) >> 2, q, row_in_tile, hand))
        break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
      if (++acc == num_acc) { acc = 0; acc_phase ^= 1; }
    }
    if (EPI == EPI_SWIGLU_BWD_MX && gu_inflight)  // a G/U load left by an aborted tile lands first
      mbar_drain(&gu_bar[warp - 2], gu_phase, WAIT_LIMIT_CYCLES);
    if (EPI == EPI_STORE && lane == 0) bulk_wait_all();  // the tensor stores are complete
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace moe
