// Persistent grouped GEMM with MXFP8 operands over CTA pairs (tcgen05 cta_group::2,
// kind::mxf8f6f4.block_scale, M = 256 per MMA), for the products with a plain bf16
// output (EPI_STORE); the layer runs its weight gradients on it (launch_gemm_mx).
//
// Across a pair each SM holds 128 rows of A and half of B's 256 rows, so per SM the operand
// bytes staged and read per FLOP drop by a third against the single-CTA kernel (M = 128,
// N = 256).  Measured on the weight gradients: +3 % (2048-row experts) to +11 % (1024-row
// experts); not on the row-scheduled products, where pair tiles waste odd half tiles.
//
// Roles and schedule are those of the bf16 pair kernel (gemm2.cuh): warp 0 of both CTAs
// loads this CTA's halves (completions counted on the leader's barriers), warp 1 of the
// leader issues the pair's MMAs and multicasts the commits, eight epilogue warps per CTA
// drain their 128 accumulator rows, hand the accumulator back as soon as they have read
// it (a CTA-scope arrive on the leader's barrier) and then store it through staging boxes
// and tensor stores.  Block scales: each CTA fetches, by tensor loads counted on the
// leader's barrier, the SF tile of its own 128 A rows and the SF tiles of all BN rows of
// B; the leader's pair copies (tcgen05.cp.cta_group::2) move each CTA's tiles into its own
// TMEM.  A copy's cost is per instruction, not per byte, and a third copy a stage cost this
// mainloop ~16 % (dense timing variants: 2.5 PFLOP/s with three, 2.9-3.2 with two or one, the
// same with one 4 KB 128x256b copy in place of two 32x128b.warpx4).  So where the producers of
// B left its SF tiles also in a replicated form (each 512-byte tile four times over: the weight
// gradients' B, x's and h's column-wise codes), both of a 256-row B tile's SF tiles arrive by
// two 2 KB tensor loads and go into all four TMEM lane quarters by one 128x256b copy.  TMEM holds one 256-column accumulator (two of 128 at BN = 128) in columns
// 0..255 and the scale factors of each stage from column 256 on.  B may be E2M1 (FP4
// weights) as in the single-CTA kernel.
#pragma once

#include "gemm2.cuh"
#include "gemm_mx.cuh"

namespace moe {

constexpr int MXP_A_BYTES = BM * MX_BK;                       // 16 KB
constexpr int MXP_STAGE_BYTES = MXP_A_BYTES + 128 * MX_BK;    // + half of a 256-row B tile
constexpr int MXP_STAGES = 5;
// SF tiles of a stage: SFA (512 B), then SFB: with p.sfb_rep each of B's two 128-row tiles in
// its replicated form (2 KB), else up to two plain tiles.
constexpr int MXP_SF_STAGE = 512 + 2 * SF_REP_TILE_BYTES;
constexpr int MXP_SF_OFF = MXP_STAGES * MXP_STAGE_BYTES;
constexpr int MXP_EPI_OFF = MXP_SF_OFF + MXP_STAGES * MXP_SF_STAGE;
constexpr int MXP_EPI_WARPS = 8;
constexpr int MXP_THREADS = 64 + 32 * MXP_EPI_WARPS;
constexpr int MXP_SMEM_BYTES = MXP_EPI_OFF + MXP_EPI_WARPS * 2048 + 1024;

template <int SCHED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MXP_THREADS, 1)
    grouped_gemm_mx_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                const __grid_constant__ CUtensorMap tmSFA,
                                const __grid_constant__ CUtensorMap tmSFB,
                                const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full_bar[MXP_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[MXP_STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_ro[MAX_EXPERTS + 1];
  __shared__ int s_pt[MAX_EXPERTS + 1];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~static_cast<uintptr_t>(1023));

  const int E = p.row_offsets ? p.E : 1;
  const int dense_rows =
      (SCHED == SCHED_KGROUP) ? (p.K + MX_BK - 1) / MX_BK * MX_BK : (p.M + BM - 1) / BM * BM;
  for (int i = threadIdx.x; i <= E; i += blockDim.x)
    s_ro[i] = p.row_offsets ? p.row_offsets[i] : (i == 0 ? 0 : dense_rows);
  const int BN = p.BN;  // 128 or 256
  const int n_tiles = p.N / BN;
  const int num_acc = BN <= 128 ? 2 : 1;
  __syncthreads();
  // SCHED_KGROUP: s_pt holds the experts in their visiting order (kgroup_order);
  // complete at the cluster barrier below
  const bool snake =
      SCHED == SCHED_KGROUP && kgroup_order(s_ro, E, (p.M / (2 * BM)) * n_tiles, npairs, s_pt);
  if (threadIdx.x == 0) {
    if (SCHED == SCHED_ROWS) {
      int run = 0;  // pair tiles per expert, exclusive prefix
      for (int e = 0; e < E; ++e) {
        s_pt[e] = run;
        run += ((s_ro[e + 1] - s_ro[e]) / BM + 1) / 2 * n_tiles;
      }
      s_pt[E] = run;
    }
    for (int s = 0; s < MXP_STAGES; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull_bar[a], 1); mbar_init(&tempty_bar[a], 2 * MXP_EPI_WARPS); }
    mbar_init(&drain_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSFA);
    tma_prefetch_desc(&tmSFB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) { tmem_alloc_pair(&s_tmem_base, TMEM_COLS); tmem_relinquish_pair(); }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int total = (SCHED == SCHED_ROWS) ? s_pt[E] : E * (p.M / (2 * BM)) * n_tiles;
  volatile int* abort_flag = &s_abort;
  const int n_sfb = BN / 128;  // SF tiles of the BN rows of B
  const bool sfb_rep = p.sfb_rep != 0 && n_sfb == 2;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint32_t b_row_tx = p.b_fmt == MX_FMT_E2M1 ? MX_W4_TX_ROW_BYTES : MX_BK;
      const uint32_t cta_tx = MXP_A_BYTES + (BN / 2) * b_row_tx + 512 + n_sfb * (sfb_rep ? SF_REP_TILE_BYTES : 512);
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int rnd = 0, tile = sched_tile(0, pair, npairs, snake); ok && tile < total;
           tile = sched_tile(++rnd, pair, npairs, snake)) {
        const PairTile t = pair_tile<SCHED, EPI_STORE, false, MX_BK>(p, s_ro, s_pt, E, n_tiles, tile, rank);
        const TileCoord& c = t.c;
        const int b0 = c.b_n - rank * (BN / 2);  // first B row of the whole pair tile
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          uint8_t* sa = smem + stage * MXP_STAGE_BYTES;
          uint8_t* sb = sa + MXP_A_BYTES;
          uint8_t* sf = smem + MXP_SF_OFF + stage * MXP_SF_STAGE;
          const uint32_t bar = mapa_shared(smem_u32(&full_bar[stage]), 0);  // the leader's
          if (rank == 0) {
            mbar_arrive_expect_tx(&full_bar[stage], 2 * cta_tx);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          const int ka = c.a_k + kb * MX_BK;
          const int kbb = c.b_k + kb * MX_BK;
          tma_load_2d_pair(sa, &tmA, bar, ka, c.a_m);
          tma_load_2d_pair(sb, &tmB, bar, kbb, c.b_n);
          // SF tile (r / 128, k / 128) is rows 2t, 2t + 1 of the [bytes / 256][256] view
          tma_load_2d_pair(sf, &tmSFA, bar, 0, 2 * ((c.a_m / 128) * p.a_sf_ktiles + ka / MX_BK));
          // SF tile (r / 128, k / 128) is rows 2t, 2t + 1 (replicated: rows 8t .. 8t + 7) of its view
          for (int i = 0; i < n_sfb; ++i) {
            const int t_sf = (b0 / 128 + i) * p.b_sf_ktiles + kbb / MX_BK;
            if (sfb_rep) tma_load_2d_pair(sf + 512 + SF_REP_TILE_BYTES * i, &tmSFB, bar, 0, 8 * t_sf);
            else tma_load_2d_pair(sf + 512 + 512 * i, &tmSFB, bar, 0, 2 * t_sf);
          }
          if (++stage == MXP_STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (rank == 0)
        for (int s = 0; s < MXP_STAGES; ++s)
          if ((armed >> s) & 1u) mbar_drain(&full_bar[s], (armed_parity >> s) & 1u, WAIT_LIMIT_CYCLES);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && rank == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int rnd = 0, tile = sched_tile(0, pair, npairs, snake); ok && tile < total;
           tile = sched_tile(++rnd, pair, npairs, snake)) {
        const PairTile t = pair_tile<SCHED, EPI_STORE, false, MX_BK>(p, s_ro, s_pt, E, n_tiles, tile, 0);
        if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1, abort_flag, p.status, WAIT_LIMIT_CYCLES)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < t.c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * MXP_STAGE_BYTES);
          const uint32_t sb = sa + MXP_A_BYTES;
          const uint32_t sf = smem_u32(smem + MXP_SF_OFF + stage * MXP_SF_STAGE);
          const uint32_t sfa_t = tmem_base + MX_SF_TMEM_COL + stage * MX_SF_COLS_PER_STAGE;
          const uint32_t sfb_t = sfa_t + 4;
          // scale tiles: 32 rows x 16 B each, 8-row core matrices 128 B apart
          tc_cp_32x128b_x4_pair(sfa_t, smem_desc_plain(sf, 0, 128));
          if (sfb_rep)  // row r of both tiles: 16 bytes at sf + 512 + 16 r and 2048 bytes on
            tc_cp_128x256b_pair(sfb_t, smem_desc_plain(sf + 512, SF_REP_TILE_BYTES, 128));
          else
            for (int i = 0; i < n_sfb; ++i)
              tc_cp_32x128b_x4_pair(sfb_t + 4 * i, smem_desc_plain(sf + 512 + 512 * i, 0, 128));
#pragma unroll
          for (int kk = 0; kk < MX_BK / 32; ++kk) {
            const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_mxf8_pair(d_tmem, ad, bd, idesc_mxf8(2 * BM, BN, kk, p.b_fmt), sfa_t, sfb_t,
                             (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(&empty_bar[stage], 0x3);  // frees the stage in both CTAs
          if (++stage == MXP_STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair_mc(&tfull_bar[acc], 0x3);      // both halves of the accumulator ready
        if (++acc == num_acc) { acc = 0; acc_phase ^= 1; }
      }
      tc_commit_pair(&drain_bar);
      mbar_drain(&drain_bar, 0, WAIT_LIMIT_CYCLES);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint8_t* stg = smem + MXP_EPI_OFF + (warp - 2) * 2048;
    for (int rnd = 0, tile = sched_tile(0, pair, npairs, snake); tile < total;
         tile = sched_tile(++rnd, pair, npairs, snake)) {
      const PairTile t = pair_tile<SCHED, EPI_STORE, false, MX_BK>(p, s_ro, s_pt, E, n_tiles, tile, rank);
      if (!mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, p.status, WAIT_LIMIT_CYCLES)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      // this warp's half of the columns: read, hand the accumulator back, then store
      const int col0 = ((warp - 2) >> 2) * (BN / 2);
      uint32_t r[4][32];
      acc_load_chunks(tbase, col0, BN / 64, t.c.kblocks > 0, r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
      if (++acc == num_acc) { acc = 0; acc_phase ^= 1; }
      if (t.c.out_row + q * 32 < t.row_end) {  // 32-row blocks never straddle an expert's end
        const long long y0 =
            (SCHED == SCHED_KGROUP ? static_cast<long long>(t.c.e) * p.M : 0ll) + t.c.out_row + q * 32;
        store_chunks_tma(&tmC, r, BN / 64, t.c.out_col + col0, static_cast<int>(y0), lane, stg);
      }
    }
    if (lane == 0) bulk_wait_all();  // tensor stores complete
  }

  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while the other may still signal its barriers
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace moe
