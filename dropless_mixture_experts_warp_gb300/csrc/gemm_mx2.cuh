// Persistent grouped GEMM with MXFP8 operands over CTA pairs (tcgen05 cta_group::2,
// kind::mxf8f6f4.block_scale, M = 256 per MMA).
//
// The pair schedule and roles are those of the bf16 pair kernel (gemm2.cuh): each
// CTA holds 128 rows of A and half of B's BN rows, so a stage is 32 KB of codes per
// CTA instead of 48 KB.  Scale tiles are fetched with tensor loads of two 256-byte
// rows (one 512-byte SF tile) so that both CTAs' bytes count on the leader's full
// barrier: each CTA fetches the tile of its own A rows and the tiles of all BN rows
// of B, and the leader's tcgen05.cp moves them into each CTA's TMEM.  The epilogue
// is the single-CTA MX kernel's on each CTA's 128 accumulator rows; rows of a pair
// half that lies beyond its expert's segment are neither stored nor quantised.
#pragma once

#include "gemm2.cuh"
#include "gemm_mx.cuh"

namespace moe {

constexpr int MXP_A_BYTES = BM * MX_BK;                      // 16 KB
constexpr int MXP_STAGE_BYTES = MXP_A_BYTES + 128 * MX_BK;   // + half of a 256-row B tile
constexpr int MXP_SF_STAGE = 1536;                           // SFA 512 B, SFB up to 1 KB
__host__ __device__ constexpr int mxp_stages(int epi) { return epi == 0 ? 6 : 5; }
__host__ __device__ constexpr int mxp_sf_off(int epi) { return mxp_stages(epi) * MXP_STAGE_BYTES; }
__host__ __device__ constexpr int mxp_epi_off(int epi) { return mxp_sf_off(epi) + mxp_stages(epi) * MXP_SF_STAGE; }
__host__ __device__ constexpr int mxp_smem_bytes(int epi) {
  return mxp_epi_off(epi) + (epi_quantises(epi) ? epi_warps(epi) * XBUF_FLOATS * 4 : 0) +
         (epi == 0 ? epi_warps(epi) * 4096 : 0) + 1024;
}

template <int SCHED, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gemm_threads(EPI), 1)
    grouped_gemm_mx_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                const __grid_constant__ CUtensorMap tmSFA,
                                const __grid_constant__ CUtensorMap tmSFB,
                                const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  constexpr int STAGES = mxp_stages(EPI);
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
  const int n_tiles = gu_split(EPI) ? p.N / (BN / 2) : p.N / BN;
  const int num_acc = BN <= 128 ? 2 : 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;  // pair tiles per expert, exclusive prefix
    for (int e = 0; e < E; ++e) {
      s_pt[e] = run;
      run += ((s_ro[e + 1] - s_ro[e]) / BM + 1) / 2 * n_tiles;
    }
    s_pt[E] = run;
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull_bar[a], 1); mbar_init(&tempty_bar[a], 2 * epi_warps(EPI)); }
    mbar_init(&drain_bar, 1);
    for (int q = 0; q < 4; ++q) { mbar_init(&dw_full_bar[q], 1); mbar_init(&dw_empty_bar[q], 1); }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSFA);
    tma_prefetch_desc(&tmSFB);
    if (EPI == EPI_STORE) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) { tmem_alloc_pair(&s_tmem_base, TMEM_COLS); tmem_relinquish_pair(); }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int total = (SCHED == SCHED_ROWS) ? s_pt[E] : E * (p.M / (2 * BM)) * n_tiles;
  volatile int* abort_flag = &s_abort;
  const int n_sfb = gu_split(EPI) ? 2 : BN / 128;  // SF tiles of the BN rows of B

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint32_t cta_tx = MXP_A_BYTES + (BN / 2) * MX_BK + 512 + n_sfb * 512;
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total; tile += npairs) {
        const PairTile t = pair_tile<SCHED, EPI, false, MX_BK>(p, s_ro, s_pt, E, n_tiles, tile, rank);
        const TileCoord& c = t.c;
        // first B row of the whole pair tile (gate rows for the split epilogue)
        const int b0 = gu_split(EPI) ? c.b_n - rank * p.f : c.b_n - rank * (BN / 2);
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          uint8_t* sa = smem + stage * MXP_STAGE_BYTES;
          uint8_t* sb = sa + MXP_A_BYTES;
          uint8_t* sf = smem + mxp_sf_off(EPI) + stage * MXP_SF_STAGE;
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
          if (gu_split(EPI)) {
            tma_load_2d_pair(sf + 512, &tmSFB, bar, 0, 2 * ((b0 / 128) * p.b_sf_ktiles + kbb / MX_BK));
            tma_load_2d_pair(sf + 1024, &tmSFB, bar, 0, 2 * (((b0 + p.f) / 128) * p.b_sf_ktiles + kbb / MX_BK));
          } else {
            for (int i = 0; i < n_sfb; ++i)
              tma_load_2d_pair(sf + 512 + 512 * i, &tmSFB, bar, 0,
                               2 * ((b0 / 128 + i) * p.b_sf_ktiles + kbb / MX_BK));
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (rank == 0)
        for (int s = 0; s < STAGES; ++s)
          if ((armed >> s) & 1u) mbar_drain(&full_bar[s], (armed_parity >> s) & 1u, WAIT_LIMIT_CYCLES);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && rank == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total; tile += npairs) {
        const PairTile t = pair_tile<SCHED, EPI, false, MX_BK>(p, s_ro, s_pt, E, n_tiles, tile, 0);
        if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1, abort_flag, p.status, WAIT_LIMIT_CYCLES)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < t.c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * MXP_STAGE_BYTES);
          const uint32_t sb = sa + MXP_A_BYTES;
          const uint32_t sf = smem_u32(smem + mxp_sf_off(EPI) + stage * MXP_SF_STAGE);
          const uint32_t sfa_t = tmem_base + MX_SF_TMEM_COL + stage * MX_SF_COLS_PER_STAGE;
          const uint32_t sfb_t = sfa_t + 4;
          tc_cp_32x128b_x4_pair(sfa_t, smem_desc_plain(sf, 0, 128));
          for (int i = 0; i < n_sfb; ++i)
            tc_cp_32x128b_x4_pair(sfb_t + 4 * i, smem_desc_plain(sf + 512 + 512 * i, 0, 128));
#pragma unroll
          for (int kk = 0; kk < MX_BK / 32; ++kk) {
            const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_mxf8_pair(d_tmem, ad, bd, idesc_mxf8(2 * BM, BN, kk), sfa_t, sfb_t, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(&empty_bar[stage], 0x3);  // frees the stage in both CTAs
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
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
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0, dw_phase = 0;
    float* xbuf = reinterpret_cast<float*>(smem + mxp_epi_off(EPI)) + (warp - 2) * XBUF_FLOATS;
    uint8_t* stg = smem + mxp_epi_off(EPI) + (warp - 2) * 4096;
    uint32_t nstore = 0;
    const DwHandoff hand{s_dw, dw_full_bar, dw_empty_bar, &dw_phase, abort_flag, xbuf};
    for (int tile = pair; tile < total; tile += npairs) {
      const PairTile t = pair_tile<SCHED, EPI, false, MX_BK>(p, s_ro, s_pt, E, n_tiles, tile, rank);
      if (!mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, p.status, WAIT_LIMIT_CYCLES)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      const long long row = t.c.out_row + row_in_tile;
      if (EPI == EPI_STORE) {
        if (t.c.out_row + q * 32 < t.row_end) {  // 32-row blocks never straddle row_end
          const long long y0 =
              (SCHED == SCHED_KGROUP ? static_cast<long long>(t.c.e) * p.M : 0ll) + t.c.out_row + q * 32;
          store_tile_tma(&tmC, t.c, tbase, BN, lane, static_cast<int>(y0), stg, nstore);
        }
      } else if (!tile_epilogue<EPI>(p, t.c, tbase, row, row < t.row_end, BN, (warp - 2) >> 2, q, row_in_tile,
                                     hand)) {
        break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
      if (++acc == num_acc) { acc = 0; acc_phase ^= 1; }
    }
    if (EPI == EPI_STORE && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while the other may still signal its barriers
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace moe
