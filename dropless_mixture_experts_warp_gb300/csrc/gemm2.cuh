// Persistent grouped GEMM over CTA pairs (tcgen05 cta_group::2, M = 256 per MMA).
//
// A cluster of two CTAs on neighbouring SMs computes one 256 x BN tile: each CTA
// holds 128 rows of A and half of B's BN rows in its shared memory and receives its
// 128 rows of the accumulator in its own TMEM.  Compared with the single-CTA kernel
// each SM stages half as many B bytes per FLOP, so a stage is 32 KB and six of them
// fit, which hides more load latency.
//   warp 0 (both CTAs)  TMA producer for this CTA's halves; completions are counted on
//                       the leader CTA's full barrier (.cta_group::2 loads)
//   warp 1 (leader)     issues the pair's MMAs; commits multicast to both CTAs
//   warps 2..           epilogue on this CTA's 128 accumulator rows (shared epilogue)
// Row tiles of the grouped (ragged-M) mode stay inside an expert: an expert with an
// odd number of 128-row tiles ends with a pair whose second half is discarded, so
// the epilogue never writes past the expert's segment.  For the gate/up GEMM the
// leader holds the gate rows and the peer the up rows of W_gu, so the accumulator's
// columns are [G | U] as in the single-CTA kernel.
#pragma once

#include "gemm.cuh"

namespace moe {

constexpr int P_STAGES = 6;  // at most; pair_stages(epi) per epilogue
constexpr int P_A_BYTES = BM * BK * 2;                // 16 KB
constexpr int P_B_BYTES_MAX = 128 * BK * 2;           // half of a 256-row B tile
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES_MAX;
// STORE runs eight epilogue warps (two per TMEM lane quarter, splitting the columns)
// that read their accumulator columns at once and write them through 2 KB staging
// buffers and tensor stores; the SwiGLU epilogues keep the shared epilogue's warp
// count (eight for SwiGLU', four for SwiGLU: measured faster than eight) and also
// write through staging boxes and tensor stores.
__host__ __device__ constexpr int pair_epi_warps(int epi) { return epi == 0 ? 8 : epi_warps(epi); }
__host__ __device__ constexpr int pair_threads(int epi) { return 64 + 32 * pair_epi_warps(epi); }
// Operand stages: six, five for SwiGLU' (whose warps also hold a G/U box).
__host__ __device__ constexpr int pair_stages(int epi) { return epi == 2 ? 5 : P_STAGES; }
// per epilogue warp: STORE 2 KB (staging box); SwiGLU 6 KB (its G, U and h boxes);
// SwiGLU' 6 KB (a dG/dU staging box and the 4 KB box of the saved G and U)
__host__ __device__ constexpr int pair_epi_bytes(int epi) { return epi == 0 ? 2048 : 6144; }
__host__ __device__ constexpr int p_smem_bytes(int epi) {
  return pair_stages(epi) * P_STAGE_BYTES + pair_epi_warps(epi) * pair_epi_bytes(epi) + 1024;
}

// A row coordinate past every tensor's rows: a tensor load there reads the zero fill.
constexpr int DEAD_ROW = 1 << 30;

struct PairTile {
  TileCoord c;
  long long row_end;  // rows at or beyond this are not stored
};

// s_pt[e]: first pair tile of expert e (SCHED_ROWS) or the experts in their visiting
// order (SCHED_KGROUP, kgroup_order); rank: 0 (leader) or 1; KB: K
// elements per stage.
template <int SCHED, int EPI, bool B_MN, int KB = BK>
__device__ __forceinline__ PairTile pair_tile(const GemmParams& p, const int* s_ro, const int* s_pt, int E,
                                              int n_tiles, int tile, int rank) {
  PairTile t;
  TileCoord& c = t.c;
  const int half_n = p.BN / 2;
  if (SCHED == SCHED_ROWS) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pt[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int local = tile - s_pt[e];
    const int mt2 = ((s_ro[e + 1] - s_ro[e]) / BM + 1) / 2;
    banded(local, mt2, n_tiles, rows_m_fastest(p.m_fastest, mt2, n_tiles), band_of(p, p.K), c.m, c.n);
    c.e = e;
    c.kblocks = p.K / KB;
    c.a_m = s_ro[e] + c.m * 2 * BM + rank * BM;
    c.a_k = 0;
    c.out_col = gu_split(EPI) ? c.n * half_n : c.n * p.BN;
    if (gu_split(EPI))  // leader: gate rows, peer: up rows
      c.b_n = e * p.b_rows_per_expert + c.out_col + rank * p.f;
    else
      c.b_n = (B_MN ? 0 : e * p.b_rows_per_expert) + c.out_col + rank * half_n;
    c.b_k = B_MN ? e * p.b_k_per_expert : 0;
    c.out_row = c.a_m;
    c.out_base = 0;
    t.row_end = s_ro[e + 1] < p.row_limit ? s_ro[e + 1] : p.row_limit;
  } else {
    const int mt2 = p.M / (2 * BM);
    const int per = mt2 * n_tiles;
    const int e = s_pt[tile / per];  // the experts in their visiting order
    const int local = tile - (tile / per) * per;
    if (p.m_fastest) { c.m = local % mt2; c.n = local / mt2; }
    else { c.n = local % n_tiles; c.m = local / n_tiles; }
    c.e = e;
    c.kblocks = (s_ro[e + 1] - s_ro[e]) / KB;
    c.a_m = c.m * 2 * BM + rank * BM;
    c.a_k = s_ro[e];
    c.out_col = c.n * p.BN;
    c.b_n = c.out_col + rank * half_n;
    c.b_k = s_ro[e];
    c.out_row = c.a_m;
    c.out_base = static_cast<long long>(e) * p.M * p.N;
    t.row_end = p.row_limit;
  }
  return t;
}

template <int SCHED, int EPI, bool A_MN, bool B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads(EPI), 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                             const GemmParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full_bar[P_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[P_STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t dw_full_bar[4];
  __shared__ __align__(8) uint64_t dw_empty_bar[4];
  __shared__ __align__(8) uint64_t gu_bar[EPI == EPI_SWIGLU_BWD ? 8 : 1];  // per epilogue warp
  __shared__ float s_dw[BM];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_ro[MAX_EXPERTS + 1];
  __shared__ int s_pt[MAX_EXPERTS + 1];
  constexpr int STAGES = pair_stages(EPI);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~static_cast<uintptr_t>(1023));

  const int E = p.row_offsets ? p.E : 1;
  const int dense_rows = (SCHED == SCHED_KGROUP) ? (p.K + BK - 1) / BK * BK : (p.M + BM - 1) / BM * BM;
  for (int i = threadIdx.x; i <= E; i += blockDim.x)
    s_ro[i] = p.row_offsets ? p.row_offsets[i] : (i == 0 ? 0 : dense_rows);
  const int BN = p.BN;  // 128 or 256
  const int n_tiles = gu_split(EPI) ? p.N / (BN / 2) : p.N / BN;
  __syncthreads();
  // SCHED_KGROUP: s_pt holds the experts in their visiting order (kgroup_order);
  // complete at the cluster barrier below
  const bool snake =
      SCHED == SCHED_KGROUP && kgroup_order(s_ro, E, (p.M / (2 * BM)) * n_tiles, npairs, s_pt);
  if (threadIdx.x == 0) {
    if (SCHED == SCHED_ROWS) {
      // pair tiles per expert, exclusive prefix (E <= 1024, once per launch)
      int run = 0;
      for (int e = 0; e < E; ++e) {
        s_pt[e] = run;
        run += ((s_ro[e + 1] - s_ro[e]) / BM + 1) / 2 * n_tiles;
      }
      s_pt[E] = run;
    }
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    if (EPI == EPI_SWIGLU_BWD)
      for (int w = 0; w < 8; ++w) mbar_init(&gu_bar[w], 1);
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull_bar[a], 1); mbar_init(&tempty_bar[a], 2 * pair_epi_warps(EPI)); }
    mbar_init(&drain_bar, 1);
    for (int q = 0; q < 4; ++q) { mbar_init(&dw_full_bar[q], 1); mbar_init(&dw_empty_bar[q], 1); }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    if (EPI == EPI_SWIGLU_FWD || EPI == EPI_SWIGLU_BWD) tma_prefetch_desc(&tmD);
  }
  if (warp == 1) { tmem_alloc_pair(&s_tmem_base, TMEM_COLS); tmem_relinquish_pair(); }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int total = (SCHED == SCHED_ROWS) ? s_pt[E] : E * (p.M / (2 * BM)) * n_tiles;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint32_t cta_tx = P_A_BYTES + (BN / 2) * BK * 2;
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int rnd = 0, tile = sched_tile(0, pair, npairs, snake); ok && tile < total;
           tile = sched_tile(++rnd, pair, npairs, snake)) {
        const PairTile t = pair_tile<SCHED, EPI, B_MN>(p, s_ro, s_pt, E, n_tiles, tile, rank);
        const TileCoord& c = t.c;
        for (int kb = 0; kb < c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          uint8_t* sa = smem + stage * P_STAGE_BYTES;
          uint8_t* sb = sa + P_A_BYTES;
          const uint32_t bar = mapa_shared(smem_u32(&full_bar[stage]), 0);  // the leader's
          if (rank == 0) {
            mbar_arrive_expect_tx(&full_bar[stage], 2 * cta_tx);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          const int k0 = kb * BK;
          if (!A_MN) {
            // The upper half of an expert's last pair tile when it has an odd number of 128-row
            // tiles lies past the expert's rows: its results are never stored, so it reads the
            // zero fill of rows beyond the tensor instead of the next expert's rows.
            const int a_row = (SCHED == SCHED_ROWS && c.a_m >= t.row_end) ? DEAD_ROW : c.a_m;
            tma_load_2d_pair(sa, &tmA, bar, c.a_k + k0, a_row);
          } else {
            tma_load_2d_pair(sa, &tmA, bar, c.a_m, c.a_k + k0);
            tma_load_2d_pair(sa + 8192, &tmA, bar, c.a_m + 64, c.a_k + k0);
          }
          if (!B_MN) {
            tma_load_2d_pair(sb, &tmB, bar, c.b_k + k0, c.b_n);
          } else {
            for (int i = 0; i < BN / 128; ++i)
              tma_load_2d_pair(sb + i * 8192, &tmB, bar, c.b_n + 64 * i, c.b_k + k0);
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
      const uint32_t idesc = idesc_bf16(2 * BM, BN, A_MN ? 1 : 0, B_MN ? 1 : 0);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int rnd = 0, tile = sched_tile(0, pair, npairs, snake); ok && tile < total;
           tile = sched_tile(++rnd, pair, npairs, snake)) {
        const PairTile t = pair_tile<SCHED, EPI, B_MN>(p, s_ro, s_pt, E, n_tiles, tile, 0);
        if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1, abort_flag, p.status, WAIT_LIMIT_CYCLES)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_STRIDE;
        for (int kb = 0; kb < t.c.kblocks; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, p.status,
                                 WAIT_LIMIT_CYCLES)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * P_STAGE_BYTES);
          const uint32_t sb = sa + P_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_f16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(&empty_bar[stage], 0x3);  // frees the stage in both CTAs
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair_mc(&tfull_bar[acc], 0x3);      // both halves of the accumulator ready
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
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
    const DwHandoff hand{s_dw, dw_full_bar, dw_empty_bar, &dw_phase, abort_flag};
    uint8_t* stg = smem + STAGES * P_STAGE_BYTES + (warp - 2) * pair_epi_bytes(EPI);
    uint32_t gu_phase = 0;
    bool gu_inflight = false;  // a G/U box load not yet waited for
    for (int rnd = 0, tile = sched_tile(0, pair, npairs, snake); tile < total;
         tile = sched_tile(++rnd, pair, npairs, snake)) {
      const PairTile t = pair_tile<SCHED, EPI, B_MN>(p, s_ro, s_pt, E, n_tiles, tile, rank);
      if (!mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, p.status, WAIT_LIMIT_CYCLES)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_STRIDE;
      const long long row = t.c.out_row + row_in_tile;
      if (EPI == EPI_STORE) {
        // this warp's half of the columns: read, release the accumulator, then store
        const int col0 = ((warp - 2) >> 2) * (BN / 2);
        uint32_t r[4][32];
        acc_load_chunks(tbase, col0, BN / 64, t.c.kblocks > 0, r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        if (t.c.out_row + q * 32 < t.row_end) {  // 32-row blocks never straddle an expert's end
          const long long y0 =
              (SCHED == SCHED_KGROUP ? static_cast<long long>(t.c.e) * p.M : 0ll) + t.c.out_row + q * 32;
          store_chunks_tma(&tmC, r, BN / 64, t.c.out_col + col0, static_cast<int>(y0), lane, stg);
        }
        continue;
      }
      if (EPI == EPI_SWIGLU_FWD) {
        // G | U (tmC) and h (tmD) through three 2 KB staging boxes and tensor stores: the
        // warp's 32 rows, h columns out_col + c0 .. + 31 (G at c0, U at BN / 2 + c0)
        const bool row_ok = row < t.row_end;
        const float w = !row_ok ? 0.0f : (p.w_rows ? p.w_rows[row] : 1.0f);
        const bool blk_ok = t.c.out_row + q * 32 < t.row_end;  // 32-row blocks never straddle it
        const int y0 = static_cast<int>(t.c.out_row + q * 32);
        for (int c0 = 0; c0 < BN / 2; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tbase + c0, g);
          tmem_ld32(tbase + BN / 2 + c0, u);
          tmem_wait_ld();
          float gv[32], uv[32], hv[32];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            gv[i] = __uint_as_float(g[i]);
            gv[i + 1] = __uint_as_float(g[i + 1]);
            uv[i] = __uint_as_float(u[i]);
            uv[i + 1] = __uint_as_float(u[i + 1]);
            const F2 h = swiglu_pair(F2{gv[i], gv[i + 1]}, F2{uv[i], uv[i + 1]}, F2{w, w});
            hv[i] = h.x;
            hv[i + 1] = h.y;
          }
          if (lane == 0) bulk_wait_read<0>();  // the previous chunk's stores have read the boxes
          __syncwarp();
          stage_row_bf16(stg, lane, gv);
          stage_row_bf16(stg + 2048, lane, uv);
          stage_row_bf16(stg + 4096, lane, hv);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && blk_ok) {
            tma_store_2d(&tmC, stg, t.c.out_col + c0, y0);
            tma_store_2d(&tmC, stg + 2048, p.f + t.c.out_col + c0, y0);
            tma_store_2d(&tmD, stg + 4096, t.c.out_col + c0, y0);
            bulk_commit();
          }
        }
      } else if (EPI == EPI_SWIGLU_BWD) {
        // dG then dU (tmC, a map of dG|dU) through the warp's 2 KB staging box and tensor
        // stores; the saved G and U of each 32-column chunk arrive one chunk ahead by
        // tensor loads (tmD, a map of G|U) in the warp's 4 KB G/U box, which keeps the
        // row-by-row reads off the L1 path; this warp takes half of the tile's h columns
        const bool row_ok = row < t.row_end;
        const float w = !row_ok ? 0.0f : (p.w_rows ? p.w_rows[row] : 1.0f);
        const bool blk_ok = t.c.out_row + q * 32 < t.row_end;
        const int y0 = static_cast<int>(t.c.out_row + q * 32);
        const int half = (warp - 2) >> 2;
        const int cb = half * (BN / 2);
        uint64_t* gbar = &gu_bar[warp - 2];
        uint8_t* gub = stg + 2048;
        const uint32_t grow = smem_u32(gub) + lane * 64;  // this lane's row of the G box
        const int sw = (lane >> 1) & 3;                     // 64-byte swizzle of the box
        if (lane == 0) {
          mbar_arrive_expect_tx(gbar, 4096);
          tma_load_2d(gub, &tmD, gbar, t.c.out_col + cb, y0);
          tma_load_2d(gub + 2048, &tmD, gbar, p.f + t.c.out_col + cb, y0);
        }
        gu_inflight = true;
        float dwp = 0.0f;
        bool ok = true;
        for (int c0 = cb; c0 < cb + BN / 2; c0 += 32) {
          if (!mbar_wait_bounded(gbar, gu_phase, abort_flag, p.status, WAIT_LIMIT_CYCLES)) { ok = false; break; }
          gu_phase ^= 1u;
          gu_inflight = false;
          GuChunk cur;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            cur.g[v] = ld_shared_v4(grow + ((v ^ sw) << 4));
            cur.u[v] = ld_shared_v4(grow + 2048 + ((v ^ sw) << 4));
          }
          __syncwarp();  // every lane has its rows: the box may be refilled
          if (c0 + 32 < cb + BN / 2) {
            if (lane == 0) {
              fence_proxy_async_smem();
              mbar_arrive_expect_tx(gbar, 4096);
              tma_load_2d(gub, &tmD, gbar, t.c.out_col + c0 + 32, y0);
              tma_load_2d(gub + 2048, &tmD, gbar, p.f + t.c.out_col + c0 + 32, y0);
            }
            gu_inflight = true;
          }
          uint32_t r[32];
          tmem_ld32(tbase + c0, r);
          tmem_wait_ld();
          float dg[32], du[32];
          dwp += swiglu_bwd_values(r, cur, w, dg, du);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (lane == 0) bulk_wait_read<0>();  // the previous store has read the box
            __syncwarp();
            stage_row_bf16(stg, lane, j == 0 ? dg : du);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && blk_ok) {
              tma_store_2d(&tmC, stg, (j == 0 ? 0 : p.f) + t.c.out_col + c0, y0);
              bulk_commit();
            }
          }
        }
        if (!ok) break;
        if (!dw_combine<2>(p, t.c, row, row_ok, half, q, row_in_tile, hand, dwp)) break;
      } else if (!tile_epilogue<EPI, pair_epi_warps(EPI) / 4>(p, t.c, tbase, row, row < t.row_end, BN,
                                                              (warp - 2) >> 2, q, row_in_tile, hand)) {
        break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if (EPI == EPI_SWIGLU_BWD && gu_inflight)  // a G/U load left by an aborted tile lands first
      mbar_drain(&gu_bar[warp - 2], gu_phase, WAIT_LIMIT_CYCLES);
    if (lane == 0) bulk_wait_all();  // tensor stores complete
  }

  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while the other may still signal its barriers
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace moe
