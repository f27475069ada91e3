// Routing (top-k, weights, per-expert counts, padded offsets), dispatch (permute),
// combine and their backward passes.  All are HBM- or latency-bound; every global
// access of a token row is a 16-byte vector, a warp reading or writing one row.
#include "kernels.h"

namespace moe {

// ============================================================================ route

// Order-preserving map of a finite fp32 (or -inf) to a nonzero uint32: a > b as
// floats iff key(a) > key(b); -0 is taken as +0 so that the two tie.  0 = no candidate.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// One block owns ROUTE_TOKENS consecutive tokens; each warp takes ROUTE_TOKENS / 8
// of them, one at a time, with the E logits spread over the lanes (PL per lane,
// expert lane + 32 c in slot c).  Selection is k rounds of a warp argmax: the
// largest order key over the warp (one redux), then the lowest expert index among
// the lanes holding it (a second redux), so ties go to the lower expert index.
// Per-block stable ranks come from a bitmask per expert over the block's tokens:
// rank of token t for expert e = number of set bits below t.  The last block to
// finish turns the per-block counts into split_sizes, offsets and row_offsets.
// GROUPED: the group-limited sigmoid router -- selection on c = sigmoid(l) + bias
// (fp32); a group's score is the sum of its two largest c; the topk_group best groups
// (ties to the lower group) are eligible; weights routed_scale * s / sum of the k s.
template <int PL, bool GROUPED>
__global__ void __launch_bounds__(256) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, int score, GroupedRoute gr,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ block_hist,
    int32_t* __restrict__ block_base, int32_t* __restrict__ local_rank, int32_t* __restrict__ counter,
    int32_t* __restrict__ split_sizes, int32_t* __restrict__ offsets, int32_t* __restrict__ row_offsets,
    int32_t* __restrict__ status) {
  extern __shared__ uint32_t masks[];  // [E][ROUTE_TOKENS / 32], then the E totals of the last block
  __shared__ int s_last;
  constexpr int WORDS = ROUTE_TOKENS / 32;
  constexpr int TPW = ROUTE_TOKENS / 8;  // tokens per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tok0 = blockIdx.x * ROUTE_TOKENS;

  for (int i = threadIdx.x; i < E * WORDS; i += blockDim.x) masks[i] = 0u;
  __syncthreads();

  // GROUPED: the group of each of this lane's expert slots (fixed for the launch)
  int grp[PL];
#pragma unroll
  for (int c = 0; c < PL; ++c) grp[c] = GROUPED ? (lane + 32 * c) / (E / gr.n_group) : 0;

  for (int i = 0; i < TPW; ++i) {
    const int tl = warp * TPW + i;
    const int t = tok0 + tl;
    if (t >= T) break;
    const float* row = logits + static_cast<long long>(t) * E;
    uint32_t key[PL];
    float sv[PL];  // GROUPED: the sigmoid scores
#pragma unroll
    for (int c = 0; c < PL; ++c) {
      const int e = lane + 32 * c;
      if (GROUPED) {
        sv[c] = e < E ? 1.0f / (1.0f + expf(-row[e])) : 0.0f;
        key[c] = e < E ? order_key(sv[c] + (gr.bias ? gr.bias[e] : 0.0f)) : 0u;
      } else {
        key[c] = e < E ? order_key(row[e]) : 0u;
      }
    }
    if (GROUPED) {
      // group scores (lane g keeps group g's), then the topk_group best groups
      float my_gscore = 0.0f;
      for (int g = 0; g < gr.n_group; ++g) {
        uint32_t b1 = 0u, b2 = 0u;  // this lane's two best keys in group g
#pragma unroll
        for (int c = 0; c < PL; ++c) {
          if (lane + 32 * c < E && grp[c] == g) {
            if (key[c] > b1) { b2 = b1; b1 = key[c]; } else if (key[c] > b2) { b2 = key[c]; }
          }
        }
        const uint32_t m1 = __reduce_max_sync(0xffffffffu, b1);
        const int own = __reduce_min_sync(0xffffffffu, (b1 == m1 && b1 != 0u) ? lane : 32);
        const uint32_t m2 = __reduce_max_sync(0xffffffffu, lane == own ? b2 : b1);
        if (lane == g) my_gscore = key_value(m1) + key_value(m2);
      }
      uint32_t gkey = lane < gr.n_group ? order_key(my_gscore) : 0u;
      uint32_t chosen = 0u;
      for (int r = 0; r < gr.topk_group; ++r) {
        const uint32_t wk = __reduce_max_sync(0xffffffffu, gkey);
        const int wg = __reduce_min_sync(0xffffffffu, (gkey == wk && gkey != 0u) ? lane : 32);
        chosen |= 1u << (wg & 31);
        if (lane == wg) gkey = 0u;
      }
#pragma unroll
      for (int c = 0; c < PL; ++c) {
        if (lane + 32 * c < E && !((chosen >> grp[c]) & 1u)) key[c] = 0u;
      }
    }
    int my_e = -1;
    float my_l = 0.0f;
    for (int j = 0; j < k; ++j) {
      // this lane's best remaining slot: strict > keeps the lowest slot (lowest index) on ties
      uint32_t bk = 0u;
      int bc = 0;
#pragma unroll
      for (int c = 0; c < PL; ++c)
        if (key[c] > bk) { bk = key[c]; bc = c; }
      const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
      const int cand = (bk == wk && bk != 0u) ? lane + 32 * bc : 0x7fffffff;
      const int we = __reduce_min_sync(0xffffffffu, cand);
      if (we == cand && cand != 0x7fffffff) {
#pragma unroll
        for (int c = 0; c < PL; ++c)
          if (c == bc) key[c] = 0u;  // taken
      }
      if (GROUPED) {
        float bs = 0.0f;  // the owner lane's sigmoid score of the chosen expert
#pragma unroll
        for (int c = 0; c < PL; ++c)
          if (c == bc) bs = sv[c];
        const float ws = __shfl_sync(0xffffffffu, bs, we & 31);
        if (lane == j) { my_e = we; my_l = ws; }
      } else if (lane == j) {
        my_e = we;
        my_l = key_value(wk);
      }
    }
    // weights of the selected experts, lanes 0..k-1
    const float top = __shfl_sync(0xffffffffu, my_l, 0);  // slot 0 holds the largest logit
    float s = 0.0f;
    if (lane < k) {
      if (GROUPED) s = my_l;  // already the sigmoid score
      else s = (score == MOE_SCORE_SOFTMAX) ? expf(my_l - top) : 1.0f / (1.0f + expf(-my_l));
    }
    float tot = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    if (lane < k) {
      topk_idx[static_cast<long long>(t) * k + lane] = my_e;
      topk_w[static_cast<long long>(t) * k + lane] = GROUPED ? gr.scale * s / tot : s / tot;
      atomicOr(&masks[my_e * WORDS + (tl >> 5)], 1u << (tl & 31));
    }
  }
  __syncthreads();

  // stable rank inside the block, and the block's histogram
  const int ntok = min(ROUTE_TOKENS, T - tok0);
  for (int pidx = threadIdx.x; pidx < ntok * k; pidx += blockDim.x) {
    const int tl = pidx / k;
    const long long gi = static_cast<long long>(tok0) * k + pidx;
    const int e = topk_idx[gi];
    const uint32_t* m = masks + e * WORDS;
    int r = __popc(m[tl >> 5] & ((1u << (tl & 31)) - 1u));
    for (int w = 0; w < (tl >> 5); ++w) r += __popc(m[w]);
    local_rank[gi] = r;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int cnt = 0;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) cnt += __popc(masks[e * WORDS + w]);
    block_hist[static_cast<long long>(blockIdx.x) * E + e] = cnt;
  }

  // last block: per-expert exclusive scan over blocks, then over experts
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counter, 1) == static_cast<int>(gridDim.x) - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int nb = gridDim.x;
  int* s_tot = reinterpret_cast<int*>(masks);  // the masks are no longer needed
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0, b = 0;
    for (; b + 16 <= nb; b += 16) {  // 16 loads in flight per thread
      int h[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = __ldcg(&block_hist[static_cast<long long>(b + i) * E + e]);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        block_base[static_cast<long long>(b + i) * E + e] = run;
        run += h[i];
      }
    }
    for (; b < nb; ++b) {
      block_base[static_cast<long long>(b) * E + e] = run;
      run += __ldcg(&block_hist[static_cast<long long>(b) * E + e]);
    }
    split_sizes[e] = run;
    s_tot[e] = run;
  }
  __syncthreads();
  if (warp == 0) {
    // lane l owns experts [l * per, (l + 1) * per): local sums, warp exclusive scan, write
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    long long cnt = 0, pad = 0;
    for (int e = e0; e < e1; ++e) {
      cnt += s_tot[e];
      pad += (s_tot[e] + ROW_ALIGN - 1) / ROW_ALIGN * ROW_ALIGN;
    }
    long long ic = cnt, ip = pad;  // inclusive scans
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long oc = __shfl_up_sync(0xffffffffu, ic, off);
      const long long op = __shfl_up_sync(0xffffffffu, ip, off);
      if (lane >= off) { ic += oc; ip += op; }
    }
    long long off = ic - cnt, roff = ip - pad;
    for (int e = e0; e < e1; ++e) {
      offsets[e] = static_cast<int32_t>(off);
      row_offsets[e] = static_cast<int32_t>(roff);
      off += s_tot[e];
      roff += (s_tot[e] + ROW_ALIGN - 1) / ROW_ALIGN * ROW_ALIGN;
    }
    if (lane == 31) {
      offsets[E] = static_cast<int32_t>(ic);
      row_offsets[E] = static_cast<int32_t>(ip);
      if (ic != static_cast<long long>(T) * k) set_status(status, MOE_ERR_INVARIANT);
      *counter = 0;
    }
  }
}

// ============================================================================ permute

// Warp per token: read x[t] once (16-byte vectors), write it to its k rows.  Blocks
// past the token blocks zero the padding rows of one expert each.
template <bool FROM_ROUTE>
__global__ void __launch_bounds__(256) scatter_rows_kernel(
    const uint4* __restrict__ src, int T, int d8, int E, int k, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_w, const int32_t* __restrict__ split_sizes,
    const int32_t* __restrict__ row_offsets, const int32_t* __restrict__ block_base,
    const int32_t* __restrict__ local_rank, uint4* __restrict__ dst,
    int32_t* __restrict__ row_to_token, int32_t* __restrict__ token_to_row,
    float* __restrict__ w_rows, int token_blocks, int rows_cap, int32_t* __restrict__ status) {
  __shared__ int s_rows[8][32];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  if (static_cast<int>(blockIdx.x) < token_blocks) {
    const int t = blockIdx.x * 8 + wib;
    if (t >= T) return;
    if (lane < k) {
      const long long gi = static_cast<long long>(t) * k + lane;
      int r;
      if (FROM_ROUTE) {
        const int e = topk_idx[gi];
        r = row_offsets[e] + block_base[static_cast<long long>(t / ROUTE_TOKENS) * E + e] +
            local_rank[gi];
        if (r < 0 || r >= rows_cap) {  // cannot happen unless the routing scratch is stale
          set_status(status, MOE_ERR_INVARIANT);
          r = -1;
        } else {
          row_to_token[r] = t;
          w_rows[r] = topk_w[gi];
        }
        token_to_row[gi] = r;
      } else {
        r = token_to_row[gi];
        if (r < 0 || r >= rows_cap) r = -1;
      }
      s_rows[wib][lane] = r;
    }
    __syncwarp();
    const uint4* s = src + static_cast<long long>(t) * d8;
    for (int c = lane; c < d8; c += 32) {
      const uint4 v = s[c];
      for (int j = 0; j < k; ++j) {
        const int r = s_rows[wib][j];
        if (r >= 0) dst[static_cast<long long>(r) * d8 + c] = v;
      }
    }
  } else {
    const int e = blockIdx.x - token_blocks;
    const int r0 = max(0, row_offsets[e] + split_sizes[e]);
    const int r1 = min(rows_cap, row_offsets[e + 1]);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (long long i = threadIdx.x; i < static_cast<long long>(r1 - r0) * d8; i += blockDim.x)
      dst[static_cast<long long>(r0) * d8 + i] = z;
    if (FROM_ROUTE) {
      for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        row_to_token[r] = -1;
        w_rows[r] = 0.0f;
      }
    }
  }
}

// ============================================================================ combine

// Warp per token: out[t] = sum_j rows[token_to_row[t][j]] (+ shared[t]) in fp32,
// slot order, one rounding to bf16.
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ rows, int T, int d8,
                                                      int k, const int32_t* __restrict__ token_to_row,
                                                      const uint4* __restrict__ shared,
                                                      uint4* __restrict__ out, int rows_cap) {
  __shared__ int s_rows[8][32];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + wib;
  if (t >= T) return;
  if (lane < k) {
    const int r = token_to_row[static_cast<long long>(t) * k + lane];
    s_rows[wib][lane] = (r >= 0 && r < rows_cap) ? r : -1;
  }
  __syncwarp();
  for (int c = lane; c < d8; c += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int r = s_rows[wib][j];
      if (r < 0) continue;
      const uint4 v = rows[static_cast<long long>(r) * d8 + c];
      acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x);
      acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
      acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z);
      acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
    }
    if (shared) {
      const uint4 v = shared[static_cast<long long>(t) * d8 + c];
      acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x);
      acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
      acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z);
      acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
    }
    out[static_cast<long long>(t) * d8 + c] =
        make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]),
                   pack_bf16(acc[4], acc[5]), pack_bf16(acc[6], acc[7]));
  }
}

// ============================================================================ backward

// dw_rows[r] = sum over N tiles of the per-tile partials, fixed order.
__global__ void dw_reduce_kernel(const float* __restrict__ part, int stride,
                                 const int32_t* __restrict__ row_offsets, int E,
                                 float* __restrict__ dw_rows, int rows_cap) {
  const int nrows = min(row_offsets[E], rows_cap);
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < nrows; r += gridDim.x * blockDim.x) {
    float s = 0.0f;
    for (int i = 0; i < stride; ++i) s += part[static_cast<long long>(r) * stride + i];
    dw_rows[r] = s;
  }
}

// Warp per token.  c = sum_j w_j dw_j;  softmax: dl_j = w_j (dw_j - c);
// sigmoid: dl_j = (dw_j - c) / sum_j s_j * s_j (1 - s_j).  Other experts get 0.
__global__ void __launch_bounds__(256) route_bwd_kernel(
    const float* __restrict__ logits, int T, int E, int k, int score,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
    const float* __restrict__ dw_rows, const int32_t* __restrict__ token_to_row,
    float* __restrict__ d_logits, int rows_cap, float scale) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const long long base = static_cast<long long>(t) * k;
  int e = 0;
  float w = 0.0f, dw = 0.0f, s = 0.0f;
  if (lane < k) {
    e = topk_idx[base + lane];
    w = topk_w[base + lane];
    const int r = token_to_row[base + lane];
    dw = (r >= 0 && r < rows_cap) ? dw_rows[r] : 0.0f;
    if (score == MOE_SCORE_SIGMOID) s = 1.0f / (1.0f + expf(-logits[static_cast<long long>(t) * E + e]));
  }
  float c = w * dw, z = s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    c += __shfl_xor_sync(0xffffffffu, c, off);
    z += __shfl_xor_sync(0xffffffffu, z, off);
  }
  float* out = d_logits + static_cast<long long>(t) * E;
  for (int i = lane; i < E; i += 32) out[i] = 0.0f;
  __syncwarp();
  if (lane < k) {
    // sigmoid weights w = scale * s_j / z: dL/ds_i = (scale dw_i - sum w dw) / z
    const float g = (score == MOE_SCORE_SOFTMAX) ? w * (dw - c) : (scale * dw - c) / z * s * (1.0f - s);
    out[e] = g;
  }
}

// ============================================================================ launchers

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int score, int32_t* topk_idx,
                              float* topk_w, int32_t* split_sizes, int32_t* offsets,
                              int32_t* row_offsets, const RouteScratch& ws, int32_t* status,
                              cudaStream_t stream, const GroupedRoute* grouped) {
  const int nb = route_blocks(T);
  cudaError_t err = cudaMemsetAsync(ws.counter, 0, sizeof(int32_t), stream);
  if (err != cudaSuccess) return err;
  // the masks [E][ROUTE_TOKENS / 32] and, in the last block, the E totals
  const size_t smem = static_cast<size_t>(E) * (ROUTE_TOKENS / 32 > 1 ? ROUTE_TOKENS / 32 : 1) * sizeof(uint32_t);
  GroupedRoute gr{};
  if (grouped) gr = *grouped;
#define MOE_ROUTE_PICK(G)                                                                                   \
  (E <= 32 ? route_topk_kernel<1, G> : E <= 64 ? route_topk_kernel<2, G> : E <= 128 ? route_topk_kernel<4, G> \
   : E <= 256 ? route_topk_kernel<8, G> : E <= 512 ? route_topk_kernel<16, G> : route_topk_kernel<32, G>)
  auto kern = grouped ? MOE_ROUTE_PICK(true) : MOE_ROUTE_PICK(false);
#undef MOE_ROUTE_PICK
  kern<<<nb, 256, smem, stream>>>(logits, T, E, k, score, gr, topk_idx, topk_w, ws.block_hist, ws.block_base,
                                  ws.local_rank, ws.counter, split_sizes, offsets, row_offsets, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_permute(const void* x, int T, int d, int E, int k, const int32_t* topk_idx,
                           const float* topk_w, const int32_t* split_sizes, const int32_t* row_offsets,
                           const RouteScratch& ws, void* xp, int32_t* row_to_token,
                           int32_t* token_to_row, float* w_rows, int rows_cap, int32_t* status,
                           cudaStream_t stream) {
  const int token_blocks = (T + 7) / 8;
  const int grid = token_blocks + E;
  scatter_rows_kernel<true><<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(x), T, d / 8, E, k, topk_idx, topk_w, split_sizes, row_offsets,
      ws.block_base, ws.local_rank, static_cast<uint4*>(xp), row_to_token, token_to_row, w_rows,
      token_blocks, rows_cap, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const void* dy, int T, int d, int E, int k, const int32_t* token_to_row,
                               const int32_t* split_sizes, const int32_t* row_offsets, void* dy_rows,
                               int rows_cap, cudaStream_t stream) {
  const int token_blocks = (T + 7) / 8;
  const int grid = token_blocks + E;
  scatter_rows_kernel<false><<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(dy), T, d / 8, E, k, nullptr, nullptr, split_sizes, row_offsets,
      nullptr, nullptr, static_cast<uint4*>(dy_rows), nullptr, const_cast<int32_t*>(token_to_row),
      nullptr, token_blocks, rows_cap, nullptr);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* rows, int T, int d, int k, const int32_t* token_to_row,
                           const void* shared, void* out, int rows_cap, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  combine_kernel<<<(T + 7) / 8, 256, 0, stream>>>(static_cast<const uint4*>(rows), T, d / 8, k,
                                                  token_to_row, static_cast<const uint4*>(shared),
                                                  static_cast<uint4*>(out), rows_cap);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_dw_reduce(const float* part, int stride, const int32_t* row_offsets, int E,
                             float* dw_rows, int max_rows, cudaStream_t stream) {
  const int grid = max(1, min((max_rows + 255) / 256, 4 * num_sms()));
  dw_reduce_kernel<<<grid, 256, 0, stream>>>(part, stride, row_offsets, E, dw_rows, max_rows);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_route_bwd(const float* logits, int T, int E, int k, int score,
                             const int32_t* topk_idx, const float* topk_w, const float* dw_rows,
                             const int32_t* token_to_row, float* d_logits, int rows_cap,
                             cudaStream_t stream, float scale) {
  if (T == 0) return cudaSuccess;
  route_bwd_kernel<<<(T + 7) / 8, 256, 0, stream>>>(logits, T, E, k, score, topk_idx, topk_w, dw_rows,
                                                    token_to_row, d_logits, rows_cap, scale);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe

namespace moe {

// One thread waits on an mbarrier that nothing ever arrives on, through the same
// bounded wait the GEMM pipeline uses; it must give up after `limit` cycles and
// leave MOE_ERR_TIMEOUT in the status word.
__global__ void wait_timeout_kernel(int32_t* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  mbar_wait_bounded(&bar, 0, &abort_flag, status, limit);
}

cudaError_t launch_wait_timeout(int32_t* status, long long limit, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(status, limit);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
