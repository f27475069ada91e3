/*
 * Dropless mixture-of-experts layer, forward and backward, on one GB300 (sm_103a).
 *
 * C ABI of libmoe.so.  Plain pointers and sizes only.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Ownership: every pointer argument is caller-owned memory; the library keeps
 *    no pointer after a call returns and allocates no device memory.  Pointers
 *    named like tensors are DEVICE pointers; `dims` is a HOST pointer.
 *  - Execution: work is enqueued on `stream` (a cudaStream_t, NULL = legacy default
 *    stream) and runs asynchronously; no call synchronises the host except
 *    moe_check_status.
 *  - Errors: argument problems are found on the host and returned synchronously
 *    (nothing is enqueued then).  Problems found while kernels run (a broken
 *    invariant, a pipeline wait that gave up) are written to the caller's
 *    `dev_status` word (int32, device memory, must start at 0; the first error
 *    sticks) and are read back by moe_check_status.  No kernel traps.
 *  - Layouts are row-major.  bf16 tensors are passed as moe_bf16 bit patterns.
 *    Weights follow the [out, in] convention: W_gu[E][2f][d] holds the gate rows
 *    [0,f) then the up rows [f,2f) of every expert; W_d[E][d][f].
 *  - Routed rows live in a padded, expert-contiguous row space of
 *    moe_row_capacity() rows: expert e owns rows [row_offsets[e], row_offsets[e+1]),
 *    row_offsets[e] being a multiple of MOE_ROW_ALIGN; its first split_sizes[e]
 *    rows hold its tokens (in token order) and the rest are padding rows that the
 *    library fills with zeros where they are read.
 *  - Alignment: all device pointers 16-byte aligned; d a multiple of 128 and f a
 *    multiple of 64 (tensor-memory tiles; 32-element MX blocks); 1 <= k <= min(E,32);
 *    E <= 1024; T >= 0.
 *
 * Sources (web pages describing the method; quoted by title and section):
 *  [DROPLESS] NVIDIA dropless MoE in JAX: "Az NVIDIA szerint tízszer gyorsabb lett a
 *             dropless MoE tanítása JAX-ban".
 *  [BIO]      NVIDIA MoE training for biology models: "NVIDIA מציגה דרך יעילה לאמן
 *             מודלי MoE בביולוגיה".
 *  [MEGA]     DeepGEMM Mega MoE article (itsolotime.com, Thai).
 *  [PRIME]    "Prime Mega MoE: tanításra is jó a DeepSeek MoE kernele".
 */
#ifndef DROPLESS_MOE_H
#define DROPLESS_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16; /* bfloat16 bit pattern */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad size, NULL pointer, k > E, ... */
  MOE_ERR_UNSUPPORTED = 2, /* valid but not supported (d % 128, f % 64 (% 128 for MXFP8), E > 1024, ...) */
  MOE_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned */
  MOE_ERR_WORKSPACE = 4,   /* workspace NULL while needed */
  MOE_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed */
  MOE_ERR_TIMEOUT = 6,     /* a bounded device wait gave up (written to dev_status) */
  MOE_ERR_INVARIANT = 7,   /* sum(split_sizes) != T*k seen on the device */
  MOE_ERR_SCRATCH_LIMIT = 8 /* too large for moe_gemm_down_dgrad_noalloc's static scratch */
} moe_status;

enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
/* MOE_PREC_MXFP8_W4: FP8 x FP4 experts -- activations and gradients MXFP8 (E4M3), the
 * expert weights MXFP4 (E2M1 codes with one E8M0 scale per 32 elements); see the MXFP8
 * layer calls below. */
enum { MOE_PREC_BF16 = 0, MOE_PREC_MXFP8 = 1, MOE_PREC_MXFP8_W4 = 2 };
enum { MOE_ROW_ALIGN = 128 };

typedef struct moe_dims {
  int32_t T;        /* tokens */
  int32_t d;        /* hidden size */
  int32_t f;        /* expert intermediate size */
  int32_t E;        /* routed experts */
  int32_t k;        /* experts per token */
  int32_t f_shared; /* shared-expert width, 0 = none */
  int32_t score;    /* MOE_SCORE_* */
  int32_t prec;     /* MOE_PREC_* */
} moe_dims;

/* Library version of this ABI (increments on any signature change). */
int32_t moe_abi_version(void);

/* Text of a status code; never NULL. */
const char* moe_status_string(int32_t status);

/* Validates dims against the limits above.  Host only. */
moe_status moe_check_dims(const moe_dims* dims);

/* Rows of the padded routed-row space: roundup(T*k,128) + 128*E.  Every [rows, .]
 * routed buffer (xp, gu, h, y_rows, dy_rows, dgu, dxp, w_rows, row_to_token) has
 * this many rows.  Returns -1 for invalid dims. */
int64_t moe_row_capacity(const moe_dims* dims);

/* Bytes of scratch the route and backward calls need (one buffer may serve both;
 * the route scratch must survive from moe_route_topk to moe_permute). */
size_t moe_workspace_size(const moe_dims* dims);

/* Number of kernels this library has launched since it was loaded. */
uint64_t moe_launch_count(void);

/*
 * Step 1 -- learned top-k routing [DROPLESS "A dropless MoE minden tokent
 * feldolgoz": each token is processed only by its top-K experts] and the per-expert
 * token counts handed to the grouped GEMM as split_sizes [BIO "מומחים מקובצים
 * במקום לולאת Python"].
 *   logits      [T][E] fp32   router logits (input)
 *   topk_idx    [T][k] int32  selected experts, best first; ties go to the lower index
 *   topk_w      [T][k] fp32   routing weights: softmax (or sigmoid) of the logits,
 *                             renormalised over the k selected experts
 *   split_sizes [E]    int32  tokens routed to each expert (dropless: sum = T*k)
 *   offsets     [E+1]  int32  exclusive prefix sum of split_sizes
 *   row_offsets [E+1]  int32  exclusive prefix sum of split_sizes rounded up to 128
 *   workspace   >= moe_workspace_size bytes; keeps per-block ranks for moe_permute
 * dev_status gets MOE_ERR_INVARIANT if the counts do not add up to T*k.
 */
moe_status moe_route_topk(const moe_dims* dims, const float* logits, int32_t* topk_idx,
                          float* topk_w, int32_t* split_sizes, int32_t* offsets,
                          int32_t* row_offsets, void* workspace, int32_t* dev_status,
                          void* stream);

/*
 * Group-limited routing (the DeepSeek-V3 router variant; neither page states it -- a
 * NEXT step of the route of step 1): dims->score must be MOE_SCORE_SIGMOID.
 *   s = sigmoid(logit); selection score c = s + bias[e] (fp32; bias may be NULL = 0 and
 *   steers selection only); the E experts form n_group groups of E / n_group
 *   consecutive experts; a group's score is the sum of its two largest c; the
 *   topk_group best groups are eligible (ties to the lower group); the top-k of c over
 *   their experts are chosen (ties to the lower expert, slot j the j-th best);
 *   topk_w = routed_scale * s_j / sum_j s_j.
 * Requirements: 1 <= n_group <= 32, E % n_group == 0, E / n_group >= 2,
 *   1 <= topk_group <= n_group, k <= topk_group * E / n_group, routed_scale > 0;
 *   otherwise MOE_ERR_INVALID_ARG.  Outputs, workspace and errors as moe_route_topk.
 */
moe_status moe_route_topk_grouped(const moe_dims* dims, const float* logits, const float* bias, int32_t n_group,
                                  int32_t topk_group, float routed_scale, int32_t* topk_idx, float* topk_w,
                                  int32_t* split_sizes, int32_t* offsets, int32_t* row_offsets, void* workspace,
                                  int32_t* dev_status, void* stream);

/*
 * Step 2 -- dispatch: copy every token to one row per selected expert, experts
 * contiguous, tokens of one expert in token order [DROPLESS "Az egyenetlen terhelés
 * lassítja a tanítást": ragged per-expert tensors; MEGA "Mega MoE คืออะไร?":
 * dispatch step].  Row of (t, j) = row_offsets[e] + number of tokens t' < t that
 * also chose e.
 *   x            [T][d] bf16            token activations
 *   topk_idx, topk_w, split_sizes, row_offsets: from moe_route_topk
 *   workspace    the one given to moe_route_topk (read only)
 *   xp           [rows][d] bf16         permuted rows; padding rows set to 0
 *   row_to_token [rows] int32           token of each row, -1 for padding rows
 *   token_to_row [T][k] int32           row of each (token, slot)
 *   w_rows       [rows] fp32            routing weight of each row, 0 for padding
 * (rows = moe_row_capacity; entries at or beyond row_offsets[E] are not written.)
 * dev_status gets MOE_ERR_INVARIANT if a computed row falls outside the row space
 * (stale or foreign workspace); such a row is skipped, never written.
 */
moe_status moe_permute(const moe_dims* dims, const moe_bf16* x, const int32_t* topk_idx,
                       const float* topk_w, const int32_t* split_sizes,
                       const int32_t* row_offsets, const void* workspace, moe_bf16* xp,
                       int32_t* row_to_token, int32_t* token_to_row, float* w_rows,
                       int32_t* dev_status, void* stream);

/*
 * Steps 3-5 -- grouped GEMM gate/up, SwiGLU scaled by the routing weight, grouped
 * GEMM down, each expert using its actual token count [DROPLESS "Csoportosított
 * mátrixszorzás és összevont adatmozgatás": one grouped GEMM call for all experts,
 * no padding to a maximum capacity; BIO "צמצום הזיכרון ותקורות הכימות":
 * GroupedLinear -> ScaledSwiGLU -> GroupedLinear as one fused operation].
 * For each row r of expert e:
 *   G = xp[r] W_gate[e]^T, U = xp[r] W_up[e]^T, h = w_rows[r] * silu(G) * U,
 *   y_rows[r] = h W_d[e]^T                       (fp32 accumulation, bf16 outputs)
 *   xp [rows][d], w_gu [E][2f][d], w_d [E][d][f]  (inputs, bf16)
 *   gu [rows][2f] bf16  saved G (cols [0,f)) and U (cols [f,2f)) for the backward
 *   h  [rows][f]  bf16  saved scaled activation
 *   y_rows [rows][d] bf16
 * Tiles are scheduled on the device from row_offsets (no host synchronisation).
 */
moe_status moe_grouped_mlp_fwd(const moe_dims* dims, const moe_bf16* xp,
                               const int32_t* row_offsets, const float* w_rows,
                               const moe_bf16* w_gu, const moe_bf16* w_d, moe_bf16* gu,
                               moe_bf16* h, moe_bf16* y_rows, int32_t* dev_status,
                               void* stream);

/*
 * The two GEMMs of moe_grouped_mlp_fwd as separate calls (same kernels, same
 * results; lets a caller time or interleave them):
 *   moe_gemm_gate_up: gu and h from xp (steps 3-4);  moe_gemm_down: y_rows from h (step 5).
 */
moe_status moe_gemm_gate_up(const moe_dims* dims, const moe_bf16* xp,
                            const int32_t* row_offsets, const float* w_rows,
                            const moe_bf16* w_gu, moe_bf16* gu, moe_bf16* h,
                            int32_t* dev_status, void* stream);
moe_status moe_gemm_down(const moe_dims* dims, const moe_bf16* h, const int32_t* row_offsets,
                         const moe_bf16* w_d, moe_bf16* y_rows, int32_t* dev_status, void* stream);

/*
 * Step 6 -- combine back to token order [MEGA "Mega MoE คืออะไร?": combine step;
 * DROPLESS "Az egyenetlen terhelés lassítja a tanítást": restore the original
 * order]:  out[t] = sum_{j<k} rows[token_to_row[t][j]]  (+ shared[t] if given),
 * summed in fp32 in slot order, rounded once to bf16.  The routing weight was
 * already applied in the SwiGLU step, so the sum is unweighted.  Also serves as
 * the un-permute of the backward (dX from dXp).
 *   rows [rows][d] bf16, token_to_row [T][k], shared [T][d] bf16 or NULL, out [T][d].
 */
moe_status moe_combine_fwd(const moe_dims* dims, const moe_bf16* rows,
                           const int32_t* token_to_row, const moe_bf16* shared,
                           moe_bf16* out, void* stream);

/*
 * Backward of step 6 (the adjoint of the combine sum) [BIO "צמצום הזיכרון ותקורות
 * הכימות": the fused grouped-MLP operation has a backward counterpart; MEGA "Mega MoE
 * คืออะไร?": combine returns expert outputs to their tokens, so its adjoint hands each
 * token's output gradient back to every row it was combined from]:
 * dy_rows[r] = dY[token of r], padding rows set to 0.
 *   dy [T][d] bf16, token_to_row [T][k], split_sizes, row_offsets, dy_rows [rows][d].
 */
moe_status moe_combine_bwd(const moe_dims* dims, const moe_bf16* dy,
                           const int32_t* token_to_row, const int32_t* split_sizes,
                           const int32_t* row_offsets, moe_bf16* dy_rows, void* stream);

/*
 * Backward of steps 3-5 [BIO "צמצום הזיכרון ותקורות הכימות": the fused grouped MLP
 * has a backward counterpart; PRIME "Mit csinált a Prime Intellect?": a backward
 * pass for the fused MoE kernel].  Per expert e, rows r of e:
 *   dH = dy_rows[r] W_d[e]; dw_rows[r] = sum_n silu(G)U dH; dA = w dH;
 *   dG = dA U silu'(G); dU = dA silu(G)               -> dgu[r] = [dG | dU]
 *   dxp[r] = dgu[r] W_gu[e]
 *   dW_d[e] = sum_r dy_rows[r]^T h[r];  dW_gu[e] = sum_r dgu[r]^T xp[r]
 * Experts with no rows get dW = 0.  Sums over rows run in a fixed order (no atomics).
 *   inputs: xp, row_offsets, w_rows, w_gu, w_d, gu, h (saved by the forward), dy_rows
 *   dgu [rows][2f] bf16 (output, also consumed internally), dxp [rows][d] bf16,
 *   dw_gu [E][2f][d] bf16, dw_d [E][d][f] bf16, dw_rows [rows] fp32,
 *   workspace >= moe_workspace_size bytes.
 */
moe_status moe_grouped_mlp_bwd(const moe_dims* dims, const moe_bf16* xp,
                               const int32_t* row_offsets, const float* w_rows,
                               const moe_bf16* w_gu, const moe_bf16* w_d,
                               const moe_bf16* gu, const moe_bf16* h,
                               const moe_bf16* dy_rows, moe_bf16* dgu, moe_bf16* dxp,
                               moe_bf16* dw_gu, moe_bf16* dw_d, float* dw_rows,
                               void* workspace, int32_t* dev_status, void* stream);

/*
 * The four GEMMs of moe_grouped_mlp_bwd as separate calls, in the order the
 * composite runs them:
 *   moe_gemm_down_dgrad     dH = dy_rows W_d[e] with the SwiGLU' epilogue -> dgu, dw_rows
 *                           (workspace holds the per-tile dw partials)
 *   moe_gemm_down_wgrad     dW_d[e]  = dy_rows_e^T h_e
 *   moe_gemm_gate_up_dgrad  dxp      = dgu W_gu[e]
 *   moe_gemm_gate_up_wgrad  dW_gu[e] = dgu_e^T xp_e
 */
moe_status moe_gemm_down_dgrad(const moe_dims* dims, const moe_bf16* dy_rows,
                               const int32_t* row_offsets, const float* w_rows,
                               const moe_bf16* w_d, const moe_bf16* gu, moe_bf16* dgu,
                               float* dw_rows, void* workspace, int32_t* dev_status,
                               void* stream);
moe_status moe_gemm_down_wgrad(const moe_dims* dims, const moe_bf16* dy_rows, const moe_bf16* h,
                               const int32_t* row_offsets, moe_bf16* dw_d, int32_t* dev_status,
                               void* stream);
moe_status moe_gemm_gate_up_dgrad(const moe_dims* dims, const moe_bf16* dgu,
                                  const int32_t* row_offsets, const moe_bf16* w_gu, moe_bf16* dxp,
                                  int32_t* dev_status, void* stream);
moe_status moe_gemm_gate_up_wgrad(const moe_dims* dims, const moe_bf16* dgu, const moe_bf16* xp,
                                  const int32_t* row_offsets, moe_bf16* dw_gu, int32_t* dev_status,
                                  void* stream);

/*
 * The always-on shared expert of the DeepSeek-V3-shaped layer (dims->f_shared > 0):
 * a dense SwiGLU MLP on every token with weight 1, whose output is added in the
 * combine after the k routed terms (pass y_s as `shared` to moe_combine_fwd, and dx_s
 * as `shared` to the un-permute).  It runs through the same tcgen05 grouped-GEMM
 * kernel with one dense group of T rows.  Not a step the pages describe: the layer
 * shape comes from DeepSeek-V3, whose training the pages report.
 *   fwd: gu_s [T][2fs] = x W_gu_s^T (saved G|U), h_s [T][fs] = silu(G) U, y_s [T][d] = h_s W_d_s^T
 *   bwd: dgu_s = [dG|dU] from dH = dy W_d_s; dx_s [T][d] = dgu_s W_gu_s;
 *        dw_d_s [d][fs] = dy^T h_s; dw_gu_s [2fs][d] = dgu_s^T x   (zero when T = 0)
 * W_gu_s [2fs][d] (gate rows first), W_d_s [d][fs]; all bf16, fp32 accumulation.
 */
moe_status moe_shared_mlp_fwd(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_gu_s,
                              const moe_bf16* w_d_s, moe_bf16* gu_s, moe_bf16* h_s, moe_bf16* y_s,
                              int32_t* dev_status, void* stream);
moe_status moe_shared_mlp_bwd(const moe_dims* dims, const moe_bf16* x, const moe_bf16* w_gu_s,
                              const moe_bf16* w_d_s, const moe_bf16* gu_s, const moe_bf16* h_s,
                              const moe_bf16* dy, moe_bf16* dgu_s, moe_bf16* dx_s,
                              moe_bf16* dw_gu_s, moe_bf16* dw_d_s, int32_t* dev_status,
                              void* stream);

/*
 * Backward of step 1 [DROPLESS "A dropless MoE minden tokent feldolgoz": the router is
 * learned, so the loss reaches its logits through the top-K routing weights; PRIME
 * "Mit csinált a Prime Intellect?": a backward pass for the fused MoE layer]:
 * router-logit gradient from the routing-weight gradient.
 * dw[t][j] = dw_rows[token_to_row[t][j]];  c = sum_j w dw;
 *   softmax: dl[e_j] = w_j (dw_j - c)
 *   sigmoid: dl[e_j] = (dw_j - c) / sum_j s_j * s_j (1 - s_j),  s = sigmoid(logit)
 * and dl = 0 for experts not selected.  d_logits [T][E] fp32.
 */
moe_status moe_route_topk_bwd(const moe_dims* dims, const float* logits,
                              const int32_t* topk_idx, const float* topk_w,
                              const float* dw_rows, const int32_t* token_to_row,
                              float* d_logits, void* stream);

/*
 * Router backward of moe_route_topk_grouped (sigmoid scores, weights scaled by
 * routed_scale; the bias has no gradient): as moe_route_topk_bwd with
 *   dL/ds_i = (routed_scale * dw_i - sum_j w_j dw_j) / sum_j s_j for the chosen i.
 */
moe_status moe_route_topk_bwd_scaled(const moe_dims* dims, const float* logits, const int32_t* topk_idx,
                                     const float* topk_w, float routed_scale, const float* dw_rows,
                                     const int32_t* token_to_row, float* d_logits, void* stream);

/*
 * moe_gemm_down_dgrad without a workspace, for callers that cannot allocate device
 * memory (a host program that owns all device memory through its own pool and gives
 * plugins no allocator, or a latency-critical loop where cudaMalloc/cudaFree and the
 * synchronisation they may bring are not allowed).  The pages have no counterpart:
 * this is an interface convenience, not a step of the method.
 *
 * Same arguments, kernels (the CTA-pair kernel where f allows it, else the single-CTA
 * one, chosen exactly as moe_gemm_down_dgrad chooses) and therefore the same bits as
 * moe_gemm_down_dgrad minus `workspace`: the per-tile partial sums of dw go to a
 * static device array of
 * moe_noalloc_scratch_bytes() bytes (8 MiB) that every GPU loading the library holds
 * until the process exits.  Requires moe_row_capacity(dims) * (f / BN) <= 2^21,
 * BN = 256, 128 or 64 (the largest dividing f); larger problems get
 * MOE_ERR_SCRATCH_LIMIT before anything is enqueued.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library call.
 *
 * The first call on a device looks up the array's device address (once per device,
 * with that device current) and keeps it for the life of the process; make that first
 * call before any stream capture, and do not use this call after cudaDeviceReset (or
 * anything else that destroys and recreates the device's primary context): the kept
 * address would then be stale.  All
 * calls share the one array, which keeps the last call's contents (nothing in it has
 * to start at zero); calls that overlap on the GPU race on it and give wrong dw_rows.
 */
moe_status moe_gemm_down_dgrad_noalloc(const moe_dims* dims, const moe_bf16* dy_rows,
                                       const int32_t* row_offsets, const float* w_rows,
                                       const moe_bf16* w_d, const moe_bf16* gu, moe_bf16* dgu,
                                       float* dw_rows, int32_t* dev_status, void* stream);

/* Bytes of the static array moe_gemm_down_dgrad_noalloc uses. */
size_t moe_noalloc_scratch_bytes(void);

/* Synchronises `stream`, then returns the status word written by the kernels
 * (MOE_OK if none failed) or MOE_ERR_CUDA if the stream itself failed. */
moe_status moe_check_status(const int32_t* dev_status, void* stream);

/*
 * The same dense GEMM as moe_gemm_bf16 on the CTA-pair kernel (tcgen05 cta_group::2,
 * M = 256 per MMA across two SMs), which the layer uses where shapes allow.
 * N % 128 == 0, K % 64 == 0.
 */
moe_status moe_gemm_bf16_pair(const moe_bf16* A, const moe_bf16* B, moe_bf16* C, int32_t M, int32_t N,
                              int32_t K, int32_t a_layout, int32_t b_layout, int32_t* dev_status, void* stream);

/*
 * Test hook for failure detection: one thread waits, through the same bounded
 * mbarrier wait as the GEMM pipeline, on a barrier that nothing arrives on.  After
 * limit_cycles (1 .. 2^32) it gives up and writes MOE_ERR_TIMEOUT to dev_status; the
 * CUDA context stays usable.  Lets a test make a device wait run out on purpose.
 */
moe_status moe_test_wait_timeout(int32_t* dev_status, int64_t limit_cycles, void* stream);

/*
 * MXFP8 building blocks (E4M3 codes, one E8M0 scale per 32 elements along the GEMM's
 * contraction axis) [BIO "צמצום הזיכרון ותקורות הכימות": one scale per block of 32
 * consecutive values, block-scaled Blackwell tensor-core instructions; DROPLESS
 * "Csoportosított mátrixszorzás és összevont adatmozgatás": group-aware MXFP8
 * quantisation for the expert GEMMs].
 * Scale rule: e = floor(log2(amax)) - 8 clamped to [-127,127], byte e + 127 (0 for an
 * all-zero block); codes = E4M3(x * 2^-e), round to nearest even, saturating at 448.
 * Scale layout ("SF tiles"): for an operand of R rows (M or N) and K columns the
 * scales form 512-byte tiles, tile (r/128, k/128) at byte (r/128 * K/128 + k/128)*512;
 * inside, byte ((r%32)*4 + (r%128)/32)*4 + (k%128)/32 is the scale of row r's block k/32.
 * Scale arrays therefore hold roundup(R,128) * K/32 bytes.
 *
 * moe_mx_quantize_rows: src bf16 [rows][ld] (first C columns) -> codes [rows][C] and
 *   SF tiles with K = C (blocks along each row).  C % 128 == 0.  Rows at or beyond
 *   *nrows_dev (if not NULL) are skipped.
 * moe_mx_quantize_cols: src bf16 [batch][rows][C] -> codes_t [batch][C][rows] and, per
 *   batch, SF tiles of an operand with C rows and K = rows (blocks of 32 rows down each
 *   column).  rows % 128 == 0, C % 128 == 0; 128-row tiles at or beyond *nrows_dev are
 *   skipped.  Per batch, scales take C * rows / 32 bytes.
 * moe_gemm_mxfp8: C[M][N] bf16 = sum_k deq(A)(m,k) deq(B)(n,k) with A codes [M][K],
 *   B codes [N][K] (both K-major) and their SF tiles; fp32 accumulation on the
 *   block-scaled tensor cores.  M, N, K multiples of 128.
 */
moe_status moe_mx_quantize_rows(const moe_bf16* src, int64_t rows, int32_t C, int64_t ld,
                                const int32_t* nrows_dev, uint8_t* codes, uint8_t* scales, void* stream);
moe_status moe_mx_quantize_cols(const moe_bf16* src, int32_t batch, int64_t rows, int32_t C,
                                const int32_t* nrows_dev, uint8_t* codes_t, uint8_t* scales, void* stream);
moe_status moe_gemm_mxfp8(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b, const uint8_t* b_sf,
                          moe_bf16* c, int32_t M, int32_t N, int32_t K, int32_t* dev_status, void* stream);

/*
 * FP8 x FP4 building blocks [MEGA "ทิศทางการปรับปรุงในระดับลึกยิ่งขึ้น": FP8 x FP4 mixed
 * precision as the next step for the expert GEMMs].  The weight operand is MXFP4: E2M1
 * codes (sign, two exponent bits with bias 1, one mantissa bit: magnitudes 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6) with one E8M0 scale per 32 elements along the contraction, scale rule
 * e = floor(log2(amax)) - 2 clamped to [-127,127] (byte e + 127, 0 for an all-zero
 * block), codes = E2M1(x * 2^-e), round to nearest even, saturating at 6.  Codes are
 * packed two a byte, the element with the lower index in the lower four bits; the SF
 * tiles are laid out as for MXFP8.
 *
 * moe_mx4_quantize_cols: src bf16 [batch][rows][C] -> codes_t [batch][C][rows / 2] bytes
 *   with per-batch SF tiles (blocks of 32 rows down each column; K = rows), and codes
 *   [batch * rows][C / 2] bytes with SF tiles of K = C (blocks along each row), from one
 *   read.  rows % 128 == 0, C % 128 == 0; pointers 16-byte aligned.
 * moe_gemm_mxf8f4: C[M][N] bf16 = sum_k deq(A)(m,k) deq(B)(n,k), A E4M3 codes [M][K] and
 *   B E2M1 codes [N][K / 2] bytes (both K-major, B 32-byte aligned) with their SF tiles;
 *   the block-scaled tcgen05 MMA with an E2M1 B operand, fp32 accumulation.  M, N, K
 *   multiples of 128.
 */
moe_status moe_mx4_quantize_cols(const moe_bf16* src, int32_t batch, int64_t rows, int32_t C, uint8_t* codes_t,
                                 uint8_t* scales_t, uint8_t* codes, uint8_t* scales, void* stream);
moe_status moe_gemm_mxf8f4(const uint8_t* a, const uint8_t* a_sf, const uint8_t* b4, const uint8_t* b_sf,
                           moe_bf16* c, int32_t M, int32_t N, int32_t K, int32_t* dev_status, void* stream);

/*
 * The layer with MXFP8 GEMM operands (dims->prec may be any value; f % 128 == 0).
 * With dims->prec == MOE_PREC_MXFP8_W4 the experts are FP8 x FP4: wq (and wq_s) hold the
 * weights as MXFP4 codes (moe_mx_weights_size shrinks accordingly; wq and wq_s must be
 * 32-byte aligned) and the four products with a weight operand (gate/up and down
 * forward, their input gradients) run with an E2M1 B operand; the weight gradients
 * stay FP8 x FP8.
 * Every GEMM operand is quantised along its own contraction axis, in the kernel that
 * produces it: the routed token rows by moe_permute_mx and dY's routed rows by
 * moe_combine_bwd_mx, each in one gathered pass that writes both the row-wise codes
 * (blocks along d, for the row GEMMs) and the column-wise codes (blocks of 32 rows
 * down each column of the 128-aligned expert segments, for the weight gradients);
 * h and dG|dU in the epilogues of the gate/up and SwiGLU' GEMMs, from fp32, in both
 * orientations.  bf16 copies of Xp, h, dY rows and dG|dU are never written.  The
 * GEMMs are the block-scaled tcgen05 kernel with fp32 accumulation and the same bf16
 * outputs (gu, y_rows, dxp, dW) as the bf16 calls.  The backward treats
 * quantisation as the identity.
 *   wq:    >= moe_mx_weights_size bytes, filled by moe_mx_quantize_weights from the
 *          bf16 master weights (W_gu along d and along 2f, W_d along f and along d;
 *          one read of each weight); refill it whenever the weights change.
 *   mx_ws: >= moe_mx_workspace_size bytes of caller scratch holding the quantised
 *          activations of one step; all the calls of the step share it, in this order:
 *          moe_permute_mx, moe_gemm_gate_up_mx, moe_gemm_down_mx, (combine),
 *          moe_combine_bwd_mx, moe_gemm_down_dgrad_mx, moe_gemm_down_wgrad_mx,
 *          moe_gemm_gate_up_dgrad_mx, moe_gemm_gate_up_wgrad_mx.
 *   moe_permute_mx writes the routing maps (row_to_token, token_to_row, w_rows) as
 *          moe_permute does; moe_combine_bwd_mx gathers dY through its row_to_token.
 *   The weight-gradient calls take their operands from mx_ws only.
 * Other arguments as in the bf16 calls of the same names without "_mx".
 */
size_t moe_mx_weights_size(const moe_dims* dims);
size_t moe_mx_workspace_size(const moe_dims* dims);
moe_status moe_mx_quantize_weights(const moe_dims* dims, const moe_bf16* w_gu, const moe_bf16* w_d, void* wq,
                                   void* stream);
moe_status moe_permute_mx(const moe_dims* dims, const moe_bf16* x, const int32_t* topk_idx, const float* topk_w,
                          const int32_t* split_sizes, const int32_t* row_offsets, const void* workspace,
                          void* mx_ws, int32_t* row_to_token, int32_t* token_to_row, float* w_rows,
                          int32_t* dev_status, void* stream);
moe_status moe_gemm_gate_up_mx(const moe_dims* dims, const int32_t* row_offsets, const float* w_rows,
                               const void* wq, void* mx_ws, moe_bf16* gu, int32_t* dev_status, void* stream);
moe_status moe_gemm_down_mx(const moe_dims* dims, const int32_t* row_offsets, const void* wq, void* mx_ws,
                            moe_bf16* y_rows, int32_t* dev_status, void* stream);
moe_status moe_combine_bwd_mx(const moe_dims* dims, const moe_bf16* dy, const int32_t* row_to_token,
                              const int32_t* split_sizes, const int32_t* row_offsets, void* mx_ws, void* stream);
moe_status moe_gemm_down_dgrad_mx(const moe_dims* dims, const int32_t* row_offsets, const float* w_rows,
                                  const void* wq, void* mx_ws, const moe_bf16* gu, float* dw_rows, void* workspace,
                                  int32_t* dev_status, void* stream);
moe_status moe_gemm_down_wgrad_mx(const moe_dims* dims, const int32_t* row_offsets, void* mx_ws, moe_bf16* dw_d,
                                  int32_t* dev_status, void* stream);
moe_status moe_gemm_gate_up_dgrad_mx(const moe_dims* dims, const int32_t* row_offsets, const void* wq,
                                     void* mx_ws, moe_bf16* dxp, int32_t* dev_status, void* stream);
moe_status moe_gemm_gate_up_wgrad_mx(const moe_dims* dims, const int32_t* row_offsets, void* mx_ws,
                                     moe_bf16* dw_gu, int32_t* dev_status, void* stream);

/*
 * Steps 3-5 with MXFP8 operands as one call, and their backward as one call
 * [BIO "צמצום הזיכרון ותקורות הכימות": GroupedLinear -> ScaledSwiGLU -> GroupedLinear
 * as one fused MXFP8 operation with a backward counterpart; DROPLESS "Csoportosított
 * mátrixszorzás és összevont adatmozgatás": group-aware MXFP8 quantisation for the
 * expert GEMMs].  The MXFP8 counterparts of moe_grouped_mlp_fwd / moe_grouped_mlp_bwd:
 *   moe_grouped_mlp_fwd_mx = moe_gemm_gate_up_mx + moe_gemm_down_mx.  Reads the routed
 *     x codes that moe_permute_mx left in mx_ws and the weight codes in wq; writes gu
 *     (saved G|U, bf16 [rows][2f]), y_rows (bf16 [rows][d]) and h's codes (in mx_ws).
 *   moe_grouped_mlp_bwd_mx = moe_gemm_down_dgrad_mx + moe_gemm_down_wgrad_mx +
 *     moe_gemm_gate_up_dgrad_mx + moe_gemm_gate_up_wgrad_mx.  Reads dY's routed codes
 *     (moe_combine_bwd_mx), h's and x's codes in mx_ws, gu and wq; writes dw_rows (fp32
 *     [rows]), dW_d [E][d][f], dxp [rows][d], dW_gu [E][2f][d] (bf16) and dG|dU's codes
 *     (in mx_ws); workspace >= moe_workspace_size bytes.
 * Same kernels and results as the per-GEMM calls; an argument error is returned
 * before any kernel is enqueued.
 */
moe_status moe_grouped_mlp_fwd_mx(const moe_dims* dims, const int32_t* row_offsets, const float* w_rows,
                                  const void* wq, void* mx_ws, moe_bf16* gu, moe_bf16* y_rows, int32_t* dev_status,
                                  void* stream);
moe_status moe_grouped_mlp_bwd_mx(const moe_dims* dims, const int32_t* row_offsets, const float* w_rows,
                                  const void* wq, void* mx_ws, const moe_bf16* gu, moe_bf16* dxp, moe_bf16* dw_gu,
                                  moe_bf16* dw_d, float* dw_rows, void* workspace, int32_t* dev_status,
                                  void* stream);

/*
 * The shared expert with MXFP8 GEMM operands (DeepSeek-V3 shape in MXFP8; f_shared and
 * T multiples of 128).  wq_s (>= moe_mx_shared_weights_size bytes) holds W_gu_s and
 * W_d_s quantised along both of their axes, filled by moe_mx_quantize_shared_weights;
 * mx_ws_s (>= moe_mx_shared_workspace_size bytes) is scratch for the quantised
 * activations (h_s and dG|dU of the shared expert are kept only as codes there); the
 * forward quantises x in both orientations there, so the backward takes no x.
 * Otherwise as moe_shared_mlp_fwd / moe_shared_mlp_bwd.
 */
size_t moe_mx_shared_weights_size(const moe_dims* dims);
size_t moe_mx_shared_workspace_size(const moe_dims* dims);
moe_status moe_mx_quantize_shared_weights(const moe_dims* dims, const moe_bf16* w_gu_s, const moe_bf16* w_d_s,
                                          void* wq_s, void* stream);
moe_status moe_shared_mlp_fwd_mx(const moe_dims* dims, const moe_bf16* x, const void* wq_s, void* mx_ws_s,
                                 moe_bf16* gu_s, moe_bf16* y_s, int32_t* dev_status, void* stream);
moe_status moe_shared_mlp_bwd_mx(const moe_dims* dims, const void* wq_s, void* mx_ws_s, const moe_bf16* gu_s,
                                 const moe_bf16* dy, moe_bf16* dx_s, moe_bf16* dw_gu_s, moe_bf16* dw_d_s,
                                 int32_t* dev_status, void* stream);

/*
 * Dense GEMM through the same tcgen05 kernel (one group), for unit tests of the
 * tensor-core core: C[m][n] = sum_k A(m,k) B(n,k), fp32 accumulation, bf16 out.
 *   a_layout 0: A stored [M][K];  1: A stored [K][M]
 *   b_layout 0: B stored [N][K];  1: B stored [K][N]
 *   C [M][N].  N % 64 == 0, K % 64 == 0, M >= 1.
 */
moe_status moe_gemm_bf16(const moe_bf16* A, const moe_bf16* B, moe_bf16* C, int32_t M,
                         int32_t N, int32_t K, int32_t a_layout, int32_t b_layout,
                         int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DROPLESS_MOE_H */
