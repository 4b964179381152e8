/*
 * w4a8moe.h -- C ABI of the GB300 (sm_103a) W4AFP8 mixture-of-experts hot path.
 *
 * W4AFP8: int4 weights with fp32 scales per 128 consecutive K, times FP8 E4M3
 * activations quantised per token per 128 columns, fp32 accumulation, bf16
 * outputs.  The layer is the workflow of the SGLang PR #7762 page ("support
 * DeepSeek-R1-W4AFP8 model with ep-moe mode", Modifications: Workflow and
 * Kernel): routing ids -> permutation preprocess -> FP8 scaling of the hidden
 * states -> int4 x FP8 grouped GEMM w13 (group size 128) -> SiLU and Mul with
 * FP8 re-scaling -> grouped GEMM w2 -> unpermutation weighted by the routing
 * weights.  The dense Linear is the same mixed-input GEMM with one weight
 * matrix (lyraW4AFp8 page, "LyraW4fp8": W4AFP8 MoE and GEMMs).
 *
 * Conventions for every entry point below
 *  - Pointers are DEVICE pointers owned by the caller, unless stated.  The
 *    library never allocates, frees or synchronises; every call only enqueues
 *    kernels on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *    and returns.  Results are valid once the stream has reached that point.
 *  - Sizes are int64_t element counts.  bf16 tensors are passed as uint16_t
 *    bit patterns.  All matrices are row-major and densely packed unless a
 *    leading dimension is given.
 *  - Return value: a w4a8_status.  Shapes, null pointers and alignment are
 *    checked on the host before anything is launched (W4A8_ERR_INVALID_ARG /
 *    W4A8_ERR_UNSUPPORTED, nothing enqueued).  A failed launch returns
 *    W4A8_ERR_CUDA.  w4a8_last_error() gives a text for the calling thread.
 *  - Device pointers passed to a GEMM must be 16-byte aligned (TMA).
 *  - Calls on the same stream are ordered; calls on different streams that
 *    share output buffers race.
 *
 * Packed weight layout (canonical): uint8 [E][N][K/2].  Byte b of a row
 * holds element k = 2b in bits 0-3 and k = 2b+1 in bits 4-7, each a two's
 * complement nibble in -8..7 (lower k in lower bits, the unpack order of the
 * SGLang PR #37796 page, Modifications).  The GEMMs take weights prepacked once
 * by w4a8_prepack_weights (same size and row layout, another code per nibble;
 * the post-load weight processing step of the PR #7762 page,
 * process_weights_after_loading).  Weight scales: fp32 [E][K/128][N]
 * (N contiguous, the [E, K/128, N] scale layout of the PR #37796 page).
 * Activation scales: fp32 [K/128][ld], element (row m, group g) at
 * scales[g*ld + m], ld >= M and ld % 4 == 0 (group-major, so a tile of rows of
 * one group is contiguous for TMA).  Activation corrections gcorr: same layout,
 * gcorr[g][m] = -1/2 * scales[g][m] * S, S = sum_{k in g} e4m3(q[m][k]) summed
 * exactly, rounded once to fp32 (exact while |S| < 2^15), then one rounded
 * fp32 product.  The quantisation calls emit them and the GEMMs consume them
 * (the prepacked weights encode v + 1/2, whose products the correction
 * removes); a GEMM given a_gcorr = NULL computes them from A itself, in its
 * workspace, with the same arithmetic (so the result is the same, bit for bit).
 */
#ifndef W4A8MOE_H
#define W4A8MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4A8MOE_ABI_VERSION 4

typedef enum {
  W4A8_OK = 0,
  W4A8_ERR_INVALID_ARG = 1, /* bad shape, null or misaligned pointer, k > E, ...  */
  W4A8_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement       */
  W4A8_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed             */
  W4A8_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (see below)     */
} w4a8_status;

/* Static text of a status code. */
const char* w4a8_status_string(int status);
/* Detail of the last non-OK status returned on the calling host thread. */
const char* w4a8_last_error(void);
/* W4A8MOE_ABI_VERSION of the loaded library. */
int w4a8_abi_version(void);

/*
 * Reads and clears the device-side error word of the current device
 * (synchronises the device).  Bit 0 (1): a kernel's bounded wait on an
 * mbarrier gave up (W4A8_ERR_TIMEOUT) and that kernel's outputs are invalid.
 * Bit 1 (2): a routed expert id or an expert_map entry was out of range and
 * those pairs were left out.  Bit 2 (4): after such a give-up, waiting for
 * the GEMM's own in-flight MMAs also ran out of time.  For tests and
 * diagnostics, not for the hot path.
 */
int w4a8_device_error(void);

/*
 * (1) Router top-k.  For each token t: the k experts with the largest logits
 * in descending order (equal logits: lower expert id first), and weights
 * p_j = softmax(logits[t])_j; with renormalize != 0 the weights are divided by
 * their sum over the selected experts, i.e. exp(l_j - l_max) / sum_sel.
 * The ids are what the permutation preprocess of the PR #7762 page consumes
 * (run_cutlass_moe_ep_preproess(topk_ids, ...)).
 *   logits   fp32 [T][E]     topk_ids int32 [T][k]     topk_w fp32 [T][k]
 *   1 <= k <= min(E, 32), 1 <= E <= 1024, T >= 0.  NaN logits: undefined order.
 */
int moe_route_topk(const float* logits, int64_t T, int64_t E, int k, int renormalize,
                   int32_t* topk_ids, float* topk_w, void* stream);

/*
 * (2) Permutation preprocess (PR #7762 page, review of ep_moe/kernels.py:
 * stable sort of the flat ids, seg_indptr[E+1] int64, src2dst int32).
 * Flat pair f = t*k + j is routed to expert topk_ids[f].  Pairs are ordered by
 * expert, and within an expert by ascending f (a stable sort).
 *   seg_indptr int64 [E+1]: seg_indptr[e] = first sorted position of expert e,
 *                           seg_indptr[E] = T*k.
 *   src2dst    int32 [T*k]: sorted position of pair f.
 *   dst2src    int32 [T*k]: pair at sorted position j (the inverse).
 * Ids outside [0, E) make the kernel set the device error word (code 2) and
 * the outputs undefined.  1 <= E <= 1024, T*k < 2^31.
 * ws / ws_bytes: workspace of at least w4a8_workspace_bytes(W4A8_OP_PERMUTE,
 * T*k, 0, 0, E) bytes (may be 0 and NULL when that is 0).
 */
int moe_permute(const int32_t* topk_ids, int64_t T, int k, int64_t E, int64_t* seg_indptr,
                int32_t* src2dst, int32_t* dst2src, void* ws, size_t ws_bytes, void* stream);

/*
 * (2') The same preprocess for one expert-parallel shard (PR #7762 page,
 * review of ep_moe/layer.py: with an expert_map the routed ids are translated
 * to local ids before the preprocess, which then runs over the local experts).
 *   expert_map int32 [E] (device): local id in [0, E_local) of each global
 *     expert held by this shard, -1 for an expert held elsewhere; NULL means
 *     the identity (then E_local must equal E and this is moe_permute).
 *   seg_indptr int64 [E_local+1]: segments of the local experts; seg_indptr[E_local]
 *     = P_local, the number of pairs routed to local experts (device side only).
 *   src2dst int32 [T*k]: sorted position of pair f, or -1 when its expert is remote.
 *   dst2src int32 [T*k]: the local pairs at [0, P_local), -1 from P_local on.
 * Local pairs are ordered by local id, and within one by ascending f.  Routed
 * ids outside [0, E) or map entries outside [-1, E_local) set the device error
 * word (code 2) and those pairs are left out.  1 <= E_local <= 1024.
 * ws / ws_bytes: w4a8_workspace_bytes(W4A8_OP_PERMUTE, T*k, 0, 0, E_local).
 */
int moe_permute_ep(const int32_t* topk_ids, int64_t T, int k, int64_t E, const int32_t* expert_map,
                   int64_t E_local, int64_t* seg_indptr, int32_t* src2dst, int32_t* dst2src, void* ws,
                   size_t ws_bytes, void* stream);

/*
 * (3) FP8 E4M3 activation quantisation per token per group of 128 columns
 * ("scale operations on the input hidden states", PR #7762 page, Cutlass W4A8
 * MoE): amax = max|x| over the group, clamped to >= 1e-12 (DeepGEMM PR #53
 * page: clamp amax before the reciprocal), s = amax / 448 (fp32 division),
 * q = E4M3(x / s) (fp32 division; round to nearest even, saturating at +-448
 * as on the PR #37796 page's fp8 write path).
 * Optional gather: output row j reads input row (row_index[j] / row_div); with
 * row_index = NULL output row j reads input row j and M_out must equal M_src.
 * In the MoE this quantises the permuted copy directly (row_index = dst2src,
 * row_div = k); quantisation is per row, so it equals permuting quantised rows.
 * Output rows whose row_index is negative (the -1 tail of an expert-parallel
 * shard's dst2src) are skipped: q, scales and gcorr keep their old contents.
 *   x bf16 [M_src][K]   q uint8 [M_out][K]   scales, gcorr fp32 [K/128][scale_ld]
 *   K % 128 == 0, scale_ld >= M_out, scale_ld % 4 == 0.  gcorr may be NULL.
 *   x and q 16-byte aligned, scales and gcorr 4-byte aligned.
 */
int fp8_quant_per_token_group(const uint16_t* x, int64_t M_src, int64_t K,
                              const int32_t* row_index, int64_t row_div, int64_t M_out,
                              uint8_t* q, float* scales, float* gcorr, int64_t scale_ld, void* stream);

/*
 * (3') The same quantisation of the permuted copy, scattered from the source
 * rows: each row t of x [T][K] is quantised once and its codes, scales and
 * gcorr are written to rows src2dst[t*k + j] of q (j < k); entries of -1 (a
 * pair of another expert-parallel shard) or >= M_out are skipped.  With
 * src2dst from (2) this writes exactly what (3) with row_index = dst2src,
 * row_div = k writes, computing each token's row once instead of k times.
 *   x bf16 [T][K]   src2dst int32 [T*k]   q uint8 [M_out][K]
 *   scales, gcorr fp32 [K/128][scale_ld]   1 <= k <= 32; x and q 16-byte aligned,
 *   scales and gcorr 4-byte aligned; other rules as (3).
 */
int fp8_quant_scatter_per_token_group(const uint16_t* x, int64_t T, int64_t K, const int32_t* src2dst, int k,
                                      int64_t M_out, uint8_t* q, float* scales, float* gcorr, int64_t scale_ld,
                                      void* stream);

/*
 * (4) Grouped int4 x FP8 GEMM (PR #7762 page: CUTLASS W4A8 grouped GEMM,
 * chunk_size 128).  For expert e and rows j in [seg_indptr[e], seg_indptr[e+1]):
 *   C[j][n] = bf16( sum_g a_s[g][j] * b_s[e][g][n] *
 *                   sum_{k in group g} e4m3(A[j][k]) * int4(B[e][n][k]) )
 * accumulated in fp32 per group on the tensor cores and promoted in fp32.
 *   A uint8 [M_total][K] (E4M3 codes)   a_scales, a_gcorr fp32 [K/128][a_scale_ld]
 *   B_prepacked uint8 [E][N][K/2] (w4a8_prepack_weights)   b_scales fp32 [E][K/128][N]
 *   seg_indptr int64 [E+1] (device; seg_indptr[E] must equal M_total)
 *   C bf16 [M_total][N]
 *   K % 128 == 0, N % 128 == 0, 1 <= E <= 1024, M_total < 2^31.
 * Rows outside every segment are not written.
 * a_gcorr may be NULL: the call then first computes the corrections of all
 * M_total rows from A and a_scales (one extra pass over A) into ws, which must
 * hold (K/128) * a_scale_ld fp32 (16-byte aligned; w4a8_workspace_bytes(
 * W4A8_OP_GROUPED_GEMM, M_total, N, K, E) for a_scale_ld = M_total rounded up
 * to 4).  With a_gcorr given, ws may be NULL (none needed).
 * The kernel configuration follows w4a8_grouped_gemm_plan(M_total, E, K):
 * 16-row token tiles, 128-row tiles, or two launches over disjoint experts
 * (those with at most theta rows, counted on the device, on 16-row tiles).
 * Every configuration computes each output element with the same fp32
 * operations.
 */
int w4a8_grouped_gemm(const uint8_t* A, const float* a_scales, const float* a_gcorr,
                      int64_t a_scale_ld, const uint8_t* B_prepacked, const float* b_scales,
                      const int64_t* seg_indptr, int64_t E, int64_t N, int64_t K, int64_t M_total,
                      uint16_t* C, void* ws, size_t ws_bytes, void* stream);

/*
 * (4) for w13 followed by (5), with N = 2I: q, h_scales, h_gcorr are what
 * silu_mul_requant writes for the Y13 that (4) computes (gate rows [0, I),
 * up rows [I, 2I) of each expert's w13).  When the plan of (4) takes the
 * 128-row tiles only, the SiLU and Mul with FP8 requantisation runs in the
 * GEMM's epilogue (the fused L1 epilogue of the DeepGEMM PR #53 page, Changes:
 * L1 GEMM -> SwiGLU -> per-token FP8 requant): a CTA computes the gate block
 * and the up block of the same 128 h-columns in turn, rounds both to bf16
 * (as Y13 would hold them), and forms h, the 128-column amax, the codes, the
 * scale and the correction with the SiLU-and-Mul kernel's arithmetic, so the
 * results equal the unfused ones bit for bit; Y13 is not written.  Otherwise
 * (4) writes Y13 into ws and (5) reads it.
 *   A, a_scales, a_gcorr (may be NULL), B_prepacked, b_scales, seg_indptr, E, K,
 *   M_total as in (4) with N = 2I   q uint8 [M_total][I] (16-byte aligned)
 *   h_scales, h_gcorr fp32 [I/128][h_scale_ld] (h_gcorr may be NULL)
 *   ws: w4a8_workspace_bytes(W4A8_OP_GROUPED_GEMM_SILU, M_total, 2I, K, E)
 *   bytes, 16-byte aligned (Y13 [M_total][2I] bf16, or the bf16 gate values of
 *   the fused epilogue, then the corrections of A when a_gcorr is NULL).
 */
int w4a8_grouped_gemm_silu(const uint8_t* A, const float* a_scales, const float* a_gcorr, int64_t a_scale_ld,
                           const uint8_t* B_prepacked, const float* b_scales, const int64_t* seg_indptr, int64_t E,
                           int64_t I, int64_t K, int64_t M_total, uint8_t* q, float* h_scales, float* h_gcorr,
                           int64_t h_scale_ld, void* ws, size_t ws_bytes, void* stream);
/* The same with the fusion switched off (always (4) then (5)); for comparisons. */
int w4a8_grouped_gemm_silu_unfused(const uint8_t* A, const float* a_scales, const float* a_gcorr,
                                   int64_t a_scale_ld, const uint8_t* B_prepacked, const float* b_scales,
                                   const int64_t* seg_indptr, int64_t E, int64_t I, int64_t K, int64_t M_total,
                                   uint8_t* q, float* h_scales, float* h_gcorr, int64_t h_scale_ld, void* ws,
                                   size_t ws_bytes, void* stream);

/*
 * One-time weight re-layout for the GEMMs (the post-load weight processing of
 * the PR #7762 page, process_weights_after_loading).  Canonical packed int4
 * rows [rows][K/2] -> prepacked rows of the same shape: within each 32-bit
 * word of 8 weights, nibble p holds in bits 0-2 the index m with |v + 1/2| =
 * m + 1/2 and in bit 3 the sign of v of element 4 + p/2 (p even) or (p-1)/2
 * (p odd).  w and out must not overlap.  K % 8 == 0 (K % 128 for the GEMMs).
 */
int w4a8_prepack_weights(const uint8_t* w, int64_t rows, int64_t K, uint8_t* out, void* stream);

/*
 * (5) SiLU and Mul with FP8 re-quantisation of the intermediate (PR #7762
 * page: "handling SiLU and Mul activation functions", scale operations on the
 * intermediate values).  gate_up row m holds gate in columns [0, I) and up in
 * [I, 2I); h = silu(gate) * up = gate / (1 + exp(-gate)) * up in fp32, then
 * the quantisation of (3) on h.
 *   gate_up bf16 [M][2I]   q uint8 [M][I]   scales, gcorr fp32 [I/128][scale_ld]
 *   I % 128 == 0, scale_ld >= M, scale_ld % 4 == 0.  gcorr may be NULL.
 *   gate_up 16-byte aligned, q 8-byte aligned, scales and gcorr 4-byte aligned.
 */
int silu_mul_requant(const uint16_t* gate_up, int64_t M, int64_t I, uint8_t* q, float* scales,
                     float* gcorr, int64_t scale_ld, void* stream);

/*
 * (5') The same over the rows [0, min(M, *m_dev)) only: m_dev (device, int64;
 * NULL = all M rows) is a row count known only on the device, such as
 * seg_indptr[E_local] of an expert-parallel shard (the pairs routed to the
 * shard's experts).  Rows past it are left unwritten.
 */
int silu_mul_requant_rows(const uint16_t* gate_up, int64_t M, const int64_t* m_dev, int64_t I, uint8_t* q,
                          float* scales, float* gcorr, int64_t scale_ld, void* stream);

/*
 * (6) Unpermute and combine (PR #7762 page: post-reordering of the outputs):
 *   out[t][c] = bf16( sum_{j=0..k-1} topk_w[t][j] * Y[src2dst[t*k+j]][c] ),
 * fp32 accumulation in j order.  Slots with src2dst = -1 (pairs of another
 * expert-parallel shard) add nothing; a token with none left gets zeros.
 *   Y bf16 [T*k][H]   src2dst int32 [T*k]   topk_w fp32 [T][k]   out bf16 [T][H]
 *   H % 8 == 0.
 */
int moe_unpermute_combine(const uint16_t* Y, const int32_t* src2dst, const float* topk_w,
                          int64_t T, int k, int64_t H, uint16_t* out, void* stream);

/*
 * (7) Dense W4AFP8 Linear: (4) with one weight matrix and no routing
 * (lyraW4AFp8 page: Machete mixed-input GEMM for the Linear layers).
 *   A uint8 [M][K]   a_scales, a_gcorr fp32 [K/128][a_scale_ld]
 *   B_prepacked uint8 [N][K/2]   b_scales fp32 [K/128][N]   C bf16 [M][N]
 *   K % 128 == 0, N % 128 == 0.
 * ws: w4a8_workspace_bytes(W4A8_OP_LINEAR, M, N, K, 1) bytes, 16-byte
 * aligned, always suffice for a_scale_ld = M rounded up to 4: the split-K
 * partial sums of small-M shapes (w4a8_linear_split_k(M, N, K) > 1), then, at
 * the next 256-byte boundary, the corrections when a_gcorr is NULL (as in
 * (4)).  With a_gcorr given and no split, ws may be NULL.
 */
int w4a8_linear(const uint8_t* A, const float* a_scales, const float* a_gcorr, int64_t a_scale_ld,
                const uint8_t* B_prepacked, const float* b_scales, int64_t M, int64_t N, int64_t K,
                uint16_t* C, void* ws, size_t ws_bytes, void* stream);

/*
 * K splits (1 = none) w4a8_linear uses for this shape on the current device:
 * when the 128-row tiles are fewer than the SMs, each tile's K range is cut
 * into pieces whose fp32 partial sums a second kernel adds.  Diagnostic.
 */
int w4a8_linear_split_k(int64_t M, int64_t N, int64_t K);

/*
 * Launch plan of (4) for M_total rows over E experts at this K: 1 = 16-row
 * token tiles, 2 = 128-row tiles, 3 = both, experts with at most *theta rows
 * (written when theta is not NULL) on the 16-row tiles.  The choice is the
 * expected-cost argmin of the DeepGEMM PR #53 page's tile cost model
 * (Conversation, the cost-model commit: cost = a * R + b * T over the tiles T
 * and the rows R they pad to, in expectation over Poisson row counts),
 * restated for these tiles: in units of one 16-row tile, cost_16(x) =
 * ceil(x / 16), cost_128(x) = 2 * tiles + 0.004 * (rows padded to 16 per tile)
 * (w4a8_tile_cost), theta the largest x with cost_16 <= cost_128 (32), the
 * split plan paying one launch start-up; and the split is kept whenever
 * theta * E < M_total < 128 * E, where skewed routing puts experts on both
 * sides of theta.  0 for an empty or invalid shape.  Host only, no GPU needed.
 */
int w4a8_grouped_gemm_plan(int64_t M_total, int64_t E, int64_t K, int* theta);
/* cost_16 (wide = 0) or cost_128 (wide = 1) of one expert with `rows` rows per
 * 128-row weight block, and its expectation over Poisson(mean_rows) rows. */
double w4a8_tile_cost(int wide, int64_t rows);
double w4a8_expected_tile_cost(int wide, double mean_rows);

/*
 * Test of the bounded waits: one thread waits, with the GEMMs' wait routine and a limit of limit_ns
 * (at most 2e9), on an mbarrier that nothing completes.  The wait gives up, sets *gave_up (device int)
 * to 1 and raises bit 0 of the device error word, as a GEMM wait that times out does (the GEMM then
 * lets its in-flight MMAs finish, bit 2 if that wait itself times out, and returns early; its outputs
 * are invalid).  No TMA or MMA is involved.  There is no counterpart of this call in the method.
 */
int w4a8_test_wait_timeout(uint64_t limit_ns, int* gave_up, void* stream);

/*
 * Test of the GEMMs' in-place tile decode: every CTA of a GEMM launch normally decodes its tiles once into
 * a shared-memory list, and decodes each tile in place (a search over the experts' chunk prefix) only when
 * the list would not fit, which takes launches of hundreds of thousands of rows.  This call bounds the list
 * at max_tiles tiles per CTA for the launches that follow, process-wide (0: always decode in place;
 * negative: no bound, the default).  Results do not depend on it.  Returns W4A8_OK.
 */
int w4a8_test_tile_list_limit(int max_tiles);

/* Operation ids for w4a8_workspace_bytes. */
#define W4A8_OP_PERMUTE 1
#define W4A8_OP_GROUPED_GEMM 2
#define W4A8_OP_LINEAR 3
#define W4A8_OP_GROUPED_GEMM_SILU 4

/* Workspace (bytes) an operation needs for the given shape; 0 = none. */
size_t w4a8_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int64_t E);

/*
 * The whole layer in one call: (1) route -> (2) permute -> (3') quantise the
 * hidden states into their permuted places -> (4) w13 -> (5) SiLU and Mul + requantise -> (4) w2
 * -> (6) combine.  Seven launches (plus the permutation's), nothing else.
 *   x bf16 [T][H]   logits fp32 [T][E]
 *   w13 uint8 [E][2I][H/2] prepacked (rows [0, I) gate, [I, 2I) up)   w13_s fp32 [E][H/128][2I]
 *   w2 uint8 [E][H][I/2] prepacked   w2_s fp32 [E][I/128][H]          out bf16 [T][H]
 *   ws: w4a8_moe_workspace_bytes(T, H, I, E, k) bytes, 256-byte aligned; it
 *   holds the intermediates (ids, weights, permutation, FP8 codes and scales,
 *   Y13, Y2), whose offsets are given by w4a8_moe_workspace_layout.
 */
int w4a8_moe_forward(const uint16_t* x, const float* logits, int64_t T, int64_t H, int64_t I,
                     int64_t E, int k, int renormalize, const uint8_t* w13, const float* w13_s,
                     const uint8_t* w2, const float* w2_s, uint16_t* out, void* ws,
                     size_t ws_bytes, void* stream);
size_t w4a8_moe_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int k);

/*
 * One expert-parallel shard of the layer (PR #7762 page, ep-moe mode and the
 * expert_map review of ep_moe/layer.py): routing over all E experts, then
 * (2') with expert_map, and the rest over the pairs routed to this shard's
 * E_local experts only.  out is this shard's share of the layer output (the
 * sum over the shards' shares, taken outside this call, is the layer).
 *   logits fp32 [T][E]   expert_map int32 [E] (device; see moe_permute_ep)
 *   w13, w13_s, w2, w2_s: the E_local local experts, laid out as in
 *   w4a8_moe_forward with E_local in place of E.  1 <= E_local <= E.
 *   ws: w4a8_moe_workspace_bytes(T, H, I, E, k) bytes (the same layout).
 * The row count P_local stays on the device: quantisation, SiLU and the
 * GEMMs read it from seg_indptr, so no host synchronisation is added.
 */
int w4a8_moe_forward_ep(const uint16_t* x, const float* logits, int64_t T, int64_t H, int64_t I,
                        int64_t E, int k, int renormalize, const int32_t* expert_map, int64_t E_local,
                        const uint8_t* w13, const float* w13_s, const uint8_t* w2, const float* w2_s,
                        uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/*
 * w4a8_moe_forward without a workspace: for callers that cannot allocate
 * device memory, such as a plugin whose host application owns the device
 * allocator and passes in only the layer's inputs and outputs, or a C program
 * that must not allocate after start-up.  The pages have no counterpart of
 * this call; it exists for those callers.
 *   Same arguments as w4a8_moe_forward, minus ws / ws_bytes.  The
 *   intermediates live in a fixed array of w4a8_moe_noalloc_scratch_bytes()
 *   (64 MiB) inside the library, which every GPU that loads the library keeps
 *   until the process exits.  A layer whose w4a8_moe_workspace_bytes() exceeds
 *   that is rejected with W4A8_ERR_INVALID_ARG before anything is launched.
 *   The call itself never calls cudaMalloc / cudaFree or any allocating routine.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  With CUDA's lazy module loading (the default),
 *   that first call may also be when the driver places the array in the
 *   device's memory: a caller whose allocator is to own the rest of the
 *   device should make it at start-up, before handing memory to that allocator.  All calls share the one array and it keeps the
 *   last call's contents: calls that overlap on the GPU (other streams, other
 *   host threads) race and corrupt each other; order them on one stream.
 */
int w4a8_moe_forward_noalloc(const uint16_t* x, const float* logits, int64_t T, int64_t H, int64_t I,
                             int64_t E, int k, int renormalize, const uint8_t* w13, const float* w13_s,
                             const uint8_t* w2, const float* w2_s, uint16_t* out, void* stream);
size_t w4a8_moe_noalloc_scratch_bytes(void);

/* Byte offsets of the intermediates inside the w4a8_moe_forward workspace. */
typedef struct {
  size_t topk_ids, topk_w, seg_indptr, src2dst, dst2src, xq, xs, xc, y13, hq, hs, hc, y2, permute_ws;
  int64_t scale_ld; /* leading dimension of xs and hs: T*k rounded up to 4 */
  size_t total;
} w4a8_moe_layout;
int w4a8_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int k,
                              w4a8_moe_layout* layout /* host pointer */);

#ifdef __cplusplus
}
#endif
#endif /* W4A8MOE_H */
