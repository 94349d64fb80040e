/*
 * bimoe.h -- C ABI of the batch-invariant MoE hot path for GB300 (sm_103a).
 *
 * One library, libbimoe.so, holding hand-written CUDA kernels.  Every entry
 * point takes plain device pointers owned by the caller plus sizes and a CUDA
 * stream, launches asynchronously on that stream, never synchronises the
 * host and never allocates device memory.  bi_router_gemm, bi_topk,
 * bi_moe_forward and the stage entry points are safe to capture in a CUDA
 * graph (argument checks are host-side; nothing reads device memory on the
 * host).
 *
 * Batch invariance contract: for fixed weights and fixed (N,K) resp.
 * (H,E,top_k,I), every output row of every entry point is bit-identical
 * whatever M is and whatever other rows share the call.  Nothing in the
 * library keys any arithmetic on M; M only sizes grids and schedules.
 *
 * Layouts are row-major and contiguous.  "bf16" arguments are bfloat16
 * values stored as 16-bit patterns.  Device pointers must be 16-byte
 * aligned where stated (TMA operands).
 *
 * Errors: entry points return bi_status.  BI_ERR_INVALID_ARG for a null
 * required pointer, a negative size, a misaligned pointer or top_k outside
 * its range; BI_ERR_UNSUPPORTED for a shape that has no kernel (the library
 * never falls back to another recipe); BI_ERR_WORKSPACE for a workspace that
 * is too small; BI_ERR_CUDA when a launch fails.  M == 0 returns BI_OK and
 * launches nothing.  A kernel that detects bad data (an expert id outside
 * [0,E), repeated experts in one row, offsets / perm handed to a stage call
 * that are not a grouping of the pairs) or whose bounded wait times out
 * records a code in a device-side error word and skips what it cannot do
 * safely; bi_device_error() reads it.
 * bi_last_error_message() returns a human-readable detail of the last
 * failing call on this host thread.
 */
#ifndef BIMOE_H_
#define BIMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define BI_API __attribute__((visibility("default")))
#else
#define BI_API
#endif

/* A cudaStream_t (NULL = legacy default stream). */
typedef struct CUstream_st *bi_stream_t;
/* bfloat16 storage. */
typedef uint16_t bi_bf16;

typedef enum {
  BI_OK = 0,
  BI_ERR_INVALID_ARG = 1,
  BI_ERR_UNSUPPORTED = 2,
  BI_ERR_WORKSPACE = 3,
  BI_ERR_CUDA = 4,
  BI_ERR_DEVICE = 5 /* bad data or a bounded wait timed out on the device */
} bi_status;

/* Device error codes recorded by kernels (bi_device_error). */
#define BI_DEVERR_NONE 0
#define BI_DEVERR_BAD_EXPERT_ID 1   /* id outside [0,E) */
#define BI_DEVERR_REPEATED_EXPERT 2 /* one row routed twice to one expert */
#define BI_DEVERR_WAIT_TIMEOUT 3    /* an mbarrier wait exceeded its limit */
#define BI_DEVERR_BAD_PERMUTATION 4 /* offsets / perm given to a stage call are not
                                       a grouping of the M*top_k pairs */

BI_API const char *bi_status_str(bi_status s);
BI_API const char *bi_last_error_message(void);
BI_API const char *bi_version(void);

/*
 * bi_device_error -- read and clear the device error word of the current
 * device.  Synchronises the device.  *code receives a BI_DEVERR_* value.
 * Returns BI_ERR_CUDA if the read fails.
 */
BI_API bi_status bi_device_error(int32_t *code);

/*
 * bi_cast_bf16_to_f32 -- y[i] = float(x[i]) for i < n, exact.
 * The router reads fp32 activations: MoE-layer activations arrive in bf16
 * and widen exactly, so scores never round through bf16 (GateLinear router
 * page, section "What").  x: n bf16, y: n fp32 (device).
 */
BI_API bi_status bi_cast_bf16_to_f32(const bi_bf16 *x, float *y, int64_t n,
                                     bi_stream_t stream);

/*
 * bi_router_gemm -- fp32 router GEMM  y = x W^T (+ bias).
 * Source: "[BI][DSv4] Batch-invariant GateLinear router with fp32
 * persistent matmul", sections "What" and "A correction to why the key
 * excludes M": fp32 scores, bias preserved, one reduction recipe that does
 * not depend on M.
 *   x    [M,K] fp32 row-major (device), ld = K
 *   w    [N,K] fp32 row-major (device), the nn.Linear weight used as W^T
 *   bias [N] fp32 (device) or NULL
 *   y    [M,N] fp32 row-major (device), written
 * Reduction recipe (fixed by K alone, never by M): K is cut into K/128
 * contiguous slices; slice s is an fp32 fused-multiply-add chain over
 * k = 128s .. 128s+127 in increasing k starting from +0.0; the slice results
 * are added in slice order starting from +0.0; the bias is added last.  All
 * schedules (chosen from M) evaluate exactly this sequence per element.
 * Requirements: K % 128 == 0, 1 <= N <= 4096, x/w 16-byte aligned.
 * Otherwise BI_ERR_UNSUPPORTED / BI_ERR_INVALID_ARG.
 */
BI_API bi_status bi_router_gemm(const float *x, const float *w, const float *bias,
                                float *y, int64_t M, int64_t K, int64_t N,
                                bi_stream_t stream);

/*
 * bi_router_gemm_bf16 -- bi_router_gemm with bf16 x: y[i,n] from the fp32
 * values of x[i,:] (a bf16 value converts to fp32 exactly), so the result is
 * bit for bit bi_router_gemm(float(x)) under every schedule.  The MoE layer's
 * tokens are bf16 and the router wants fp32 scores ("[BI][DSv4]
 * Batch-invariant GateLinear router with fp32 persistent matmul", section
 * "What": routing through bf16 would round the scores): reading x as bf16
 * removes the separate fp32 copy of the tokens and halves their reads.
 *   x [M,K] bf16 row-major (device, 16-byte aligned); w, bias, y, M, K, N and
 *   errors as bi_router_gemm.
 */
BI_API bi_status bi_router_gemm_bf16(const bi_bf16 *x, const float *w, const float *bias,
                                     float *y, int64_t M, int64_t K, int64_t N,
                                     bi_stream_t stream);
/*
 * bi_topk -- sigmoid scoring and deterministic top-k expert selection.
 * Source: "[BI][DSv4] Pin sparse-MLA decode and prefill scheduling under
 * batch invariance", commit log, deterministic per-row top-k commit: score
 * descending, exact ties broken by ascending index, -0.0 equal to +0.0,
 * ranking on a monotone int32 key of the fp32 score, no shared-memory
 * atomics.
 *   scores [M,E] fp32 (device): router outputs
 *   probs  [M,E] fp32 (device) or NULL: sigmoid of every score, written
 *   ids    [M,top_k] int32 (device), written: ids[m,t] = rank-t expert
 *   wts    [M,top_k] fp32 (device), written: sigmoid(scores[m, ids[m,t]])
 * Selection is on the fp32 score (sigmoid is monotone, so this is the
 * selection by probability without ties manufactured by rounding the
 * sigmoid).  One warp per row.  Requirements: 1 <= E <= 512,
 * 1 <= top_k <= min(E, 16).
 */
BI_API bi_status bi_topk(const float *scores, float *probs, int32_t *ids,
                         float *wts, int64_t M, int64_t E, int32_t top_k,
                         bi_stream_t stream);

/*
 * bi_topk_window -- deterministic per-row top-k over a column window (the
 * sparse-MLA indexer's selection): "[BI][DSv4] Pin sparse-MLA decode and
 * prefill scheduling under batch invariance", commit log (the deterministic
 * per-row top-k commit, the masked-lane fix and the validity-first ranking
 * commits).
 *   scores    [n_rows, ld] fp32 (device), the first num_cols columns used;
 *   row_start, row_end  [n_rows] int64 (device) or NULL (whole rows); the
 *             window of row i is [rs, re) with rs = clamp(row_start[i], 0,
 *             num_cols), re = clamp(row_end[i], 0, num_cols), empty if re <= rs;
 *   out       [n_rows, k] int32 (device, written): the chosen columns as
 *             window-relative indices (column - rs) in ascending order, then
 *             -1 up to k.
 * Chosen: the min(k, window size) in-window columns ranked first by the
 * monotone int32 key of the fp32 score (descending; -0.0 equals +0.0; NaN
 * patterns are ordered by their bits, +NaN above +inf, -NaN below -inf), equal
 * keys by ascending column.  Out-of-window columns are never chosen, whatever
 * they hold.  A pure function of each row: no atomics decide ties.
 * Limits: num_cols <= 8192 (else BI_ERR_UNSUPPORTED), 1 <= k <= 8192,
 * ld >= num_cols.  n_rows == 0 is a no-op.
 */
BI_API bi_status bi_topk_window(const float *scores, int64_t ld,
                                const int64_t *row_start, const int64_t *row_end,
                                int64_t n_rows, int64_t num_cols, int32_t k,
                                int32_t *out, bi_stream_t stream);

/*
 * bi_router_topk -- bi_router_gemm followed by bi_topk on its scores, as one
 * call for the decode path.  The scores y are exactly bi_router_gemm's (same
 * recipe, same bits) and ids / wts / probs exactly bi_topk's on y.
 * The selection grid is launched as a programmatic dependent of the router
 * grid (programmatic stream serialization: it waits in hardware for the
 * router's completion before reading y).  A one-kernel path exists for up
 * to 4 rows (N a multiple of 16 up to 256, K a multiple of 1024): a
 * thread-block cluster of N/16 CTAs owns all N scores of the rows (CTA c
 * computes columns 16c..16c+15 with the same per-element recipe) and after a
 * cluster barrier one warp per row selects from the scores in the cluster's
 * shared memory (bi_router_topk_schedule, schedule 10).  Both give the same
 * bits.  The pages keep the router
 * ("[BI][DSv4] Batch-invariant GateLinear router with fp32 persistent
 * matmul", whose Perf table puts the decode-size router cost in microseconds
 * per layer) and the selection as separate ops; they have no combined
 * counterpart.
 *   x, w, bias, y, M, K, N  as bi_router_gemm (N <= 512);
 *   probs, ids, wts, top_k  as bi_topk on y (top_k <= min(16, N)).
 * Errors as bi_router_gemm / bi_topk.  Stream-ordered, graph-capturable.
 */
BI_API bi_status bi_router_topk(const float *x, const float *w, const float *bias,
                                float *y, float *probs, int32_t *ids, float *wts,
                                int64_t M, int64_t K, int64_t N, int32_t top_k,
                                bi_stream_t stream);
/*
 * bi_router_topk_bf16 -- bi_router_topk with bf16 x, i.e. bi_router_gemm_bf16
 * followed by bi_topk on its scores (same bits as bi_router_topk(float(x))).
 */
BI_API bi_status bi_router_topk_bf16(const bi_bf16 *x, const float *w, const float *bias,
                                     float *y, float *probs, int32_t *ids, float *wts,
                                     int64_t M, int64_t K, int64_t N, int32_t top_k,
                                     bi_stream_t stream);
/*
 * bi_moe_workspace_bytes -- bytes of device workspace bi_moe_forward needs
 * for these sizes (a multiple of 256).  Returns 0 for invalid sizes.  The
 * pages have no counterpart: their fused-MoE keeps its buffers inside the
 * framework; this library leaves every allocation to the caller, so it states
 * the size.  The workspace holds the permutation (offsets, pair ids, a mask of
 * valid slots per token), the gathered token rows, the activations and the
 * fp32 per-slot contributions.
 */
BI_API size_t bi_moe_workspace_bytes(int64_t M, int64_t H, int64_t E,
                                     int32_t top_k, int64_t I);

/*
 * bi_moe_forward -- batch-invariant fused-MoE expert path.
 * Source: "Batch-invariance generation with vLLM fused-MoE backend at
 * improved performance", section "What's included" and the strict-review
 * summary: permute tokens by expert; gate/up grouped GEMM with fp32
 * accumulation, a fixed K step and no split-K; SwiGLU with the routing
 * probability applied at the activation (fp32 math, one bf16 round, gate
 * half = rows [0,I) of each expert's W13, up half = rows [I,2I)); down
 * grouped GEMM (fp32 accumulation, fixed K step, no split-K); top-k sum with
 * unit weights in slot order t = 0..top_k-1 in fp32, one bf16 round.
 *   x    [M,H] bf16 (device, 16-byte aligned)
 *   ids  [M,top_k] int32 (device): distinct experts per row in [0,E)
 *   wts  [M,top_k] fp32 (device): routing probabilities
 *   w13  [E,2I,H] bf16 (device, 16-byte aligned)
 *   w2   [E,H,I] bf16 (device, 16-byte aligned)
 *   out  [M,H] bf16 (device), written
 *   workspace: >= bi_moe_workspace_bytes(...) bytes of device memory,
 *   256-byte aligned, owned by the caller, contents need not be initialised.
 * Requirements: H % 128 == 0, I % 128 == 0, 1 <= E <= 1024,
 * 1 <= top_k <= 16, M * top_k < 2^31.
 * Bad routing data: a slot whose expert id is outside [0,E), or repeats an
 * earlier slot of its row, is skipped (BI_DEVERR_BAD_EXPERT_ID /
 * BI_DEVERR_REPEATED_EXPERT in the device error word) and adds nothing: that
 * token's output is the slot-order sum over its valid slots (+0 if none).
 * Launches: the permutation, gather, gate/up, down and combine kernels; for
 * decode-sized batches (M * top_k <= 32) two kernels, gate/up and down, each
 * deriving the same routing from ids in every CTA, gate/up gathering its
 * token rows itself and down summing each token's contributions in slot
 * order as the last of them lands.  Same bits either way.
 */
BI_API bi_status bi_moe_forward(const bi_bf16 *x, const int32_t *ids,
                                const float *wts, const bi_bf16 *w13,
                                const bi_bf16 *w2, bi_bf16 *out, int64_t M,
                                int64_t H, int64_t E, int32_t top_k, int64_t I,
                                void *workspace, size_t workspace_bytes,
                                bi_stream_t stream);

/*
 * bi_moe_layer -- the whole hot path of one MoE layer in one call: the fp32
 * router on the bf16 tokens (read as their exact fp32 values), sigmoid top-k,
 * and the expert path; the bits of bi_router_topk_bf16 followed by
 * bi_moe_forward, whose contracts it combines.  The pages' router and
 * fused-MoE are separate ops; this library adds the combination so that a
 * decode-sized batch (M * top_k <= 32) runs in two or three launches: the
 * router, then the expert GEMMs, whose every CTA selects the rows' experts
 * from the scores itself (bi_topk's selection; one CTA writes ids / wts),
 * with the combine fused into the down GEMM: one launch for both GEMMs
 * where the gate/up tiles fit one wave on the SMs (bi_moe_decode_fused),
 * else a gate/up launch and a down launch.  Larger batches: router,
 * selection grid, bi_moe_forward's kernels.
 *   x        [M,H] bf16 (device, 16-byte aligned)
 *   w_router [E,H] fp32 (device, 16-byte aligned); bias [E] fp32 or NULL
 *   w13, w2, out, workspace: as bi_moe_forward (workspace >=
 *            bi_moe_workspace_bytes(M, H, E, top_k, I))
 *   scores   [M,E] fp32, ids [M,top_k] int32, wts [M,top_k] fp32 (device,
 *            written): as bi_router_topk's y, ids, wts
 * Requirements: those of bi_moe_forward and bi_router_gemm, and E <= 512.
 */
BI_API bi_status bi_moe_layer(const bi_bf16 *x, const float *w_router, const float *bias,
                              const bi_bf16 *w13, const bi_bf16 *w2, bi_bf16 *out,
                              float *scores, int32_t *ids, float *wts, int64_t M,
                              int64_t H, int64_t E, int32_t top_k, int64_t I,
                              void *workspace, size_t workspace_bytes, bi_stream_t stream);

/* ---- the stages of bi_moe_forward, callable one by one (same contracts) --
 *
 * bi_moe_permute -- group the M*top_k (token, slot) pairs by expert, stable
 * (by expert, then token, then slot).  offsets [E+1] int32 written:
 * offsets[e] = first position of expert e, offsets[E] = M*top_k.
 * perm [M*top_k] int32 written: perm[p] = token*top_k + slot at position p.
 * workspace: >= bi_moe_permute_workspace_bytes(M, E) bytes.
 * Integer-only and deterministic (counts and bit masks, no ordering by
 * atomics).
 */
BI_API size_t bi_moe_permute_workspace_bytes(int64_t M, int64_t E);
BI_API bi_status bi_moe_permute(const int32_t *ids, int32_t *offsets,
                                int32_t *perm, int64_t M, int64_t E,
                                int32_t top_k, void *workspace,
                                size_t workspace_bytes, bi_stream_t stream);

/*
 * bi_moe_gather -- x_perm[p, :] = x[perm[p] / top_k, :] for every permuted
 * position p < offsets[E]: the token rows in expert order, contiguous so the
 * gate/up GEMM can stream them with TMA.  x [M,H] bf16; x_perm [M*top_k, H]
 * bf16 (device, written; 16-byte aligned).  Rows at positions >= offsets[E]
 * are left untouched.
 * Bad grouping (offsets[E] outside [0, M*top_k], or a perm entry outside
 * [0, M*top_k)): those positions are not copied and BI_DEVERR_BAD_PERMUTATION
 * is recorded in the device error word.
 */
BI_API bi_status bi_moe_gather(const bi_bf16 *x, const int32_t *offsets,
                               const int32_t *perm, bi_bf16 *x_perm, int64_t M,
                               int64_t H, int64_t E, int32_t top_k,
                               bi_stream_t stream);

/*
 * bi_moe_gate_up -- act[p, j] = bf16(silu(g) * u * wts[perm[p]]) for every
 * permuted position p < M*top_k, with g/u the gate/up projections of row p
 * of x_perm by the expert owning position p (tcgen05 bf16 MMA, fp32
 * accumulation in tensor memory, K step 64, no split-K).
 *   x_perm [M*top_k, H] bf16 from bi_moe_gather (16-byte aligned);
 *   offsets/perm from bi_moe_permute; wts [M,top_k] fp32;
 *   w13 [E,2I,H] bf16 (16-byte aligned); act [M*top_k, I] bf16 (written).
 * Bad grouping: offsets that are not non-decreasing inside [0, M*top_k]
 * make the kernel compute nothing; a perm entry outside [0, M*top_k) gets
 * probability 0.  Either records BI_DEVERR_BAD_PERMUTATION (device error
 * word); nothing is read or written outside the arguments' extents.
 */
BI_API bi_status bi_moe_gate_up(const bi_bf16 *x_perm, const int32_t *offsets,
                                const int32_t *perm, const float *wts,
                                const bi_bf16 *w13, bi_bf16 *act, int64_t M,
                                int64_t H, int64_t E, int32_t top_k, int64_t I,
                                bi_stream_t stream);

/*
 * bi_moe_gate_up_tokens -- bi_moe_gate_up reading the token rows straight
 * from x [M,H] bf16 (16-byte aligned) instead of a gathered copy: the GEMM
 * fetches row perm[p] / top_k of x for position p with TMA gather loads
 * (tile::gather4).  Same result bits as bi_moe_gather + bi_moe_gate_up;
 * other arguments, requirements and bad-grouping behaviour as
 * bi_moe_gate_up.  Slower than the gathered copy for large batches (the TMA
 * gathers 128-byte rows far slower than the MMAs consume them), so
 * bi_moe_forward uses it only when bi_moe_gate_up_feed selects it.
 */
BI_API bi_status bi_moe_gate_up_tokens(const bi_bf16 *x, const int32_t *offsets,
                                       const int32_t *perm, const float *wts,
                                       const bi_bf16 *w13, bi_bf16 *act, int64_t M,
                                       int64_t H, int64_t E, int32_t top_k, int64_t I,
                                       bi_stream_t stream);

/*
 * bi_moe_down -- contrib[perm[p], h] = sum_j act[p,j] * W2[e,h,j] for every
 * permuted position p (tcgen05 bf16 MMA, fp32 accumulation, K step 64, no
 * split-K).  act [M*top_k, I] bf16 (16-byte aligned); w2 [E,H,I] bf16;
 * contrib [M*top_k, H] fp32 (row = token*top_k + slot), written.
 * Bad grouping: offsets that are not non-decreasing inside [0, M*top_k]
 * make the kernel compute nothing; a position whose perm entry is outside
 * [0, M*top_k) is not stored.  Either records BI_DEVERR_BAD_PERMUTATION.
 */
BI_API bi_status bi_moe_down(const bi_bf16 *act, const int32_t *offsets,
                             const int32_t *perm, const bi_bf16 *w2,
                             float *contrib, int64_t M, int64_t H, int64_t E,
                             int32_t top_k, int64_t I, bi_stream_t stream);

/*
 * bi_moe_combine -- out[m,h] = bf16(((c[m,0,h] + c[m,1,h]) + ...) +
 * c[m,top_k-1,h]) in fp32, slot order, unit weights (the top-k sum of the
 * fused-MoE page, section "What's included": a fixed `for t in range(topk)`
 * order, the probabilities already applied at the activation).
 * contrib [M,top_k,H] fp32; out [M,H] bf16 (device, written).
 */
BI_API bi_status bi_moe_combine(const float *contrib, bi_bf16 *out, int64_t M,
                                int64_t H, int32_t top_k, bi_stream_t stream);

/*
 * bi_moe_combine_consume -- bi_moe_combine (same arguments, checks and
 * result bits) for a caller that never reads contrib again: once a line of
 * contrib has been summed it is dropped from L2 without being written back
 * to memory (discard.global.L2), so contributions still cached when the
 * combine runs cost no DRAM write.  contrib's contents are indeterminate
 * afterwards.  The drop applies when H is a multiple of 32 and contrib is
 * 128-byte aligned (each 128-byte line then belongs to one (token, slot)
 * row); otherwise the call is exactly bi_moe_combine.  bi_moe_forward
 * combines this way into its own workspace.
 */
BI_API bi_status bi_moe_combine_consume(float *contrib, bi_bf16 *out, int64_t M,
                                        int64_t H, int32_t top_k, bi_stream_t stream);

/* ---- expert parallelism: the two data-layout steps around the exchange --
 *
 * With the experts split over R ranks (rank r owns experts
 * [r*E/R, (r+1)*E/R)), a token's k contributions are computed on the ranks
 * that own its experts and must return to the token's home rank, where they
 * are summed in slot order: then every output bit is the single-GPU layer's
 * ("Batch-invariance generation with vLLM fused-MoE backend at improved
 * performance", sections "Summary" and "Usage": expert parallelism over 8
 * GPUs with the fused-MoE backend).  The home rank groups its pairs by expert
 * (bi_moe_permute, which also groups them by destination rank), gathers the
 * token rows (bi_moe_gather) and their routing (bi_moe_gather_routing), and
 * sends each rank its contiguous range of positions; the receiving rank runs
 * the expert GEMMs on the rows it received (top_k = 1, pair id = row) and
 * sends the fp32 contribution rows back in the order it received them; the
 * home rank puts them back in (token, slot) order (bi_moe_scatter_contrib)
 * and combines them in slot order (bi_moe_combine).
 *
 * bi_moe_gather_routing -- for every permuted position p < offsets[E]:
 *   lid[p] = ids[perm[p]] % experts_per_rank   (the expert's index on its rank)
 *   pw[p]  = wts[perm[p]]                      (the routing probability)
 *   ids [M,top_k] int32, wts [M,top_k] fp32, offsets [E+1] / perm [M*top_k]
 *   from bi_moe_permute; lid [M*top_k] int32 and pw [M*top_k] fp32 (device,
 *   written for p < offsets[E]).  experts_per_rank must divide E.
 *   A perm entry outside [0, M*top_k) or offsets[E] outside that range:
 *   the position is skipped and BI_DEVERR_BAD_PERMUTATION recorded.
 */
BI_API bi_status bi_moe_gather_routing(const int32_t *ids, const float *wts,
                                       const int32_t *offsets, const int32_t *perm,
                                       int32_t *lid, float *pw, int64_t M, int64_t E,
                                       int32_t top_k, int64_t experts_per_rank,
                                       bi_stream_t stream);

/*
 * bi_moe_scatter_contrib -- contrib[perm[p], :] = rows[p, :] for every
 * permuted position p < offsets[E]: fp32 contribution rows that came back in
 * the permuted order, put back at row token*top_k + slot.
 *   rows [M*top_k, H] fp32, contrib [M*top_k, H] fp32 (device, 16-byte
 *   aligned; rows of pairs that were skipped are not written).  H % 4 == 0.
 *   Bad grouping as bi_moe_gather_routing.
 */
BI_API bi_status bi_moe_scatter_contrib(const float *rows, const int32_t *offsets,
                                        const int32_t *perm, float *contrib, int64_t M,
                                        int64_t H, int64_t E, int32_t top_k,
                                        bi_stream_t stream);

/*
 * bi_moe_forward_noalloc -- bi_moe_forward without a caller-provided
 * workspace, for callers that cannot allocate device memory where they run
 * the layer (code inside an allocator or memory-pool callback, runtimes that
 * own all device memory and forbid allocations behind their back).  This
 * entry point has no counterpart in the papers; it exists only for such
 * callers.
 *
 * Arguments, layouts, requirements and results are those of bi_moe_forward
 * (same kernels, same bits).  The scratch space is a fixed array of
 * BI_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library's device code: every
 * GPU that loads the library holds it until the process exits.  Sizes whose
 * bi_moe_workspace_bytes() exceeds it are rejected with BI_ERR_WORKSPACE and
 * a message naming both sizes (64 MiB covers e.g. 605 tokens of H=2048,
 * E=128, top-8, I=768, or 291 tokens of H=4096, E=256, top-8, I=2048).
 * The call never allocates or frees device memory.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it for the
 * current CUDA context; the first call after the context changes (after a
 * cudaDeviceReset, or from a context other than the device's primary one)
 * looks it up again.  Make the first call of each context before any stream
 * capture begins.
 *
 * All calls on a device share the one array and it keeps the previous
 * call's contents; nothing in it needs to start at zero, because every call
 * writes each scratch byte it reads before reading it.  Calls whose
 * executions overlap on the GPU (different streams, or host threads issuing
 * concurrently without ordering) race on the array and give undefined
 * results: order them on one stream.
 */
#define BI_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
BI_API bi_status bi_moe_forward_noalloc(const bi_bf16 *x, const int32_t *ids,
                                        const float *wts, const bi_bf16 *w13,
                                        const bi_bf16 *w2, bi_bf16 *out,
                                        int64_t M, int64_t H, int64_t E,
                                        int32_t top_k, int64_t I,
                                        bi_stream_t stream);

/* ======================================================================
 * TEST AND MEASUREMENT HOOKS.  Not part of the hot path and not needed to
 * use it: the test-suite and the benchmark call these to force schedules
 * (and show the bits do not depend on them), to run the negative control,
 * to measure the FP32 peak and to exercise the bounded-wait discipline.
 * ====================================================================== */

/*
 * bi_router_gemm_schedule -- test hook: bi_router_gemm with the schedule
 * forced (0 = automatic by M, 1 = per-row warp kernel, 2 = slice-parallel
 * tile kernel, 3 = register-tiled kernel, 4 = slices spread over a cluster
 * of CTAs with the lane tile picked from M, 5..8 = the same with the lane
 * tile forced to 2x2, 4x2, 4x4, 8x4 outputs, 9 = register-tiled kernel
 * with 7x8 outputs per thread).  Schedules 4..8 need K/128 to split into
 * 2..8 CTAs of 4 or 8 slices, schedule 9 K/128 even (N > 128) or a multiple
 * of 4 (N <= 128) (else BI_ERR_UNSUPPORTED).  Every schedule computes the same recipe; tests use
 * this to show that the bits do not depend on it.
 */
BI_API bi_status bi_router_gemm_schedule(const float *x, const float *w,
                                         const float *bias, float *y, int64_t M,
                                         int64_t K, int64_t N, int32_t schedule,
                                         bi_stream_t stream);

/* test hook: bi_router_gemm_bf16 with the schedule forced (as bi_router_gemm_schedule) */
BI_API bi_status bi_router_gemm_bf16_schedule(const bi_bf16 *x, const float *w,
                                              const float *bias, float *y, int64_t M,
                                              int64_t K, int64_t N, int32_t schedule,
                                              bi_stream_t stream);


/*
 * bi_router_gemm_splitk_negctl -- NEGATIVE CONTROL, test use only.  Same
 * signature as bi_router_gemm but its K split depends on M (one chain over
 * all of K for M > 16, sixteen 256-long slices for M <= 16), the kind of
 * batch-dependent reduction the GateLinear page diagnoses in the default
 * route.  Row bits change across that boundary; the tests assert that they
 * do, to prove the invariance tests can fail.
 */
BI_API bi_status bi_router_gemm_splitk_negctl(const float *x, const float *w,
                                              const float *bias, float *y,
                                              int64_t M, int64_t K, int64_t N,
                                              bi_stream_t stream);

/*
 * bi_router_topk_schedule -- test hook: bi_router_topk with the path forced:
 * 0 automatic, 1..9 the router schedule of bi_router_gemm_schedule followed
 * by the selection grid, 10 the one-kernel cluster path (BI_ERR_UNSUPPORTED
 * for a shape it does not take, M > 4, or a cluster the device cannot
 * schedule).  bi_router_topk_bf16_schedule: the same for bf16 x.
 */
BI_API bi_status bi_router_topk_schedule(const float *x, const float *w,
                                         const float *bias, float *y, float *probs,
                                         int32_t *ids, float *wts, int64_t M, int64_t K,
                                         int64_t N, int32_t top_k, int32_t schedule,
                                         bi_stream_t stream);
BI_API bi_status bi_router_topk_bf16_schedule(const bi_bf16 *x, const float *w,
                                              const float *bias, float *y, float *probs,
                                              int32_t *ids, float *wts, int64_t M, int64_t K,
                                              int64_t N, int32_t top_k, int32_t schedule,
                                              bi_stream_t stream);

/*
 * bi_moe_gemm_variant -- selects how the expert GEMMs (bi_moe_gate_up,
 * bi_moe_down and the two GEMMs inside bi_moe_forward) are scheduled, for
 * the whole process, from the next call on:
 *   0  automatic (the default): for batches of at most 16 (token, expert)
 *      pairs per expert on average (M * top_k <= 16 E), one CTA per tile
 *      with narrow token tiles (for gate/up with interleaved rows, as 4,
 *      when min(E, M * top_k) * I / 64 tiles fit on the SMs); otherwise CTA pairs whenever the GEMM's
 *      output features (I for gate/up, H for down) are a multiple of 256,
 *      else one CTA per tile, and for gate/up with H >= 4096 and at least
 *      64 pairs per expert on average, CTA pairs with interleaved gate/up
 *      rows;
 *   1  one CTA per tile (128 weight rows), tcgen05 cta_group::1;
 *   2  CTA pairs (256 weight rows over two SMs of a cluster), cta_group::2;
 *      a call whose output features are not a multiple of 256 then fails
 *      with BI_ERR_UNSUPPORTED;
 *   3  gate/up: CTA pairs whose CTAs each hold 64 gate rows and the matching
 *      64 up rows (one M=256 x N=256 MMA per K step, any I % 128 == 0);
 *      down: as 2;
 *   4  gate/up: one CTA per tile holding 64 gate rows and the matching 64 up
 *      rows (one M=128 MMA per K step, any I % 64 == 0); down: as 1.
 * All variants evaluate the same per-element K order, so the bits do not
 * depend on the choice (tests compare them).  *previous (may be NULL)
 * receives the old setting.  Other values: BI_ERR_INVALID_ARG.  Not
 * synchronised with calls in flight on other host threads.
 */
BI_API bi_status bi_moe_gemm_variant(int32_t variant, int32_t *previous);

/*
 * bi_moe_gate_up_feed -- how bi_moe_forward feeds the gate/up GEMM its token
 * rows, for the whole process from the next call on: 0 automatic (the
 * default: the copy), 1 a contiguous copy made by the gather kernel first
 * (bi_moe_gather + bi_moe_gate_up), 2 gathered by the GEMM
 * (bi_moe_gate_up_tokens).  Same bits either way (tests compare them).
 * *previous (may be NULL) receives the old setting; other values
 * BI_ERR_INVALID_ARG.
 */
BI_API bi_status bi_moe_gate_up_feed(int32_t mode, int32_t *previous);

/*
 * bi_moe_decode_fused -- how bi_moe_layer runs the expert GEMMs of a
 * decode-sized batch (M * top_k <= 32 under the automatic variant, with
 * 64-feature interleaved gate/up tiles, i.e. min(E, M * top_k) * I / 64 at
 * most the SM count), for the whole process from the next call on:
 *   0  automatic (the default): one launch (its gate/up tiles, then the
 *      down tiles with the fused combine, each K block of a down tile
 *      waiting for the gate/up tile that stores its activations);
 *   1  two launches (the gate/up GEMM, then the down GEMM with the fused
 *      combine), as bi_moe_forward's decode path.
 * Same bits either way (tests compare them).  *previous (may be NULL)
 * receives the old setting; other values BI_ERR_INVALID_ARG.
 */
BI_API bi_status bi_moe_decode_fused(int32_t mode, int32_t *previous);

/*
 * bi_fp32_fma_probe -- MEASUREMENT ONLY, not part of the MoE path: blocks x
 * 256 threads, each running 16 independent fp32 FMA chains for `iters`
 * steps (2 * 16 * iters flop per thread, no memory traffic in the loop).
 * The benchmark times it to measure the FP32 (non-tensor) peak that the
 * router's FFMA roofline is reported against.  out: blocks * 256 floats
 * (device), written.
 */
BI_API bi_status bi_fp32_fma_probe(float *out, int64_t blocks, int32_t iters,
                                   bi_stream_t stream);

/*
 * bi_wait_timeout_probe -- TEST USE ONLY, not part of the MoE path and not on
 * the pages (it exercises this library's bounded-wait discipline): one CTA
 * waits on something that never happens, through one of the bounded waits
 * the GEMM kernels use: which = 0, the mbarrier wait of the stage rings, on
 * a barrier phase that nothing completes; which = 1, the arrival-count wait
 * of the one-launch decode layer, on a count that nothing raises.  The wait
 * gives up after its limit (one second of the GPU's global timer), records
 * BI_DEVERR_WAIT_TIMEOUT in the device error word and the kernel returns;
 * nothing faults or traps and the context stays usable.  Read the outcome
 * with bi_device_error.  Other values of which: BI_ERR_INVALID_ARG.
 */
BI_API bi_status bi_wait_timeout_probe(int32_t which, bi_stream_t stream);


#ifdef __cplusplus
}
#endif

#endif /* BIMOE_H_ */
