/*
 * lp.h -- C ABI of the bit-consistent sampled-token logprob engine (GB300, sm_103a).
 *
 * The engine turns final hidden states X[T,H] (bf16) into the logprob of each
 * sampled token under an lm_head W[V,H] (bf16):
 *
 *   P_j[t,v] = sum_{k in leaf j} X[t,k] W[v,k]      fp32 accumulation, K cut into
 *                                                   N contiguous leaves of H/N
 *   z[t,v]   = fixed pairwise tree over P_0..P_{N-1} (adjacent pairs first)
 *   logZ[t]  = fixed-order log-sum-exp of z[t,:]: (max, sum-exp) per 64-column tile, then a
 *              fixed pairwise tree over the tiles
 *   logp[t]  = z[t, y_t] - logZ[t]
 *
 * and, from a learner logprob log pi and a rollout logprob log mu, the unclipped
 * importance weight w = exp(log pi - log mu) and D3 = mean over valid tokens of
 * w - 1 - log w.
 *
 * Sources (the pages the method comes from):
 *  - diff = 0: the rollout logprob of every valid sampled token must equal the
 *    trainer's recomputed one exactly, with the same weights and prefix; results
 *    must not depend on batch composition, prefill versus decode, or the
 *    parallel layout (vLLM blog "Finish RL training faster: bit-consistent,
 *    high-throughput, agent-driven", section 2).
 *  - K cut into N contiguous FP32 leaves combined by a fixed binary tree, with a
 *    fixed rank->leaf map and partials only transported between ranks
 *    (IsoExec, SkyRL blog summary, section "Parallelism-invariant kernels";
 *    contract example: leaves = 8, leaf_dtype = fp32).  Unproven parallel sizes
 *    are rejected (same page, "Claims").
 *  - w = pi / mu, unclipped, per sampled token (REINFORCE Zero summary,
 *    sections 2 and 4); D3 = per-update token mean of w - 1 - log w (same page,
 *    section 3).
 *  - workspaces sized by static limits before any CUDA-graph capture, no host
 *    synchronisation inside a step, weights updated in place (vLLM blog,
 *    section 4.6).
 *
 * Every call on a handle is asynchronous on the caller's CUDA stream (cudaStream_t
 * passed as void*; NULL = legacy default stream), performs no host synchronisation and
 * no allocation (except lp_init, lp_free, lp_check and the *_host variants, which
 * are documented as synchronous), and can be captured in a CUDA graph.  The calls on one
 * handle share its device workspace (tile partials, block sums, the block counter of the
 * one-launch epilogues), so the kernels of two calls on the same handle must not overlap on
 * the GPU: issue them on one stream, or order their streams.
 *
 * Errors: every function returns an lp_status.  Argument errors are detected on
 * the host and returned before anything is enqueued; lp_last_error() gives a
 * thread-local message.  Problems found on the device (a sampled id outside
 * [0, V), a bounded wait that expired) set a sticky status word in the handle;
 * lp_check() synchronises and reports it.
 */
#ifndef LP_H_
#define LP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LP_API __attribute__((visibility("default")))
#else
#define LP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lp_status {
    LP_OK = 0,
    LP_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, sampled id outside [0,V) */
    LP_ERR_UNSUPPORTED = 2, /* configuration outside the proven set (see lp_config) */
    LP_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    LP_ERR_OOM = 4,         /* workspace allocation failed */
    LP_ERR_TIMEOUT = 5      /* a device-side bounded wait expired (kernel returned early) */
} lp_status;

/* Phase hint of lp_logprobs.  It selects a launch schedule only: every phase runs
 * the same per-element arithmetic, so results are bit-identical across phases. */
enum { LP_PHASE_AUTO = 0, LP_PHASE_PREFILL = 1, LP_PHASE_DECODE = 2 };

/*
 * Static configuration, fixed for the lifetime of a handle.
 *   H           hidden size (K of the lm_head GEMM); H % (64 * n_leaves) == 0.
 *   V           vocabulary size, 1 <= V < 2^31.
 *   n_leaves    N, number of contiguous K leaves: 1, 2, 4 or 8 (the proven set).
 *   tp_slices   emulated tensor-parallel split of K used by lp_logprobs: 1 (fused
 *               path), or 2, 4, 8 with tp_slices dividing n_leaves.  Slice r owns
 *               leaves [r*N/s, (r+1)*N/s) and produces that node of the leaf tree.
 *   max_tokens  row chunk: lp_logprobs processes at most this many rows per pass
 *               (larger T is split into chunks, which changes no bits because every
 *               row is computed alone).  The workspace is sized by it.
 */
typedef struct lp_config {
    int32_t H;
    int32_t V;
    int32_t n_leaves;
    int32_t tp_slices;
    int64_t max_tokens;
} lp_config;

typedef struct lp_handle lp_handle; /* opaque, owned by the library */

/*
 * Create a handle.  W: device pointer to the lm_head, bf16 [V, H] row-major
 * (row v = token v), 16-byte aligned, owned by the caller, referenced (not
 * copied): in-place updates of W are seen by later calls.  stream: used for the
 * one-time workspace initialisation (synchronised before return).  Allocates the
 * workspace (device memory sized by max_tokens and V, plus pinned staging for the
 * *_host call).  Returns LP_ERR_UNSUPPORTED for a configuration outside the
 * proven set or a device that is not sm_103.
 *
 * Environment variables read here, for this handle's lifetime.  The first group changes only
 * which CTA computes a tile and how data moves, never a bit of any output (the tests prove
 * each against the default layout):
 *   LP_FORCE_SINGLE_CTA=1    one CTA per tile instead of CTA pairs (cta_group::2) for
 *                            launches of more than 128 rows;
 *   LP_FORCE_SHORT_STAGES=1  64-K pipeline stages for every launch;
 *   LP_BAND_AXIS=rows        schedule bf16 launches in bands of rows (X kept in L2, W read
 *                            once per band) instead of bands of vocabulary tiles;
 *   LP_BAND_ROWS=<n>         scheduling rows (row tiles, or row-tile pairs) per row band;
 *   LP_BAND=<even n>         vocabulary tiles per scheduling band of bf16 handles (2..1024).
 *   LP_WAIT_TIMEOUT_MS=<ms>  bound on every in-kernel wait (default 2000); on expiry the
 *                            sticky status reads LP_ERR_TIMEOUT.
 *   LP_TEST_FAIL_ALLOC=<name> test hook: the named workspace allocation reports failure.
 *   LP_TEST_STOP_AFTER_STAGES=<n> test hook: the leaf GEMM's copy producer (bf16 or
 *                            block-FP8) stops after n
 *                            pipeline stages, as if its own wait had run out; the other warps'
 *                            bounded waits then expire, the kernel drains and returns, and the
 *                            sticky status reads LP_ERR_TIMEOUT.
 */
LP_API int lp_init(const lp_config* cfg, const void* W, void* stream, lp_handle** out);

/*
 * Sampled-token logprobs.
 *   X         device, bf16 [T, ldx] row-major (row t = hidden state of token t),
 *             16-byte aligned, ldx >= H and ldx % 8 == 0.
 *   ids       device, int32 [T], sampled token of each row.
 *   out_logp  device, fp32 [T]: z[t, ids[t]] - logZ[t]; NaN for an id outside
 *             [0, V) (which also sets the sticky LP_ERR_INVALID_ARG status).
 *   out_logZ  device, fp32 [T], or NULL: the log-partition logZ[t].
 *   phase     LP_PHASE_*; a schedule hint only (see above).
 * T == 0 is a no-op.  All buffers are caller-owned.
 */
LP_API int lp_logprobs(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids, int64_t T,
                float* out_logp, float* out_logZ, int phase, void* stream);

/*
 * lp_logprobs plus the entropy of each row's softmax, H[t] = -sum_v p log p = logZ - sum_v p z
 * (the actor entropy the pages track beside the KL; vLLM blog "Finish RL training faster",
 * section 3.2 results).  Per 64-column tile the epilogue also forms
 * u = sum e^(z-m) (z - m), merged by the same tile tree with the (m, s) partials:
 * H = log s - u / s.  logp and logZ are bit-equal to lp_logprobs's; H obeys the same
 * invariance (batch, position, phase, TP split).  out_entropy: device, fp32 [T].
 */
LP_API int lp_logprobs_entropy(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids,
                               int64_t T, float* out_logp, float* out_logZ, float* out_entropy,
                               int phase, void* stream);

/*
 * Same as lp_logprobs with HOST buffers (X: bf16 [T, ldx]; ids, out_logp,
 * out_logZ as above but in host memory; pinned memory is fastest).  Rows are
 * staged through the handle's device workspace in pieces (512 rows, then 8
 * times the previous piece, at most half of max_tokens, alternating between the
 * two halves of the workspace when max_tokens >= 256): the host-to-device copy
 * of the next piece runs on a stream the handle owns, under the kernels of the
 * current piece on `stream`.
 * Results do not depend on the split.  The call returns after the results are
 * in host memory (it synchronises `stream`).
 */
LP_API int lp_logprobs_host(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids, int64_t T,
                     float* out_logp, float* out_logZ, void* stream);

/*
 * One node of the leaf tree: the fp32 tree over leaves
 * [leaf_begin, leaf_begin + leaf_count) of every logit (what tensor-parallel
 * rank r contributes when it owns those leaves).  leaf_count must be a power of
 * two and leaf_begin a multiple of it (an aligned subtree), leaf_begin +
 * leaf_count <= N.  With leaf_count == 1 this exports the raw leaf partials P_j.
 *   X, ldx, T  as in lp_logprobs.
 *   out        device, fp32 [T, ldo] row-major, ldo >= V, 16-byte aligned rows.
 */
LP_API int lp_logits_partial(lp_handle* h, const void* X, int64_t ldx, int64_t T, int32_t leaf_begin,
                      int32_t leaf_count, float* out, int64_t ldo, void* stream);

/*
 * Finish the logprob from n_parts tree nodes that together cover the N leaves
 * in order (the partials gathered from all ranks): the upper levels of the same
 * fixed tree, then the same log-sum-exp and gather as lp_logprobs.
 *   partials    device, fp32; part p of row t, vocab v at
 *               partials[p * part_stride + t * ldp + v]; ldp >= V.
 *   n_parts     1, 2, 4 or 8, dividing N.
 *   ids, T, out_logp, out_logZ as in lp_logprobs (T <= max_tokens).
 * Bit-identical to lp_logprobs when the parts come from lp_logits_partial with
 * leaf_count = N / n_parts.
 */
LP_API int lp_logprobs_from_partials(lp_handle* h, const float* partials, int32_t n_parts,
                              int64_t part_stride, int64_t ldp, const int32_t* ids, int64_t T,
                              float* out_logp, float* out_logZ, void* stream);

/*
 * Importance weights and D3.
 *   logp_pi, logp_mu  device, fp32 [T]: learner and rollout logprobs.
 *   mask              device, uint8 [T] (nonzero = valid token), or NULL (all valid).
 *   out_w             device, fp32 [T]: exp(logp_pi - logp_mu) for every token.
 *   out_d3            device, one double: sum over valid tokens of
 *                     (w - 1 - log w) / n_valid, 0 when n_valid == 0.  The sum is
 *                     fp64 over a fixed tree of 1024-token blocks, independent of
 *                     the launch.
 *   out_nvalid        device, one int64: number of valid tokens (may be NULL).
 * T may exceed max_tokens (no row-chunk limit) up to 2^31 - 1.
 */
LP_API int lp_importance_weights(lp_handle* h, const float* logp_pi, const float* logp_mu,
                          const uint8_t* mask, int64_t T, float* out_w, double* out_d3,
                          int64_t* out_nvalid, void* stream);

/*
 * Vocabulary-parallel split of the lm_head (the pages' rule for parallel layouts: ranks only
 * transport partials, which a fixed schedule then combines; IsoExec summary,
 * "Parallelism-invariant kernels").  A rank holding the rows [v0, v0 + V) of the full lm_head
 * opens a bf16 handle over that slice (lp_init with this V and W pointing at row v0).
 *   lp_vocab_partials: the fused leaf GEMM of the slice for T <= max_tokens rows, writing the
 *     (max, sum-exp) partial of each of its ceil(V / 64) vocabulary tiles to out_ms (device,
 *     float pairs [ceil(V / 64)][ld_ms], ld_ms >= T, 16-byte aligned) and the sampled logit
 *     to out_zy [T].  ids_local[t] = sampled id - v0; out_zy[t] is the sampled logit for rows
 *     with ids_local[t] in [0, V), whose sampled token this rank owns, and NaN for the others.
 *   lp_logprobs_from_vocab_partials: on any handle (it lends its status word), logp and logZ
 *     for the full vocabulary of V_full tokens from the gathered partials: every rank's tile
 *     rows concatenated in vocabulary order (ms: float pairs [ceil(V_full / 64)][ld_ms]) and,
 *     per row, the sampled logit from the rank owning its id (zy [T]); ids are global.
 * When every slice starts at a multiple of 128 rows, the results are bit-identical to
 * lp_logprobs on the full lm_head (each tile partial is the same computation, and the tile
 * tree is the same).  A block-FP8 or TP-split handle returns LP_ERR_UNSUPPORTED.
 */
LP_API int lp_vocab_partials(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids_local,
                             int64_t T, void* out_ms, int64_t ld_ms, float* out_zy, void* stream);
LP_API int lp_logprobs_from_vocab_partials(lp_handle* h, int32_t V_full, const void* ms,
                                           int64_t ld_ms, const float* zy, const int32_t* ids,
                                           int64_t T, float* out_logp, float* out_logZ,
                                           void* stream);

/*
 * D3 over a token stream split across data-parallel ranks, with one exchange step.  D3 is a
 * per-update mean over all valid tokens (REINFORCE Zero summary, section 3), so ranks must
 * combine their tokens; the pages let the collective only move partials, never reduce them
 * (IsoExec summary, "Parallelism-invariant kernels": NCCL transports partials).
 *   lp_importance_weights_partials: out_w as in lp_importance_weights, and per 1024-token
 *     block (LP_IS_BLOCK) of this rank's range the fp64 sum of the D3 term over its valid
 *     tokens (out_blk_sum) and their count (out_blk_cnt); both device arrays of
 *     ceil(T / 1024) entries, caller-owned.
 *   lp_d3_from_partials: D3 and n_valid from num_blocks gathered blocks (device arrays, in
 *     stream order; num_blocks <= 2^21), by the same fixed fp64 tree over blocks as
 *     lp_importance_weights.
 * When every rank but the last holds a multiple of 1024 tokens and the partials are gathered
 * in rank order (an all-gather: data movement only), D3 and n_valid are bit-identical to one
 * lp_importance_weights call over the whole stream, for any number of ranks.  Both calls are
 * asynchronous on `stream`.
 */
#define LP_IS_BLOCK 1024
LP_API int lp_importance_weights_partials(lp_handle* h, const float* logp_pi,
                                          const float* logp_mu, const uint8_t* mask, int64_t T,
                                          float* out_w, double* out_blk_sum, int64_t* out_blk_cnt,
                                          void* stream);
LP_API int lp_d3_from_partials(lp_handle* h, const double* blk_sum, const int64_t* blk_cnt,
                               int64_t num_blocks, double* out_d3, int64_t* out_nvalid,
                               void* stream);

/*
 * Same as lp_importance_weights with HOST buffers (logp_pi, logp_mu, mask, out_w in
 * host memory; out_d3 and out_nvalid are host scalars).  Tokens are staged through
 * the device workspace in chunks of whole 1024-token blocks, so D3 is the same tree
 * as the device call.  Synchronises `stream` before returning.
 */
LP_API int lp_importance_weights_host(lp_handle* h, const float* logp_pi, const float* logp_mu,
                                      const uint8_t* mask, int64_t T, float* out_w,
                                      double* out_d3, int64_t* out_nvalid, void* stream);

/*
 * Block-FP8 (W8A8) handle.  The deployment recipe keeps the lm_head GEMM in block FP8 on both
 * sides: the trainer quantises its master bf16 weights by the deployment rule and calls the
 * inference GEMM (vLLM blog "Finish RL training faster", section 4.1).  The rule (DeepSeek's
 * block rule): activations in 1 x 128 blocks, weights in 128 x 128 blocks, scale
 * s = amax / 448 (fp32; 1 for an all-zero block), q = e4m3(x / s) rounded to nearest even and
 * saturated to +-448.  Then, per 128-K block kb, B_kb = sum qx qw (tcgen05 kind::f8f6f4, fp32);
 * per leaf P_j = sum over its blocks, ascending, of (sx sw) B_kb (a product, then one fma
 * per block); z = the same fixed pairwise leaf tree, and the same log-sum-exp and combine.
 *
 * lp_init_fp8 takes the same arguments as lp_init (W: the bf16 master lm_head, referenced) and
 * additionally requires H % (128 * n_leaves) == 0.  It quantises W into
 * a handle-owned e4m3 copy with its scales (synchronises `stream`).  lp_logprobs and
 * lp_logprobs_host on such a handle quantise each chunk of X (1 x 128 blocks) and run the
 * block-scaled GEMM; results obey the same invariance (batch, position, phase, chunking).
 * lp_logprobs_entropy also runs on such a handle (the same tile entropy partial and merge;
 * logp and logZ keep the bits of lp_logprobs), and so does the emulated tensor-parallel split
 * (tp_slices > 1: each slice's node of the leaf tree from the block-scaled leaves, the same
 * upper levels) with lp_logits_partial and lp_logprobs_from_partials.  lp_logprobs_backward
 * returns LP_ERR_UNSUPPORTED on a block-FP8 handle.
 * lp_fp8_requantize re-quantises W after an in-place update (asynchronous on `stream`).
 * lp_fp8_weights exposes the handle's e4m3 weights [V][H] and scales [ceil(V/128)][H/128]
 * (device pointers owned by the handle) for verification.
 */
LP_API int lp_init_fp8(const lp_config* cfg, const void* W, void* stream, lp_handle** out);
LP_API int lp_fp8_requantize(lp_handle* h, void* stream);
LP_API int lp_fp8_weights(const lp_handle* h, const uint8_t** wq, const float** sw);
/* The activation rule alone: X bf16 [T][ldx] -> xq e4m3 [T][H] (4-byte aligned) and
 * sx fp32 [T][H/128], on `stream`.  Any handle with H % 128 == 0. */
LP_API int lp_fp8_quantize_x(lp_handle* h, const void* X, int64_t ldx, int64_t T, uint8_t* xq,
                             float* sx, void* stream);

/*
 * Logprob backward.  For a loss L with upstream gradient g[t] = dL/dlogp[t] (fp32, device
 * [T]), with logp = lp_logprobs(X, ids) and logZ its out_logZ (device [T]):
 *   dl[t,v] = g[t] (1[v = y_t] - exp(z[t,v] - logZ[t]))      rounded to bf16, row chunks
 *   dX[t,:] = sum_v dl[t,v] W[v,:]                            fp32 [T][H] (row stride H)
 *   dW[v,:] = sum_t dl[t,v] X[t,:]  (added to dW if accumulate) fp32 [V][H]
 * z is recomputed by the forward's leaf GEMM and tree (the same kernel, a third epilogue),
 * so dl uses exactly the forward's logits.  The two products are the library's own tcgen05
 * GEMMs (bf16 operands, fp32 accumulation in TMEM); dX may be split over K = V into at most 4
 * fp32 partials that are added in slice order, and every dW element has one writer per row
 * chunk.  The pages' recipe keeps forward values from the inference kernel and
 * differentiates a separate training graph, whose backward need only be correct, not
 * deterministic (vLLM blog "Finish RL training faster", section 3.1); this backward is
 * deterministic for a given T and chunking but is not covered by the invariance guarantees.
 *   dX or dW may be NULL (not computed).  Requires lp_backward_reserve.
 * Uses the reserved gradient buffer: calls on one handle must be stream-ordered.
 */
LP_API int lp_logprobs_backward(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids,
                                const float* logZ, const float* grad_logp, int64_t T, float* dX,
                                float* dW, int accumulate, void* stream);

/*
 * Reserve the backward's workspace for row chunks of max_rows rows: a bf16 buffer
 * [max_rows][ceil(V/8)*8] (e.g. 4096 rows at V = 151936: 1.24 GB) and fp32 K-split partials
 * of dX [4][max_rows][H] (e.g. 134 MB at H = 2048).  Allocates and may synchronise the device: call it before any graph
 * capture.  A smaller request than the current reservation is a no-op.
 */
LP_API int lp_backward_reserve(lp_handle* h, int64_t max_rows);

/*
 * Acceptance statistics between two logprob vectors (vLLM blog "Finish RL training
 * faster", section 2: acceptance asks the max, mean and std of the per-token difference
 * over every valid sampled token to be 0; section 3.2: the k3 KL estimator r - 1 - log r).
 *   logp_a, logp_b  device, fp32 [T]: learner (log pi) and rollout (log mu) logprobs.
 *   mask            device, uint8 [T] (nonzero = valid), or NULL (all valid).
 *   out_stats       device, double [LP_STAT_COUNT]:
 *     [LP_STAT_MAX_ABS]   max |d| over valid tokens, d = fp32(logp_a - logp_b)
 *     [LP_STAT_MEAN_ABS]  mean |d|
 *     [LP_STAT_STD_ABS]   population std of |d|: sqrt(max(0, mean d^2 - mean^2))
 *     [LP_STAT_K3]        mean of e^d - 1 - d (r = pi/mu); bit-equal to the D3 of
 *                         lp_importance_weights on the same inputs
 *     [LP_STAT_N_VALID]   number of valid tokens
 *   Sums are fp64 over the same fixed tree of 1024-token blocks as D3.  A NaN |d| on a
 *   valid token makes the max NaN (and the sums with it); no valid token gives all 0.
 * T up to 2^31 - 1.  Uses the handle's block workspace: calls on one handle must be
 * stream-ordered.
 */
enum { LP_STAT_MAX_ABS = 0, LP_STAT_MEAN_ABS, LP_STAT_STD_ABS, LP_STAT_K3, LP_STAT_N_VALID,
       LP_STAT_COUNT };

LP_API int lp_acceptance_stats(lp_handle* h, const float* logp_a, const float* logp_b,
                               const uint8_t* mask, int64_t T, double* out_stats, void* stream);

/*
 * The same statistics over a token stream split across data-parallel ranks (acceptance is
 * over every valid sampled token of the update), with the one exchange step of
 * lp_importance_weights_partials / lp_d3_from_partials:
 *   lp_acceptance_stats_partials: per 1024-token block of this rank's range, out_blk
 *     [3][nb] doubles (sum |d|, sum d^2, sum of e^d - 1 - d), out_blk_max [nb] floats
 *     (max |d|, NaN kept) and out_blk_cnt [nb] valid counts; nb = ceil(T / 1024), device
 *     arrays, caller-owned.
 *   lp_acceptance_stats_from_partials: out_stats as lp_acceptance_stats from num_blocks
 *     gathered blocks (each of the three rows of blk concatenated in stream order).
 * With every rank but the last holding a multiple of 1024 tokens and the blocks gathered in
 * rank order, the statistics are bit-identical to one lp_acceptance_stats call.
 */
LP_API int lp_acceptance_stats_partials(lp_handle* h, const float* logp_a, const float* logp_b,
                                        const uint8_t* mask, int64_t T, double* out_blk,
                                        float* out_blk_max, int64_t* out_blk_cnt, void* stream);
LP_API int lp_acceptance_stats_from_partials(lp_handle* h, const double* blk,
                                             const float* blk_max, const int64_t* blk_cnt,
                                             int64_t num_blocks, double* out_stats, void* stream);

/*
 * REINFORCE Zero loss (REINFORCE Zero summary, section 4) for B responses packed back to
 * back, with the corrections the pages list beside it as options (vLLM blog, section 1:
 * TIS truncates the ratio at an upper bound, MIS drops whole sequences whose ratio passes
 * a threshold; REINFORCE Zero summary, results table: sequence and token gates):
 *
 *   L = -(1/B) sum_i (1/T_i) sum_t A_i w_hat_it,   dL/dlog pi_it = -(1/B)(1/T_i) A_i w_hat_it
 *
 *   w_it   = exp(d_it), d_it = fp32(logp_pi - logp_mu), unclipped (the plain recipe);
 *   w_hat  = w, then 0 if LP_RZ_TOKEN_GATE and d is outside [token_log_lo, token_log_hi],
 *            then min(., tis_cap) if LP_RZ_TIS, then 0 for the whole response if
 *            LP_RZ_SEQ_GATE and its log-ratio sum_t d_it (fp64, valid tokens) is outside
 *            [seq_log_lo, seq_log_hi]; masked tokens get w_hat = 0.  The modified weight
 *            is the coefficient of grad log pi, so the gradient uses w_hat in every mode;
 *   A_i    = R_i - mean of R over the response's group (groups of group_size consecutive
 *            responses), fp64;
 *   T_i    = valid tokens of response i; a response with T_i = 0 adds 0.
 *
 *   logp_pi, logp_mu  device, fp32 [T];   mask  device, uint8 [T] or NULL (all valid).
 *   seq_offsets       device, int64 [B+1]: response i holds tokens [offs[i], offs[i+1]);
 *                     expected offs[0] = 0 and offs[B] = T.  A range outside [0, T) sets
 *                     the sticky status (lp_check: LP_ERR_INVALID_ARG) and is treated as
 *                     empty; tokens outside every range are not written.
 *   rewards           device, fp32 [B];  group_size >= 1 dividing B;  B <= 2^21.
 *   opt               host, or NULL for the plain recipe.
 *   out_w_hat         device, fp32 [T] or NULL;  out_grad  device, fp32 [T].
 *   out_adv           device, double [B] or NULL: A_i.
 *   out_loss          device, one double: L (sum over responses by a fixed fp64 tree).
 *   out_n_kept        device, one int64 or NULL: responses that passed the sequence gate.
 * Per-token outputs depend only on the token's response and its group, never on the
 * rest of the batch or the launch.  Uses the handle's block workspace: calls on one handle
 * must be stream-ordered.
 */
enum { LP_RZ_TIS = 1, LP_RZ_TOKEN_GATE = 2, LP_RZ_SEQ_GATE = 4 };
typedef struct lp_rz_options {
    int32_t flags;                    /* OR of LP_RZ_*; 0 = unclipped token-level IS */
    float tis_cap;                    /* LP_RZ_TIS: cap C > 0 */
    float token_log_lo, token_log_hi; /* LP_RZ_TOKEN_GATE: bounds on d (fp32) */
    double seq_log_lo, seq_log_hi;    /* LP_RZ_SEQ_GATE: bounds on sum_t d (fp64) */
} lp_rz_options;
LP_API int lp_reinforce_zero(lp_handle* h, const float* logp_pi, const float* logp_mu,
                             const uint8_t* mask, int64_t T, const int64_t* seq_offsets,
                             int64_t B, const float* rewards, int32_t group_size,
                             const lp_rz_options* opt, float* out_w_hat, float* out_grad,
                             double* out_adv, double* out_loss, int64_t* out_n_kept,
                             void* stream);

/*
 * Kernel timing for profiling.  While enabled, every leaf-GEMM launch (the dominant
 * kernel), and each of the backward's two GEMMs (dX with its K-split sum; dW), is bracketed
 * by a pair of CUDA events recorded on the launch stream (at most 4096 pairs are kept).
 * lp_profile_read_kind synchronises and returns the summed duration in milliseconds and the
 * number of pairs of one kind (LP_PROFILE_*) recorded since the last lp_profile_read;
 * lp_profile_read does the same for the leaf GEMM and clears the record.  Enabling creates
 * the events (not graph-capturable).
 */
enum { LP_PROFILE_LEAF_GEMM = 0, LP_PROFILE_GRAD_DX = 1, LP_PROFILE_GRAD_DW = 2 };
LP_API int lp_profile_enable(lp_handle* h, int enable);
LP_API int lp_profile_read(lp_handle* h, double* gemm_ms_total, int32_t* gemm_launches);
LP_API int lp_profile_read_kind(lp_handle* h, int kind, double* ms_total, int32_t* count);

/*
 * lp_logprobs without a handle and without any device allocation.  (The pages have no
 * counterpart; this is a deployment entry point.)  For callers that cannot call
 * cudaMalloc: runtimes whose device memory is planned ahead by their own allocator (an
 * allocation behind its back breaks its plan), and hosts that forbid allocation after
 * start-up.  The scratch (per-tile max/sum-exp pairs, sampled logits, a status word) is a
 * fixed 8.13 MiB file-scope device array that every GPU loading the library holds until exit.
 *   W, H, V, n_leaves  as in lp_config / lp_init (W referenced, bf16 [V, H]).
 *   X, ldx, ids, T, out_logp, out_logZ  as in lp_logprobs.
 * Limits: T <= 32768 and T * ceil(V / 64) <= 1048576 (e.g. 441 rows at V = 151936);
 * larger calls return LP_ERR_INVALID_ARG and must use lp_logprobs with a handle.
 * The first call on a device resolves the array's device address, sets kernel attributes
 * and reads LP_WAIT_TIMEOUT_MS (no allocation); make that first call before any stream
 * capture.  Every call shares the array and overwrites what the last call left there:
 * calls whose kernels may overlap on the GPU (other streams, other threads) race and must
 * be serialised by the caller.
 * Errors found on the GPU are reported in the outputs (this entry point keeps no sticky
 * status): an id outside [0, V) gives NaN logp on that row; if a bounded in-kernel wait
 * expires (LP_WAIT_TIMEOUT_MS, default 2000 ms), every row's logp and logZ are NaN.
 * Bit-identical to lp_logprobs with tp_slices = 1.  Host-side errors are described by
 * lp_noalloc_last_error().  LP_TEST_NOALLOC_MARK_TIMEOUT=1 (read with the first call) is a
 * test hook: every call then reports as if a wait had expired.
 */
LP_API int lp_logprobs_noalloc(const void* W, int32_t H, int32_t V, int32_t n_leaves,
                               const void* X, int64_t ldx, const int32_t* ids, int64_t T,
                               float* out_logp, float* out_logZ, void* stream);
LP_API const char* lp_noalloc_last_error(void);

/*
 * Execution contract (IsoExec, SkyRL blog summary, "unified execution contract"): a canonical
 * JSON description of every execution choice that can change a bit, and SHA-256 identities
 * of its three sections, so that two runtimes (a trainer and a rollout engine) can prove they
 * run the same numerics by comparing digests.
 *   semantic          the logical computation (op, lm_head shape, outputs);
 *   numerical_policy  cases, composition (implementation ids and versions, pinned constants:
 *                     leaves, leaf dtype, MMA shape and order, tree shapes, LSE tile and order,
 *                     exp/log functions, D3 blocks) and claims (proven TP sizes, phases,
 *                     tolerances);
 *   deployment        settings proven not to change bits (max_tokens, tp_slices).
 * Pure host code: no device, no handle.  The configuration is validated as by lp_init.
 *
 * lp_contract writes the JSON (NUL-terminated) into buf[cap]; with buf == NULL it only sets
 * *len (the length without the NUL).  lp_contract_digest writes one 32-byte SHA-256 of the
 * canonical section.  lp_contract_check compares this configuration's semantic and
 * numerical_policy digests with a peer's and returns LP_ERR_UNSUPPORTED on a mismatch.
 * lp_sha256 is the library's SHA-256 (FIPS 180-4), exported for verification.
 */
enum { LP_DIGEST_SEMANTIC = 0, LP_DIGEST_NUMERICAL_POLICY = 1, LP_DIGEST_DEPLOYMENT = 2 };
/* precision: the handle kind the contract describes (lp_init or lp_init_fp8). */
enum { LP_PRECISION_BF16 = 0, LP_PRECISION_FP8_BLOCK = 1 };
LP_API int lp_contract(const lp_config* cfg, int precision, char* buf, size_t cap, size_t* len);
LP_API int lp_contract_digest(const lp_config* cfg, int precision, int which, uint8_t out[32]);
LP_API int lp_contract_check(const lp_config* cfg, int precision, const uint8_t peer_semantic[32],
                             const uint8_t peer_numerical_policy[32]);
LP_API void lp_sha256(const void* data, size_t n, uint8_t out[32]);

/*
 * Failure-detection self-test: launches a one-warp kernel that waits, with the same bounded
 * wait as every pipeline barrier, on an mbarrier nothing ever arrives on.  After timeout_us
 * (1 .. 2e6) it raises the sticky timeout status and returns; lp_check then reports
 * LP_ERR_TIMEOUT and lp_clear_status resets it.  Nothing else is in flight in that kernel, so
 * the context stays usable.
 */
LP_API int lp_selftest_wait_timeout(lp_handle* h, int64_t timeout_us, void* stream);

/* Synchronise the stream last used with the handle and return the sticky device
 * status (LP_OK, LP_ERR_INVALID_ARG for a bad id, LP_ERR_TIMEOUT). */
LP_API int lp_check(lp_handle* h);

/* Clear the sticky device status (asynchronous on `stream`). */
LP_API int lp_clear_status(lp_handle* h, void* stream);

/* Thread-local message describing the last error returned on this thread. */
LP_API const char* lp_last_error(void);

/* Workspace bytes held by the handle (device), for capacity planning. */
LP_API int64_t lp_workspace_bytes(const lp_handle* h);

/* Number of kernel launches the last lp_* compute call on this handle enqueued. */
LP_API int32_t lp_last_launch_count(const lp_handle* h);

/* ABI version (major * 100 + minor). */
LP_API int lp_version(void);

/* Synchronise and release the handle and its workspace.  NULL is a no-op. */
LP_API void lp_free(lp_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* LP_H_ */
