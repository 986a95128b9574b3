/*
 * rlk.h -- C ABI of the deterministic, batch-invariant selected-token
 * log-probability operator `linear_logp` for NVIDIA GB300 (sm_103a).
 *
 * Operation ("Announcing RL-Kernel for vime", section "Key Capabilities", first
 * bullet, and the operator boundary "hidden + lm_head_weight + target_ids ->
 * selected logprob" in section "Why the Fused Path Wins"):
 *
 *   z[t][v]  = h[t] . W[v]                        (bf16 inputs, fp32 accumulation)
 *   lse[t]   = log sum_{v < V_true} exp(z[t][v])   (columns >= V_true are masked:
 *              "true vocabulary range", table "Boundary Fixes in the RL-Kernel
 *              Strict Path", row "Linear logprob", of "vLLM RL-Kernel v0.1.0:
 *              Bitwise Train-Rollout Consistency on ROCm")
 *   logp[t]  = z[t][y[t]] - lse[t]
 *
 * computed without materialising the [T, V] logits (the fused kernel keeps
 * running max / sum-exp / target-logit statistics while it walks vocab tiles,
 * second reason in "Why the Fused Path Wins"). The backward returns dH and dW of
 * L = sum_t g[t] * logp[t] ("Full-gradient support" bullet), recomputing the
 * logits tile by tile and forming dz = g * (onehot - softmax).
 *
 * Numerical contract (the six observables of "The Numerical Execution
 * Contract" in the ROCm consistency article, fixed here once for every shape):
 *  1. Input dependency: logp[t], lse[t] and dH[t] depend only on h[t], y[t], W,
 *     V_true (and g[t], lse[t] for dH[t]); never on T, on other rows, on the
 *     stream, on the launch shape or on the GPU's SM count.
 *  2. Partitioning: the hidden dimension is reduced in steps of 64 (one K=16
 *     tensor-core instruction at a time, ascending). The vocabulary is cut into
 *     leaves of RLK_LEAF_WIDTH = 1024 global columns, each walked in 256-column
 *     tiles in ascending order. No split-K, no atomics on data (one atomic
 *     counter per launch only hands out work items; which CTA pair computes an
 *     output tile never changes how it is computed).
 *  3. Merge order: leaves are merged by a balanced pairwise tree defined on
 *     global leaf indices: nLeaves = ceil(V_true / 1024) leaves are grouped into
 *     RLK_MAX_SHARDS = 8 super-shards of L = ceil(nLeaves / 8) leaves; inside a
 *     super-shard the leaves sit in P = next_pow2(L) slots (missing leaves are
 *     the identity) and are merged pairwise; the 8 super-shard results are then
 *     merged pairwise (8 -> 4 -> 2 -> 1). Because the tree depends only on V_true,
 *     a vocab-sharded run (S in {1, 2, 4, 8} contiguous shards, each a
 *     power-of-two-aligned run of super-shards) followed by rlk_lse_merge gives
 *     bit-identical logp and lse to the unsharded run.
 *  4. Precision: bf16 inputs; fp32 accumulation, statistics, logp and lse; dz
 *     is rounded once to bf16 (it is an operand of the dH/dW products); dH is
 *     rounded once to bf16 from its fp32 accumulator; dW is fp32.
 *  5. Rounding: every floating-point step is an explicitly rounded operation
 *     (round-to-nearest fmul / fadd / fma); nothing is left to compiler contraction.
 *  6. Primitives: e(x) = ex2.approx.ftz(fma(x, log2 e, -rn(b * log2 e))) for
 *     exp(x - b) everywhere; log is logf (fp32, CUDA math library).
 *
 * Conventions for every entry point:
 *  - The caller owns every buffer. The library allocates and frees nothing and
 *    keeps no state between calls (apart from per-device kernel attributes),
 *    so calls are re-entrant.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) with no host synchronisation. Device pointers must be valid in the
 *    current CUDA context.
 *  - Argument errors are returned before anything is launched; T == 0 returns
 *    RLK_OK and launches nothing (per-token pointers may then be NULL). A
 *    launch failure returns RLK_ERR_CUDA.
 *  - Row-major, contiguous tensors. h, W and dz-style bf16 rows need a 16-byte
 *    aligned base and H % 8 == 0 (tensor-memory-access strides).
 *  - Targets outside [0, V_true) cannot be checked on the host without a sync:
 *    their logp is NaN, their gradient row is zero, and RLK_FLAG_BAD_TARGET is
 *    ORed into *err_flag when err_flag is not NULL.
 *  - Every internal wait of a kernel is bounded; on expiry the kernel stops,
 *    ORs RLK_FLAG_TIMEOUT into *err_flag (if given) and the outputs are invalid.
 */
#ifndef RLK_H_
#define RLK_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RLK_API __attribute__((visibility("default")))
#else
#define RLK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RLK_OK = 0,
  RLK_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned pointer, H % 8 != 0 */
  RLK_ERR_UNSUPPORTED = 2, /* a shard split the fixed merge tree cannot express; sizes beyond limits */
  RLK_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the query returns */
  RLK_ERR_CUDA = 4         /* a CUDA runtime/driver call failed (launch, tensor-map encode) */
} rlk_status;

/* bits ORed into *err_flag by the kernels */
#define RLK_FLAG_BAD_TARGET 1
#define RLK_FLAG_TIMEOUT 2
#define RLK_FLAG_NONFINITE 4 /* rlk_quantize_rows_e4m3: a row held a NaN or an infinity */
#define RLK_FLAG_BOUNDS 8    /* debug-checks builds only: an index or tensor-copy coordinate
                                check failed; the access was skipped (see rlk_debug_checks) */

/* tiling constants that are part of the numerical contract */
#define RLK_LEAF_WIDTH 1024
#define RLK_MAX_SHARDS 8

/* size limits (RLK_ERR_UNSUPPORTED beyond them) */
#define RLK_MAX_VOCAB (1 << 24)
#define RLK_MAX_HIDDEN (1 << 16)

/*
 * Per-token statistics of one vocab shard, natural-log units: m is the largest
 * logit of the shard's valid columns, s = sum exp(z - m) over them, zt the
 * target logit if the shard owns y[t], else -inf (NaN for an invalid target).
 * The identity (empty shard) is {-inf, 0, -inf}. Layout: 12 bytes, no padding.
 * ("Why the Fused Path Wins", third reason: only statistics cross shards.)
 */
typedef struct {
  float m;
  float s;
  float zt;
} rlk_lse_partial;

/* Bytes of device workspace rlk_linear_logp_fwd needs (256-byte aligned base): the
 * per-(token, leaf) statistics, then 256 bytes of work-item counters that the call
 * zeroes on its stream before its kernels use them. */
RLK_API size_t rlk_linear_logp_fwd_workspace(int64_t T, int64_t H, int64_t V_local);

/*
 * Forward. The shard holds W rows for global vocab columns
 * [vocab_start, vocab_start + V_local); the unsharded call is vocab_start = 0,
 * V_local = V >= V_true.
 *
 *   h        device bf16 [T][H]
 *   W        device bf16 [V_local][H] (this shard's rows)
 *   y        device int64 [T], global vocab ids
 *   V_true   global true-vocab bound; columns >= V_true are masked
 *   logp,lse device fp32 [T] each, or NULL; used when partial == NULL, which
 *            requires the shard to cover [0, V_true)
 *   partial  device rlk_lse_partial [T] or NULL: when given, the call writes
 *            this shard's triple per token instead of logp / lse; combine the
 *            shards with rlk_lse_merge
 *   err_flag device int32 or NULL (RLK_FLAG_* bits are ORed in, never cleared)
 *   workspace, workspace_bytes: device scratch of at least
 *            rlk_linear_logp_fwd_workspace(T, H, V_local) bytes, 256-byte aligned
 *
 * A shard must start at a multiple of the super-shard width
 * L * RLK_LEAF_WIDTH (L = ceil(ceil(V_true / 1024) / 8)), cover n = ceil(V_local /
 * (L * 1024)) super-shards with n a power of two and vocab_start / (L * 1024) a
 * multiple of n, and contain every column of those super-shards below V_true;
 * otherwise RLK_ERR_UNSUPPORTED.
 */
RLK_API rlk_status rlk_linear_logp_fwd(const void* h, const void* W, const int64_t* y, int64_t T,
                               int64_t H, int64_t V_local, int64_t vocab_start, int64_t V_true,
                               float* logp, float* lse, rlk_lse_partial* partial,
                               int32_t* err_flag, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Merge S per-shard triples per token (partials laid out [S][T], shards in
 * ascending vocab order) by the top levels of the fixed tree, then
 * lse = m + log(s), logp = zt - lse. S must be 1, 2, 4 or 8. logp, lse: device
 * fp32 [T]. ("vLLM RL-Kernel v0.1.0 ... on ROCm", "Boundary Fixes" table,
 * "Linear logprob" row: cross-rank LSE merge; fixed merge order, item 3 of
 * "The Numerical Execution Contract".)
 */
RLK_API rlk_status rlk_lse_merge(const rlk_lse_partial* partials, int32_t S, int64_t T, float* logp,
                         float* lse, void* stream);

/* Bytes of device workspace rlk_linear_logp_bwd needs: the bf16 dz tile store
 * [T][round_up(V_local, 256)] (the "controlled workspace" of the fourth reason
 * in "Why the Fused Path Wins"), plus, when V_local > 65536, an fp32 [T][H]
 * running sum for dH's chunked accumulation, plus 256 bytes of work-item counters
 * (zeroed by the call on its stream). */
RLK_API size_t rlk_linear_logp_bwd_workspace(int64_t T, int64_t H, int64_t V_local);

/*
 * Backward of L = sum_t g[t] logp[t] for one shard (or the whole vocabulary).
 *
 *   h, W, y, T, H, V_local, vocab_start, V_true: as in the forward
 *   lse      device fp32 [T], the GLOBAL log-sum-exp from the forward / merge
 *   g        device fp32 [T], upstream gradient
 *   dH       device [T][H] or NULL: bf16 when dH_fp32_partial == 0, else fp32
 *            (a shard's partial; sum the shards with rlk_shard_sum_bf16)
 *   dW       device fp32 [V_local][H] or NULL; rows at or above V_true get 0
 *   err_flag, workspace, workspace_bytes, stream: as in the forward
 *
 * dz[t][v] = g[t] (1[v == y[t]] - exp(z[t][v] - lse[t])) is recomputed from a
 * fresh z tile with the forward's exact tensor-core sequence, rounded once to
 * bf16; dH = dz W sums the vocabulary in ascending 64-column steps, dW = dz^T h
 * sums the tokens in ascending 64-row steps, each output tile by one CTA pair.
 * Both reductions run in fixed chunks of 65536 (tensor-core fp32 accumulation
 * within a chunk, then round-to-nearest fp32 adds of the chunk results in
 * ascending order), which keeps the accumulation bias of very long reductions
 * bounded; the chunking depends on neither T's batch composition nor the launch.
 */
RLK_API rlk_status rlk_linear_logp_bwd(const void* h, const void* W, const int64_t* y, const float* lse,
                               const float* g, int64_t T, int64_t H, int64_t V_local,
                               int64_t vocab_start, int64_t V_true, void* dH,
                               int32_t dH_fp32_partial, float* dW, int32_t* err_flag,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * The same backward, launched in separate stages. The backward's three products
 * meet in its workspace ("tiled logits / dlogits and linear-gradient work ... with
 * a controlled workspace", "Announcing RL-Kernel for vime", section "Why the Fused
 * Path Wins", fourth reason): the dz tiles are written there once and read by both
 * gradient products. `stages` is a nonzero OR of
 *   RLK_BWD_DZ  recompute the logits and write dz into the workspace
 *   RLK_BWD_DH  dH = dz W from the dz the workspace holds (dH must not be NULL)
 *   RLK_BWD_DW  dW = dz^T h from the dz the workspace holds (dW must not be NULL)
 * and every other argument is as in rlk_linear_logp_bwd. A stage launches the kernel
 * that rlk_linear_logp_bwd launches for it, on the same operands in the same work order
 * (only how it follows the launch before it differs), so stages run one call at a time
 * in the order DZ, DH, DW with one workspace give the bits of a single
 * rlk_linear_logp_bwd call. The workspace must stay untouched
 * from the DZ call until the last call that reads its dz. Each stage has its own
 * work-item counter in the workspace and only RLK_BWD_DH uses its fp32 running sum,
 * so once the DZ stage has completed, the DH and DW stages may run on two streams
 * at the same time. Uses: pipeline schedules that need the input gradient dH at once
 * and defer the weight gradient dW; timing each stage on its own.
 */
#define RLK_BWD_DZ 1
#define RLK_BWD_DH 2
#define RLK_BWD_DW 4

RLK_API rlk_status rlk_linear_logp_bwd_stages(const void* h, const void* W, const int64_t* y,
                                              const float* lse, const float* g, int64_t T,
                                              int64_t H, int64_t V_local, int64_t vocab_start,
                                              int64_t V_true, void* dH, int32_t dH_fp32_partial,
                                              float* dW, int32_t stages, int32_t* err_flag,
                                              void* workspace, size_t workspace_bytes,
                                              void* stream);

/*
 * Saved-logits variant of the pair above: the forward also stores the fp32
 * logits it computed and the backward forms dz from them instead of recomputing
 * the logits GEMM (the "save-logits fused-tile full-gradient path" named in
 * "Announcing RL-Kernel for vime", section "Validation and Benchmarks"). The
 * saved logits are the accumulator values bit for bit and dz uses the same
 * arithmetic, so logp, lse, dH and dW are bit-identical to the recompute path;
 * the price is rlk_saved_logits_bytes of device memory between the two calls.
 *
 *   z_saved  device fp32 [T][round_up(V_local, 256)], 16-byte aligned, caller-owned;
 *            written by rlk_linear_logp_fwd_save for the shard's columns below
 *            V_true, read by rlk_linear_logp_bwd_saved; z_saved_bytes must be at
 *            least rlk_saved_logits_bytes(T, V_local) (else RLK_ERR_INVALID_ARG)
 * Every other argument is as in rlk_linear_logp_fwd / rlk_linear_logp_bwd.
 */
RLK_API size_t rlk_saved_logits_bytes(int64_t T, int64_t V_local);

RLK_API rlk_status rlk_linear_logp_fwd_save(const void* h, const void* W, const int64_t* y,
                                            int64_t T, int64_t H, int64_t V_local,
                                            int64_t vocab_start, int64_t V_true, float* logp,
                                            float* lse, rlk_lse_partial* partial, float* z_saved,
                                            size_t z_saved_bytes, int32_t* err_flag,
                                            void* workspace, size_t workspace_bytes, void* stream);

RLK_API rlk_status rlk_linear_logp_bwd_saved(const void* h, const void* W, const int64_t* y,
                                             const float* lse, const float* g,
                                             const float* z_saved, size_t z_saved_bytes, int64_t T,
                                             int64_t H, int64_t V_local, int64_t vocab_start,
                                             int64_t V_true, void* dH, int32_t dH_fp32_partial,
                                             float* dW, int32_t* err_flag, void* workspace,
                                             size_t workspace_bytes, void* stream);

/*
 * Saved-probabilities variant (the bf16 "save probs" option of the pages'
 * linear_logp settings, "Announcing RL-Kernel for vime", section "Quick Start"):
 * the forward stores, for every logit, e(z - m) rounded to bf16 together with the
 * row's fp32 running max m after each 64-column chunk, and the backward forms
 * p = e(z - m) * e(m - lse) from them. Half the memory of the saved logits; dz
 * carries an extra relative error of at most 2^-9 (bf16) per element, so dH / dW
 * are NOT bit-identical to the recompute path (logp and lse are).
 *
 *   p_saved  device buffer of rlk_saved_probs_bytes(T, V_local) bytes, 256-byte
 *            aligned, caller-owned: bf16 [T][round_up(V_local, 256)], then fp32
 *            [T][round_up(V_local, 256) / 64] at a 256-byte aligned offset
 * Every other argument is as in rlk_linear_logp_fwd / rlk_linear_logp_bwd.
 */
RLK_API size_t rlk_saved_probs_bytes(int64_t T, int64_t V_local);

RLK_API rlk_status rlk_linear_logp_fwd_save_probs(const void* h, const void* W, const int64_t* y,
                                                  int64_t T, int64_t H, int64_t V_local,
                                                  int64_t vocab_start, int64_t V_true,
                                                  float* logp, float* lse,
                                                  rlk_lse_partial* partial, void* p_saved,
                                                  size_t p_saved_bytes, int32_t* err_flag,
                                                  void* workspace, size_t workspace_bytes,
                                                  void* stream);

RLK_API rlk_status rlk_linear_logp_bwd_saved_probs(const void* h, const void* W, const int64_t* y,
                                                   const float* lse, const float* g,
                                                   const void* p_saved, size_t p_saved_bytes,
                                                   int64_t T, int64_t H, int64_t V_local,
                                                   int64_t vocab_start, int64_t V_true, void* dH,
                                                   int32_t dH_fp32_partial, float* dW,
                                                   int32_t* err_flag, void* workspace,
                                                   size_t workspace_bytes, void* stream);

/*
 * out[i] = bf16(((p[0][i] + p[1][i]) + p[2][i]) + ...), the fixed ascending-order
 * sum of S fp32 partials laid out [S][n], rounded once to bf16 (RNE). Used to
 * combine per-shard dH partials. partials, out: device, 16-byte aligned.
 */
RLK_API rlk_status rlk_shard_sum_bf16(const float* partials, int32_t S, int64_t n, void* out,
                              void* stream);

/*
 * FP8 LM head. An RL trainer whose rollouts run an FP8 output layer reproduces it
 * in the training forward: the weights are quantized to FP8 again at every
 * forward, both sides use one quantization rounding rule and one batch-invariant
 * GEMM for every batch size, and the backward takes gradients for the bf16 master
 * weights with the quantization treated as the identity (straight-through
 * estimator) (AREX feed article on vLLM's bitwise-consistent RL training, sections
 * "训练前向直接调用推理内核" and "对齐的代价：逐算子拆解"). The pages fix neither the
 * FP8 format nor the scale granularity; this library uses OCP E4M3 (no infinities,
 * largest magnitude 448) with one power-of-two scale per row, so a token's codes
 * never depend on the rest of the batch and quantization is exactly reproducible.
 *
 * rlk_quantize_rows_e4m3: for each row r of x (bf16 [rows][cols], device, 16-byte
 * aligned, cols % 8 == 0):
 *   e       = the smallest integer with max_k |x[r][k]| <= 448 * 2^e (0 if the row is all zero)
 *   scale[r] = 2^e                                   (fp32 [rows], device)
 *   q[r][k]  = E4M3 code nearest to x[r][k] / 2^e, ties to even (uint8 [rows][cols], device,
 *             16-byte aligned)
 * A row holding a NaN or an infinity gets scale NaN and zero codes, and
 * RLK_FLAG_NONFINITE is ORed into *err_flag (device int32, or NULL). rows == 0 or
 * cols == 0 launches nothing. Asynchronous on `stream`; argument errors are returned
 * before any launch.
 */
RLK_API rlk_status rlk_quantize_rows_e4m3(const void* x, int64_t rows, int64_t cols, void* q,
                                          float* scale, int32_t* err_flag, void* stream);

/*
 * FP8 forward: the forward of rlk_linear_logp_fwd on E4M3 operands,
 *   z[t][v] = (sum_k hq[t][k] * Wq[v][k]) * h_scale[t] * W_scale[v]
 * (products exact, fp32 tensor-core accumulation over K in ascending 128-element
 * steps, then the two power-of-two scales), with the same fixed merge tree, shard
 * statistics, masking, outputs and errors.
 *   hq       E4M3 codes [T][H] (device, 16-byte aligned), h_scale fp32 [T]
 *   Wq       E4M3 codes [V_local][H] (device, 16-byte aligned), W_scale fp32 [V_local]
 *            (device, 16-byte aligned)
 * as produced by rlk_quantize_rows_e4m3; H % 16 == 0. Workspace: as
 * rlk_linear_logp_fwd_workspace(T, H, V_local).
 */
RLK_API rlk_status rlk_linear_logp_fwd_fp8(const void* hq, const float* h_scale, const void* Wq,
                                           const float* W_scale, const int64_t* y, int64_t T,
                                           int64_t H, int64_t V_local, int64_t vocab_start,
                                           int64_t V_true, float* logp, float* lse,
                                           rlk_lse_partial* partial, int32_t* err_flag,
                                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Straight-through FP8 backward: dz[t][v] = g[t] (1[v = y[t]] - e(z[t][v] - lse[t]))
 * with z the E4M3 logits of rlk_linear_logp_fwd_fp8 (recomputed tile by tile, the
 * same bits as that forward's), then dH = dz W and dW = dz^T h with the bf16
 * operands h, W exactly as in rlk_linear_logp_bwd (outputs, shard partials, workspace
 * rlk_linear_logp_bwd_workspace(T, H, V_local), errors). hq, h_scale, Wq, W_scale as
 * in rlk_linear_logp_fwd_fp8; lse is the FP8 forward's.
 */
RLK_API rlk_status rlk_linear_logp_bwd_fp8(const void* h, const void* W, const void* hq,
                                           const float* h_scale, const void* Wq,
                                           const float* W_scale, const int64_t* y,
                                           const float* lse, const float* g, int64_t T, int64_t H,
                                           int64_t V_local, int64_t vocab_start, int64_t V_true,
                                           void* dH, int32_t dH_fp32_partial, float* dW,
                                           int32_t* err_flag, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * Forward without a workspace argument, for callers that cannot allocate device
 * memory: runtimes whose device memory is fully reserved up front by another
 * allocator (a serving engine that pre-plans every buffer), or latency-critical
 * loops where cudaMalloc / cudaFree would synchronise the device and stall the
 * other streams. The pages have no counterpart to this entry point.
 *
 * Same arguments, results and errors as rlk_linear_logp_fwd, minus workspace and
 * workspace_bytes. The scratch it needs instead is one static device array of
 * RLK_FWD_NOALLOC_SCRATCH_BYTES (16 MiB), held by every GPU that loads the library
 * until the process exits; the call itself allocates nothing. A shape whose
 * rlk_linear_logp_fwd_workspace(T, H, V_local) exceeds that size is rejected with
 * RLK_ERR_WORKSPACE before anything runs (e.g. at most 9383 tokens for a 151936-row
 * W). The first call on a device looks up the array's device address (with that
 * device current) and keeps it for the life of the process; make that first call
 * before any stream capture. Calling it after cudaDeviceReset on that device is not
 * supported (the array may then live at another address). All calls on a
 * device share the array: calls that can overlap on the GPU (different streams with
 * no ordering between them) race and give wrong results.
 */
#define RLK_FWD_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

RLK_API rlk_status rlk_linear_logp_fwd_noalloc(const void* h, const void* W, const int64_t* y,
                                               int64_t T, int64_t H, int64_t V_local,
                                               int64_t vocab_start, int64_t V_true, float* logp,
                                               float* lse, rlk_lse_partial* partial,
                                               int32_t* err_flag, void* stream);

/*
 * Self-test of the kernels' bounded waits. Runs the unsharded forward (arguments
 * as rlk_linear_logp_fwd with vocab_start = 0) with the first shared-memory stage
 * of one CTA deliberately left unfilled, so the pipeline's first wait can never
 * complete. After the wait limit (2 s) the kernel gives up: it raises its abort
 * flag in both CTAs of the pair, drains the copies and tensor-core work already in
 * flight, frees its tensor memory, ORs RLK_FLAG_TIMEOUT into *err_flag (required)
 * and returns; the kernel takes about 4 s and logp / lse are undefined. No fault,
 * trap or hang is involved, and the CUDA context stays usable afterwards.
 */
RLK_API rlk_status rlk_selftest_wait_timeout(const void* h, const void* W, const int64_t* y,
                                             int64_t T, int64_t H, int64_t V, int64_t V_true,
                                             float* logp, float* lse, int32_t* err_flag,
                                             void* workspace, size_t workspace_bytes,
                                             void* stream);

/*
 * Debug-checks builds. The library can also be compiled with device-side checks
 * (RLK_DEBUG_CHECKS=1; `python -m deterministic_token_logprob_gb300.build --debug-checks`
 * writes _build_debug/librlk.so): before every global-memory access whose address the
 * kernels compute from an index (statistics, saved maxima, running sums, plain output
 * stores, the dz passes, the leaf-tree reads) they check the index against the extent of
 * the buffer, and before every tensor copy they check the rules of its coordinates (the
 * innermost one a multiple of 16 bytes, a store's never negative). A failed check ORs
 * RLK_FLAG_BOUNDS into *err_flag instead of trapping and skips the access (a load's
 * misaligned coordinate is rounded down instead, so the pipeline's byte counts still
 * complete), so the context stays usable. Results of a build with checks are bit-identical
 * to the plain build's.
 *
 * rlk_debug_checks: 1 for a library built with the checks, else 0.
 * rlk_selftest_bounds_check: the unsharded forward (arguments as rlk_linear_logp_fwd) told
 * that its statistics workspace is one (token, leaf) entry shorter than it is, so the last
 * entry's store and read fail their checks: afterwards *err_flag (required) holds
 * RLK_FLAG_BOUNDS, and every access stayed inside the real buffers. logp / lse are
 * undefined. Without the checks it returns RLK_ERR_UNSUPPORTED and launches nothing.
 */
RLK_API int32_t rlk_debug_checks(void);

RLK_API rlk_status rlk_selftest_bounds_check(const void* h, const void* W, const int64_t* y,
                                             int64_t T, int64_t H, int64_t V, int64_t V_true,
                                             float* logp, float* lse, int32_t* err_flag,
                                             void* workspace, size_t workspace_bytes,
                                             void* stream);

/* Static description of a status code. */
RLK_API const char* rlk_status_string(rlk_status s);

/* Library version string, e.g. "rlk 0.1.0 sm_103a". */
RLK_API const char* rlk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RLK_H_ */
