/*
 * lossk.h -- C ABI of liblossk.so, a fused LM-head loss for NVIDIA GB300
 * (sm_103a).
 *
 * The loss takes hidden[n_tok][d_model] and weight[vocab][d_model] and never
 * builds the [n_tok][vocab] logit tensor: the projection runs tile by tile on
 * the tensor cores and each tile is reduced on chip to the per-token
 * log-sum-exp and target logit ("Loss functions and resident-context
 * kernels", section "lossk: the loss is where the memory goes", entries
 * fused_linear_ce_flat and fused_linear_ce_bwd_flat).  A z-loss term lse^2
 * and a distillation variant against a full teacher distribution follow
 * "Fuse distillation + z-loss in the triton monolithic path (#507)", section
 * "What it does".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Return value: a status code in 580..599 (enum lossk_status).  580 means
 *    the work was enqueued (or the check passed).  Any other code means the
 *    call was refused before any output was written, except 589/590, which
 *    report a device failure.
 *  - Buffers: every tensor argument is a caller-owned DEVICE pointer to a
 *    contiguous row-major array; the library never allocates device memory.
 *    Each tensor comes with its element count (`*_len`); a count shorter than
 *    the shape needs, or a NULL required pointer, gives 582.
 *  - dtype: LOSSK_BF16 (uint16 bf16 bits), LOSSK_F16 (uint16 IEEE half bits)
 *    or LOSSK_F32 (float) for hidden, weight, logits and teacher logits.
 *    16-bit inputs are multiplied on the tcgen05 tensor cores with fp32
 *    accumulation; fp32 inputs use an FFMA path.  Per-token outputs are
 *    float, gradients are float (grad_logits take the logits' dtype), the
 *    three reduced scalars are double.  fp16 grad tiles hold the gradient
 *    without its common factor grad_scale / N_valid (applied in fp32 when the
 *    accumulators are stored), so they stay inside fp16's range; the training
 *    step's single-pass forward + d_hidden needs bf16's exponent range and is
 *    bf16 only (fp16 runs the separate passes).  The 16-bit tensor path loads
 *    operands with TMA, which needs 16-byte row pitches: d_model % 8 == 0
 *    (and, for the teacher logits, vocab % 8 == 0), else 591.  Every device
 *    pointer must be 16-byte aligned, else 591.
 *  - Scratch: `workspace` is device memory of at least
 *    lossk_workspace_bytes(...) bytes, 256-byte aligned; shorter gives 582.
 *    Calls that share a workspace must not overlap in time.
 *  - Streams: all device work is enqueued on `stream` (NULL = legacy default
 *    stream).  Each compute call synchronises `stream` once, after a small
 *    validation kernel, to read back the target-range flag and the number of
 *    counted tokens: the call refuses bad targets (586) before the main
 *    kernels run, the way the pages' functions validate first.  After that
 *    point the call returns without waiting for the GPU.  The training-step
 *    calls on the bf16 path (lossk_ce_fwd_bwd and its _ex form) synchronise
 *    once too, at their end instead: the validation is queued first, every
 *    kernel after it returns at once on the device when it found a target out
 *    of range (so a 586 still leaves every output untouched), and the end
 *    read-back carries the validation result with the range flag of the
 *    single-pass forward (see there).  Those calls also run the token mean
 *    and d_hidden's last kernel on a helper stream the library keeps for
 *    each calling stream (up to 8 streams per device; a call on a further
 *    stream runs them on `stream` itself) and join it back into `stream`
 *    before returning, so calls on different streams never wait for each
 *    other's helper work.  The
 *    read-backs go through a one-warp kernel writing into mapped pinned host
 *    memory, not through a copy engine, so large copies other streams have in
 *    flight do not delay them; the library allocates that memory (64 bytes
 *    per calling host thread) on a thread's first call and keeps it.
 *  - Check order (the first failing check wins): 581 empty dimension, 583
 *    dimension over 2^24, 584 n_tok*d_model*vocab over 2^46, 587 chunk*vocab
 *    over 2^27, 582 length / NULL pointer / short workspace, 591 alignment,
 *    585 non-finite scalar, 588 unknown objective, 586 target out of range.
 *  - Mask: `loss_mask` is an optional uint8[n_tok] (NULL = every token
 *    counts; nonzero = counts).  Reductions are means over the N_valid
 *    counted tokens; with N_valid == 0 every reduced value and gradient is 0.
 *    A masked token's target must still lie in [0, vocab).  Per-token
 *    outputs of a masked token: ce/loss 0, lse still written.
 *  - Chunk: `chunk` is the pages' peak-memory knob.  It is validated
 *    (chunk*vocab <= 2^27, else 587) but the GPU never holds a chunk of
 *    logits: tiles live in tensor memory, and the tile schedule depends only
 *    on the shape, so every output is bit-identical for every valid chunk.
 *  - Determinism: no atomics on any output; the same inputs give the same
 *    bits on every run.  The token mean is a fixed-shape double-precision
 *    tree.
 *  - Device waits are bounded: a kernel that waits too long sets an error
 *    word in the workspace and exits; lossk_device_status() (and the next
 *    call that uses the same workspace) reports it as 590.
 */
#ifndef LOSSK_H
#define LOSSK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t, without pulling in the CUDA headers. */
typedef struct CUstream_st *lossk_stream_t;

/* Status vocabulary 580-599 ("Loss functions and resident-context kernels",
 * section "Status codes").  589-592 are this library's own additions inside
 * the same range; 593-599 are unassigned. */
enum lossk_status {
    LOSSK_OK = 580,
    LOSSK_EMPTY_DIMENSION = 581,
    LOSSK_LENGTH_MISMATCH = 582,
    LOSSK_DIMENSION_TOO_LARGE = 583,
    LOSSK_WORK_BUDGET_EXCEEDED = 584,
    LOSSK_NON_FINITE_SCALAR = 585,
    LOSSK_TARGET_OUT_OF_RANGE = 586,
    LOSSK_CHUNK_EXCEEDS_LOGIT_BUDGET = 587,
    LOSSK_UNKNOWN_OBJECTIVE = 588,
    LOSSK_DEVICE_ERROR = 589,   /* a CUDA call or launch failed */
    LOSSK_DEVICE_TIMEOUT = 590, /* a device-side wait hit its time limit */
    LOSSK_UNALIGNED = 591,      /* pointer or row pitch not 16-byte aligned */
    LOSSK_UNKNOWN_FLAGS = 592   /* a flags argument with a bit this library does not define */
};

/* Flags of the _ex entry points (bitwise or; 0 = the plain call's behaviour).
 * LOSSK_ACCUMULATE_GRADS: gradients are added into d_hidden / d_weight /
 *   grad_logits instead of overwriting them (gradient accumulation across
 *   micro-batches).
 * LOSSK_REDUCE_SUM: the reduction is a sum over the counted tokens instead of
 *   their mean: total = sum_t m_t (loss_t + z_weight z_t), the other two
 *   scalars are sums too, and a_t = grad_scale m_t (no 1/N_valid).
 * Both follow the variants the pages list beside masking and scaling in the
 * parity suite of "Fuse distillation + z-loss ...", "Testing". */
enum lossk_flags { LOSSK_ACCUMULATE_GRADS = 1, LOSSK_REDUCE_SUM = 2 };

enum lossk_dtype { LOSSK_F32 = 0, LOSSK_BF16 = 1, LOSSK_F16 = 2 };

/* Distillation objective ("Fuse distillation + z-loss ...", "What it
 * does": cross-entropy, forward-KL, reverse-KL).  Any other value -> 588. */
enum lossk_direction { LOSSK_DISTILL_CE = 0, LOSSK_DISTILL_FWD_KL = 1, LOSSK_DISTILL_REV_KL = 2 };

/* Which call a workspace is sized for. */
enum lossk_kind {
    LOSSK_KIND_CE_FWD = 0,
    LOSSK_KIND_CE_BWD = 1,
    LOSSK_KIND_CE_FWD_BWD = 2,
    LOSSK_KIND_FROM_LOGITS = 3,
    LOSSK_KIND_DISTILL = 4,
    LOSSK_KIND_CE_CHUNK_CHECK = 5,
    LOSSK_KIND_SHARD_FWD = 6,      /* lossk_ce_shard_fwd, sized at (n_tok, d_model, vocab_shard) */
    LOSSK_KIND_SHARD_BWD = 7,      /* lossk_ce_shard_bwd, sized at (n_tok, d_model, vocab_shard) */
    LOSSK_KIND_SHARD_COMBINE = 8   /* lossk_ce_shard_combine, sized at (n_tok, 1, 1) */
};

/* ---- contract: host arithmetic, no device ------------------------------- */

/* Name of a status code: "ok", "empty_dimension", ... for 580-588,
 * "device_error", "device_timeout", "unaligned", "unknown_flags" for
 * 589-592, and "unknown_status" for anything else (never a neighbour's name).
 * loss_status_name in the pages' function table.  Returns a static string. */
const char *lossk_status_name(int32_t code);

/* loss_dims_check: every dimension >= 1 (581) and <= 2^24 (583), and
 * n_tok*d_model*vocab <= 2^46 (584).  The 2^24 per-dimension ceiling is this
 * library's reading: the pages name a ceiling without printing it. */
int32_t lossk_dims_check(int64_t n_tok, int64_t d_model, int64_t vocab);

/* loss_chunk_check: chunk, vocab >= 1 (581); chunk*vocab <= 2^27 (587,
 * refused, never clamped). */
int32_t lossk_chunk_check(int64_t chunk, int64_t vocab);

/* loss_logit_cells: chunk*vocab as a double; -1.0 if either is < 1. */
double lossk_logit_cells(int64_t chunk, int64_t vocab);

/* loss_work_fits: 1 when n_tok*d_model*vocab <= ceiling, decided by
 * successive division (no overflow); 0 otherwise or for any argument < 1. */
int32_t lossk_work_fits(int64_t n_tok, int64_t d_model, int64_t vocab, int64_t ceiling);

/* ce_peak_logit_cells ("Loss functions and resident-context kernels",
 * opening example): what a chunked call holds against the materialised
 * form.  chunked_cells = min(chunk, n_tok)*vocab, materialized_cells =
 * n_tok*vocab, ratio = materialized/chunked, n_chunks = ceil(n_tok/chunk),
 * status = lossk_chunk_check(chunk, vocab) (the numbers are filled in even
 * when it is 587).  Any argument < 1: cells -1, ratio 0, n_chunks 0, 581.
 * `out` is a host pointer; NULL gives 582.  Returns out->status. */
typedef struct {
    double chunked_cells;
    double materialized_cells;
    double ratio;
    int64_t n_chunks;
    int32_t status;
} lossk_peak_cells;
int32_t lossk_peak_logit_cells(int64_t n_tok, int64_t vocab, int64_t chunk, lossk_peak_cells *out);

/* Bytes of device workspace a call of `kind` needs at this shape and dtype
 * (a multiple of 256).  Returns -1 for a shape that lossk_dims_check
 * refuses. */
int64_t lossk_workspace_bytes(int32_t kind, int64_t n_tok, int64_t d_model, int64_t vocab,
                              int32_t dtype);

/* ---- device calls --------------------------------------------------------- */

/* loss_targets_in_range on device data: 580 when every one of targets[0..n)
 * lies in [0, vocab), 586 otherwise.  Synchronises `stream`. */
int32_t lossk_targets_check(int64_t n_tok, int64_t vocab, const int64_t *targets,
                            int64_t targets_len, void *workspace, int64_t workspace_bytes,
                            lossk_stream_t stream);

/* Fused projection + cross-entropy forward (fused_linear_ce_flat).
 *   hidden   [n_tok][d_model]  (dtype)       weight [vocab][d_model] (dtype)
 *   targets  int64[n_tok] in [0, vocab)      loss_mask uint8[n_tok] or NULL
 *   z_weight >= 0: adds z_weight * lse^2 per token ("Fuse distillation +
 *            z-loss ...": forward scalar log_sum_exp^2)
 * Outputs (device):
 *   lse_out     float[n_tok], required: log-sum-exp of each token's logits
 *               (the backward takes it back)
 *   ce_out      float[n_tok] or NULL: lse - target logit (0 if masked)
 *   scalars_out double[3], required: {total, ce_mean, z_mean} with
 *               total = sum_t m_t (ce_t + z_weight lse_t^2) / N_valid. */
int32_t lossk_ce_fwd(int64_t n_tok, int64_t d_model, int64_t vocab, int64_t chunk, int32_t dtype,
                     const void *hidden, int64_t hidden_len, const void *weight, int64_t weight_len,
                     const int64_t *targets, int64_t targets_len, const uint8_t *loss_mask,
                     double z_weight, float *lse_out, float *ce_out, double *scalars_out,
                     void *workspace, int64_t workspace_bytes, lossk_stream_t stream);

/* Backward of grad_scale * total (fused_linear_ce_bwd_flat; not chunked).
 * Takes lse from lossk_ce_fwd on the same inputs.  Recomputes the logit
 * tiles, forms grad_logits = a_t((1 + 2 z_weight lse_t) softmax - onehot),
 * a_t = grad_scale m_t / N_valid, in registers, and folds it into
 *   d_hidden float[n_tok][d_model] = G W      (NULL to skip)
 *   d_weight float[vocab][d_model] = G^T H    (NULL to skip)
 * Both are overwritten (not accumulated). */
int32_t lossk_ce_bwd(int64_t n_tok, int64_t d_model, int64_t vocab, int32_t dtype,
                     const void *hidden, int64_t hidden_len, const void *weight, int64_t weight_len,
                     const int64_t *targets, int64_t targets_len, const uint8_t *loss_mask,
                     double z_weight, double grad_scale, const float *lse, int64_t lse_len,
                     float *d_hidden, float *d_weight, void *workspace, int64_t workspace_bytes,
                     lossk_stream_t stream);

/* lossk_ce_fwd followed by lossk_ce_bwd on the same inputs, with one
 * validation sync instead of two: the training-step call.  lse_out is
 * required (it is also the backward's input).
 *
 * On the bf16 path with d_hidden requested, the forward is folded into the
 * d_hidden pass: every logit is exponentiated against a per-token reference
 * shift r_t = target logit * log2(e) + 64 instead of the (not yet known)
 * log-sum-exp, which saves one full logit pass.  A row whose maximum logit
 * lies more than about 110 nats above its target logit would leave the range
 * the shift covers; the call detects that (and any non-finite d_hidden) on
 * the device, reads the flag back at its end (with the validation result, in
 * the call's one synchronisation of `stream`) and then recomputes every
 * output on the separate passes.  The outputs are the same quantities either
 * way, within the tolerances. */
int32_t lossk_ce_fwd_bwd(int64_t n_tok, int64_t d_model, int64_t vocab, int64_t chunk,
                         int32_t dtype, const void *hidden, int64_t hidden_len, const void *weight,
                         int64_t weight_len, const int64_t *targets, int64_t targets_len,
                         const uint8_t *loss_mask, double z_weight, double grad_scale,
                         float *lse_out, float *ce_out, double *scalars_out, float *d_hidden,
                         float *d_weight, void *workspace, int64_t workspace_bytes,
                         lossk_stream_t stream);

/* Cross-entropy from materialised logits [n_tok][vocab] (ce_from_logits_flat).
 * Same outputs as lossk_ce_fwd; grad_logits (same dtype as logits, or NULL)
 * receives grad_scale * d total / d logits. */
int32_t lossk_ce_from_logits(int64_t n_tok, int64_t vocab, int32_t dtype, const void *logits,
                             int64_t logits_len, const int64_t *targets, int64_t targets_len,
                             const uint8_t *loss_mask, double z_weight, double grad_scale,
                             float *lse_out, float *ce_out, double *scalars_out, void *grad_logits,
                             int64_t grad_len, void *workspace, int64_t workspace_bytes,
                             lossk_stream_t stream);

/* Distillation against a full teacher distribution, forward and backward in
 * one call ("Fuse distillation + z-loss ...", "What it does").  With
 * a = logits/T, b = teacher/T, q = softmax(a), p = softmax(b):
 *   LOSSK_DISTILL_CE:     L_t = -sum p log q
 *   LOSSK_DISTILL_FWD_KL: L_t = sum p (log p - log q)
 *   LOSSK_DISTILL_REV_KL: L_t = sum q (log q - log p)
 *   z_t = lse(a)^2 over the same student softmax
 *   total = sum_t m_t (L_t + z_weight z_t) / N_valid
 * Gradients of grad_scale * total: d/dlogits = (q - p)/T (CE, fKL) or
 * q (log q - log p - L_t)/T (rKL), plus 2 z_weight lse(a) q / T; no T^2
 * factor.  temperature must be finite and > 0 (585).
 *   teacher_logits [n_tok][vocab] (dtype)
 *   scalars_out double[3] {total, distill_mean, z_mean}, required
 *   per_token_out float[n_tok] or NULL: L_t (0 if masked)
 *   lse_out float[n_tok] or NULL: lse(a)
 *   d_hidden, d_weight: float gradients or NULL to skip. */
int32_t lossk_distill_fwd_bwd(int64_t n_tok, int64_t d_model, int64_t vocab, int64_t chunk,
                              int32_t dtype, const void *hidden, int64_t hidden_len,
                              const void *weight, int64_t weight_len, const void *teacher_logits,
                              int64_t teacher_len, const uint8_t *loss_mask, int32_t direction,
                              double temperature, double z_weight, double grad_scale,
                              double *scalars_out, float *per_token_out, float *lse_out,
                              float *d_hidden, float *d_weight, void *workspace,
                              int64_t workspace_bytes, lossk_stream_t stream);

/* lossk_ce_fwd_bwd with flags (lossk_flags).  With LOSSK_ACCUMULATE_GRADS
 * the call adds into d_hidden and d_weight, and touches them only after the
 * end read-back has come back clean (the d_weight pass and the addition of
 * d_hidden then follow it).  Unknown flag bits give 592 (checked after 585). */
int32_t lossk_ce_fwd_bwd_ex(int64_t n_tok, int64_t d_model, int64_t vocab, int64_t chunk,
                            int32_t dtype, const void *hidden, int64_t hidden_len, const void *weight,
                            int64_t weight_len, const int64_t *targets, int64_t targets_len,
                            const uint8_t *loss_mask, double z_weight, double grad_scale,
                            uint32_t flags, float *lse_out, float *ce_out, double *scalars_out,
                            float *d_hidden, float *d_weight, void *workspace, int64_t workspace_bytes,
                            lossk_stream_t stream);

/* lossk_distill_fwd_bwd with flags (lossk_flags). */
int32_t lossk_distill_fwd_bwd_ex(int64_t n_tok, int64_t d_model, int64_t vocab, int64_t chunk,
                                 int32_t dtype, const void *hidden, int64_t hidden_len,
                                 const void *weight, int64_t weight_len, const void *teacher_logits,
                                 int64_t teacher_len, const uint8_t *loss_mask, int32_t direction,
                                 double temperature, double z_weight, double grad_scale, uint32_t flags,
                                 double *scalars_out, float *per_token_out, float *lse_out,
                                 float *d_hidden, float *d_weight, void *workspace,
                                 int64_t workspace_bytes, lossk_stream_t stream);

/* ce_chunk_invariance_flat ("Loss functions and resident-context kernels",
 * lossk function table and "Chunk invariance is checked to the last bit"):
 * runs lossk_ce_fwd at chunk = 1 and at chunk = n_tok and writes to the host
 * double *max_abs_delta the largest absolute difference between the two
 * runs over the three reduced scalars and every token's lse and ce (0.0 is
 * the property).  When n_tok*vocab exceeds the 2^27 logit budget, the second
 * chunk is the largest the budget allows (this library's reading: the check
 * would otherwise be refused at every realistic size).  Workspace kind
 * LOSSK_KIND_CE_CHUNK_CHECK.  Synchronises `stream`. */
int32_t lossk_ce_chunk_invariance(int64_t n_tok, int64_t d_model, int64_t vocab, int32_t dtype,
                                  const void *hidden, int64_t hidden_len, const void *weight,
                                  int64_t weight_len, const int64_t *targets, int64_t targets_len,
                                  const uint8_t *loss_mask, double z_weight, double *max_abs_delta,
                                  void *workspace, int64_t workspace_bytes, lossk_stream_t stream);

/* Distillation from materialised student logits [n_tok][vocab] (the
 * (loss, z_loss, grad_logits) shape of "Fuse distillation + z-loss ...",
 * "Changes": the from-distribution forward/backward with its optional z
 * slot).  Same objectives, temperature, mask, divisor and scalars as
 * lossk_distill_fwd_bwd, with the student logits given instead of hidden and
 * weight.  logits and teacher_logits share `dtype`; grad_logits (same dtype,
 * or NULL to skip) receives grad_scale * d total / d logits.  flags as in
 * lossk_flags (LOSSK_ACCUMULATE_GRADS adds into grad_logits).  An HBM
 * stream: one block per token row.  Workspace kind LOSSK_KIND_FROM_LOGITS. */
int32_t lossk_distill_from_logits(int64_t n_tok, int64_t vocab, int32_t dtype, const void *logits,
                                  int64_t logits_len, const void *teacher_logits, int64_t teacher_len,
                                  const uint8_t *loss_mask, int32_t direction, double temperature,
                                  double z_weight, double grad_scale, uint32_t flags,
                                  double *scalars_out, float *per_token_out, float *lse_out,
                                  void *grad_logits, int64_t grad_len, void *workspace,
                                  int64_t workspace_bytes, lossk_stream_t stream);

/* Synchronises `stream`, then reports and clears the workspace's device
 * error word: 580 (none), 590 (a bounded device wait timed out) or 589. */
int32_t lossk_device_status(void *workspace, int64_t workspace_bytes, lossk_stream_t stream);

/* ---- vocabulary-parallel cross-entropy ---------------------------------------
 * The weight's vocabulary rows split into contiguous shards, one per rank
 * ("Fuse distillation + z-loss ...", "Changes": its tests add a
 * tensor-parallel distributed subtest; "Validation": the world_size=2
 * tensor-parallel subtests).  Shard p holds rows [v0, v0 + vocab_shard) of a
 * vocabulary of vocab_total.  A step runs, per rank:
 *   1. lossk_ce_shard_fwd on the rank's shard -> partials float[3][n_tok];
 *   2. an exchange the caller makes (an all-gather of the 3 n_tok floats of
 *      every rank, in shard order, over NCCL or any other transport) ->
 *      partials_all float[n_shards][3][n_tok];
 *   3. lossk_ce_shard_combine -> lse, ce and the three scalars, exactly the
 *      outputs of lossk_ce_fwd on the whole vocabulary (every rank gets them);
 *   4. lossk_ce_shard_bwd with that lse -> the shard's d_weight rows and its
 *      share of d_hidden; the caller's all-reduce (sum) of the shares over the
 *      ranks gives d_hidden.
 * Partials of one shard, per token t:
 *   partials[0][t] = log sum_{v in shard} exp(s_tv)  (the shard's lse)
 *   partials[1][t] = s_{t,y_t} if the shard holds y_t, else 0
 *   partials[2][t] = 1 if the shard holds y_t, else 0
 * The shard's partials depend on the shard alone (its lse comes from the
 * same CTA-pair statistics pass as lossk_ce_fwd, on the shard's rows).
 * Targets are global ids: each must lie in [0, vocab_total) (586).
 * Shape checks: the fused calls' checks at (n_tok, d_model, vocab_shard);
 * vocab_total < 1: 581, > 2^24: 583; v0 < 0 or v0 + vocab_shard >
 * vocab_total: 582. */
int32_t lossk_ce_shard_fwd(int64_t n_tok, int64_t d_model, int64_t vocab_shard, int64_t v0, int64_t vocab_total,
                           int32_t dtype, const void *hidden, int64_t hidden_len, const void *weight_shard,
                           int64_t weight_len, const int64_t *targets, int64_t targets_len, float *partials,
                           int64_t partials_len, void *workspace, int64_t workspace_bytes, lossk_stream_t stream);

/* Combines the gathered partials float[n_shards][3][n_tok] (device) into
 * lse_out, ce_out (or NULL) and scalars_out {total, ce_mean, z_mean}, as
 * lossk_ce_fwd defines them: lse = M + log sum_p exp(lse_p - M) over the
 * shards, ce = lse - the target logit of the one shard whose flag is set.  A
 * token whose flags do not sum to 1 (no shard, or two, held its target: the
 * shards do not tile the vocabulary) gives 586 before any output is written.
 * Synchronises `stream` once, after that check. */
int32_t lossk_ce_shard_combine(int64_t n_tok, int64_t n_shards, const float *partials_all, int64_t partials_len,
                               const uint8_t *loss_mask, double z_weight, float *lse_out, float *ce_out,
                               double *scalars_out, void *workspace, int64_t workspace_bytes, lossk_stream_t stream);

/* The shard's backward, given the whole row's lse (from
 * lossk_ce_shard_combine): grad_logits restricted to the shard's columns,
 * a_t((1 + 2 z_weight lse_t) softmax - onehot) with a_t = grad_scale m_t /
 * N_valid, folded into
 *   d_hidden_part  float[n_tok][d_model] = sum over the shard's columns of G W
 *                  (NULL to skip; summed over the shards it is d_hidden)
 *   d_weight_shard float[vocab_shard][d_model] = G^T H for the shard's rows
 *                  (NULL to skip)
 * Both are overwritten. */
int32_t lossk_ce_shard_bwd(int64_t n_tok, int64_t d_model, int64_t vocab_shard, int64_t v0, int64_t vocab_total,
                           int32_t dtype, const void *hidden, int64_t hidden_len, const void *weight_shard,
                           int64_t weight_len, const int64_t *targets, int64_t targets_len, const uint8_t *loss_mask,
                           double z_weight, double grad_scale, const float *lse, int64_t lse_len,
                           float *d_hidden_part, float *d_weight_shard, void *workspace, int64_t workspace_bytes,
                           lossk_stream_t stream);

/* Self-test of the failure detection every tensor-core kernel carries: each
 * device-side wait gives up after a time limit, records a timeout in the
 * workspace's error word and lets its kernel unwind (copies drained, tensor
 * memory freed, every thread exits), so a stalled pipeline surfaces as 590
 * instead of a hung GPU.  This call runs that mechanism on purpose in one
 * small block with the kernels' roles: a producer arrives on n_arrive of
 * n_stages (1..8) pipeline barriers and a consumer waits on each of them in
 * turn with a limit of limit_ns (1e3..1e9 ns, else 585).  With n_arrive <
 * n_stages the consumer's wait on stage n_arrive runs out after limit_ns.
 * Writes the number of stages the consumer saw complete to the host int
 * *stages_seen (may be NULL).  Synchronises `stream`.  Returns 590 when the
 * wait ran out (the error word stays set, as after a real timeout:
 * lossk_device_status reports and clears it, and until then every call on
 * this workspace returns 590), else 580.  Stage counts out of range, or a
 * workspace of fewer than 256 bytes or NULL: 582; a workspace not 256-byte
 * aligned: 591; limit_ns out of range: 585. */
int32_t lossk_selftest_wait(int32_t n_stages, int32_t n_arrive, int64_t limit_ns, int32_t *stages_seen,
                            void *workspace, int64_t workspace_bytes, lossk_stream_t stream);

/* lossk_ce_from_logits without a workspace, for callers that cannot allocate
 * device memory.  The pages have no counterpart to this entry point.
 *
 * Some callers have no way to give the library scratch memory: a plug-in
 * inside another framework whose device memory is all owned by that
 * framework's arena, or a runtime whose memory plan is fixed at start-up and
 * which treats any allocation made during a step as an error.  This variant
 * computes exactly what lossk_ce_from_logits computes (same kernels, same
 * outputs, same status codes) but keeps its scratch -- a 256-byte header and
 * three doubles per token -- in a device array built into the library, so
 * the call allocates nothing (no cudaMalloc, no cudaFree, no allocating
 * library routine).  The caller still passes every input and output.
 *
 * Limits and rules:
 *  - n_tok <= 16384 (the array holds 256 + 3*8*16384 bytes, about 384 KB,
 *    held by every GPU that loads the library until the process exits);
 *    larger n_tok returns 583.  Every other check, its order and its status
 *    code are those of lossk_ce_from_logits (the two share them), 590
 *    included.
 *  - The first call on each device looks up the array's device address with
 *    that device current (cudaGetSymbolAddress) and caches it.  The cached
 *    address is that of the device's primary context: after a
 *    cudaDeviceReset of a device, do not call this entry point on it again
 *    in the same process.
 *  - Like lossk_ce_from_logits, each call synchronises `stream` once, after
 *    its validation kernel, to read back the target-range flag, so a call
 *    cannot be recorded into a CUDA graph.
 *  - All calls share the one array, which keeps the previous call's
 *    contents; each call clears the header before use.  Calls that overlap
 *    on the GPU (two streams, or two host threads on one device) race on it
 *    and must be serialised by the caller.
 *  - Its kernels are counted and traced like every other launch
 *    (lossk_launch_count, lossk_profile_read). */
int32_t lossk_ce_from_logits_static(int64_t n_tok, int64_t vocab, int32_t dtype, const void *logits,
                                    int64_t logits_len, const int64_t *targets, int64_t targets_len,
                                    const uint8_t *loss_mask, double z_weight, double grad_scale,
                                    float *lse_out, float *ce_out, double *scalars_out,
                                    void *grad_logits, int64_t grad_len, lossk_stream_t stream);

/* ---- tracing ----------------------------------------------------------------
 * Every kernel the library launches belongs to one of LOSSK_N_KERNELS kinds
 * (lossk_kernel_name gives its name).  lossk_launch_count() is the number of
 * kernels launched by this process so far.  With lossk_profile_enable(1),
 * each launch is bracketed by a CUDA event pair recorded on its own stream
 * (no synchronisation is added); lossk_profile_read() waits for the recorded
 * events, adds their durations per kind into total_ms[kind] and
 * launches[kind] (host arrays of `cap` entries), and clears them if `reset`.
 * Returns the number of kinds written, or -1 on a CUDA error. */
#define LOSSK_N_KERNELS 23
const char *lossk_kernel_name(int32_t kind);
int64_t lossk_launch_count(void);
int32_t lossk_profile_enable(int32_t on);
int32_t lossk_profile_read(double *total_ms, int64_t *launches, int32_t cap, int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* LOSSK_H */
