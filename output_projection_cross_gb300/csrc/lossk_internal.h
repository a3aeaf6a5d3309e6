// lossk_internal.h -- shared between the host entry points and the kernels:
// the workspace layout, the per-token parameter records and the launcher
// declarations.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace lossk {

constexpr double LN2 = 0.69314718055994530942;
constexpr double LOG2E = 1.44269504088896340736;

// Tile geometry of the tensor-core path.
constexpr int TC_BM = 128;         // rows of X per tile (MMA M, TMEM lanes)
constexpr int TC_BN_FWD = 256;     // logit tile width of the label-CE forward
constexpr int TC_BN_ACC = 128;     // vocabulary tile width the d_hidden splits are counted in
constexpr int TC_BK = 64;          // K per pipeline stage (one 128-byte swizzle row)
constexpr int TC_SLICE = 256;      // d_model columns one backward CTA accumulates
// Tile geometry of the fp32 FFMA path.
constexpr int FP_BM = 64, FP_BN = 64, FP_BK = 16, FP_SLICE = 64;

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
    int err;          // device error word (ERR_* in ptx.cuh)
    int bad_targets;  // count of targets outside [0, vocab)
    int n_valid;      // counted tokens
    int redo;         // fused pass: a row left the range its reference shift covers
    int pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Per-(token, logit tile) partial statistics written by the forward pass
// (structure of arrays, each [n_ct][n_pad]).  Label CE: m2 (running max of
// logit*log2e) and z (sum of 2^(logit*log2e - m2)).  Distillation: the same
// pair for logit/T and one direction-dependent cross term with the teacher.
constexpr int NSTAT_CE = 2;
constexpr int NSTAT_DISTILL = 3;

struct WsLayout {
    int64_t n_pad = 0;       // n_tok rounded up to 128
    int64_t n_ct = 0;        // logit tiles across the vocabulary in the forward
    int64_t bn = 0;          // their width
    int64_t nstat = 0;
    int64_t nsplit = 0;      // vocabulary splits of the d_hidden pass
    size_t off_tokp = 0;     // float4 [n_pad]   per-token backward parameters
    size_t off_tgt = 0;      // float  [n_pad]   target logit
    size_t off_tokacc = 0;   // double [3][n_pad] per-token reduction terms
    size_t off_part = 0;     // float  [nstat][n_ct][n_pad]
    size_t off_dhpart = 0;   // float  [nsplit][n_tok][d_model] (nsplit > 1)
    size_t off_zpart = 0;    // float  [nsplit * BWD_MAX_CL][n_pad] fused pass: sums of G' per (split, CTA)
    size_t off_dhc = 0;      // float2 [n_pad] fused pass: d_hidden coefficients per token
    size_t off_gring = 0;    // bf16 [G_RING_ROWS][128] grad-tile ring of the group passes
    size_t off_gsig = 0;     // unsigned [2][G_MAX_CTAS][G_SLOTS] the ring's hand-off counters
    size_t off_tstat = 0;    // double2 [n_pad] distillation: teacher (lse_t2, Eb) per token
    size_t off_dhacc = 0;    // float [n_tok][d_model] training step with accumulation: d_hidden before it is added
    size_t off_chk = 0;      // chunk self-check: two runs' lse and ce, float [4][n_pad], + double [8]
    size_t off_red = 0;      // double [8] reduction output scratch
    size_t total = 0;
};

// kind: lossk_kind; dtype: lossk_dtype.  Returns false for an invalid shape.
bool ws_layout(int kind, int64_t n, int64_t d, int64_t V, int dtype, WsLayout *L);
int64_t dh_splits(int64_t n, int64_t d, int64_t V, int dtype);

// ---- tensor-core kernel arguments ------------------------------------------
enum TcMode : int { TC_STATS = 0, TC_ROWS = 1, TC_COLS = 2 };
enum Direction : int { DIR_CE = 0, DIR_FKL = 1, DIR_RKL = 2 };

struct TcArgs {
    CUtensorMap map_x;     // X operand (K-major), box {64, 128}
    CUtensorMap map_y;     // Y operand (K-major), box {64, BN}
    CUtensorMap map_ys;    // Y rows x d-slice as the MN-major B operand, box {64, 64}
    int n_x;               // rows of X (n_tok in STATS/ROWS, vocab in COLS)
    int n_y;               // rows of Y
    int d;                 // contraction length (d_model)
    int n_tok, vocab;
    int n_xt;              // X tiles
    int n_yt;              // Y tiles
    int n_items;           // STATS: (x tile, y tile) pairs
    int n_slices;          // ROWS/COLS: d_model slices
    int n_split;           // ROWS: vocabulary splits
    int direction;         // distillation objective
    float inv_t_l2e;       // log2(e) / temperature
    const int64_t *targets;
    const uint16_t *teacher; // distillation forward: teacher logits [n_tok][vocab] (bf16)
    const double2 *tstat;  // distillation forward: per token (lse_t2, Eb) from teacher_stats
    const float4 *tokp;    // per-token backward parameters
    float *part;           // STATS output (structure of arrays)
    float *tgt;            // STATS (label CE): target logit per token
    int64_t part_stride;   // n_pad
    int64_t part_plane;    // n_ct * n_pad
    float *out;            // ROWS/COLS output
    int64_t out_split_stride;
    int *err;
};

// ---- backward (cluster-shared grad tiles) kernel arguments -------------------
// BWD_FUSED: the d_hidden schedule run as the forward pass as well, with a
// per-token reference shift in place of the log-sum-exp (k_bwp.cu).
enum BwdMode : int { BWD_ROWS = 1, BWD_COLS = 2, BWD_FUSED = 3 };

// The fused pass's reference: r_t = s[t][y_t] log2e + FUSED_SHIFT (log2 units).
constexpr float FUSED_SHIFT = 64.f;

// Loop supertile: the logit tile of the cluster passes is 128 fixed rows x
// BWD_BN loop columns.  Grad-tile ring: G_SLOTS slots of one supertile
// (2 x 128 x 128 bf16) per CTA, for at most G_MAX_CTAS CTAs.
constexpr int BWD_BN = 256;
constexpr int BWD_MAX_CL = 16;     // CTAs per group at most
constexpr int G_SLOTS = 2;
constexpr int G_MAX_CTAS = 160;
constexpr int64_t G_RING_ROWS = int64_t(G_MAX_CTAS) * G_SLOTS * 2 * 128;   // rows of 128 bf16

struct BwdArgs {
    CUtensorMap map_fix;   // the fixed tensor (hidden for d_hidden, weight for d_weight), box {64, 128} (a CTA's half)
    CUtensorMap map_loop;  // the loop tensor as the logit MMA's B operand (a CTA's half), box {64, 128}
    CUtensorMap map_ys;    // the loop tensor rows x d-slice (MN-major B of the accumulate), box {64, 64}
    CUtensorMap map_g;     // the grad-tile ring [G_RING_ROWS][128] bf16, box {64, 128}
    CUtensorMap map_ys3;   // map_ys as [64-column blocks][rows][64] (d_model % 64 == 0): one box {64, 64, 2}
    int ys3;               // map_ys3 is valid
    CUtensorMap map_teach; // distillation d_weight: teacher [n_tok][vocab] bf16, box {32, 32}
    CUtensorMap map_gst;   // the grad-tile ring for stores, box {32, 32} bf16, 64-byte swizzle
    int g_tma;             // map_gst is valid: grad tiles leave through shared memory and TMA
    CUtensorMap map_out;   // d_weight output [vocab][d_model] fp32, box {16, 32}, 64-byte swizzle
    int out_tma;           // d_weight: store (or, accumulating, add) through map_out
    CUtensorMap map_out3;  // d_hidden passes: `out` as fp32 [planes][n_tok][d_model], box {32, 32, 1}, 128-byte swizzle
    int out3_tma;          // the d_hidden passes store (or add) their accumulators through map_out3
    uint16_t *gscr;        // the grad-tile ring itself
    const uint16_t *teacher; // teacher logits [n_tok][vocab] (bf16), read by the epilogue
    int n_tok, vocab, d;
    int n_fixed;           // fixed tiles: token tiles (d_hidden) or vocabulary tiles (d_weight)
    int n_loop;            // loop supertiles (BWD_BN columns): vocabulary (d_hidden) or tokens (d_weight)
    int n_split;           // splits of the loop range (d_hidden)
    int n_cl;              // CTAs per group (consecutive blocks sharing grad tiles) = 256-column d-slices
    int n_dg;              // d-groups (clusters per fixed tile and split)
    int direction;
    float inv_t_l2e;
    const float4 *tokp;
    float *out;
    int64_t out_split_stride;
    float *zpart;          // BWD_FUSED: sums of G' [n_split * n_cl][zpart_stride]
    int64_t zpart_stride;
    int accumulate;        // add the accumulator into `out` instead of overwriting it
    float out_scale;       // fp16 operands: the factor the stored accumulator is multiplied by
    const int *refused;    // nonzero: the validation before found a bad target; return at once
    unsigned *gsig;        // grad-tile ring hand-off counters [2][G_MAX_CTAS][G_SLOTS] (ready, free)
    int *err;
};

// Group geometry of the backward for a d_model: slices of 256 columns, one
// per CTA of a group of at most BWD_MAX_CL CTAs, d-groups beyond that (each
// d-group recomputes the logits); chosen from the shape alone.
// The passes run on CTA pairs (k_bwp.cu): n_cl pairs per group, fixed tiles of
// 256 rows.
struct BwdGeom {
    int n_cl, n_dg;
};
BwdGeom bwd_geometry(int64_t d, bool distill);

// Kernel kinds, for the launch counter and the optional per-kernel timing.
enum KernelKind : int {
    KK_VALIDATE = 0,
    KK_TC_STATS,
    KK_TC_ROWS,
    KK_TC_COLS,
    KK_FP_STATS,
    KK_FP_ROWS,
    KK_FP_COLS,
    KK_MERGE_CE,
    KK_MERGE_DISTILL,
    KK_REDUCE,
    KK_TOKP,
    KK_SUM_SPLITS,
    KK_FROM_LOGITS,
    KK_TC_FUSED,
    KK_TGT_LOGIT,
    KK_MERGE_FUSED,
    KK_COMBINE_DH,
    KK_TEACHER_STATS,
    KK_DISTILL_LOGITS,
    KK_READBACK,
    KK_SELFTEST,
    KK_SHARD_TGT,
    KK_SHARD_COMBINE,
    KK_N
};

// Brackets one kernel launch: counts it (lossk_launch_count) and, when
// profiling is on, records a CUDA event pair around it on its stream
// (lossk_profile_read).  Every launch of the library goes through one.
class Launch {
  public:
    Launch(int kind, cudaStream_t st);
    ~Launch();
    Launch(const Launch &) = delete;
    Launch &operator=(const Launch &) = delete;

  private:
    int kind_;
    cudaStream_t st_;
    cudaEvent_t a_ = nullptr, b_ = nullptr;
    bool active_ = false;
};

// ---- cross-entropy from given logits, shared by its two entry points --------
// The argument checks of lossk_ce_from_logits in the documented order (581,
// 583, 582, 591, 585).  With `workspace` the scratch is the caller's workspace
// (null, size and alignment checked, its layout returned in *L); without it
// the scratch is a built-in array holding at most max_tok tokens (more: 583).
int32_t check_from_logits(int64_t n, int64_t V, int32_t dtype, const void *logits, int64_t logits_len,
                          const int64_t *targets, int64_t targets_len, const float *lse_out,
                          const double *scalars_out, const void *grad, int64_t grad_len, double wz,
                          double gs, const void *workspace, int64_t workspace_bytes, int64_t max_tok,
                          WsLayout *L);
// Validation (586, or 590 for a device error word already set in hdr), the
// row stream and the token mean, on scratch hdr (256 bytes) + tokacc
// (3 x n_pad doubles).  Synchronises `st` once, after the validation.
int32_t run_from_logits(int64_t n, int64_t V, int32_t dtype, const void *logits, const int64_t *targets,
                        const uint8_t *mask, double wz, double gs, float *lse_out, float *ce_out,
                        double *scalars_out, void *grad, WsHeader *hdr, double *tokacc, int64_t n_pad,
                        cudaStream_t st);

// ---- launchers (all enqueue on `st`) -----------------------------------------
cudaError_t launch_validate(const int64_t *targets, const uint8_t *mask, int64_t n, int64_t V,
                            WsHeader *hdr, cudaStream_t st);
// One block: a producer arrives on n_arrive of n_stages barriers, a consumer
// waits on each with the bounded wait (limit_ns); an expired wait sets *err.
cudaError_t launch_wait_selftest(int n_stages, int n_arrive, uint64_t limit_ns, int *err, int *seen,
                                 cudaStream_t st);
// The group passes on CTA pairs (k_bwp.cu): persistent groups, at most as many
// as fit at once, walking `n_units` units.  f16: fp16 operands (BWD_ROWS /
// BWD_COLS only); otherwise bf16.
cudaError_t launch_bwp(int mode, bool distill, bool f16, const BwdArgs &a, int n_units, cudaStream_t st);
cudaError_t launch_fwd2(const TcArgs &a, bool distill, bool f16, int grid, cudaStream_t st);
cudaError_t launch_fp(int mode, bool distill, const void *X, const void *Y, const float *teach,
                      int n_x, int n_y, int d, int n_tok, int vocab, int n_split, int direction,
                      float inv_t, const int64_t *targets, const float4 *tokp, const double2 *tstat,
                      float *part,
                      float *tgt, int64_t part_stride, int64_t part_plane, float *out,
                      int64_t out_split_stride, cudaStream_t st, bool accumulate = false);
// precise: exact exp2 rescales (the fp32 inputs path); else ex2.approx.
cudaError_t launch_merge_ce(const float *part, const float *tgt, const int64_t *targets,
                            const uint8_t *mask, int64_t n, int64_t n_ct, int64_t n_pad,
                            double wz, float *lse_out, float *ce_out, double *tokacc,
                            cudaStream_t st, bool precise);
cudaError_t launch_merge_distill(const float *part, const double2 *tstat, const uint8_t *mask, int64_t n,
                                 int64_t n_ct, int64_t n_pad, int direction, double wz, float *lse_out,
                                 float *per_token, double *tokacc, float4 *tokp, double alpha,
                                 double temperature, cudaStream_t st);
// Teacher log-sum-exp and sum p*logit per token (one block per token row).
// dtype: lossk_dtype (0 fp32, 1 bf16, 2 fp16) here and in the other row-stream launchers.
cudaError_t launch_teacher_stats(int dtype, const void *teach, int64_t n, int64_t V, double temperature,
                                 double2 *out, cudaStream_t st);
// sum: the three scalars are sums over the tokens instead of means over N_valid.
cudaError_t launch_reduce(const double *tokacc, int64_t n, int64_t n_pad, const WsHeader *hdr,
                          double wz, double *scalars_out, cudaStream_t st, bool sum = false);
// v0, n_rows: the weight rows the passes see are vocabulary rows [v0, v0 + n_rows)
// (a shard); a target outside them gets no one-hot term.
cudaError_t launch_tokp_ce(const float *lse, const int64_t *targets, const uint8_t *mask,
                           int64_t n, int64_t n_pad, double alpha, double wz, float4 *tokp,
                           cudaStream_t st, int64_t v0, int64_t n_rows);
// Vocabulary shards: the target logit and its flag per token; the gathered
// partials' check (bad_targets, n_valid into the header) and their combination
// into lse, ce and the token-mean terms.
cudaError_t launch_shard_tgt(int dtype, const void *H, const void *Ws, const int64_t *targets, int64_t n,
                             int64_t d, int64_t v0, int64_t n_rows, float *tgt, float *flag, cudaStream_t st);
cudaError_t launch_shard_check(const float *parts, int64_t P, int64_t n, const uint8_t *mask, WsHeader *hdr,
                               cudaStream_t st);
cudaError_t launch_shard_combine(const float *parts, int64_t P, int64_t n, int64_t n_pad, const uint8_t *mask,
                                 double wz, float *lse_out, float *ce_out, double *tokacc, cudaStream_t st);
// accumulate: out += the sum instead of out = the sum.
cudaError_t launch_sum_splits(const float *part, int64_t nsplit, int64_t count, float *out,
                              cudaStream_t st, bool accumulate = false);
// The fused forward + d_hidden path (label CE, bf16): target logit and
// reference shift per token; merge of the fused pass's sums into lse, ce, z
// and the backward parameters; d_hidden from the split partials.
// Copies the header's first four words (err, bad_targets, n_valid, redo) to
// `dst`, a device view of mapped pinned host memory (one warp, no copy engine).
cudaError_t launch_publish_header(const WsHeader *hdr, int *dst, cudaStream_t st);
// Validation and the target logit / reference shift in one launch (the bf16 training step).
cudaError_t launch_validate_tgt(const uint16_t *H, const uint16_t *W, const int64_t *targets,
                                const uint8_t *mask, int64_t n, int64_t d, int64_t V, int64_t n_pad,
                                WsHeader *hdr, float *tgt, float4 *tokp, cudaStream_t st);
cudaError_t launch_tgt_logit(bool f16, const uint16_t *H, const uint16_t *W, const int64_t *targets, int64_t n,
                             int64_t d, int64_t n_pad, float *tgt, float4 *tokp, cudaStream_t st);
// gs, sum: the gradient scale and the reduction; alpha comes from the header's N_valid.
cudaError_t launch_merge_fused(const float *zpart, int64_t nz, const float *tgt, const int64_t *targets,
                               const uint8_t *mask, int64_t n, int64_t n_pad, double gs, bool sum, double wz,
                               float *lse_out, float *ce_out, double *tokacc, float4 *tokp,
                               float2 *dhc, WsHeader *hdr, cudaStream_t st);
cudaError_t launch_combine_dh(const float *part, int64_t nsplit, int64_t n, int64_t d,
                              const uint16_t *W, const int64_t *targets, const float2 *dhc,
                              float *out, WsHeader *hdr, cudaStream_t st);
// Distillation from given student logits: per token row the losses, lse and
// backward parameters, and grad_logits (or nothing when grad is NULL).
// at_on: the gradient scale of a counted token before the 1/T factor.
cudaError_t launch_distill_logits(int dtype, const void *student, const void *teacher, const uint8_t *mask,
                                  int64_t n, int64_t V, int direction, double temperature, double wz,
                                  double at_on, float *lse_out, float *per_token, double *tokacc,
                                  int64_t n_pad, void *grad, bool accumulate, cudaStream_t st);
cudaError_t launch_from_logits(int dtype, const void *logits, const int64_t *targets,
                               const uint8_t *mask, int64_t n, int64_t V, double wz,
                               double alpha, float *lse_out, float *ce_out, double *tokacc,
                               void *grad, cudaStream_t st);

} // namespace lossk
