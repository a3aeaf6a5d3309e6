// k_simt.cu -- the CUDA-core kernels of the fused LM-head loss:
//   validate       target-range guard and counted-token count
//                  ("Loss functions and resident-context kernels", lossk
//                  function table: loss_targets_in_range)
//   merge_ce       per token: combine the per-tile (max, sum-exp) partials in
//                  tile order into lse, then ce = lse - target logit and
//                  z = lse^2 ("Fuse distillation + z-loss ...", "What it does")
//   teacher_stats  per token, the teacher's log-sum-exp and sum p*logit over its
//                  whole row: an HBM stream over the teacher logits
//   merge_distill  the student's partials with the teacher's statistics, for
//                  the three distillation objectives, plus the backward parameters
//   reduce         fixed-shape double-precision tree over tokens -> the means
//   tokp_ce        per-token backward parameters of the label loss
//   sum_splits     d_hidden partials of the vocabulary splits, in split order
//   tgt_logit      the target logit s[t][y_t] per token and the reference
//                  shift r_t the fused pass exponentiates against
//   validate_tgt   the training step's first launch: validate and tgt_logit
//                  in one pass
//   merge_fused    fused path: per token, the pass's sums of 2^(s log2e - r_t)
//                  -> lse, ce, z and the backward parameters; flags a row
//                  whose sum left the range the shift covers
//   combine_dh     fused path: d_hidden = coef_t * (sum of split partials)
//                  - a_t W[y_t], in split order
//   from_logits    cross-entropy from materialised logits (ce_from_logits_flat):
//                  a row-streaming, HBM-bound kernel with an optional
//                  grad_logits write
//   fp_kernel      the fp32 inputs path: the same three passes as the tensor
//                  core kernel (statistics, d_hidden, d_weight) on FFMA tiles.
#include "lossk_internal.h"
#include "ptx.cuh"

#include <cfloat>
#include <type_traits>

namespace lossk {

// ---------------------------------------------------------------------------
__global__ void validate_kernel(const int64_t *__restrict__ targets, const uint8_t *__restrict__ mask,
                                int64_t n, int64_t V, WsHeader *hdr)
{
    int bad = 0, valid = 0;
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < n;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (targets) {
            const int64_t y = targets[t];
            bad += (y < 0 || y >= V) ? 1 : 0;
        }
        valid += mask ? (mask[t] != 0) : 1;
    }
    for (int o = 16; o > 0; o >>= 1) {
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
        valid += __shfl_xor_sync(0xffffffffu, valid, o);
    }
    if ((threadIdx.x & 31) == 0) {
        if (bad) atomicAdd(&hdr->bad_targets, bad);
        if (valid) atomicAdd(&hdr->n_valid, valid);
    }
}

// The host's read-back of a call's header words goes through mapped host
// memory written by this one warp, not through a copy engine (where the
// 16-byte copy would queue behind other streams' large copies).
__global__ void __launch_bounds__(32) publish_header_kernel(const WsHeader *__restrict__ hdr, int *__restrict__ dst)
{
    if (threadIdx.x < 4) dst[threadIdx.x] = reinterpret_cast<const volatile int *>(hdr)[threadIdx.x];
}

cudaError_t launch_publish_header(const WsHeader *hdr, int *dst, cudaStream_t st)
{
    publish_header_kernel<<<1, 32, 0, st>>>(hdr, dst);
    return cudaGetLastError();
}

cudaError_t launch_validate(const int64_t *targets, const uint8_t *mask, int64_t n, int64_t V,
                            WsHeader *hdr, cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(&hdr->bad_targets, 0, 3 * sizeof(int), st);   // bad, n_valid, redo
    if (e != cudaSuccess) return e;
    int grid = static_cast<int>((n + 255) / 256);
    if (grid > 1024) grid = 1024;
    validate_kernel<<<grid, 256, 0, st>>>(targets, mask, n, V, hdr);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Failure-detection self-test: the tensor-core kernels' role structure in
// miniature.  Thread 0 of warp 0 (the producer) arrives on the first n_arrive
// of n_stages single-arrival barriers; lane 0 of warp 1 (the consumer, also
// the tensor-memory owner's warp) waits on every stage with the same bounded
// wait the real kernels use, here with a limit of limit_ns.  When the
// producer skipped a stage, that wait runs out, sets ERR_TIMEOUT in the error
// word and returns false, and the block unwinds the way the real kernels do:
// every thread reaches the final barrier and the tensor memory is freed.
// seen[0] = the number of stages the consumer saw complete.
__global__ void __launch_bounds__(64) wait_selftest_kernel(int n_stages, int n_arrive, uint64_t limit_ns,
                                                           int *err, int *seen)
{
    __shared__ uint64_t full[8];
    __shared__ uint32_t slot;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 8; ++s) mbar_init(&full[s], 1);
        fence_mbarrier_init();
    }
    if (warp == 1) tmem_alloc(&slot, 32);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = slot;
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < n_arrive && s < n_stages; ++s) mbar_arrive(&full[s]);
    } else if (warp == 1 && lane == 0) {
        int k = 0;
        for (; k < n_stages; ++k)
            if (!mbar_wait(&full[k], 0, err, limit_ns)) break;
        seen[0] = k;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
}

cudaError_t launch_wait_selftest(int n_stages, int n_arrive, uint64_t limit_ns, int *err, int *seen,
                                 cudaStream_t st)
{
    wait_selftest_kernel<<<1, 64, 0, st>>>(n_stages, n_arrive, limit_ns, err, seen);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Merging the per-tile partials of each token.  A block covers 32 tokens
// (threadIdx.x, so every load of one tile's partials is a 128-byte line) and
// splits the tiles into MG contiguous groups (threadIdx.y).  Pass 1 takes the
// maximum; pass 2 sums z_c * 2^(m_c - M) per group in double (the exp2 is
// the fp32 ex2.approx, relative error about 2^-22 per term); the MG group
// sums are then added in group order.  The tile-to-thread map depends only
// on n_ct, so the result is the same bits for every run.
constexpr int MG = 8;

__device__ __forceinline__ void tile_range(int64_t n_ct, int g, int64_t &c0, int64_t &c1)
{
    c0 = n_ct * g / MG;
    c1 = n_ct * (g + 1) / MG;
}

// PRECISE (the fp32 inputs path, tolerance 1e-6 relative): the rescale
// factors are exp2 in double instead of ex2.approx.
template <bool PRECISE>
__global__ void __launch_bounds__(32 * MG) merge_ce_kernel(
    const float *__restrict__ part, const float *__restrict__ tgt, const uint8_t *__restrict__ mask,
    int64_t n, int64_t n_ct, int64_t n_pad, double wz, float *__restrict__ lse_out,
    float *__restrict__ ce_out, double *__restrict__ tokacc)
{
    __shared__ float smax[MG][32];
    __shared__ double ssum[MG][32];
    const int tx = threadIdx.x, g = threadIdx.y;
    const int64_t t = blockIdx.x * 32 + tx;
    const bool live = t < n;
    const float *m2 = part;
    const float *zz = part + n_ct * n_pad;
    int64_t c0, c1;
    tile_range(n_ct, g, c0, c1);
    float M = -INFINITY;
    if (live)
        for (int64_t c = c0; c < c1; ++c) M = fmaxf(M, m2[c * n_pad + t]);
    smax[g][tx] = M;
    __syncthreads();
    M = smax[0][tx];
    for (int k = 1; k < MG; ++k) M = fmaxf(M, smax[k][tx]);
    double Z = 0.0;
    if (live)
        for (int64_t c = c0; c < c1; ++c)
            Z += PRECISE ? static_cast<double>(zz[c * n_pad + t]) *
                               exp2(static_cast<double>(m2[c * n_pad + t]) - static_cast<double>(M))
                         : static_cast<double>(zz[c * n_pad + t] * ex2_approx(m2[c * n_pad + t] - M));
    ssum[g][tx] = Z;
    __syncthreads();
    if (g != 0 || !live) return;
    Z = ssum[0][tx];
    for (int k = 1; k < MG; ++k) Z += ssum[k][tx];
    const double lse = (static_cast<double>(M) + log2(Z)) * LN2;
    const bool on = mask ? (mask[t] != 0) : true;
    const double ce = on ? lse - static_cast<double>(tgt[t]) : 0.0;
    const double z2 = on ? lse * lse : 0.0;
    lse_out[t] = static_cast<float>(lse);
    if (ce_out) ce_out[t] = static_cast<float>(ce);
    tokacc[t] = ce + wz * z2;
    tokacc[n_pad + t] = ce;
    tokacc[2 * n_pad + t] = z2;
}

cudaError_t launch_merge_ce(const float *part, const float *tgt, const int64_t *targets,
                            const uint8_t *mask, int64_t n, int64_t n_ct, int64_t n_pad,
                            double wz, float *lse_out, float *ce_out, double *tokacc,
                            cudaStream_t st, bool precise)
{
    (void)targets;
    if (precise)
        merge_ce_kernel<true><<<static_cast<unsigned>((n + 31) / 32), dim3(32, MG), 0, st>>>(
            part, tgt, mask, n, n_ct, n_pad, wz, lse_out, ce_out, tokacc);
    else
        merge_ce_kernel<false><<<static_cast<unsigned>((n + 31) / 32), dim3(32, MG), 0, st>>>(
            part, tgt, mask, n, n_ct, n_pad, wz, lse_out, ce_out, tokacc);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// The teacher's own statistics (teacher_stats, one block per token row, an
// HBM stream): in log2 units of b = teacher * log2(e) / T,
//   lse_t2 = log2 sum_v 2^b   and   Eb = sum_v p_v b_v,  p = 2^(b - lse_t2),
// so that sum p log p = ln2 (Eb - lse_t2).  Each thread keeps an online
// (max, sum, weighted sum) over 16-byte groups of its row; the threads are then
// merged by a fixed tree.  The sums are fp32 per thread for bf16 teachers and
// fp64 for fp32 teachers (whose tolerance is 1e-6).
// T: float, uint16_t (bf16 bits) or h16_t (fp16 bits).
template <typename T> constexpr bool kIsF16 = false;
template <> constexpr bool kIsF16<h16_t> = true;

template <typename T> struct TeachAcc { using type = float; };
template <> struct TeachAcc<float> { using type = double; };

template <typename T>
__device__ __forceinline__ float teach_exp2(float x)
{
    if constexpr (sizeof(T) == 2) return ex2_approx(x);
    else return exp2f(x);
}

// The largest of a 16-byte vector's values (as fmaxf: a NaN loses to a
// number), the 16-bit ones compared two at a time in their own format
// (exact: the maximum is one of the values).
template <typename T> __device__ __forceinline__ float raw_max(const uint4 &v)
{
    if constexpr (sizeof(T) == 4) {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    } else {
        uint32_t a, b, m;
        if constexpr (kIsF16<T>) {
            asm("max.f16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
            asm("max.f16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z), "r"(v.w));
            asm("max.f16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
        } else {
            asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
            asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z), "r"(v.w));
            asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
        }
        return fmaxf(h16_lo<kIsF16<T>>(m), h16_hi<kIsF16<T>>(m));
    }
}

// One warp's scan of a teacher row into (M, Z, E), merged over the lanes:
// b = x kT for raw logits x, M the running maximum of b, Z = sum 2^(b - M) and
// E = sum 2^(b - M) x (scaled by kT at the end), so each element costs one FFMA
// into the exponent, one exp2, one add and one FFMA.
// GUARD: a -inf logit (a vocabulary entry masked out of the row) has
// probability 0 and adds nothing (0 log 0 = 0).  Without GUARD such a logit
// leaves a NaN in Z or E (0 * -inf, or -inf - -inf while every entry so far
// was -inf), so a row is scanned without it first and again with it only if
// its sums come out non-finite.
template <typename T, bool GUARD, typename A>
__device__ __forceinline__ void teacher_scan(const T *__restrict__ row, int64_t V, int lane, float kT, float &M,
                                             A &Z, A &E)
{
    constexpr int VEC = 16 / sizeof(T);
    constexpr int UNR = 8;
    M = -INFINITY;
    Z = 0;
    E = 0;
    // cm: the largest of the nv raw values x
    auto absorb = [&](const float (&x)[VEC], int nv, float cm) {
        cm *= kT;                                   // kT > 0: the maximum commutes with the scale
        if (cm > M) {
            const A f = static_cast<A>(teach_exp2<T>(M - cm));
            Z *= f;
            E *= f;
            M = cm;
        }
#pragma unroll
        for (int i = 0; i < VEC; ++i)
            if (i < nv && (!GUARD || x[i] != -INFINITY)) {
                const A e = static_cast<A>(teach_exp2<T>(fmaf(x[i], kT, -M)));
                Z += e;
                E += e * static_cast<A>(x[i]);
            }
    };
    if constexpr (sizeof(T) == 2) {
        // 16-bit: V % 8 == 0, so every row starts 16-byte aligned
        const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
        const int64_t nvec = V / VEC;
        for (int64_t v0 = lane; v0 < nvec; v0 += UNR * 32) {
            uint4 w[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int64_t v = v0 + u * 32;
                w[u] = v < nvec ? __ldg(r4 + v) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                if (v0 + u * 32 >= nvec) break;
                const uint32_t q[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
                float x[VEC];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[2 * i] = h16_lo<kIsF16<T>>(q[i]);
                    x[2 * i + 1] = h16_hi<kIsF16<T>>(q[i]);
                }
                absorb(x, VEC, raw_max<T>(w[u]));
            }
        }
    } else {
        for (int64_t v0 = lane * VEC; v0 < V; v0 += 32 * VEC) {
            float x[VEC];
            const int nv = V - v0 < VEC ? static_cast<int>(V - v0) : VEC;
#pragma unroll
            for (int i = 0; i < VEC; ++i) x[i] = i < nv ? static_cast<float>(row[v0 + i]) : 0.f;
            float cm = -INFINITY;
#pragma unroll
            for (int i = 0; i < VEC; ++i)
                if (i < nv) cm = fmaxf(cm, x[i]);
            absorb(x, nv, cm);
        }
    }
    E *= static_cast<A>(kT);
    // fixed xor tree over the lanes, in the accumulation type (fp64 is slow on
    // this part, so bf16 rows merge in fp32); every lane ends with the row
    for (int o = 16; o > 0; o >>= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
        const A zo = __shfl_xor_sync(0xffffffffu, Z, o), eo = __shfl_xor_sync(0xffffffffu, E, o);
        const float Mn = fmaxf(M, Mo);
        const A f1 = M == -INFINITY ? A(0) : static_cast<A>(teach_exp2<T>(M - Mn));
        const A f2 = Mo == -INFINITY ? A(0) : static_cast<A>(teach_exp2<T>(Mo - Mn));
        Z = Z * f1 + zo * f2;
        E = E * f1 + eo * f2;
        M = Mn;
    }
}

// One warp per token row, all rows at once (no block-level merge and no
// partial last wave of blocks): 8 x 16 bytes in flight per lane.
template <typename T>
__global__ void __launch_bounds__(256) teacher_stats_kernel(const T *__restrict__ teach, int64_t n, int64_t V,
                                                           float kT, double2 *__restrict__ out)
{
    using A = typename TeachAcc<T>::type;
    const int64_t t = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= n) return;
    const T *row = teach + t * V;
    float M;
    A Z, E;
    teacher_scan<T, false>(row, V, lane, kT, M, Z, E);
    if (!(isfinite(static_cast<float>(Z)) && isfinite(static_cast<float>(E))))
        teacher_scan<T, true>(row, V, lane, kT, M, Z, E);
    if (lane == 0) {
        const double Zd = static_cast<double>(Z);
        out[t] = make_double2(static_cast<double>(M) + log2(Zd), static_cast<double>(E) / Zd);
    }
}

cudaError_t launch_teacher_stats(int dtype, const void *teach, int64_t n, int64_t V, double temperature,
                                 double2 *out, cudaStream_t st)
{
    const float kT = static_cast<float>(LOG2E / temperature);
    const unsigned grid = static_cast<unsigned>((n + 7) / 8);
    if (dtype == 1)
        teacher_stats_kernel<uint16_t><<<grid, 256, 0, st>>>(static_cast<const uint16_t *>(teach), n, V, kT, out);
    else if (dtype == 2)
        teacher_stats_kernel<h16_t><<<grid, 256, 0, st>>>(static_cast<const h16_t *>(teach), n, V, kT, out);
    else
        teacher_stats_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float *>(teach), n, V, kT, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Distillation merge.  Per (token, vocabulary tile) the forward wrote the
// student's (m_c, z_c) in log2 units of a = s log2(e) / T and one cross term
// x_c: CE and forward KL sum p a (the teacher's p exact); reverse KL sums
// 2^(a - m_c) (a - b).  With lse_s2 = M + log2 sum z_c 2^(m_c - M) and the
// teacher's (lse_t2, Eb), in natural units:
//   CE   L = ln2 (lse_s2 - sum_c x_c)
//   fKL  L = ln2 (Eb - lse_t2 - sum_c x_c + lse_s2)
//   rKL  L = ln2 (sum_c x_c 2^(m_c - M) / Z_s - lse_s2 + lse_t2)
// (the three definitions of "Fuse distillation + z-loss ...", "What it does",
// with q = softmax(a), p = softmax(b)).  Tiles are combined in tile order, as
// in merge_ce.
__global__ void __launch_bounds__(32 * MG) merge_distill_kernel(
    const float *__restrict__ part, const double2 *__restrict__ tstat, const uint8_t *__restrict__ mask,
    int64_t n, int64_t n_ct, int64_t n_pad, int direction, double wz, float *__restrict__ lse_out,
    float *__restrict__ per_token, double *__restrict__ tokacc, float4 *__restrict__ tokp,
    double alpha, double temperature)
{
    __shared__ float smax[MG][32];
    __shared__ double ssum[2][MG][32];
    const int tx = threadIdx.x, g = threadIdx.y;
    const int64_t t = blockIdx.x * 32 + tx;
    const bool live = t < n;         // the grid covers exactly n_pad tokens
    const int64_t pl = n_ct * n_pad;
    const float *ms = part, *zs = part + pl, *xx = part + 2 * pl;
    int64_t c0, c1;
    tile_range(n_ct, g, c0, c1);
    float Ms = -INFINITY;
    if (live)
        for (int64_t c = c0; c < c1; ++c) Ms = fmaxf(Ms, ms[c * n_pad + t]);
    smax[g][tx] = Ms;
    __syncthreads();
    Ms = smax[0][tx];
    for (int k = 1; k < MG; ++k) Ms = fmaxf(Ms, smax[k][tx]);
    double Zs = 0.0, X = 0.0;
    if (live)
        for (int64_t c = c0; c < c1; ++c) {
            const int64_t o = c * n_pad + t;
            const float fs = ex2_approx(ms[o] - Ms);
            Zs += static_cast<double>(zs[o] * fs);
            X += static_cast<double>(direction == DIR_RKL ? xx[o] * fs : xx[o]);
        }
    ssum[0][g][tx] = Zs;
    ssum[1][g][tx] = X;
    __syncthreads();
    if (g != 0) return;
    if (!live) {
        tokp[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    Zs = ssum[0][0][tx];
    X = ssum[1][0][tx];
    for (int k = 1; k < MG; ++k) {
        Zs += ssum[0][k][tx];
        X += ssum[1][k][tx];
    }
    const double lse_s2 = static_cast<double>(Ms) + log2(Zs);
    const double2 ts = tstat[t];
    const double lse_t2 = ts.x;
    double L2;
    if (direction == DIR_CE) L2 = lse_s2 - X;
    else if (direction == DIR_FKL) L2 = ts.y - lse_t2 - X + lse_s2;
    else L2 = X / Zs - lse_s2 + lse_t2;
    const double L = L2 * LN2, lse_s = lse_s2 * LN2, lse_t = lse_t2 * LN2;
    const bool on = mask ? (mask[t] != 0) : true;
    const double Lm = on ? L : 0.0;
    const double z2 = on ? lse_s * lse_s : 0.0;
    if (lse_out) lse_out[t] = static_cast<float>(lse_s);
    if (per_token) per_token[t] = static_cast<float>(Lm);
    tokacc[t] = Lm + wz * z2;
    tokacc[n_pad + t] = Lm;
    tokacc[2 * n_pad + t] = z2;
    const double at = on ? alpha / temperature : 0.0;
    float4 P;
    P.x = static_cast<float>(lse_s2);
    P.y = static_cast<float>(lse_t2);
    if (direction == DIR_RKL) {
        P.z = static_cast<float>(at);
        P.w = static_cast<float>(lse_t - lse_s - L + 2.0 * wz * lse_s);
    } else {
        P.z = static_cast<float>(at * (1.0 + 2.0 * wz * lse_s));
        P.w = static_cast<float>(at);
    }
    tokp[t] = P;
}

cudaError_t launch_merge_distill(const float *part, const double2 *tstat, const uint8_t *mask, int64_t n,
                                 int64_t n_ct, int64_t n_pad, int direction, double wz, float *lse_out,
                                 float *per_token, double *tokacc, float4 *tokp, double alpha,
                                 double temperature, cudaStream_t st)
{
    merge_distill_kernel<<<static_cast<unsigned>((n_pad + 31) / 32), dim3(32, MG), 0, st>>>(
        part, tstat, mask, n, n_ct, n_pad, direction, wz, lse_out, per_token, tokacc, tokp, alpha,
        temperature);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Fixed-shape tree: thread i sums tokens i, i+1024, i+2048, ... in that
// order, then the 1024 partials are added pairwise (i += i + stride, stride
// halving).  The shape depends on n only, so the result is the same bits for
// every chunk, grid and run.
__global__ void __launch_bounds__(1024) reduce_kernel(const double *__restrict__ tokacc, int64_t n,
                                                      int64_t n_pad, const WsHeader *hdr,
                                                      double *__restrict__ out, int sum)
{
    __shared__ double sh[3][1024];
    // a refused call (a target out of range, found by the validation queued
    // before) leaves its outputs untouched
    if (*reinterpret_cast<const volatile int *>(&hdr->bad_targets)) return;
    const int i = threadIdx.x;
    for (int s = 0; s < 3; ++s) {
        double acc = 0.0;
        for (int64_t t = i; t < n; t += 1024) acc += tokacc[s * n_pad + t];
        sh[s][i] = acc;
    }
    __syncthreads();
    for (int stride = 512; stride > 0; stride >>= 1) {
        if (i < stride)
            for (int s = 0; s < 3; ++s) sh[s][i] += sh[s][i + stride];
        __syncthreads();
    }
    if (i == 0) {
        const int nv = hdr->n_valid;
        for (int s = 0; s < 3; ++s) out[s] = sum ? sh[s][0] : (nv > 0 ? sh[s][0] / nv : 0.0);
    }
}

cudaError_t launch_reduce(const double *tokacc, int64_t n, int64_t n_pad, const WsHeader *hdr,
                          double wz, double *scalars_out, cudaStream_t st, bool sum)
{
    (void)wz;
    reduce_kernel<<<1, 1024, 0, st>>>(tokacc, n, n_pad, hdr, scalars_out, sum ? 1 : 0);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// P.w holds the target's column in the weight rows the passes see: y - v0
// when that lies in [0, n_rows) (a vocabulary shard starting at row v0), else
// -1, which matches no column (the one-hot term then belongs to another shard).
__global__ void tokp_ce_kernel(const float *__restrict__ lse, const int64_t *__restrict__ targets,
                               const uint8_t *__restrict__ mask, int64_t n, int64_t n_pad,
                               double alpha, double wz, int64_t v0, int64_t n_rows, float4 *__restrict__ tokp)
{
    const int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (t >= n_pad) return;
    if (t >= n) {
        tokp[t] = make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
        return;
    }
    const double l = lse[t];
    const double at = (mask ? (mask[t] != 0) : true) ? alpha : 0.0;
    const int64_t col = targets[t] - v0;
    tokp[t] = make_float4(static_cast<float>(l * LOG2E), static_cast<float>(at * (1.0 + 2.0 * wz * l)),
                          static_cast<float>(at),
                          __int_as_float(col >= 0 && col < n_rows ? static_cast<int>(col) : -1));
}

cudaError_t launch_tokp_ce(const float *lse, const int64_t *targets, const uint8_t *mask,
                           int64_t n, int64_t n_pad, double alpha, double wz, float4 *tokp,
                           cudaStream_t st, int64_t v0, int64_t n_rows)
{
    tokp_ce_kernel<<<static_cast<int>((n_pad + 127) / 128), 128, 0, st>>>(lse, targets, mask, n, n_pad, alpha,
                                                                          wz, v0, n_rows, tokp);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Element i of the nsplit partial planes (count4 float4 apart), added in split
// order.  The planes are read once, so the loads stream past L2, eight (then
// four, then one) at a time so that each thread keeps several in flight.
__device__ __forceinline__ float4 split_sum(const float4 *__restrict__ part, int64_t nsplit, int64_t count4,
                                            int64_t i)
{
    auto add = [](float4 &a, const float4 &v) {
        a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
    };
    float4 acc = __ldcs(part + i);
    int64_t s = 1;
    for (; s + 8 <= nsplit; s += 8) {
        float4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = __ldcs(part + (s + q) * count4 + i);
#pragma unroll
        for (int q = 0; q < 8; ++q) add(acc, v[q]);
    }
    if (s + 4 <= nsplit) {
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = __ldcs(part + (s + q) * count4 + i);
#pragma unroll
        for (int q = 0; q < 4; ++q) add(acc, v[q]);
        s += 4;
    }
    for (; s < nsplit; ++s) add(acc, __ldcs(part + s * count4 + i));
    return acc;
}

__global__ void sum_splits_kernel(const float4 *__restrict__ part, int64_t nsplit, int64_t count4,
                                  float4 *__restrict__ out, int accumulate)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 acc = split_sum(part, nsplit, count4, i);
        if (accumulate) {
            const float4 o = out[i];
            acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
        }
        out[i] = acc;
    }
}

cudaError_t launch_sum_splits(const float *part, int64_t nsplit, int64_t count, float *out,
                              cudaStream_t st, bool accumulate)
{
    const int64_t c4 = count / 4;  // count is a multiple of 4 (d_model % 8 == 0)
    int64_t grid = (c4 + 255) / 256;
    if (grid > 4096) grid = 4096;
    sum_splits_kernel<<<static_cast<int>(grid), 256, 0, st>>>(
        reinterpret_cast<const float4 *>(part), nsplit, c4, reinterpret_cast<float4 *>(out), accumulate ? 1 : 0);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// The fused forward + d_hidden path.  See k_bwp.cu (BWD_FUSED) for the pass
// itself: it exponentiates every logit against r_t = s[t][y_t] log2e + 64 and
// reports, per (split, CTA, token), the sum of those terms.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One warp per token: 16-byte loads of the hidden row and the target's weight
// row, fp32 products summed per lane in k order, then a fixed xor tree.
template <bool F16>
__global__ void __launch_bounds__(256) tgt_logit_kernel(const uint16_t *__restrict__ H,
                                                        const uint16_t *__restrict__ W,
                                                        const int64_t *__restrict__ targets, int64_t n,
                                                        int64_t d, int64_t n_pad, float *__restrict__ tgt,
                                                        float4 *__restrict__ tokp)
{
    const int64_t t = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= n_pad) return;
    if (t >= n) {
        if (lane == 0) {
            tgt[t] = 0.f;
            tokp[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const uint4 *h = reinterpret_cast<const uint4 *>(H + t * d);
    const uint4 *w = reinterpret_cast<const uint4 *>(W + targets[t] * d);
    float acc = 0.f;
    for (int64_t k = lane; k < d / 8; k += 32) {
        const uint4 a = h[k], b = w[k];
        acc = fmaf(h16_lo<F16>(a.x), h16_lo<F16>(b.x), acc);
        acc = fmaf(h16_hi<F16>(a.x), h16_hi<F16>(b.x), acc);
        acc = fmaf(h16_lo<F16>(a.y), h16_lo<F16>(b.y), acc);
        acc = fmaf(h16_hi<F16>(a.y), h16_hi<F16>(b.y), acc);
        acc = fmaf(h16_lo<F16>(a.z), h16_lo<F16>(b.z), acc);
        acc = fmaf(h16_hi<F16>(a.z), h16_hi<F16>(b.z), acc);
        acc = fmaf(h16_lo<F16>(a.w), h16_lo<F16>(b.w), acc);
        acc = fmaf(h16_hi<F16>(a.w), h16_hi<F16>(b.w), acc);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
        tgt[t] = acc;
        tokp[t] = make_float4(fmaf(acc, static_cast<float>(LOG2E), FUSED_SHIFT), 0.f, 0.f, 0.f);
    }
}

// The training step's first kernel: validation (target range, counted
// tokens) and the target logit with its reference shift in one pass, one
// warp per token.  An out-of-range target is counted and its weight row never
// read (the call then refuses with 586 before anything else runs).
template <bool F16>
__global__ void __launch_bounds__(256) validate_tgt_kernel(const uint16_t *__restrict__ H,
                                                           const uint16_t *__restrict__ W,
                                                           const int64_t *__restrict__ targets,
                                                           const uint8_t *__restrict__ mask, int64_t n,
                                                           int64_t d, int64_t V, int64_t n_pad,
                                                           WsHeader *hdr, float *__restrict__ tgt,
                                                           float4 *__restrict__ tokp)
{
    __shared__ int sbad, svalid;
    if (threadIdx.x == 0) { sbad = 0; svalid = 0; }
    __syncthreads();
    const int64_t t = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t < n_pad) {
        float acc = 0.f;
        bool in = false;
        if (t < n) {
            const int64_t y = targets[t];
            in = y >= 0 && y < V;
            if (lane == 0) {
                if (!in) atomicAdd(&sbad, 1);
                if (mask ? (mask[t] != 0) : true) atomicAdd(&svalid, 1);
            }
            if (in) {
                const uint4 *h = reinterpret_cast<const uint4 *>(H + t * d);
                const uint4 *w = reinterpret_cast<const uint4 *>(W + y * d);
                // d_model 1024: four 16-byte pairs per lane, all loads in flight at once
#pragma unroll 4
                for (int64_t k = lane; k < d / 8; k += 32) {
                    const uint4 a = h[k], b = w[k];
                    acc = fmaf(h16_lo<F16>(a.x), h16_lo<F16>(b.x), acc);
                    acc = fmaf(h16_hi<F16>(a.x), h16_hi<F16>(b.x), acc);
                    acc = fmaf(h16_lo<F16>(a.y), h16_lo<F16>(b.y), acc);
                    acc = fmaf(h16_hi<F16>(a.y), h16_hi<F16>(b.y), acc);
                    acc = fmaf(h16_lo<F16>(a.z), h16_lo<F16>(b.z), acc);
                    acc = fmaf(h16_hi<F16>(a.z), h16_hi<F16>(b.z), acc);
                    acc = fmaf(h16_lo<F16>(a.w), h16_lo<F16>(b.w), acc);
                    acc = fmaf(h16_hi<F16>(a.w), h16_hi<F16>(b.w), acc);
                }
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            }
        }
        if (lane == 0) {
            tgt[t] = in ? acc : 0.f;
            tokp[t] = make_float4(in ? fmaf(acc, static_cast<float>(LOG2E), FUSED_SHIFT) : 0.f, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (sbad) atomicAdd(&hdr->bad_targets, sbad);
        if (svalid) atomicAdd(&hdr->n_valid, svalid);
    }
}

cudaError_t launch_validate_tgt(const uint16_t *H, const uint16_t *W, const int64_t *targets,
                                const uint8_t *mask, int64_t n, int64_t d, int64_t V, int64_t n_pad,
                                WsHeader *hdr, float *tgt, float4 *tokp, cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(&hdr->bad_targets, 0, 3 * sizeof(int), st);   // bad, n_valid, redo
    if (e != cudaSuccess) return e;
    validate_tgt_kernel<false><<<static_cast<unsigned>((n_pad + 7) / 8), 256, 0, st>>>(H, W, targets, mask, n, d,
                                                                                     V, n_pad, hdr, tgt, tokp);
    return cudaGetLastError();
}

cudaError_t launch_tgt_logit(bool f16, const uint16_t *H, const uint16_t *W, const int64_t *targets, int64_t n,
                             int64_t d, int64_t n_pad, float *tgt, float4 *tokp, cudaStream_t st)
{
    const unsigned grid = static_cast<unsigned>((n_pad + 7) / 8);
    if (f16) tgt_logit_kernel<true><<<grid, 256, 0, st>>>(H, W, targets, n, d, n_pad, tgt, tokp);
    else tgt_logit_kernel<false><<<grid, 256, 0, st>>>(H, W, targets, n, d, n_pad, tgt, tokp);
    return cudaGetLastError();
}

// One thread per token.  Z = sum of the nz partials in index order (fp32);
// with r_t the shift, lse_t = (r_t + log2 Z) ln 2.  The row is flagged for the
// exact recomputation when Z is outside [2^-80, 2^90] (or not a number): the
// shifted terms are only trusted while the largest stays far from the fp32
// and bf16 limits.  The flag is raised for masked rows too, since their lse is
// an output.
// The counted-token total comes from the validation's header (the call does
// not wait for it on the host): alpha = grad_scale / N_valid, or grad_scale
// for the sum.  A refused call returns at once.
__global__ void __launch_bounds__(32) merge_fused_kernel(const float *__restrict__ zpart, int64_t nz,
                                                         const float *__restrict__ tgt,
                                                         const int64_t *__restrict__ targets,
                                                         const uint8_t *__restrict__ mask, int64_t n,
                                                         int64_t n_pad, double gs, int sum, double wz,
                                                         float *__restrict__ lse_out, float *__restrict__ ce_out,
                                                         double *__restrict__ tokacc, float4 *__restrict__ tokp,
                                                         float2 *__restrict__ dhc, WsHeader *hdr)
{
    if (*reinterpret_cast<const volatile int *>(&hdr->bad_targets)) return;
    const int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (t >= n_pad) return;
    if (t >= n) {
        tokp[t] = make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
        dhc[t] = make_float2(0.f, 0.f);
        return;
    }
    const int nv = hdr->n_valid;
    const float alpha = static_cast<float>(sum ? gs : (nv > 0 ? gs / nv : 0.0));
    // The partials in index order, loaded sixteen at a time so the loads
    // overlap.  fp32 throughout: this path takes bf16 inputs only (tolerance
    // 2e-3), and fp64 arithmetic is slow enough on this part to make the merge
    // a visible share of the step.
    float Z = 0.f;
    int64_t j = 0;
    for (; j + 16 <= nz; j += 16) {
        float v[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] = zpart[(j + q) * n_pad + t];
#pragma unroll
        for (int q = 0; q < 16; ++q) Z += v[q];
    }
    for (; j < nz; ++j) Z += zpart[j * n_pad + t];
    if (!(Z >= 0x1p-80f && Z <= 0x1p90f)) hdr->redo = 1;
    const float lse = (tokp[t].x + log2f(Z)) * static_cast<float>(LN2);
    const bool on = mask ? (mask[t] != 0) : true;
    const float ce = on ? lse - tgt[t] : 0.f;
    const float z2 = on ? lse * lse : 0.f;
    lse_out[t] = lse;
    if (ce_out) ce_out[t] = ce;
    tokacc[t] = static_cast<double>(ce) + wz * static_cast<double>(z2);
    tokacc[n_pad + t] = static_cast<double>(ce);
    tokacc[2 * n_pad + t] = static_cast<double>(z2);
    const float at = on ? alpha : 0.f;
    const float cz = at * (1.f + 2.f * static_cast<float>(wz) * lse);
    tokp[t] = make_float4(lse * static_cast<float>(LOG2E), cz, at, __int_as_float(static_cast<int>(targets[t])));
    dhc[t] = make_float2(cz / Z, at);
}

cudaError_t launch_merge_fused(const float *zpart, int64_t nz, const float *tgt, const int64_t *targets,
                               const uint8_t *mask, int64_t n, int64_t n_pad, double gs, bool sum, double wz,
                               float *lse_out, float *ce_out, double *tokacc, float4 *tokp,
                               float2 *dhc, WsHeader *hdr, cudaStream_t st)
{
    merge_fused_kernel<<<static_cast<unsigned>((n_pad + 31) / 32), 32, 0, st>>>(
        zpart, nz, tgt, targets, mask, n, n_pad, gs, sum ? 1 : 0, wz, lse_out, ce_out, tokacc, tokp, dhc, hdr);
    return cudaGetLastError();
}

// d_hidden[t][k] = coef_t * sum_s part[s][t][k] - a_t W[y_t][k], the splits
// added in split order.  `part` may be `out` itself (one split): every
// element is read before the same thread writes it.  A non-finite result
// flags the call for the exact recomputation (it would also come out of
// non-finite inputs, where the recomputation gives the same values).
__global__ void combine_dh_kernel(const float4 *part, int64_t nsplit, int64_t n, int64_t d4,
                                  const uint16_t *__restrict__ W, const int64_t *__restrict__ targets,
                                  const float2 *__restrict__ dhc, float4 *out, WsHeader *hdr)
{
    if (*reinterpret_cast<const volatile int *>(&hdr->bad_targets)) return;   // a refused call
    const int64_t count4 = n * d4;
    bool bad = false;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / d4, k4 = i - t * d4;
        const float4 acc = split_sum(part, nsplit, count4, i);
        const float2 c = dhc[t];
        const uint2 wv = *reinterpret_cast<const uint2 *>(W + targets[t] * (d4 * 4) + k4 * 4);
        float4 o;
        o.x = fmaf(c.x, acc.x, -c.y * bf_lo(wv.x));
        o.y = fmaf(c.x, acc.y, -c.y * bf_hi(wv.x));
        o.z = fmaf(c.x, acc.z, -c.y * bf_lo(wv.y));
        o.w = fmaf(c.x, acc.w, -c.y * bf_hi(wv.y));
        bad |= !(isfinite(o.x) && isfinite(o.y) && isfinite(o.z) && isfinite(o.w));
        out[i] = o;
    }
    if (bad) hdr->redo = 1;
}

cudaError_t launch_combine_dh(const float *part, int64_t nsplit, int64_t n, int64_t d,
                              const uint16_t *W, const int64_t *targets, const float2 *dhc,
                              float *out, WsHeader *hdr, cudaStream_t st)
{
    const int64_t c4 = n * (d / 4);   // d_model % 8 == 0 on this path
    int64_t grid = (c4 + 255) / 256;
    if (grid > 4096) grid = 4096;
    combine_dh_kernel<<<static_cast<int>(grid), 256, 0, st>>>(
        reinterpret_cast<const float4 *>(part), nsplit, n, d / 4, W, targets, dhc,
        reinterpret_cast<float4 *>(out), hdr);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Cross-entropy from materialised logits.  One block per row: pass 1 streams
// the row with 16-byte loads and keeps an online (max, sum) per thread, merged
// by a fixed tree; pass 2 (optional) writes grad_logits.
template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<uint16_t> { static constexpr int N = 8; };
template <> struct Vec<h16_t> { static constexpr int N = 8; };

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }
__device__ __forceinline__ float to_f(h16_t x) { return f16_to_f(x.bits); }
// One gradient value rounded to the element type.
__device__ __forceinline__ void from_f(float v, float &o) { o = v; }
__device__ __forceinline__ void from_f(float v, uint16_t &o) { o = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu); }
__device__ __forceinline__ void from_f(float v, h16_t &o) { o.bits = static_cast<uint16_t>(pack_f16x2(v, 0.f) & 0xFFFFu); }

// ---------------------------------------------------------------------------
// Vocabulary-parallel cross-entropy ("Fuse distillation + z-loss ...",
// "Changes": the tensor-parallel subtest).  A shard holds weight rows
// [v0, v0 + n_rows) of the vocabulary.  shard_tgt: per token (one warp), the
// target logit when the shard holds the target, else 0, and that 1/0 flag,
// written into the shard's partials (rows 1 and 2 of [3][n]; row 0 is its
// log-sum-exp, from the statistics pass and merge_ce).  The dot product runs
// in fp32, lanes strided over k, then a fixed xor tree.
template <typename T>
__global__ void __launch_bounds__(256) shard_tgt_kernel(const T *__restrict__ H, const T *__restrict__ Ws,
                                                        const int64_t *__restrict__ targets, int64_t n, int64_t d,
                                                        int64_t v0, int64_t n_rows, float *__restrict__ tgt,
                                                        float *__restrict__ flag)
{
    const int64_t t = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= n) return;
    const int64_t col = targets[t] - v0;
    const bool in = col >= 0 && col < n_rows;
    float acc = 0.f, err = 0.f;
    if (in) {
        // compensated (Dot2, as in the fp32 statistics pass): the rounding
        // residuals of every product and sum are added on the side
        const T *h = H + t * d, *w = Ws + col * d;
        for (int64_t k = lane; k < d; k += 32) {
            const float a = to_f(h[k]), b = to_f(w[k]);
            const float p = __fmul_rn(a, b), pe = __fmaf_rn(a, b, -p);
            const float u = __fadd_rn(acc, p), z = __fsub_rn(u, acc);
            err = __fadd_rn(err, __fadd_rn(pe, __fadd_rn(__fsub_rn(acc, __fsub_rn(u, z)), __fsub_rn(p, z))));
            acc = u;
        }
        for (int o = 16; o > 0; o >>= 1) {
            const float q = __shfl_xor_sync(0xffffffffu, acc, o), qe = __shfl_xor_sync(0xffffffffu, err, o);
            const float u = __fadd_rn(acc, q), z = __fsub_rn(u, acc);
            err = __fadd_rn(__fadd_rn(err, qe), __fadd_rn(__fsub_rn(acc, __fsub_rn(u, z)), __fsub_rn(q, z)));
            acc = u;
        }
        acc = __fadd_rn(acc, err);
    }
    if (lane == 0) {
        tgt[t] = in ? acc : 0.f;
        flag[t] = in ? 1.f : 0.f;
    }
}

cudaError_t launch_shard_tgt(int dtype, const void *H, const void *Ws, const int64_t *targets, int64_t n,
                             int64_t d, int64_t v0, int64_t n_rows, float *tgt, float *flag, cudaStream_t st)
{
    const unsigned grid = static_cast<unsigned>((n + 7) / 8);
    if (dtype == 2)
        shard_tgt_kernel<h16_t><<<grid, 256, 0, st>>>(static_cast<const h16_t *>(H), static_cast<const h16_t *>(Ws),
                                                      targets, n, d, v0, n_rows, tgt, flag);
    else if (dtype == 1)
        shard_tgt_kernel<uint16_t><<<grid, 256, 0, st>>>(static_cast<const uint16_t *>(H),
                                                         static_cast<const uint16_t *>(Ws), targets, n, d, v0,
                                                         n_rows, tgt, flag);
    else
        shard_tgt_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float *>(H), static_cast<const float *>(Ws),
                                                      targets, n, d, v0, n_rows, tgt, flag);
    return cudaGetLastError();
}

// The gathered partials [P][3][n] of every shard: count the tokens whose
// target is held by no shard or by more than one (flags not summing to 1)
// into bad_targets, and the counted tokens into n_valid, as the validation
// does (the header's counters are cleared first).
__global__ void shard_check_kernel(const float *__restrict__ parts, int64_t P, int64_t n,
                                   const uint8_t *__restrict__ mask, WsHeader *hdr)
{
    int bad = 0, valid = 0;
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < n;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float f = 0.f;
        for (int64_t p = 0; p < P; ++p) f += parts[(p * 3 + 2) * n + t];
        bad += f == 1.f ? 0 : 1;
        valid += mask ? (mask[t] != 0) : 1;
    }
    for (int o = 16; o > 0; o >>= 1) {
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
        valid += __shfl_xor_sync(0xffffffffu, valid, o);
    }
    if ((threadIdx.x & 31) == 0) {
        if (bad) atomicAdd(&hdr->bad_targets, bad);
        if (valid) atomicAdd(&hdr->n_valid, valid);
    }
}

cudaError_t launch_shard_check(const float *parts, int64_t P, int64_t n, const uint8_t *mask, WsHeader *hdr,
                               cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(&hdr->bad_targets, 0, 3 * sizeof(int), st);
    if (e != cudaSuccess) return e;
    int grid = static_cast<int>((n + 255) / 256);
    if (grid > 1024) grid = 1024;
    shard_check_kernel<<<grid, 256, 0, st>>>(parts, P, n, mask, hdr);
    return cudaGetLastError();
}

// One thread per token: lse = M + log sum_p exp(lse_p - M) over the shards in
// shard order (double), the target logit from the shard whose flag is set,
// then ce, z and the token-mean terms as in merge_ce.
__global__ void shard_combine_kernel(const float *__restrict__ parts, int64_t P, int64_t n, int64_t n_pad,
                                     const uint8_t *__restrict__ mask, double wz, float *__restrict__ lse_out,
                                     float *__restrict__ ce_out, double *__restrict__ tokacc)
{
    const int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (t >= n) return;
    double M = parts[t], tgt = 0.0;
    for (int64_t p = 1; p < P; ++p) M = fmax(M, static_cast<double>(parts[p * 3 * n + t]));
    double Z = 0.0;
    for (int64_t p = 0; p < P; ++p) {
        Z += exp(static_cast<double>(parts[p * 3 * n + t]) - M);
        if (parts[(p * 3 + 2) * n + t] != 0.f) tgt = parts[(p * 3 + 1) * n + t];
    }
    const double lse = M + log(Z);
    const bool on = mask ? (mask[t] != 0) : true;
    const double ce = on ? lse - tgt : 0.0;
    const double z2 = on ? lse * lse : 0.0;
    lse_out[t] = static_cast<float>(lse);
    if (ce_out) ce_out[t] = static_cast<float>(ce);
    tokacc[t] = ce + wz * z2;
    tokacc[n_pad + t] = ce;
    tokacc[2 * n_pad + t] = z2;
}

cudaError_t launch_shard_combine(const float *parts, int64_t P, int64_t n, int64_t n_pad, const uint8_t *mask,
                                 double wz, float *lse_out, float *ce_out, double *tokacc, cudaStream_t st)
{
    shard_combine_kernel<<<static_cast<unsigned>((n + 127) / 128), 128, 0, st>>>(parts, P, n, n_pad, mask, wz,
                                                                                lse_out, ce_out, tokacc);
    return cudaGetLastError();
}

// 16-byte loads of a logit row.  `keep` leaves the line in L2 (the row is read
// again for its gradient); otherwise the load streams past L2.
template <typename T>
__device__ __forceinline__ void load_vec(const T *p, float *f, bool keep);
template <>
__device__ __forceinline__ void load_vec<float>(const float *p, float *f, bool keep)
{
    const float4 *q = reinterpret_cast<const float4 *>(p);
    const float4 v = keep ? __ldg(q) : __ldcs(q);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
template <bool F16>
__device__ __forceinline__ void load_vec16(const void *p, float *f, bool keep)
{
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    const uint4 v = keep ? __ldg(q) : __ldcs(q);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = h16_lo<F16>(w[i]);
        f[2 * i + 1] = h16_hi<F16>(w[i]);
    }
}
template <>
__device__ __forceinline__ void load_vec<uint16_t>(const uint16_t *p, float *f, bool keep)
{
    load_vec16<false>(p, f, keep);
}
template <>
__device__ __forceinline__ void load_vec<h16_t>(const h16_t *p, float *f, bool keep)
{
    load_vec16<true>(p, f, keep);
}

// 16-byte streaming store of NV gradient values.
__device__ __forceinline__ void store_vec(float *p, const float *g)
{
    __stcs(reinterpret_cast<float4 *>(p), make_float4(g[0], g[1], g[2], g[3]));
}
__device__ __forceinline__ void store_vec(uint16_t *p, const float *g)
{
    __stcs(reinterpret_cast<uint4 *>(p), make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]),
                                                    pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7])));
}
__device__ __forceinline__ void store_vec(h16_t *p, const float *g)
{
    __stcs(reinterpret_cast<uint4 *>(p), make_uint4(pack_f16x2(g[0], g[1]), pack_f16x2(g[2], g[3]),
                                                    pack_f16x2(g[4], g[5]), pack_f16x2(g[6], g[7])));
}

// One term into a running (max m, sum z) in log2 units.  A -inf term (a
// vocabulary entry masked out of the row) adds nothing; skipping it also
// avoids 2^(-inf - (-inf)) while every term so far has been -inf.
__device__ __forceinline__ void online_add(float &m, float &z, float x2)
{
    if (x2 > m) {
        z = z * ex2_approx(m - x2) + 1.f;
        m = x2;
    } else if (x2 != -INFINITY) {
        z += ex2_approx(x2 - m);
    }
}

__device__ __forceinline__ void online_merge(float &m, float &z, float m_o, float z_o)
{
    const float M = fmaxf(m, m_o);
    if (M == -INFINITY) return;
    z = z * ex2_approx(m - M) + z_o * ex2_approx(m_o - M);
    m = M;
}

// 16 bytes of a row as raw bits (`keep`: leave the line in L2 for a second
// read; otherwise stream it past L2), and their NV values as fp32.
__device__ __forceinline__ uint4 ld16(const void *p, bool keep)
{
    const uint4 *q = static_cast<const uint4 *>(p);
    return keep ? __ldg(q) : __ldcs(q);
}
template <typename T> __device__ __forceinline__ void cvt16(const uint4 &v, float *f)
{
    if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = h16_lo<kIsF16<T>>(w[i]);
            f[2 * i + 1] = h16_hi<kIsF16<T>>(w[i]);
        }
    }
}

// One 16-byte vector of raw values f into a running (max m, sum z) of
// f * scale in log2 units (scale > 0): the vector's maximum lm (raw_max of
// the same vector; scaling commutes with it) first, one rescale if it rose,
// then its exponentials, which do not depend on one another, each argument
// one FFMA.
template <int NV>
__device__ __forceinline__ void online_vec(float &m, float &z, const float (&f)[NV], float scale, float lm)
{
    if (lm == -INFINITY) return;                   // every term is zero
    lm *= scale;
    if (lm > m) {
        z *= ex2_approx(m - lm);
        m = lm;
    }
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int u = 0; u < NV; u += 2) {
        z0 += ex2_approx(fmaf(f[u], scale, -m));
        z1 += ex2_approx(fmaf(f[u + 1], scale, -m));
    }
    z += z0 + z1;
}

// The streaming row kernels run one block per row, each thread with FL_U
// 16-byte loads in flight.  With a gradient, one 1024-thread block per SM:
// enough bytes in flight to cover HBM latency, while the rows in flight (one
// per SM, 46 MB at 152k bf16 logits) stay well inside L2, so the gradient
// pass re-reads its row from L2 (four 512-thread blocks per SM kept 185 MB of
// rows in flight, and the second read went back to HBM).  Without one, two
// 512-thread blocks per SM, so that one block's end-of-row merge overlaps the
// other's stream.
constexpr int FL_THREADS_GRAD = 1024;
constexpr int FL_THREADS_STAT = 512;
constexpr int FL_U = 4;
// Cross-entropy without a gradient streams one array: eight loads in flight
// per thread keep as many bytes in flight per SM as the distillation stream's
// two arrays of four (0.104 against 0.114 ms at 2048 x 151936 bf16).  With a
// gradient it stays at four (eight were no faster).
constexpr int FL_U_CE = 8;
static_assert(FL_THREADS_GRAD / 32 <= 32 && FL_THREADS_STAT / 32 <= 32, "warp 0 merges one partial per warp");

template <typename T, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) from_logits_kernel(const T *__restrict__ logits,
                                                                   const int64_t *__restrict__ targets,
                                                                   const uint8_t *__restrict__ mask, int64_t V,
                                                                   double wz, double alpha,
                                                                   float *__restrict__ lse_out,
                                                                   float *__restrict__ ce_out,
                                                                   double *__restrict__ tokacc, int64_t n_pad,
                                                                   T *__restrict__ grad)
{
    constexpr int NV = Vec<T>::N;
    constexpr int FU = NT == FL_THREADS_STAT ? FL_U_CE : FL_U;     // 16-byte loads in flight per thread
    const int64_t t = blockIdx.x;
    const T *x = logits + t * V;
    const int tid = threadIdx.x;
    const float L2E = static_cast<float>(LOG2E);
    const bool vec_ok = ((V * static_cast<int64_t>(sizeof(T))) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    const bool keep = grad != nullptr;
    float m = -INFINITY, z = 0.f;
    if (vec_ok) {
        const int64_t nvec = V / NV;
        for (int64_t base = 0; base < nvec; base += NT * FU) {
            uint4 v[FU];
#pragma unroll
            for (int u = 0; u < FU; ++u) {
                const int64_t i = base + u * NT + tid;
                if (i < nvec) v[u] = ld16(x + i * NV, keep);
            }
#pragma unroll
            for (int u = 0; u < FU; ++u) {
                if (base + u * NT + tid >= nvec) continue;
                float f[NV];
                cvt16<T>(v[u], f);
                online_vec<NV>(m, z, f, L2E, raw_max<T>(v[u]));
            }
        }
    } else {
        for (int64_t i = tid; i < V; i += NT) online_add(m, z, to_f(x[i]) * L2E);
    }
    // fixed-shape merge: a butterfly within each warp, then one over the 32
    // warp partials in warp 0
    for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, o);
        const float zo = __shfl_xor_sync(0xffffffffu, z, o);
        online_merge(m, z, mo, zo);
    }
    __shared__ float sm[NT / 32], sz[NT / 32];
    __shared__ float s_par[3];
    const int w = tid >> 5, l = tid & 31;
    if (l == 0) {
        sm[w] = m;
        sz[w] = z;
    }
    __syncthreads();
    if (w == 0) {
        m = l < NT / 32 ? sm[l] : -INFINITY;
        z = l < NT / 32 ? sz[l] : 0.f;
        for (int o = 16; o > 0; o >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m, o);
            const float zo = __shfl_xor_sync(0xffffffffu, z, o);
            online_merge(m, z, mo, zo);
        }
        if (l == 0) {
            // fp32 row statistics for 16-bit logits (far inside their 2e-3
            // tolerance, and one lane's serial work per row here), fp64 for fp32
            using M = typename std::conditional<sizeof(T) == 2, float, double>::type;
            M lse2;
            if constexpr (sizeof(T) == 2) lse2 = m + log2f(z);
            else lse2 = static_cast<double>(m) + log2(static_cast<double>(z));
            const M lse = lse2 * static_cast<M>(LN2);
            const bool on = mask ? (mask[t] != 0) : true;
            const M ce = on ? lse - static_cast<M>(to_f(x[targets[t]])) : M(0);
            const M zz = on ? lse * lse : M(0);
            lse_out[t] = static_cast<float>(lse);
            if (ce_out) ce_out[t] = static_cast<float>(ce);
            tokacc[t] = static_cast<double>(ce) + wz * static_cast<double>(zz);
            tokacc[n_pad + t] = static_cast<double>(ce);
            tokacc[2 * n_pad + t] = static_cast<double>(zz);
            const M al = on ? static_cast<M>(alpha) : M(0);
            s_par[0] = static_cast<float>(lse2);
            s_par[1] = static_cast<float>(al * (M(1) + M(2) * static_cast<M>(wz) * lse));
            s_par[2] = static_cast<float>(al);
        }
    }
    if (!grad) return;
    __syncthreads();
    const float lse2 = s_par[0], c = s_par[1], at = s_par[2];
    const int64_t y = targets[t];
    T *g = grad + t * V;
    if (vec_ok) {
        // the second read: from L2 (the row was read moments ago), then streamed out
        const int64_t nvec = V / NV;
        for (int64_t base = 0; base < nvec; base += NT * FU) {
            uint4 v[FU];
#pragma unroll
            for (int u = 0; u < FU; ++u) {
                const int64_t i = base + u * NT + tid;
                if (i < nvec) v[u] = ld16(x + i * NV, false);
            }
#pragma unroll
            for (int u = 0; u < FU; ++u) {
                const int64_t i = base + u * NT + tid;
                if (i >= nvec) continue;
                float f[NV], gv[NV];
                cvt16<T>(v[u], f);
#pragma unroll
                for (int q = 0; q < NV; ++q) gv[q] = c * ex2_approx(fmaf(f[q], L2E, -lse2));
                const int64_t dy = y - i * NV;     // the one-hot term, in one vector of the row
                if (dy >= 0 && dy < NV) {
#pragma unroll
                    for (int q = 0; q < NV; ++q)
                        if (q == dy) gv[q] -= at;
                }
                store_vec(g + i * NV, gv);
            }
        }
        return;
    }
    for (int64_t i = tid; i < V; i += NT) {
        float gv = c * ex2_approx(fmaf(to_f(x[i]), L2E, -lse2));
        if (i == y) gv -= at;
        from_f(gv, g[i]);
    }
}

template <typename T, int NT>
static void launch_fl(const void *logits, const int64_t *targets, const uint8_t *mask, int64_t n, int64_t V,
                      double wz, double alpha, float *lse_out, float *ce_out, double *tokacc, int64_t n_pad,
                      void *grad, cudaStream_t st)
{
    from_logits_kernel<T, NT><<<static_cast<unsigned>(n), NT, 0, st>>>(
        static_cast<const T *>(logits), targets, mask, V, wz, alpha, lse_out, ce_out, tokacc, n_pad,
        static_cast<T *>(grad));
}

template <typename T>
static void launch_fl_t(const void *logits, const int64_t *targets, const uint8_t *mask, int64_t n, int64_t V,
                        double wz, double alpha, float *lse_out, float *ce_out, double *tokacc, int64_t n_pad,
                        void *grad, cudaStream_t st)
{
    if (grad)
        launch_fl<T, FL_THREADS_GRAD>(logits, targets, mask, n, V, wz, alpha, lse_out, ce_out, tokacc, n_pad, grad, st);
    else
        launch_fl<T, FL_THREADS_STAT>(logits, targets, mask, n, V, wz, alpha, lse_out, ce_out, tokacc, n_pad, grad, st);
}

cudaError_t launch_from_logits(int dtype, const void *logits, const int64_t *targets,
                               const uint8_t *mask, int64_t n, int64_t V, double wz,
                               double alpha, float *lse_out, float *ce_out, double *tokacc,
                               void *grad, cudaStream_t st)
{
    const int64_t n_pad = (n + TC_BM - 1) / TC_BM * TC_BM;
    if (dtype == 1)
        launch_fl_t<uint16_t>(logits, targets, mask, n, V, wz, alpha, lse_out, ce_out, tokacc, n_pad, grad, st);
    else if (dtype == 2)
        launch_fl_t<h16_t>(logits, targets, mask, n, V, wz, alpha, lse_out, ce_out, tokacc, n_pad, grad, st);
    else
        launch_fl_t<float>(logits, targets, mask, n, V, wz, alpha, lse_out, ce_out, tokacc, n_pad, grad, st);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Distillation from materialised student logits (the from-distribution
// forward/backward with its z slot, "Fuse distillation + z-loss ...").  One
// block per token row.  Pass 1 streams the student and teacher
// rows once and keeps, per thread, online (max, sum) pairs for a = s log2e/T
// and b = t log2e/T plus the direction's cross sums; the threads merge by a
// fixed tree.  Pass 2 (optional) re-reads both rows (kept in L2 by pass 1's
// loads) and writes grad_logits.  Sums are fp32 for bf16 rows and fp64 for
// fp32 rows (whose tolerance is 1e-6).
template <typename A> struct DlState {
    float ms, mt;        // running maxima of a and b
    A zs, zt;            // sum 2^(a - ms), sum 2^(b - mt)
    A xa, xb;            // CE/fKL: sum 2^(b - mt) a, sum 2^(b - mt) b
    A xq;                // rKL: sum 2^(a - ms) (a - b)
};

template <typename T, typename A>
__device__ __forceinline__ void dl_add(DlState<A> &S, float a, float b, int direction)
{
    if (a > S.ms) {
        const A f = static_cast<A>(teach_exp2<T>(S.ms - a));
        S.zs *= f;
        S.xq *= f;
        S.ms = a;
    }
    if (b > S.mt) {
        const A f = static_cast<A>(teach_exp2<T>(S.mt - b));
        S.zt *= f;
        S.xa *= f;
        S.xb *= f;
        S.mt = b;
    }
    // a -inf logit has probability 0 and adds nothing to a sum it weights
    // (0 log 0 = 0); a term whose weight is positive keeps its +-inf
    const A es = a != -INFINITY ? static_cast<A>(teach_exp2<T>(a - S.ms)) : A(0);
    const A et = b != -INFINITY ? static_cast<A>(teach_exp2<T>(b - S.mt)) : A(0);
    S.zs += es;
    S.zt += et;
    if (direction == DIR_RKL) {
        if (es != A(0)) S.xq += es * static_cast<A>(a - b);
    } else if (et != A(0)) {
        S.xa += et * static_cast<A>(a);
        S.xb += et * static_cast<A>(b);
    }
}

template <typename T, typename A>
__device__ __forceinline__ void dl_merge(DlState<A> &S, const DlState<A> &O)
{
    const float Ms = fmaxf(S.ms, O.ms), Mt = fmaxf(S.mt, O.mt);
    const A f1 = S.ms == -INFINITY ? A(0) : static_cast<A>(teach_exp2<T>(S.ms - Ms));
    const A f2 = O.ms == -INFINITY ? A(0) : static_cast<A>(teach_exp2<T>(O.ms - Ms));
    const A g1 = S.mt == -INFINITY ? A(0) : static_cast<A>(teach_exp2<T>(S.mt - Mt));
    const A g2 = O.mt == -INFINITY ? A(0) : static_cast<A>(teach_exp2<T>(O.mt - Mt));
    S.zs = S.zs * f1 + O.zs * f2;
    S.xq = S.xq * f1 + O.xq * f2;
    S.zt = S.zt * g1 + O.zt * g2;
    S.xa = S.xa * g1 + O.xa * g2;
    S.xb = S.xb * g1 + O.xb * g2;
    S.ms = Ms;
    S.mt = Mt;
}

// One 16-byte vector of raw student and teacher logits (fa, fb; a = fa kT,
// b = fb kT) into the running maxima, sums and the direction's cross sums, as
// dl_add does element-wise: the maxima first (lms, lmt: raw_max of the two
// vectors; kT > 0 commutes with them), one rescale each if they rose, then the
// independent exponentials, each argument one FFMA.  The cross sums take the
// raw logits: a state built by dl_vec holds xa, xb and xq divided by kT (the
// row kernel scales them back once).
template <typename T, typename A, int NV, bool RKL>
__device__ __forceinline__ void dl_vec(DlState<A> &S, const float (&fa)[NV], const float (&fb)[NV], float kT,
                                       float lms, float lmt)
{
    lms *= kT;
    lmt *= kT;
    if (lms > S.ms) {
        const A f = static_cast<A>(teach_exp2<T>(S.ms - lms));
        S.zs *= f;
        S.xq *= f;
        S.ms = lms;
    }
    if (lmt > S.mt) {
        const A f = static_cast<A>(teach_exp2<T>(S.mt - lmt));
        S.zt *= f;
        S.xa *= f;
        S.xb *= f;
        S.mt = lmt;
    }
    // No -inf handling here: a -inf logit leaves a NaN or an infinity in the
    // sums (0 * -inf, -inf - -inf), and the kernel recomputes such a row with
    // dl_add, so rows of finite logits pay nothing for it.
    A zs = 0, zt = 0, x1 = 0, x2 = 0;
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const A es = static_cast<A>(teach_exp2<T>(fmaf(fa[u], kT, -S.ms)));
        const A et = static_cast<A>(teach_exp2<T>(fmaf(fb[u], kT, -S.mt)));
        zs += es;
        zt += et;
        if (RKL) {
            x1 += es * static_cast<A>(fa[u] - fb[u]);
        } else {
            x1 += et * static_cast<A>(fa[u]);
            x2 += et * static_cast<A>(fb[u]);
        }
    }
    S.zs += zs;
    S.zt += zt;
    if (RKL) {
        S.xq += x1;
    } else {
        S.xa += x1;
        S.xb += x2;
    }
}

template <typename T, typename A> __device__ __forceinline__ DlState<A> dl_shfl(const DlState<A> &x, int o)
{
    DlState<A> r;
    r.ms = __shfl_xor_sync(0xffffffffu, x.ms, o);
    r.mt = __shfl_xor_sync(0xffffffffu, x.mt, o);
    r.zs = __shfl_xor_sync(0xffffffffu, x.zs, o);
    r.zt = __shfl_xor_sync(0xffffffffu, x.zt, o);
    r.xa = __shfl_xor_sync(0xffffffffu, x.xa, o);
    r.xb = __shfl_xor_sync(0xffffffffu, x.xb, o);
    r.xq = __shfl_xor_sync(0xffffffffu, x.xq, o);
    return r;
}

// RKL: reverse KL (its own cross sum and gradient form); otherwise CE or
// forward KL, which share them.
template <typename T, int NT, bool RKL>
__global__ void __launch_bounds__(NT, 1024 / NT) distill_logits_kernel(
    const T *__restrict__ student, const T *__restrict__ teacher, const uint8_t *__restrict__ mask,
    int64_t V, int direction, float kT, double wz, double at_on, double inv_t, float *__restrict__ lse_out,
    float *__restrict__ per_token, double *__restrict__ tokacc, int64_t n_pad, T *__restrict__ grad,
    int accumulate)
{
    using A = typename TeachAcc<T>::type;
    constexpr int NV = Vec<T>::N;
    const int64_t t = blockIdx.x;
    const T *xs = student + t * V, *xt = teacher + t * V;
    const int tid = threadIdx.x;
    const bool vec_ok = ((V * static_cast<int64_t>(sizeof(T))) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(student) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(teacher) % 16 == 0);
    const bool keep = grad != nullptr;
    const DlState<A> S0{-INFINITY, -INFINITY, 0, 0, 0, 0, 0};
    DlState<A> S = S0;
    if (vec_ok) {
        const int64_t nvec = V / NV;
        for (int64_t base = 0; base < nvec; base += NT * FL_U) {
            uint4 vs[FL_U], vt[FL_U];
#pragma unroll
            for (int u = 0; u < FL_U; ++u) {
                const int64_t i = base + u * NT + tid;
                if (i < nvec) {
                    vs[u] = ld16(xs + i * NV, keep);
                    vt[u] = ld16(xt + i * NV, keep);
                }
            }
#pragma unroll
            for (int u = 0; u < FL_U; ++u) {
                if (base + u * NT + tid >= nvec) continue;
                float fa[NV], fb[NV];
                cvt16<T>(vs[u], fa);
                cvt16<T>(vt[u], fb);
                dl_vec<T, A, NV, RKL>(S, fa, fb, kT, raw_max<T>(vs[u]), raw_max<T>(vt[u]));
            }
        }
    } else {
        for (int64_t i = tid; i < V; i += NT)
            dl_add<T, A>(S, to_f(xs[i]) * kT, to_f(xt[i]) * kT, direction);
    }
    // fixed-shape merge: a butterfly within each warp, then one over the 32
    // warp partials in warp 0 (whose lanes hold the row's state after it)
    __shared__ DlState<A> sw[NT / 32];
    __shared__ float sP[4];
    __shared__ int s_redo;
    const int w = tid >> 5, l = tid & 31;
    auto block_merge = [&](DlState<A> X) {
        for (int o = 16; o > 0; o >>= 1) dl_merge<T, A>(X, dl_shfl<T, A>(X, o));
        if (l == 0) sw[w] = X;
        __syncthreads();
        DlState<A> R = S0;
        if (w == 0) {
            if (l < NT / 32) R = sw[l];
            for (int o = 16; o > 0; o >>= 1) dl_merge<T, A>(R, dl_shfl<T, A>(R, o));
        }
        return R;
    };
    DlState<A> R = block_merge(S);
    bool masked = false;
    if (vec_ok) {
        // vector sums that are not finite mean a -inf logit in the row (or an
        // overflow, which the element-wise sums reproduce): recompute the row
        // with dl_add's handling of -inf
        if (tid == 0)
            s_redo = !(isfinite(static_cast<float>(R.zs)) && isfinite(static_cast<float>(R.zt)) &&
                       isfinite(static_cast<float>(R.xa)) && isfinite(static_cast<float>(R.xb)) &&
                       isfinite(static_cast<float>(R.xq)));
        __syncthreads();
        masked = s_redo != 0;
        if (masked) {
            S = S0;
            for (int64_t i = tid; i < V; i += NT)
                dl_add<T, A>(S, to_f(xs[i]) * kT, to_f(xt[i]) * kT, direction);
            R = block_merge(S);
        }
    } else {
        masked = true;
    }
    if (w == 0) {
        if (l == 0) {
            if (!masked) {
                // dl_vec's cross sums are in raw logits
                R.xa *= static_cast<A>(kT);
                R.xb *= static_cast<A>(kT);
                R.xq *= static_cast<A>(kT);
            }
            // fp32 row statistics for 16-bit logits (far inside their 2e-3
            // tolerance, and one lane's serial work per row here), fp64 for fp32
            using M = typename std::conditional<sizeof(T) == 2, float, double>::type;
            auto lg2 = [](M v) -> M {
                if constexpr (sizeof(T) == 2) return log2f(v);
                else return log2(v);
            };
            const M lse_s2 = static_cast<M>(R.ms) + lg2(static_cast<M>(R.zs));
            const M lse_t2 = static_cast<M>(R.mt) + lg2(static_cast<M>(R.zt));
            const M pa = static_cast<M>(R.xa) / static_cast<M>(R.zt);
            const M pb = static_cast<M>(R.xb) / static_cast<M>(R.zt);
            const M qx = static_cast<M>(R.xq) / static_cast<M>(R.zs);
            M L2;
            if (direction == DIR_CE) L2 = lse_s2 - pa;
            else if (direction == DIR_FKL) L2 = pb - lse_t2 - pa + lse_s2;
            else L2 = qx - lse_s2 + lse_t2;
            const M ln2 = static_cast<M>(LN2);
            const M L = L2 * ln2, lse_s = lse_s2 * ln2, lse_t = lse_t2 * ln2;
            const M wzm = static_cast<M>(wz);
            const bool on = mask ? (mask[t] != 0) : true;
            const M Lm = on ? L : M(0), z2 = on ? lse_s * lse_s : M(0);
            if (lse_out) lse_out[t] = static_cast<float>(lse_s);
            if (per_token) per_token[t] = static_cast<float>(Lm);
            tokacc[t] = static_cast<double>(Lm) + wz * static_cast<double>(z2);
            tokacc[n_pad + t] = static_cast<double>(Lm);
            tokacc[2 * n_pad + t] = static_cast<double>(z2);
            const M at = on ? static_cast<M>(at_on * inv_t) : M(0);
            sP[0] = static_cast<float>(lse_s2);
            sP[1] = static_cast<float>(lse_t2);
            if (direction == DIR_RKL) {
                sP[2] = static_cast<float>(at);
                sP[3] = static_cast<float>(lse_t - lse_s - L + M(2) * wzm * lse_s);
            } else {
                sP[2] = static_cast<float>(at * (M(1) + M(2) * wzm * lse_s));
                sP[3] = static_cast<float>(at);
            }
        }
    }
    if (!grad) return;
    __syncthreads();
    const float ls2 = sP[0], lt2 = sP[1], pz = sP[2], pw = sP[3];
    const float ln2f = static_cast<float>(LN2), kTln2 = kT * ln2f;
    // the gradient of one element from its raw logits (a = fa kT, b = fb kT)
    auto gval = [&](float fa, float fb) {
        const float qv = teach_exp2<T>(fmaf(fa, kT, -ls2));
        if (RKL) return pz * qv * fmaf(fa - fb, kTln2, pw);
        return pz * qv - pw * teach_exp2<T>(fmaf(fb, kT, -lt2));
    };
    T *g = grad + t * V;
    // In reverse KL a -inf student logit has q = 0 and a gradient of 0, where
    // gval's product q (a - b) would be 0 * -inf: rows that held a -inf take the
    // element-wise loop, which tests for it.
    if (vec_ok && !(masked && RKL)) {
        // the second read, last rounds first: the most recently read part of the
        // rows is the most likely to be still in L2 (one loop per accumulate mode)
        const int64_t nvec = V / NV;
        const int64_t nround = (nvec + NT * FL_U - 1) / (NT * FL_U);
        auto pass2 = [&](auto acc_mode) {
        constexpr bool ACC = decltype(acc_mode)::value;
        for (int64_t rr = nround - 1; rr >= 0; --rr) {
            const int64_t base = rr * NT * FL_U;
            uint4 vs[FL_U], vt[FL_U];
#pragma unroll
            for (int u = 0; u < FL_U; ++u) {
                const int64_t i = base + u * NT + tid;
                if (i < nvec) {
                    vs[u] = ld16(xs + i * NV, false);
                    vt[u] = ld16(xt + i * NV, false);
                }
            }
#pragma unroll
            for (int u = 0; u < FL_U; ++u) {
                const int64_t i = base + u * NT + tid;
                if (i >= nvec) continue;
                float fs[NV], ft[NV], gv[NV];
                cvt16<T>(vs[u], fs);
                cvt16<T>(vt[u], ft);
                if (ACC) load_vec<T>(g + i * NV, gv, false);
#pragma unroll
                for (int q = 0; q < NV; ++q) {
                    const float v = gval(fs[q], ft[q]);
                    gv[q] = ACC ? gv[q] + v : v;
                }
                store_vec(g + i * NV, gv);
            }
        }
        };
        if (accumulate) pass2(std::true_type{});
        else pass2(std::false_type{});
        return;
    }
    for (int64_t i = tid; i < V; i += NT) {
        const float fa = to_f(xs[i]);
        float v = RKL && teach_exp2<T>(fmaf(fa, kT, -ls2)) == 0.f ? 0.f : gval(fa, to_f(xt[i]));
        if (accumulate) v += to_f(g[i]);
        from_f(v, g[i]);
    }
}

template <typename T>
static void launch_dl_t(const void *student, const void *teacher, const uint8_t *mask, int64_t n, int64_t V,
                        int direction, float kT, double wz, double at_on, double inv_t, float *lse_out,
                        float *per_token, double *tokacc, int64_t n_pad, void *grad, int accumulate, cudaStream_t st)
{
    const T *xs = static_cast<const T *>(student), *xt = static_cast<const T *>(teacher);
    T *g = static_cast<T *>(grad);
    const unsigned grid = static_cast<unsigned>(n);
    if (grad && direction == DIR_RKL)
        distill_logits_kernel<T, FL_THREADS_GRAD, true><<<grid, FL_THREADS_GRAD, 0, st>>>(
            xs, xt, mask, V, direction, kT, wz, at_on, inv_t, lse_out, per_token, tokacc, n_pad, g, accumulate);
    else if (grad)
        distill_logits_kernel<T, FL_THREADS_GRAD, false><<<grid, FL_THREADS_GRAD, 0, st>>>(
            xs, xt, mask, V, direction, kT, wz, at_on, inv_t, lse_out, per_token, tokacc, n_pad, g, accumulate);
    else if (direction == DIR_RKL)
        distill_logits_kernel<T, FL_THREADS_STAT, true><<<grid, FL_THREADS_STAT, 0, st>>>(
            xs, xt, mask, V, direction, kT, wz, at_on, inv_t, lse_out, per_token, tokacc, n_pad, g, accumulate);
    else
        distill_logits_kernel<T, FL_THREADS_STAT, false><<<grid, FL_THREADS_STAT, 0, st>>>(
            xs, xt, mask, V, direction, kT, wz, at_on, inv_t, lse_out, per_token, tokacc, n_pad, g, accumulate);
}

cudaError_t launch_distill_logits(int dtype, const void *student, const void *teacher, const uint8_t *mask,
                                  int64_t n, int64_t V, int direction, double temperature, double wz,
                                  double at_on, float *lse_out, float *per_token, double *tokacc,
                                  int64_t n_pad, void *grad, bool accumulate, cudaStream_t st)
{
    const float kT = static_cast<float>(LOG2E / temperature);
    const double inv_t = 1.0 / temperature;
    const int acc = accumulate ? 1 : 0;
    if (dtype == 2)
        launch_dl_t<h16_t>(student, teacher, mask, n, V, direction, kT, wz, at_on, inv_t, lse_out, per_token,
                           tokacc, n_pad, grad, acc, st);
    else if (dtype == 1)
        launch_dl_t<uint16_t>(student, teacher, mask, n, V, direction, kT, wz, at_on, inv_t, lse_out, per_token,
                              tokacc, n_pad, grad, acc, st);
    else
        launch_dl_t<float>(student, teacher, mask, n, V, direction, kT, wz, at_on, inv_t, lse_out, per_token,
                           tokacc, n_pad, grad, acc, st);
    return cudaGetLastError();
}


// ---------------------------------------------------------------------------
// fp32 FFMA path.  256 threads (16 x 16), 64 x 64 logit tiles, 4 x 4 per
// thread; the contraction over d_model is staged through shared memory in
// steps of 16 and summed in ascending k.  Modes mirror the tensor-core
// kernel: STATS writes per-tile partial statistics, ROWS/COLS rebuild the
// gradient tile in shared memory (fp32, never rounded) and accumulate
// G . Y[:, slice] over the loop of Y tiles.
template <int MODE, bool DISTILL>
__global__ void __launch_bounds__(256) fp_kernel(const float *__restrict__ X,
                                                 const float *__restrict__ Y,
                                                 const float *__restrict__ teach, int n_x, int n_y,
                                                 int d, int n_tok, int vocab, int n_split,
                                                 int direction, float inv_t,
                                                 const int64_t *__restrict__ targets,
                                                 const float4 *__restrict__ tokp,
                                                 const double2 *__restrict__ tstat,
                                                 float *__restrict__ part, float *__restrict__ tgt,
                                                 int64_t part_stride, int64_t part_plane,
                                                 float *__restrict__ out, int64_t out_split_stride,
                                                 int accumulate)
{
    __shared__ float xs[FP_BK][FP_BM + 4];
    __shared__ float ys[FP_BK][FP_BN + 4];
    __shared__ float gs[FP_BM][FP_BN + 1];
    __shared__ float yv[FP_BN][FP_SLICE + 4];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const float L2E = static_cast<float>(LOG2E);
    const int n_xt = (n_x + FP_BM - 1) / FP_BM, n_yt = (n_y + FP_BN - 1) / FP_BN;

    int xt, yt_begin, yt_end, slice = 0, split = 0;
    if (MODE == TC_STATS) {
        xt = blockIdx.x % n_xt;
        yt_begin = blockIdx.x / n_xt;
        yt_end = yt_begin + 1;
    } else {
        const int n_sl = (d + FP_SLICE - 1) / FP_SLICE;
        int b = blockIdx.x;
        slice = b % n_sl;
        b /= n_sl;
        xt = b % n_xt;
        split = b / n_xt;
        yt_begin = static_cast<int>((static_cast<int64_t>(split) * n_yt) / n_split);
        yt_end = static_cast<int>((static_cast<int64_t>(split + 1) * n_yt) / n_split);
    }
    const int xrow0 = xt * FP_BM;
    float acc[4][4] = {};
    // STATS: the logits are compensated dot products (Dot2 of Ogita, Rump and
    // Oishi, "Accurate sum and dot product", SIAM J. Sci. Comput. 26 (2005)):
    // each product is split exactly into its rounded value and the FMA
    // residual, each sum into its rounded value and the TwoSum residual, and
    // the residuals are added on the side, so a logit carries about one
    // rounding of its own size however much its terms cancel.  The plain
    // intrinsics keep the compiler from contracting the split operations.
    constexpr bool DOT2 = MODE == TC_STATS;

    for (int yt = yt_begin; yt < yt_end; ++yt) {
        const int ycol0 = yt * FP_BN;
        float s[4][4] = {}, sc[4][4] = {};
        for (int k0 = 0; k0 < d; k0 += FP_BK) {
            for (int e = threadIdx.x; e < FP_BM * FP_BK; e += 256) {
                const int rr = e / FP_BK, kk = e % FP_BK;
                const int gx = xrow0 + rr, gy = ycol0 + rr, gk = k0 + kk;
                xs[kk][rr] = (gx < n_x && gk < d) ? X[static_cast<int64_t>(gx) * d + gk] : 0.f;
                ys[kk][rr] = (gy < n_y && gk < d) ? Y[static_cast<int64_t>(gy) * d + gk] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < FP_BK; ++kk) {
                float xa[4], yb[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xa[i] = xs[kk][ty * 4 + i];
                    yb[i] = ys[kk][tx * 4 + i];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jx = 0; jx < 4; ++jx) {
                        if (DOT2) {
                            const float p = __fmul_rn(xa[i], yb[jx]);
                            const float pe = __fmaf_rn(xa[i], yb[jx], -p);       // a b = p + pe exactly
                            const float t = __fadd_rn(s[i][jx], p);
                            const float z = __fsub_rn(t, s[i][jx]);
                            const float se = __fadd_rn(__fsub_rn(s[i][jx], __fsub_rn(t, z)), __fsub_rn(p, z));
                            s[i][jx] = t;                                      // s + p = t + se exactly
                            sc[i][jx] = __fadd_rn(sc[i][jx], __fadd_rn(pe, se));
                        } else {
                            s[i][jx] = fmaf(xa[i], yb[jx], s[i][jx]);
                        }
                    }
            }
            __syncthreads();
        }
        if (DOT2) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jx = 0; jx < 4; ++jx) s[i][jx] = __fadd_rn(s[i][jx], sc[i][jx]);
        }
        if (MODE == TC_STATS) {
            // rows ty*4+i, columns tx*4+jx; a row's 64 columns live in 16
            // lanes of one half-warp
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = xrow0 + ty * 4 + i;
                float vs[4], vt[4];
#pragma unroll
                for (int jx = 0; jx < 4; ++jx) {
                    const int v = ycol0 + tx * 4 + jx;
                    const bool in = v < vocab && t < n_tok;
                    vs[jx] = in ? s[i][jx] : -INFINITY;
                    vt[jx] = (DISTILL && in) ? teach[static_cast<int64_t>(t) * vocab + v] : -INFINITY;
                }
                if (!DISTILL) {
                    float m = -INFINITY, z = 0.f;
#pragma unroll
                    for (int jx = 0; jx < 4; ++jx) m = fmaxf(m, vs[jx] * L2E);
                    for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
#pragma unroll
                    for (int jx = 0; jx < 4; ++jx) z += exp2f(vs[jx] * L2E - m);
                    for (int o = 1; o < 16; o <<= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
                    if (t < n_tok) {
                        if (tx == 0) {
                            const int64_t o = static_cast<int64_t>(yt) * part_stride + t;
                            part[o] = m;
                            part[part_plane + o] = z;
                        }
                        // no targets (a vocabulary shard): the target logit comes from elsewhere
                        const int64_t rel = targets ? targets[t] - ycol0 - tx * 4 : -1;
#pragma unroll
                        for (int jx = 0; jx < 4; ++jx)
                            if (rel == jx) tgt[t] = s[i][jx];
                    }
                } else {
                    // student (max, sum) of this tile and the direction's cross term:
                    // CE / forward KL: sum p a with the teacher's p exact (its lse from
                    // teacher_stats); reverse KL: sum 2^(a - max) (a - b)
                    const float lt2 = t < n_tok ? static_cast<float>(tstat[t].x) : 0.f;
                    float a2[4], b2[4], ms = -INFINITY;
#pragma unroll
                    for (int jx = 0; jx < 4; ++jx) {
                        a2[jx] = vs[jx] * inv_t * L2E;
                        b2[jx] = vt[jx] * inv_t * L2E;
                        ms = fmaxf(ms, a2[jx]);
                    }
                    for (int o = 1; o < 16; o <<= 1) ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, o));
                    float zs = 0.f, xx = 0.f;
#pragma unroll
                    for (int jx = 0; jx < 4; ++jx) {
                        if (vs[jx] == -INFINITY) continue;
                        const float es = exp2f(a2[jx] - ms);
                        zs += es;
                        if (direction == DIR_RKL) xx = fmaf(es, a2[jx] - b2[jx], xx);
                        else xx = fmaf(exp2f(b2[jx] - lt2), a2[jx], xx);
                    }
                    for (int o = 1; o < 16; o <<= 1) {
                        zs += __shfl_xor_sync(0xffffffffu, zs, o);
                        xx += __shfl_xor_sync(0xffffffffu, xx, o);
                    }
                    if (t < n_tok && tx == 0) {
                        const int64_t o = static_cast<int64_t>(yt) * part_stride + t;
                        part[o] = ms;
                        part[part_plane + o] = zs;
                        part[2 * part_plane + o] = xx;
                    }
                }
            }
        } else {
            // gradient tile (rows of X by columns of Y) into shared memory
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int jx = 0; jx < 4; ++jx) {
                    const int xr = xrow0 + ty * 4 + i, yc = ycol0 + tx * 4 + jx;
                    const int tok = (MODE == TC_ROWS) ? xr : yc;
                    const int voc = (MODE == TC_ROWS) ? yc : xr;
                    float g = 0.f;
                    if (tok < n_tok && voc < vocab) {
                        const float4 P = tokp[tok];
                        const float sv = s[i][jx];
                        if (!DISTILL) {
                            g = P.y * exp2f(fmaf(sv, L2E, -P.x));
                            if (__float_as_int(P.w) == voc) g -= P.z;
                        } else {
                            const float a2v = sv * inv_t * L2E;
                            const float b2v = teach[static_cast<int64_t>(tok) * vocab + voc] * inv_t * L2E;
                            const float qv = exp2f(a2v - P.x);
                            if (direction == DIR_RKL)
                                g = P.z * qv * fmaf(a2v - b2v, static_cast<float>(LN2), P.w);
                            else
                                g = P.z * qv - P.w * exp2f(b2v - P.y);
                        }
                    }
                    gs[ty * 4 + i][tx * 4 + jx] = g;
                }
            }
            // Y[ycol0 .. +64][slice cols]
            for (int e = threadIdx.x; e < FP_BN * FP_SLICE; e += 256) {
                const int rr = e / FP_SLICE, cc = e % FP_SLICE;
                const int gy = ycol0 + rr, gc = slice * FP_SLICE + cc;
                yv[rr][cc] = (gy < n_y && gc < d) ? Y[static_cast<int64_t>(gy) * d + gc] : 0.f;
            }
            __syncthreads();
            for (int kk = 0; kk < FP_BN; ++kk) {
                float ga[4], yb[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    ga[i] = gs[ty * 4 + i][kk];
                    yb[i] = yv[kk][tx * 4 + i];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jx = 0; jx < 4; ++jx) acc[i][jx] = fmaf(ga[i], yb[jx], acc[i][jx]);
            }
            __syncthreads();
        }
    }
    if (MODE != TC_STATS) {
        float *o = out + static_cast<int64_t>(split) * out_split_stride;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int xr = xrow0 + ty * 4 + i;
            if (xr >= n_x) continue;
#pragma unroll
            for (int jx = 0; jx < 4; ++jx) {
                const int c = slice * FP_SLICE + tx * 4 + jx;
                if (c < d) {
                    float *p = o + static_cast<int64_t>(xr) * d + c;
                    *p = accumulate ? *p + acc[i][jx] : acc[i][jx];
                }
            }
        }
    }
}

cudaError_t launch_fp(int mode, bool distill, const void *X, const void *Y, const float *teach,
                      int n_x, int n_y, int d, int n_tok, int vocab, int n_split, int direction,
                      float inv_t, const int64_t *targets, const float4 *tokp, const double2 *tstat,
                      float *part,
                      float *tgt, int64_t part_stride, int64_t part_plane, float *out,
                      int64_t out_split_stride, cudaStream_t st, bool accumulate)
{
    const int n_xt = (n_x + FP_BM - 1) / FP_BM, n_yt = (n_y + FP_BN - 1) / FP_BN;
    const int n_sl = (d + FP_SLICE - 1) / FP_SLICE;
    const int64_t grid64 = mode == TC_STATS ? static_cast<int64_t>(n_xt) * n_yt
                                            : static_cast<int64_t>(n_xt) * n_sl * n_split;
    const unsigned grid = static_cast<unsigned>(grid64);
    const float *x = static_cast<const float *>(X), *y = static_cast<const float *>(Y);
#define LOSSK_FP(M, D)                                                                             \
    fp_kernel<M, D><<<grid, 256, 0, st>>>(x, y, teach, n_x, n_y, d, n_tok, vocab, n_split,       \
                                          direction, inv_t, targets, tokp, tstat, part, tgt, part_stride, \
                                          part_plane, out, out_split_stride, accumulate ? 1 : 0)
    if (mode == TC_STATS) {
        if (distill) LOSSK_FP(TC_STATS, true); else LOSSK_FP(TC_STATS, false);
    } else if (mode == TC_ROWS) {
        if (distill) LOSSK_FP(TC_ROWS, true); else LOSSK_FP(TC_ROWS, false);
    } else {
        if (distill) LOSSK_FP(TC_COLS, true); else LOSSK_FP(TC_COLS, false);
    }
#undef LOSSK_FP
    return cudaGetLastError();
}

} // namespace lossk
