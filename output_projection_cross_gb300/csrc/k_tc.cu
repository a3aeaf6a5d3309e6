// k_tc.cu -- the tcgen05 / TMA path of the fused LM-head loss (bf16 inputs,
// fp32 accumulation in tensor memory).
//
// One warp-specialised kernel template does all three passes:
//
//   TC_STATS  forward.  S = H_tile . W_tile^T (tokens x vocabulary) lands in
//             TMEM; the epilogue reduces each row of the tile to a partial
//             (running max, sum of exp) pair -- the online log-sum-exp of
//             "Loss functions and resident-context kernels" (lossk: a chunk's
//             logits are reduced at once, never kept) -- and gathers the
//             target logit.  Distillation also reduces the teacher tile beside
//             it.
//   TC_ROWS   d_hidden.  X = hidden rows (tokens), Y = weight rows.  For each
//             vocabulary tile the logit tile is recomputed, turned into
//             grad_logits in registers (label family: softmax minus one-hot,
//             "Fuse distillation + z-loss ...", "What it does"), written to
//             shared memory as bf16, and multiplied by W_tile[:, slice] into a
//             TMEM accumulator that lives across the whole vocabulary loop.
//   TC_COLS   d_weight.  The same with X = weight rows and Y = hidden rows,
//             so the accumulator holds dW_tile[:, slice] across all tokens.
//
// Roles (192 threads): warp 0 issues TMA copies into a ring of shared-memory
// stages; warp 1 owns tensor memory and issues tcgen05.mma; warps 2-5 are the
// epilogue (warp w reads TMEM lanes 32*(w%4) .. +31, one tile row per
// thread).  Two TMEM logit buffers let the tensor core compute tile j+1
// while the epilogue reduces tile j.  Every wait is bounded (ptx.cuh).
#include "lossk_internal.h"
#include "ptx.cuh"

#include <cfloat>

namespace lossk {

template <int MODE, bool DISTILL> struct TcCfg {
    static constexpr bool ACC = MODE != TC_STATS;
    static constexpr int BN = (MODE == TC_STATS && !DISTILL) ? TC_BN_FWD : TC_BN_ACC;
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;
    static constexpr int B_BYTES = BN * TC_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (ACC && DISTILL) ? 3 : (ACC ? 5 : 4);
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int G_BYTES = ACC ? TC_BM * TC_BN_ACC * 2 : 0;
    static constexpr int T_BYTES = DISTILL ? 2 * TC_BM * TC_BN_ACC * 2 : 0;
    static constexpr int COLP_N = (MODE == TC_COLS) ? 2 * TC_BN_ACC : 0;
    static constexpr int NBARS = 2 * STAGES + 2 + 2 + 3 + 2 + 2 + 2 + 1;
    static constexpr int SMEM_BYTES =
        1024 + RING_BYTES + G_BYTES + T_BYTES + COLP_N * 16 + NBARS * 8 + 16;
    static constexpr uint32_t TMEM_COLS = ACC ? 512 : 2 * BN;
    static constexpr uint32_t ACC_COL = 2 * TC_BN_ACC;
    static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
    static_assert(!ACC || STAGE_BYTES == 4 * 64 * 64 * 2, "a backward stage also holds a d-slice");
    static_assert(SMEM_BYTES <= 232448, "fits the 227 KB per-CTA shared memory limit");
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Wait without looking at the error word: used only while unwinding, to let
// copies and MMAs that are already in flight land before the CTA exits.
__device__ __forceinline__ void mbar_wait_drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 200000000ull) return;
}

template <int MODE, bool DISTILL>
__global__ void __launch_bounds__(192, 1) tc_kernel(const __grid_constant__ TcArgs a)
{
    using C = TcCfg<MODE, DISTILL>;
    constexpr int BN = C::BN;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem;
    uint8_t *gbuf = ring + C::RING_BYTES;
    uint8_t *teach = gbuf + C::G_BYTES;
    float4 *colp = reinterpret_cast<float4 *>(teach + C::T_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(colp + C::COLP_N);
    uint64_t *full = bars;              // [S]  TMA bytes landed
    uint64_t *empty = full + S;         // [S]  MMA done reading the stage
    uint64_t *tfull = empty + S;        // [2]  logit tile in TMEM buffer ready
    uint64_t *tempty = tfull + 2;       // [2]  epilogue done with TMEM buffer
    uint64_t *gfull = tempty + 2;       // grad tile written to shared memory
    uint64_t *gempty = gfull + 1;       // grad tile consumed by the MMA
    uint64_t *accfull = gempty + 1;     // accumulator final
    uint64_t *thfull = accfull + 1;     // [2] teacher tile landed
    uint64_t *thempty = thfull + 2;     // [2] teacher tile consumed
    uint64_t *colrdy = thempty + 2;     // [2] per-column parameters staged
    uint64_t *drain = colrdy + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *err = a.err;

    // ---- work assignment ----------------------------------------------------
    int it_begin, it_end, xt_fixed = 0, slice = 0, yt_begin = 0;
    if (MODE == TC_STATS) {
        it_begin = static_cast<int>((static_cast<int64_t>(blockIdx.x) * a.n_items) / gridDim.x);
        it_end = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * a.n_items) / gridDim.x);
    } else {
        int b = blockIdx.x;
        slice = b % a.n_slices;
        b /= a.n_slices;
        xt_fixed = b % a.n_xt;
        const int split = b / a.n_xt;
        yt_begin = static_cast<int>((static_cast<int64_t>(split) * a.n_yt) / a.n_split);
        const int yt_end = static_cast<int>((static_cast<int64_t>(split + 1) * a.n_yt) / a.n_split);
        it_begin = 0;
        it_end = yt_end - yt_begin;
    }
    const int n_it = it_end - it_begin;
    const int slice0 = slice * TC_SLICE;
    auto coords = [&](int j, int &xrow0, int &ycol0, int &yt) {
        if (MODE == TC_STATS) {
            const int i = it_begin + j;
            yt = i / a.n_xt;
            xrow0 = (i - yt * a.n_xt) * TC_BM;
        } else {
            yt = yt_begin + j;
            xrow0 = xt_fixed * TC_BM;
        }
        ycol0 = yt * BN;
    };

    // ---- setup ----------------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 128);
            mbar_init(&thfull[b], 1);
            mbar_init(&thempty[b], 128);
            mbar_init(&colrdy[b], 128);
        }
        mbar_init(gfull, 128);
        mbar_init(gempty, 1);
        mbar_init(accfull, 1);
        mbar_init(drain, 1);
        fence_mbarrier_init();
    }
    if (warp == 1) tmem_alloc(tslot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0 && lane == 0) {
        // ================= TMA producer =================
        tma_prefetch_desc(&a.map_x);
        tma_prefetch_desc(&a.map_y);
        if (C::ACC) tma_prefetch_desc(&a.map_ys);
        if (DISTILL) tma_prefetch_desc(&a.map_teach);
        int st = 0;
        uint32_t ph = 0;
        uint32_t issued = 0;          // bit s: stage s has been filled at least once
        uint32_t last_ph = 0;         // bit s: parity of its last fill
        bool ok = true;
        const int nk = (a.d + TC_BK - 1) / TC_BK;
        auto acquire = [&](uint32_t bytes) -> uint8_t * {
            if (!mbar_wait(&empty[st], ph ^ 1, err)) return nullptr;
            mbar_arrive_expect_tx(&full[st], bytes);
            issued |= 1u << st;
            last_ph = (last_ph & ~(1u << st)) | (ph << st);
            return ring + st * C::STAGE_BYTES;
        };
        auto advance = [&]() {
            if (++st == S) {
                st = 0;
                ph ^= 1;
            }
        };
        for (int j = 0; j <= n_it && ok; ++j) {
            if (j < n_it) {
                int xrow0, ycol0, yt;
                coords(j, xrow0, ycol0, yt);
                if (DISTILL) {
                    const int b = j & 1;
                    if (!mbar_wait(&thempty[b], ((j >> 1) & 1) ^ 1, err)) { ok = false; break; }
                    mbar_arrive_expect_tx(&thfull[b], 2 * TC_BM * 64 * 2);
                    uint8_t *tb = teach + b * (TC_BM * TC_BN_ACC * 2);
                    if (MODE == TC_COLS) {   // tokens are the Y rows, vocabulary the X rows
                        tma_load_2d(tb, &a.map_teach, &thfull[b], xrow0, ycol0);
                        tma_load_2d(tb + 16384, &a.map_teach, &thfull[b], xrow0 + 64, ycol0);
                    } else {
                        tma_load_2d(tb, &a.map_teach, &thfull[b], ycol0, xrow0);
                        tma_load_2d(tb + 16384, &a.map_teach, &thfull[b], ycol0 + 64, xrow0);
                    }
                }
                for (int kb = 0; kb < nk; ++kb) {
                    uint8_t *sp = acquire(C::STAGE_BYTES);
                    if (!sp) { ok = false; break; }
                    tma_load_2d(sp, &a.map_x, &full[st], kb * TC_BK, xrow0);
                    tma_load_2d(sp + C::A_BYTES, &a.map_y, &full[st], kb * TC_BK, ycol0);
                    advance();
                }
                if (!ok) break;
            }
            if (C::ACC && j >= 1) {
                int xrow0, ycol0, yt;
                coords(j - 1, xrow0, ycol0, yt);
                for (int h = 0; h < 2; ++h) {
                    uint8_t *sp = acquire(C::STAGE_BYTES);
                    if (!sp) { ok = false; break; }
                    for (int q = 0; q < 4; ++q)
                        tma_load_2d(sp + q * 8192, &a.map_ys, &full[st], slice0 + q * 64,
                                    ycol0 + h * 64);
                    advance();
                }
            }
        }
        // Let every copy already issued land before the CTA can exit.
        for (int s = 0; s < S; ++s)
            if (issued & (1u << s)) mbar_wait_drain(&full[s], (last_ph >> s) & 1);
        if (DISTILL && n_it > 0) {
            mbar_wait_drain(&thfull[(n_it - 1) & 1], ((n_it - 1) >> 1) & 1);
            if (n_it > 1) mbar_wait_drain(&thfull[(n_it - 2) & 1], ((n_it - 2) >> 1) & 1);
        }
    } else if (warp == 1 && lane == 0) {
        // ================= MMA issuer =================
        constexpr uint32_t ID_S = idesc_bf16_f32(TC_BM, BN, 0, 0);
        constexpr uint32_t ID_ACC = idesc_bf16_f32(TC_BM, TC_SLICE, 0, 1);
        int st = 0;
        uint32_t ph = 0;
        bool ok = true, first_acc = true;
        const int nk = (a.d + TC_BK - 1) / TC_BK;
        const uint32_t g_base = smem_u32(gbuf);
        for (int j = 0; j <= n_it && ok; ++j) {
            if (j < n_it) {
                const int b = j & 1;
                if (!mbar_wait(&tempty[b], ((j >> 1) & 1) ^ 1, err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_s = tmem + b * BN;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&full[st], ph, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(ring + st * C::STAGE_BYTES);
                    const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < TC_BK / 16; ++k)
                        tc_mma_bf16(d_s, sdesc_sw128(sa + k * 32, 16, 1024),
                                    sdesc_sw128(sb + k * 32, 16, 1024), ID_S, (kb | k) != 0);
                    tc_commit(&empty[st]);
                    if (++st == S) { st = 0; ph ^= 1; }
                }
                if (!ok) break;
                tc_commit(&tfull[b]);
            }
            if (C::ACC && j >= 1) {
                const int jj = j - 1;
                if (!mbar_wait(gfull, jj & 1, err)) { ok = false; break; }
                tc_fence_after();
                for (int h = 0; h < 2; ++h) {
                    if (!mbar_wait(&full[st], ph, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sb = smem_u32(ring + st * C::STAGE_BYTES);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        tc_mma_bf16(tmem + C::ACC_COL,
                                    sdesc_sw128(g_base + h * 16384 + k * 32, 16, 1024),
                                    sdesc_sw128(sb + k * 2048, 8192, 1024), ID_ACC,
                                    first_acc ? 0u : 1u);
                        first_acc = false;
                    }
                    tc_commit(&empty[st]);
                    if (++st == S) { st = 0; ph ^= 1; }
                }
                if (!ok) break;
                tc_commit(gempty);
            }
        }
        if (C::ACC && ok) tc_commit(accfull);
        tc_commit(drain);
        mbar_wait_drain(drain, 0);
    } else if (warp >= 2) {
        // ================= epilogue =================
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const float L2E = static_cast<float>(LOG2E);
        const float kT = a.inv_t_l2e;
        bool ok = true;
        for (int j = 0; j < n_it && ok; ++j) {
            int xrow0, ycol0, yt;
            coords(j, xrow0, ycol0, yt);
            const int b = j & 1;
            ok = mbar_wait(&tfull[b], (j >> 1) & 1, err);
            if (DISTILL && ok) ok = mbar_wait(&thfull[b], (j >> 1) & 1, err);
            if (C::ACC && ok) ok = mbar_wait(gempty, (j & 1) ^ 1, err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const int ncols = min(BN, a.vocab - ycol0);   // valid logit columns (STATS)
            const uint32_t tbuf = trow + b * BN;
            const uint8_t *tt = teach + b * (TC_BM * TC_BN_ACC * 2);

            if (MODE == TC_STATS) {
                const int t = xrow0 + r;
                const bool row_ok = t < a.n_tok;
                if (!DISTILL) {
                    const int rel = row_ok ? static_cast<int>(a.targets[t] - ycol0) : -1;
                    float m2 = -INFINITY, z = 0.f;
#pragma unroll 1
                    for (int q = 0; q < BN / 32; ++q) {
                        if (q * 32 >= ncols) break;
                        uint32_t v[32];
                        tmem_ld32(tbuf + q * 32, v);
                        tmem_ld_wait();
                        float f[32];
                        float cm = -INFINITY;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            f[i] = (q * 32 + i < ncols) ? __uint_as_float(v[i]) * L2E : -INFINITY;
                            cm = fmaxf(cm, f[i]);
                        }
                        if (cm > m2) {
                            z *= ex2_approx(m2 - cm);
                            m2 = cm;
                        }
                        float acc = 0.f;
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc += ex2_approx(f[i] - m2);
                        z += acc;
                        if (rel >= q * 32 && rel < q * 32 + 32) {
                            float tv = 0.f;
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (rel - q * 32 == i) tv = __uint_as_float(v[i]);
                            a.tgt[t] = tv;
                        }
                    }
                    if (row_ok) {
                        const int64_t o = static_cast<int64_t>(yt) * a.part_stride + t;
                        a.part[o] = m2;
                        a.part[a.part_plane + o] = z;
                    }
                } else {
                    float ms = -INFINITY, zs = 0.f, mt = -INFINITY, zt = 0.f, X = 0.f;
                    const int dir = a.direction;
#pragma unroll 1
                    for (int q = 0; q < BN / 32; ++q) {
                        if (q * 32 >= ncols) break;
                        uint32_t v[32];
                        tmem_ld32(tbuf + q * 32, v);
                        tmem_ld_wait();
                        float sa[32], sb[32];
                        const uint8_t *rowp = tt + (q >> 1) * 16384 + r * 128;
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const int phys = (((q & 1) * 4 + c4) ^ (r & 7)) << 4;
                            const uint4 w = *reinterpret_cast<const uint4 *>(rowp + phys);
                            sb[c4 * 8 + 0] = bf16_lo(w.x); sb[c4 * 8 + 1] = bf16_hi(w.x);
                            sb[c4 * 8 + 2] = bf16_lo(w.y); sb[c4 * 8 + 3] = bf16_hi(w.y);
                            sb[c4 * 8 + 4] = bf16_lo(w.z); sb[c4 * 8 + 5] = bf16_hi(w.z);
                            sb[c4 * 8 + 6] = bf16_lo(w.w); sb[c4 * 8 + 7] = bf16_hi(w.w);
                        }
                        float cms = -INFINITY, cmt = -INFINITY;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const bool in = q * 32 + i < ncols;
                            sa[i] = in ? __uint_as_float(v[i]) * kT : -INFINITY;
                            sb[i] = in ? sb[i] * kT : -INFINITY;
                            cms = fmaxf(cms, sa[i]);
                            cmt = fmaxf(cmt, sb[i]);
                        }
                        if (cms > ms) {
                            const float f = ex2_approx(ms - cms);
                            zs *= f;
                            if (dir == DIR_RKL) X *= f;
                            ms = cms;
                        }
                        if (cmt > mt) {
                            const float f = ex2_approx(mt - cmt);
                            zt *= f;
                            if (dir != DIR_RKL) X *= f;
                            mt = cmt;
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            if (q * 32 + i < ncols) {
                                const float es = ex2_approx(sa[i] - ms);
                                const float et = ex2_approx(sb[i] - mt);
                                zs += es;
                                zt += et;
                                if (dir == DIR_CE) X = fmaf(et, sa[i], X);
                                else if (dir == DIR_FKL) X = fmaf(et, sb[i] - sa[i], X);
                                else X = fmaf(es, sa[i] - sb[i], X);
                            }
                        }
                    }
                    if (row_ok) {
                        const int64_t o = static_cast<int64_t>(yt) * a.part_stride + t;
                        a.part[o] = ms;
                        a.part[a.part_plane + o] = zs;
                        a.part[2 * a.part_plane + o] = mt;
                        a.part[3 * a.part_plane + o] = zt;
                        a.part[4 * a.part_plane + o] = X;
                    }
                }
                tc_fence_before();
                mbar_arrive(&tempty[b]);
                if (DISTILL) mbar_arrive(&thempty[b]);
            } else {
                // ---- backward: grad_logits tile -> shared memory (bf16, K-major SW128)
                const int xr = xrow0 + r;
                // parameters of a token past n_tok: zero weight (and no target)
                const float4 P0 = DISTILL ? make_float4(0.f, 0.f, 0.f, 0.f)
                                          : make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
                float4 P = P0;
                if (MODE == TC_ROWS) {
                    if (xr < a.n_tok) P = a.tokp[xr];
                } else {
                    const int tc = ycol0 + r;     // this thread stages column r's token
                    colp[b * TC_BN_ACC + r] = tc < a.n_tok ? a.tokp[tc] : P0;
                    mbar_arrive(&colrdy[b]);
                    ok = mbar_wait(&colrdy[b], (j >> 1) & 1, err);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                }
                const float4 *cp = colp + b * TC_BN_ACC;
                const int rel = (MODE == TC_ROWS) ? __float_as_int(P.w) - ycol0 : 0;
#pragma unroll 1
                for (int q = 0; q < TC_BN_ACC / 32; ++q) {
                    uint32_t v[32];
                    tmem_ld32(tbuf + q * 32, v);
                    tmem_ld_wait();
                    float tv[32];
                    if (DISTILL) {
                        if (MODE == TC_ROWS) {
                            const uint8_t *rowp = tt + (q >> 1) * 16384 + r * 128;
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                const int phys = (((q & 1) * 4 + c4) ^ (r & 7)) << 4;
                                const uint4 w = *reinterpret_cast<const uint4 *>(rowp + phys);
                                tv[c4 * 8 + 0] = bf16_lo(w.x); tv[c4 * 8 + 1] = bf16_hi(w.x);
                                tv[c4 * 8 + 2] = bf16_lo(w.y); tv[c4 * 8 + 3] = bf16_hi(w.y);
                                tv[c4 * 8 + 4] = bf16_lo(w.z); tv[c4 * 8 + 5] = bf16_hi(w.z);
                                tv[c4 * 8 + 6] = bf16_lo(w.w); tv[c4 * 8 + 7] = bf16_hi(w.w);
                            }
                        } else {
                            // element (token row jj of the tile, vocabulary column r)
                            const uint8_t *colbase = tt + (r >> 6) * 16384 + (r & 7) * 2;
                            const int c16 = (r & 63) >> 3;
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int jj = q * 32 + i;
                                const uint16_t h = *reinterpret_cast<const uint16_t *>(
                                    colbase + jj * 128 + ((c16 ^ (jj & 7)) << 4));
                                tv[i] = __uint_as_float(static_cast<uint32_t>(h) << 16);
                            }
                        }
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float g[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int jj = q * 32 + i + u;
                            const float s = __uint_as_float(v[i + u]);
                            const float4 Q = (MODE == TC_ROWS) ? P : cp[jj];
                            if (!DISTILL) {
                                float gv = Q.y * ex2_approx(fmaf(s, L2E, -Q.x));
                                const bool hit = (MODE == TC_ROWS) ? (rel == jj)
                                                                   : (__float_as_int(Q.w) == xr);
                                if (hit) gv -= Q.z;
                                g[u] = gv;
                            } else {
                                const float a2 = s * kT, b2 = tv[i + u] * kT;
                                const float qv = ex2_approx(a2 - Q.x);
                                if (a.direction == DIR_RKL)
                                    g[u] = Q.z * qv * fmaf(a2 - b2, static_cast<float>(LN2), Q.w);
                                else
                                    g[u] = Q.z * qv - Q.w * ex2_approx(b2 - Q.y);
                            }
                        }
                        pk[i >> 1] = pack_bf16x2(g[0], g[1]);
                    }
                    uint8_t *grow = gbuf + (q >> 1) * 16384 + r * 128;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int phys = (((q & 1) * 4 + c4) ^ (r & 7)) << 4;
                        *reinterpret_cast<uint4 *>(grow + phys) =
                            make_uint4(pk[c4 * 4 + 0], pk[c4 * 4 + 1], pk[c4 * 4 + 2], pk[c4 * 4 + 3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(&tempty[b]);
                if (DISTILL) mbar_arrive(&thempty[b]);
                fence_proxy_async_smem();
                mbar_arrive(gfull);
            }
        }
        if (C::ACC && ok) {
            ok = mbar_wait(accfull, 0, err);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const int xr = xt_fixed * TC_BM + r;
                float *dst = a.out +
                             static_cast<int64_t>(blockIdx.x / (a.n_slices * a.n_xt)) * a.out_split_stride +
                             static_cast<int64_t>(xr) * a.d;
#pragma unroll 1
                for (int q = 0; q < TC_SLICE / 32; ++q) {
                    uint32_t v[32];
                    tmem_ld32(trow + C::ACC_COL + q * 32, v);
                    tmem_ld_wait();
                    const int col = slice0 + q * 32;
                    if (xr < a.n_x && col < a.d) {
                        if (col + 32 <= a.d) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4 *>(dst + col + i) =
                                    make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                        } else {
                            for (int i = 0; i < 32; ++i)
                                if (col + i < a.d) dst[col + i] = __uint_as_float(v[i]);
                        }
                    }
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int MODE, bool DISTILL>
static cudaError_t launch_one(const TcArgs &a, int grid, cudaStream_t st)
{
    using C = TcCfg<MODE, DISTILL>;
    auto k = tc_kernel<MODE, DISTILL>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    k<<<grid, 192, C::SMEM_BYTES, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_tc(int mode, bool distill, const TcArgs &a, int grid, cudaStream_t st)
{
    if (mode == TC_STATS) return distill ? launch_one<TC_STATS, true>(a, grid, st)
                                         : launch_one<TC_STATS, false>(a, grid, st);
    if (mode == TC_ROWS) return distill ? launch_one<TC_ROWS, true>(a, grid, st)
                                        : launch_one<TC_ROWS, false>(a, grid, st);
    return distill ? launch_one<TC_COLS, true>(a, grid, st) : launch_one<TC_COLS, false>(a, grid, st);
}

} // namespace lossk
