// k_bwd.cu -- the backward passes of the fused LM-head loss on tcgen05, with
// each recomputed grad_logits tile shared across a thread-block cluster.
//
// d_hidden = G W and d_weight = G^T H need a [128 x d_model] fp32 accumulator
// per tile, wider than tensor memory (512 columns).  So the accumulator is
// split into 256-column d-slices, one per CTA of a cluster of c CTAs.  A unit
// of work is one "fixed" tile (token tile for d_hidden, vocabulary tile for
// d_weight) with a range of "loop" tiles; every CTA of the cluster walks the
// same loop tiles.  Loop tile y's logits S = H_tok . W_voc^T (token rows x
// vocabulary columns, contraction over the whole d_model) are computed once,
// by CTA y % c; its epilogue turns them into grad_logits G (bf16) -- "Fuse
// distillation + z-loss ...", "What it does": prob_coeff * softmax -
// label_coeff * onehot, with the z term folded into prob_coeff, or the
// distribution-family form -- writes G into grad slot y % R of its own shared
// memory and pushes it to the other CTAs with bulk shared-to-distributed-
// shared copies.  Every CTA then adds G times its d-slice of the loop tile
// into its accumulator:
//   d_hidden (BWD_ROWS): D[tok][slice] += G[tok][voc] . W[voc][slice]  (A = G, K-major)
//   d_weight (BWD_COLS): D[voc][slice] += G^T[voc][tok] . H[tok][slice] (A = G, MN-major)
// A grad slot is reused once every CTA's MMA has consumed it: each CTA's
// tcgen05.commit arrives (multicast) on the slot barrier of the CTA that fills
// the slot next.
//
// The clusters are persistent: each walks units u, u + #clusters, ... with the
// TMA ring, the TMEM logit buffers and the grad-slot phases carried across
// units, so a unit's last accumulate round overlaps the next unit's first
// logit tile and the accumulator store of one unit overlaps the next unit's
// logits.  An "emptied" barrier keeps the next unit's first accumulate from
// overwriting the accumulator before the epilogue has stored it.
//
// BWD_FUSED is the d_hidden schedule run as the forward pass too, before any
// log-sum-exp is known.  Its grad tile is the unnormalised
//   G'[t][v] = 2^(s[t][v] log2e - r_t),   r_t = s[t][y_t] log2e + 64,
// a per-token reference shift fixed before the pass (the target logit lies at
// or below the row maximum, so the largest term of a row is at least 2^-64 and
// nothing that matters underflows).  Each CTA also sums G' over the valid
// vocabulary columns of its own loop tiles (per tile in fp32, across tiles in
// fp64) and writes that sum per (split, CTA, token).  With Z_t the sum of
// those partials, p = G'/Z_t, lse_t = (r_t + log2 Z_t) ln 2 and
//   d_hidden_t = a_t (1 + 2 w_z lse_t) D_t / Z_t - a_t W[y_t],
// which a later kernel applies; that kernel, not this one, also detects a row
// whose shifted terms left the safe range.
//
// Roles per CTA (192 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 2-5 epilogue (one token row per thread).  TMEM: two 128-column
// logit buffers and the 256-column accumulator.  Every wait is bounded.
#include "lossk_internal.h"
#include "ptx.cuh"

namespace lossk {

template <bool DISTILL> struct BwdCfg {
    static constexpr int BN = 128;                  // loop-tile rows per logit tile
    static constexpr int STAGE_BYTES = 32768;       // X+Y k-slices, or 64 rows x 256-column slice
    // One grad slot per CTA of a 4-CTA cluster: with fewer slots, the grad tile
    // of a loop tile waits for the accumulate of another tile of the same
    // round in every CTA, which serialises each round.  That leaves room for
    // three 32 KB ring stages.
    static constexpr int STAGES = 3;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int G_TILE = 32768;            // 128 x 128 bf16
    static constexpr int R_MAX = 4;                 // grad slots
    static constexpr int G_BYTES = R_MAX * G_TILE;
    // Teacher logits are read by the epilogue straight from global memory (one
    // contiguous 256-byte row segment per thread and tile), so they take no
    // shared memory.
    static constexpr int NBARS = 2 * STAGES + 2 + 2 + 2 + 2 * R_MAX + 1;
    static constexpr int SMEM_BYTES = 1024 + RING_BYTES + G_BYTES + NBARS * 8 + 16;
    static_assert(SMEM_BYTES <= 232448, "fits the 227 KB per-CTA shared memory limit");
};

__device__ __forceinline__ float bw_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bw_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void bw_wait_drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 200000000ull) return;
}

// One unit of work: a fixed tile, a d-group and a range of loop tiles.
struct BwdUnit {
    int fixed, dg, yt_begin, ny;
};

__device__ __forceinline__ BwdUnit bwd_unit(const BwdArgs &a, int u)
{
    BwdUnit w;
    w.dg = u % a.n_dg;
    u /= a.n_dg;
    w.fixed = u % a.n_fixed;
    const int split = u / a.n_fixed;
    w.yt_begin = static_cast<int>((static_cast<int64_t>(split) * a.n_loop) / a.n_split);
    const int yt_end = static_cast<int>((static_cast<int64_t>(split + 1) * a.n_loop) / a.n_split);
    w.ny = yt_end - w.yt_begin;
    return w;
}

// Position in this cluster's schedule: unit u (the k-th of the cluster), round r
// of its nr rounds of c loop tiles.
struct BwdCursor {
    int u, k, r, nr;
    BwdUnit w;
};

template <int MODE, bool DISTILL>
__global__ void __launch_bounds__(192, 1) bwd_kernel(const __grid_constant__ BwdArgs a)
{
    using C = BwdCfg<DISTILL>;
    constexpr bool FUSED = MODE == BWD_FUSED;
    constexpr bool ROWS = MODE != BWD_COLS;     // the token tile is the fixed one
    static_assert(!(FUSED && DISTILL), "the fused pass is label cross-entropy only");
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem;
    uint8_t *gbuf = ring + C::RING_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(gbuf + C::G_BYTES);
    uint64_t *full = bars;                 // [S]
    uint64_t *empty = full + S;            // [S]
    uint64_t *tfull = empty + S;           // [2]  logit tile ready in TMEM buffer
    uint64_t *tempty = tfull + 2;          // [2]  epilogue done with TMEM buffer
    uint64_t *accfull = tempty + 2;        // accumulator of a unit final
    uint64_t *accempty = accfull + 1;      // accumulator of a unit stored
    uint64_t *gfull = accempty + 1;        // [R_MAX] grad slot filled (4 warp arrivals + bytes)
    uint64_t *gempty = gfull + C::R_MAX;   // [R_MAX] grad slot consumed by every CTA (c arrivals)
    uint64_t *drain = gempty + C::R_MAX;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *err = a.err;
    const int c = a.n_cl, R = a.g_slots;
    const int crank = static_cast<int>(cluster_ctarank());
    const int cluster = blockIdx.x / c, n_clusters = gridDim.x / c;
    const int n_units = a.n_fixed * a.n_split * a.n_dg;
    const int s_own = crank % R;                           // this CTA's grad slot
    auto tile_origin = [&](const BwdUnit &w, int y, int &tok0, int &voc0) {
        const int t = w.yt_begin + y;
        if (ROWS) { tok0 = w.fixed * 128; voc0 = t * 128; }
        else { voc0 = w.fixed * 128; tok0 = t * 128; }
    };
    // Step i of the schedule issues round i's own logit tile and the
    // accumulates of round i-1 (possibly of the previous unit).
    auto cursor_set = [&](BwdCursor &cu, int u, int k) {
        cu.u = u;
        cu.k = k;
        cu.r = 0;
        cu.nr = 0;
        if (u < n_units) {
            cu.w = bwd_unit(a, u);
            cu.nr = (cu.w.ny + c - 1) / c;
        }
    };
    auto cursor_next = [&](BwdCursor &cu) {
        if (++cu.r >= cu.nr) cursor_set(cu, cu.u + n_clusters, cu.k + 1);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 128);
        }
        mbar_init(accfull, 1);
        mbar_init(accempty, 128);
        for (int s = 0; s < C::R_MAX; ++s) {
            mbar_init(&gfull[s], 4);
            mbar_init(&gempty[s], c);
        }
        mbar_init(drain, 1);
        fence_mbarrier_init();
    }
    if (warp == 1) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    cluster_sync();            // every CTA's barriers exist before any remote arrive or copy
    tc_fence_after();
    const uint32_t tmem = *tslot;
    constexpr uint32_t ACC_COL = 256;
    const int nk = (a.d + TC_BK - 1) / TC_BK;

    if (warp == 0 && lane == 0) {
        // ================= TMA producer =================
        tma_prefetch_desc(&a.map_h);
        tma_prefetch_desc(&a.map_w);
        tma_prefetch_desc(&a.map_ys);
        int st = 0;
        uint32_t ph = 0, issued = 0, last_ph = 0;
        bool ok = true;
        auto acquire = [&]() -> uint8_t * {
            if (!mbar_wait(&empty[st], ph ^ 1, err)) return nullptr;
            mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
            issued |= 1u << st;
            last_ph = (last_ph & ~(1u << st)) | (ph << st);
            return ring + st * C::STAGE_BYTES;
        };
        auto advance = [&]() {
            if (++st == S) { st = 0; ph ^= 1; }
        };
        BwdCursor cur, prev;
        cursor_set(cur, cluster, 0);
        bool have_prev = false;
        while (ok && (cur.u < n_units || have_prev)) {
            if (cur.u < n_units) {
                const int y = cur.r * c + crank;
                if (y < cur.w.ny) {
                    int tok0, voc0;
                    tile_origin(cur.w, y, tok0, voc0);
                    for (int kb = 0; kb < nk; ++kb) {
                        uint8_t *sp = acquire();
                        if (!sp) { ok = false; break; }
                        tma_load_2d(sp, &a.map_h, &full[st], kb * TC_BK, tok0);
                        tma_load_2d(sp + 16384, &a.map_w, &full[st], kb * TC_BK, voc0);
                        advance();
                    }
                    if (!ok) break;
                }
            }
            if (have_prev) {
                const int slice0 = (prev.w.dg * c + crank) * TC_SLICE;
                const int y_end = min((prev.r + 1) * c, prev.w.ny);
                for (int yy = prev.r * c; yy < y_end && ok; ++yy) {
                    int tok0, voc0;
                    tile_origin(prev.w, yy, tok0, voc0);
                    const int row0 = ROWS ? voc0 : tok0;
                    for (int h = 0; h < 2; ++h) {
                        uint8_t *sp = acquire();
                        if (!sp) { ok = false; break; }
                        for (int q = 0; q < 4; ++q)
                            tma_load_2d(sp + q * 8192, &a.map_ys, &full[st], slice0 + q * 64,
                                        row0 + h * 64);
                        advance();
                    }
                }
            }
            have_prev = cur.u < n_units;
            prev = cur;
            if (cur.u < n_units) cursor_next(cur);
        }
        for (int s = 0; s < S; ++s)
            if (issued & (1u << s)) bw_wait_drain(&full[s], (last_ph >> s) & 1);
    } else if (warp == 1 && lane == 0) {
        // ================= MMA issuer =================
        constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);
        constexpr uint32_t ID_ACC = idesc_bf16_f32(128, TC_SLICE, MODE == BWD_COLS ? 1 : 0, 1);
        int st = 0;
        uint32_t ph = 0;
        bool ok = true, first_acc = true;
        int m_all = 0;                         // own logit tiles issued so far (TMEM buffer index)
        int use[4] = {0, 0, 0, 0};             // completed uses of each grad slot
        BwdCursor cur, prev;
        cursor_set(cur, cluster, 0);
        bool have_prev = false;
        while (ok && (cur.u < n_units || have_prev)) {
            if (cur.u < n_units) {
                const int y = cur.r * c + crank;
                if (y < cur.w.ny) {
                    const int b = m_all & 1;
                    if (!mbar_wait(&tempty[b], ((m_all >> 1) & 1) ^ 1, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_s = tmem + b * 128;
                    for (int kb = 0; kb < nk; ++kb) {
                        if (!mbar_wait(&full[st], ph, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t sa = smem_u32(ring + st * C::STAGE_BYTES);
#pragma unroll
                        for (int k = 0; k < TC_BK / 16; ++k)
                            tc_mma_bf16(d_s, sdesc_sw128(sa + k * 32, 16, 1024),
                                        sdesc_sw128(sa + 16384 + k * 32, 16, 1024), ID_S, (kb | k) != 0);
                        tc_commit(&empty[st]);
                        if (++st == S) { st = 0; ph ^= 1; }
                    }
                    if (!ok) break;
                    tc_commit(&tfull[b]);
                    ++m_all;
                }
            }
            if (have_prev) {
                if (prev.r == 0) {
                    // first accumulate of a unit: the previous unit's accumulator must be stored
                    if (!mbar_wait(accempty, (prev.k & 1) ^ 1, err)) { ok = false; break; }
                    tc_fence_after();
                    first_acc = true;
                }
                const bool last_round = prev.r == prev.nr - 1;
                // Loop tiles of this cluster's next unit, for the slot hand-over at the
                // end of this one.  The last tile of a slot can sit in the round
                // before the last (when ny is not a multiple of the slot count), so
                // this is needed in every round, not only the last.
                int ny_next = 0;
                if (prev.u + n_clusters < n_units) ny_next = bwd_unit(a, prev.u + n_clusters).ny;
                const int y_end = min((prev.r + 1) * c, prev.w.ny);
                for (int yy = prev.r * c; yy < y_end && ok; ++yy) {
                    const int s = yy % R;
                    int par = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q == s) par = use[q] & 1;
                    if (!mbar_wait(&gfull[s], par, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t g_base = smem_u32(gbuf + s * C::G_TILE);
                    for (int h = 0; h < 2; ++h) {
                        if (!mbar_wait(&full[st], ph, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t sb = smem_u32(ring + st * C::STAGE_BYTES);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint64_t adesc;
                            if (ROWS)               // K = vocabulary columns of G
                                adesc = sdesc_sw128(g_base + h * 16384 + k * 32, 16, 1024);
                            else                    // K = token rows of G, M = vocabulary (MN-major)
                                adesc = sdesc_sw128(g_base + h * 8192 + k * 2048, 16384, 1024);
                            tc_mma_bf16(tmem + ACC_COL, adesc, sdesc_sw128(sb + k * 2048, 8192, 1024),
                                        ID_ACC, first_acc ? 0u : 1u);
                            first_acc = false;
                        }
                        tc_commit(&empty[st]);
                        if (++st == S) { st = 0; ph ^= 1; }
                    }
                    if (!ok) break;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q == s) ++use[q];
                    // Slot s is filled next by CTA (yy + R) % c of this unit or, after the
                    // unit's last tile in the slot, by CTA s in this cluster's next unit.
                    int target = -1;
                    if (yy + R < prev.w.ny) target = (yy + R) % c;
                    else if (s < ny_next) target = s;
                    if (target >= 0) tc_commit_multicast(&gempty[s], static_cast<uint16_t>(1u << target));
                }
                if (!ok) break;
                if (last_round) tc_commit(accfull);
            }
            have_prev = cur.u < n_units;
            prev = cur;
            if (cur.u < n_units) cursor_next(cur);
        }
        tc_commit(drain);
        bw_wait_drain(drain, 0);
    } else if (warp >= 2) {
        // ================= epilogue =================
        const int quad = warp & 3;
        const int r = quad * 32 + lane;               // token row of the logit tile
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const float L2E = static_cast<float>(LOG2E);
        const float kT = a.inv_t_l2e;
        const float4 P0 = DISTILL ? make_float4(0.f, 0.f, 0.f, 0.f)
                                  : make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
        uint8_t *gslot = gbuf + s_own * C::G_TILE;
        bool ok = true;
        int m_all = 0;                                // own logit tiles consumed so far
        int gwait = 0;                                // slot hand-overs waited for so far
        int ny_prev = 0;                              // loop tiles of this cluster's previous unit
        for (int k = 0, u = cluster; u < n_units && ok; ++k, u += n_clusters) {
            const BwdUnit w = bwd_unit(a, u);
            const int n_own = crank < w.ny ? (w.ny - crank + c - 1) / c : 0;
            float4 P = P0;
            double zsum = 0.0;                        // fused pass: this CTA's sum of G' for its row
            if (ROWS) {                               // the token tile is fixed
                const int t = w.fixed * 128 + r;
                if (t < a.n_tok) P = a.tokp[t];
            }
            for (int m = 0; m < n_own && ok; ++m, ++m_all) {
                const int y = m * c + crank;
                int tok0, voc0;
                tile_origin(w, y, tok0, voc0);
                if (MODE == BWD_COLS) {
                    const int t = tok0 + r;
                    P = t < a.n_tok ? a.tokp[t] : P0;
                }
                const int b = m_all & 1;
                ok = mbar_wait(&tfull[b], (m_all >> 1) & 1, err);
                // Teacher row segment teacher[token][voc0 .. voc0+127] of this thread:
                // 16-byte loads, each chunk fetched one chunk ahead of its use.
                const int tok = tok0 + r;
                const bool trow_ok = DISTILL && tok < a.n_tok;
                const uint4 *tsrc = DISTILL ? reinterpret_cast<const uint4 *>(
                                                  a.teacher + static_cast<int64_t>(trow_ok ? tok : 0) * a.vocab + voc0)
                                            : nullptr;
                const int tvalid = min(128, a.vocab - voc0);   // columns of this tile inside the vocabulary
                auto tload = [&](int q, uint4 (&tw)[4]) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        tw[c4] = (trow_ok && q * 32 + c4 * 8 < tvalid) ? __ldg(tsrc + q * 4 + c4)
                                                                       : make_uint4(0, 0, 0, 0);
                };
                uint4 tw[4] = {};
                if (DISTILL) tload(0, tw);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                const int rel = DISTILL ? 0 : __float_as_int(P.w) - voc0;
                const uint32_t tbuf = trow + b * 128;
                uint32_t pk[64];
                float zt = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t v[32];
                    tmem_ld32(tbuf + q * 32, v);
                    float tv[32];
                    if (DISTILL) {
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            tv[c4 * 8 + 0] = bw_lo(tw[c4].x); tv[c4 * 8 + 1] = bw_hi(tw[c4].x);
                            tv[c4 * 8 + 2] = bw_lo(tw[c4].y); tv[c4 * 8 + 3] = bw_hi(tw[c4].y);
                            tv[c4 * 8 + 4] = bw_lo(tw[c4].z); tv[c4 * 8 + 5] = bw_hi(tw[c4].z);
                            tv[c4 * 8 + 6] = bw_lo(tw[c4].w); tv[c4 * 8 + 7] = bw_hi(tw[c4].w);
                        }
                        if (q < 3) tload(q + 1, tw);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float g[2];
#pragma unroll
                        for (int uu = 0; uu < 2; ++uu) {
                            const float s = __uint_as_float(v[i + uu]);
                            if (FUSED) {
                                const float gv = ex2_approx(fmaf(s, L2E, -P.x));
                                g[uu] = gv;
                                zt += (q * 32 + i + uu < tvalid) ? gv : 0.f;
                            } else if (!DISTILL) {
                                float gv = P.y * ex2_approx(fmaf(s, L2E, -P.x));
                                if (rel == q * 32 + i + uu) gv -= P.z;
                                g[uu] = gv;
                            } else {
                                const float a2 = s * kT, b2 = tv[i + uu] * kT;
                                const float qv = ex2_approx(a2 - P.x);
                                if (a.direction == DIR_RKL)
                                    g[uu] = P.z * qv * fmaf(a2 - b2, static_cast<float>(LN2), P.w);
                                else
                                    g[uu] = P.z * qv - P.w * ex2_approx(b2 - P.y);
                            }
                        }
                        pk[q * 16 + (i >> 1)] = pack_bf16x2(g[0], g[1]);
                    }
                }
                if (FUSED) zsum += static_cast<double>(zt);
                // the tile is in registers: give the TMEM buffer back
                tc_fence_before();
                mbar_arrive(&tempty[b]);
                // The grad slot must be free in every CTA: wait for the consumption of
                // the previous tile in this slot -- tile y - R of this unit, or for
                // the first tiles (y < R) the previous unit's last tile in the slot.
                const bool has_pred = y >= R || (k > 0 && ny_prev > s_own);
                if (has_pred) {
                    ok = mbar_wait(&gempty[s_own], gwait & 1, err);
                    ++gwait;
                }
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint8_t *grow = gslot + (q >> 1) * 16384 + r * 128;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int phys = (((q & 1) * 4 + c4) ^ (r & 7)) << 4;
                        *reinterpret_cast<uint4 *>(grow + phys) =
                            make_uint4(pk[q * 16 + c4 * 4 + 0], pk[q * 16 + c4 * 4 + 1],
                                       pk[q * 16 + c4 * 4 + 2], pk[q * 16 + c4 * 4 + 3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // this warp's 32 rows: 4 KB in each of the two 64-column blocks
                    mbar_arrive(&gfull[s_own]);
                    const uint32_t src0 = smem_u32(gslot) + quad * 32 * 128;
                    const uint32_t bar_local = smem_u32(&gfull[s_own]);
                    for (int qq = 1; qq < c; ++qq) {
                        const uint32_t dst = static_cast<uint32_t>((crank + qq) % c);
                        const uint32_t rbar = mapa_shared(bar_local, dst);
                        mbar_arrive_expect_tx_remote(rbar, 8192);
                        bulk_copy_s2cluster(mapa_shared(src0, dst), src0, 4096, rbar);
                        bulk_copy_s2cluster(mapa_shared(src0 + 16384, dst), src0 + 16384, 4096, rbar);
                    }
                }
            }
            if (!ok) break;
            if (FUSED && w.dg == 0) {
                // every d-group recomputes the same logits; the first one reports the sums
                const int t = w.fixed * 128 + r;
                const int split = u / (a.n_fixed * a.n_dg);
                if (t < a.n_tok)
                    a.zpart[(static_cast<int64_t>(split) * c + crank) * a.zpart_stride + t] =
                        static_cast<float>(zsum);
            }
            // the unit's accumulator: store this CTA's rows of its d-slice
            ok = mbar_wait(accfull, k & 1, err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const int slice0 = (w.dg * c + crank) * TC_SLICE;
            const int row = w.fixed * 128 + r;        // token (ROWS) or vocabulary (COLS) row
            const int n_rows = ROWS ? a.n_tok : a.vocab;
            const int split = u / (a.n_fixed * a.n_dg);
            float *dst = a.out + static_cast<int64_t>(split) * a.out_split_stride +
                         static_cast<int64_t>(row) * a.d;
            // Two 32-column chunks per TMEM wait; full chunks leave as 32-byte
            // stores (rows are d_model floats apart, d_model % 8 == 0, so every
            // chunk start is 32-byte aligned).
#pragma unroll 1
            for (int q = 0; q < TC_SLICE / 32; q += 2) {
                uint32_t v[2][32];
                tmem_ld32(trow + ACC_COL + q * 32, v[0]);
                tmem_ld32(trow + ACC_COL + (q + 1) * 32, v[1]);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int col = slice0 + (q + h) * 32;
                    if (row < n_rows && col < a.d) {
                        if (col + 32 <= a.d) {
#pragma unroll
                            for (int i = 0; i < 32; i += 8) st_global_v8(dst + col + i, &v[h][i]);
                        } else {
                            for (int i = 0; i < 32; ++i)
                                if (col + i < a.d) dst[col + i] = __uint_as_float(v[h][i]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(accempty);
            ny_prev = w.ny;
        }
        tc_fence_before();
    }
    __syncthreads();
    // No CTA leaves while another may still copy into, or arrive on, its shared memory.
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int MODE, bool DISTILL>
static cudaError_t launch_bwd_one(const BwdArgs &a, int n_units, cudaStream_t st)
{
    using C = BwdCfg<DISTILL>;
    auto k = bwd_kernel<MODE, DISTILL>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.n_cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // As many clusters as fit at once, each walking several units; the results
    // do not depend on the count, only the schedule does.
    cfg.gridDim = dim3(n_units * a.n_cl, 1, 1);
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, k, &cfg) != cudaSuccess || active < 1) {
        (void)cudaGetLastError();
        active = n_units;
    }
    const int clusters = active < n_units ? active : n_units;
    cfg.gridDim = dim3(clusters * a.n_cl, 1, 1);
    return cudaLaunchKernelEx(&cfg, k, a);
}

cudaError_t launch_bwd(int mode, bool distill, const BwdArgs &a, int n_units, cudaStream_t st)
{
    if (mode == BWD_FUSED) return launch_bwd_one<BWD_FUSED, false>(a, n_units, st);
    if (mode == BWD_ROWS)
        return distill ? launch_bwd_one<BWD_ROWS, true>(a, n_units, st) : launch_bwd_one<BWD_ROWS, false>(a, n_units, st);
    return distill ? launch_bwd_one<BWD_COLS, true>(a, n_units, st) : launch_bwd_one<BWD_COLS, false>(a, n_units, st);
}

} // namespace lossk
