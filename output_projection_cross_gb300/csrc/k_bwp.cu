// k_bwp.cu -- the backward passes of the fused LM-head loss (and the training
// step's fused forward + d_hidden pass) on CTA pairs: every MMA is one
// tcgen05 cta_group::2 unit of two CTAs, 256 fixed rows x 256 columns, each
// CTA holding its own 128 fixed rows of A and half (128 rows or columns) of
// B.  Per ring stage of 512 MMA clocks an SM then takes in 32 KB of operands
// instead of the 48 KB a single CTA's 128 x 256 tile needs; these passes are
// bound by operand bytes from L2 into the SMs.
//
// d_hidden = G W and d_weight = G^T H need a [rows x d_model] fp32 accumulator
// per fixed tile, wider than tensor memory (512 columns).  So the accumulator
// is split into 256-column d-slices, one per CTA pair of a group of c pairs
// (2c consecutive blocks of the grid).  A unit of work is one fixed tile (256
// tokens for d_hidden, 256 vocabulary rows for d_weight), one d-group and a
// range of loop supertiles of 256 columns (vocabulary for d_hidden, tokens for
// d_weight).  Every pair of the group walks the same supertiles; supertile y's
// logits -- the whole d_model contraction, one 256 x 256 pair tile -- are
// computed once, by pair y % c.  Each CTA's epilogue turns its 128 rows into
// grad_logits G in registers ("Fuse distillation + z-loss ...", "What it
// does": prob_coeff * softmax - label_coeff * onehot, with the z term folded
// into prob_coeff, or the distribution-family form), stores the bf16 half
// tile into one of that CTA's slots of a global ring that stays in L2 (each
// warp stages 32 x 32 chunks in shared memory and stores them with TMA), and
// signals the CTAs of the same parity in every pair of the group.  Those load
// it with TMA like any other operand and the pair adds G times its d-slice of
// the loop tensor into its accumulator:
//   d_hidden: D[tok][slice] += G[tok][voc] . W[voc][slice]
//   d_weight: D[voc][slice] += G^T[voc][tok] . H[tok][slice]
// In both the MMA's A operand is the stored tile (K-major: the d_weight pass
// computes its logits transposed, vocabulary rows x token columns) and B is
// the loop tensor's rows x d-slice (MN-major), 128 slice columns per CTA.
//
// Ring hand-over (per CTA, G_SLOTS slots of one half supertile each), through
// two monotonic counters per slot in global memory (the workspace; zeroed
// before each launch): the writer waits until the slot's free count shows
// that every pair of the group has loaded the slot's previous tile (one
// relaxed add per loading pair, from its MMA issuer once both halves of the
// stage have landed: it announces completed reads and never holds the
// issuer), writes, waits for its TMA stores to complete, fences and adds to
// the slot's ready count (one release add per epilogue warp: they publish the
// tile); a loader CTA's poller warp waits for the ready count (acquire) and
// passes it to the CTA's TMA producer in shared memory, which then loads the
// tile.  Groups are not clusters: only the two CTAs of a pair form a
// cluster (cta_group::2 needs one), and a group's pairs wait on each other
// through global memory, which is safe as the grid never holds more pairs
// than fit at once (every CTA of the grid is resident).  Groups of 4 pairs
// fill all 152 SMs of a GB300.
//
// BWD_FUSED is the d_hidden schedule run before any log-sum-exp is known: its
// grad tile is the unnormalised G'[t][v] = 2^(s[t][v] log2e - r_t) with the
// per-token reference shift r_t = s[t][y_t] log2e + 64 fixed before the pass
// (the target logit lies at or below the row maximum, so a row's largest term
// is at least 2^-64 and nothing that matters underflows).  Each CTA also sums
// G' over the valid vocabulary columns of its own supertiles (per supertile in
// fp32, across supertiles in fp64) and writes one sum per (split, pair, token).
// With Z_t the sum of those partials, p = G'/Z_t, lse_t = (r_t + log2 Z_t) ln 2
// and d_hidden_t = a_t (1 + 2 w_z lse_t) D_t / Z_t - a_t W[y_t], which a later
// kernel applies and checks.
//
// The groups are persistent: each walks units u, u + #groups, ... with the
// TMA ring, the TMEM logit buffer and the ring slots' counts carried across
// units.  Step i of the schedule issues round i's own logit tile and the
// accumulates of round i-1 (possibly of the previous unit).
//
// Roles per CTA (224 threads): warp 0 loads this CTA's operand halves with TMA
// (counted on the even CTA's stage barrier), warp 1 owns the pair's tensor
// memory and, in the even CTA, issues the pair's MMAs; warps 2-5 are the
// epilogue (one logit-tile row per thread); warp 6 watches the group's publish
// counts in global memory ahead of the loader and hands each writer's count to
// it in shared memory, so the L2 round trip of that check is off the loader's
// path (it otherwise held the MMAs up at the first stage of every grad tile
// but a round's first).  TMEM per CTA: one 256-column
// logit buffer and the 256-column accumulator.  Every wait is bounded.
#include "lossk_internal.h"
#include "ptx.cuh"

#include <atomic>

namespace lossk {

namespace {

constexpr int B_NST = 6;                          // operand ring stages
constexpr int B_STAGE = 32768;                    // this CTA's halves: an A part and a B part
constexpr int B_APART = 16384;                    // 128 rows x 64 K (bf16, 128-byte swizzle)
constexpr int B_MAXC = BWD_MAX_CL;                // pairs per group at most
constexpr int B_NBARS = 2 * B_NST + 4 + 1 + 8;
// The distillation d_weight pass reads its teacher block through TMA: per
// epilogue warp two 32-token x 32-vocabulary bf16 buffers (2 KB each).
// The plain d_weight pass uses the same 16 KB (four 1024-byte-aligned 4 KB
// blocks) to stage each epilogue warp's 32 x 32 fp32 block of the accumulator
// for a TMA store.
constexpr int B_TBLK = 32 * 32 * 2;
constexpr int B_TEACH = 4 * 2 * B_TBLK;
constexpr int B_STG = 32 * 32 * 4;
static_assert(4 * B_STG == B_TEACH, "the staging blocks fill the teacher-block region");
template <int MODE, bool DISTILL> constexpr int bwd_smem()
{
    return 1024 + B_NST * B_STAGE + 4 * BWD_BN * 16 + (MODE == BWD_COLS ? B_TEACH : 0) + B_NBARS * 8 + 16 +
           4 * B_MAXC;
}
static_assert(bwd_smem<BWD_COLS, true>() <= 232448, "fits the 227 KB per-CTA shared memory limit");
static_assert(B_NST <= 8, "stage masks fit a byte");
static_assert(BWD_BN == 256 && TC_SLICE == 256, "one 256-column logit buffer + one 256-column accumulator");
static_assert(TC_BK == 64, "a ring stage holds four K steps of 16");


__device__ __forceinline__ void bw_wait_drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 200000000ull) return;
}

// One unit of work: a fixed tile, a d-group and a range of loop supertiles.
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

// Position in this group's schedule: unit u (the k-th of the group), round r
// of its nr rounds of c supertiles.
struct BwdCursor {
    int u, k, r, nr;
    BwdUnit w;
};

// Per-writer counters indexed by a run-time CTA rank, kept in registers.
__device__ __forceinline__ int cnt_get(const int (&cnt)[B_MAXC], int i)
{
    int v = 0;
#pragma unroll
    for (int q = 0; q < B_MAXC; ++q)
        if (q == i) v = cnt[q];
    return v;
}
__device__ __forceinline__ void cnt_inc(int (&cnt)[B_MAXC], int i)
{
#pragma unroll
    for (int q = 0; q < B_MAXC; ++q)
        if (q == i) ++cnt[q];
}

} // namespace

// F16: fp16 operands (hidden, weight, teacher).  The grad tile then holds
// G / out_scale (every per-token coefficient without the common factor
// grad_scale / N_valid, so it stays inside fp16's range) and the accumulator
// is multiplied by out_scale when it is stored.
constexpr int B_THREADS = 224;
template <int MODE, bool DISTILL, bool F16>
__global__ void __launch_bounds__(B_THREADS, 1) bwp_kernel(const __grid_constant__ BwdArgs a)
{
    constexpr bool FUSED = MODE == BWD_FUSED;
    constexpr bool ROWS = MODE != BWD_COLS;     // token rows x vocabulary columns
    static_assert(!(FUSED && DISTILL), "the fused pass is label cross-entropy only");
    // Queued behind a validation that found a target out of range: every CTA
    // leaves before it touches anything (a refused call writes no output).
    if (a.refused && *reinterpret_cast<const volatile int *>(a.refused)) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem;
    // d_weight: per-token parameters of a supertile's columns, one copy per epilogue warp
    float4 *sPall = reinterpret_cast<float4 *>(ring + B_NST * B_STAGE);
    constexpr bool TTMA = MODE == BWD_COLS && DISTILL;     // teacher blocks through TMA
    // the accumulator staged for TMA stores (in the distillation pass through the
    // warp's teacher buffers, which hold nothing between tiles)
    constexpr bool STG = MODE == BWD_COLS;
    constexpr bool GSTG = !TTMA;                           // grad tiles staged for TMA stores
    static_assert(4 * BWD_BN * 16 == 4 * B_STG, "the parameter region holds four staging blocks");
    uint8_t *tblk = reinterpret_cast<uint8_t *>(sPall + 4 * BWD_BN);   // [4 warps][2][32][32] bf16
    uint64_t *bars = reinterpret_cast<uint64_t *>(tblk + (MODE == BWD_COLS ? B_TEACH : 0));
    uint64_t *full = bars;                 // [B_NST] even CTA's: both CTAs' bytes landed
    uint64_t *empty = full + B_NST;        // [B_NST] each CTA's: the pair's MMAs are done with the stage
    uint64_t *tfull = empty + B_NST;       // each CTA's: its logit rows are in TMEM
    uint64_t *tempty = tfull + 1;          // even CTA's: both epilogues done with the logit buffer (8 warps)
    uint64_t *accfull = tempty + 1;        // each CTA's: the unit's accumulator is final
    uint64_t *accempty = accfull + 1;      // even CTA's: both epilogues stored the accumulator (8 warps)
    uint64_t *drain = accempty + 1;
    uint64_t *tbar = drain + 1;            // [4 warps][2] teacher block landed (TTMA)
    uint32_t *tslot = reinterpret_cast<uint32_t *>(tbar + 8);
    uint32_t *gseen = tslot + 4;           // [B_MAXC] tiles of each writer seen published (the poller's)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *err = a.err;
    const int c = a.n_cl;                                  // pairs per group
    const int hh = static_cast<int>(cluster_ctarank());    // 0: even CTA (MMA issuer), 1: odd
    const bool lead = hh == 0;
    const int pid = blockIdx.x >> 1;                       // this pair
    const int crank = pid % c;                             // this pair's place in its group
    const int group = pid / c, n_groups = (gridDim.x >> 1) / c;   // the group and the group count
    const int pbase = pid - crank;                         // first pair of this group
    // the CTA of parity hh in pair wr of this group (the writer of the tiles this CTA loads)
    auto wcta = [&](int wr) { return 2 * (pbase + wr) + hh; };
    // per (CTA, slot): tiles published (4 per tile) and loads completed (c per tile)
    unsigned *const gready = a.gsig;
    unsigned *const gfree = a.gsig + G_MAX_CTAS * G_SLOTS;
    const int n_units = a.n_fixed * a.n_split * a.n_dg;
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
        if (++cu.r >= cu.nr) cursor_set(cu, cu.u + n_groups, cu.k + 1);
    };
    // First row of slot g of grid CTA `cta` in the global grad-tile array
    // (a slot holds two 128 x 128 sub-tiles).
    auto slot_row = [&](int cta, int g) { return (cta * G_SLOTS + g) * 2 * 128; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < B_NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, 8);
        mbar_init(accfull, 1);
        mbar_init(accempty, 8);
        mbar_init(drain, 1);
        for (int i = 0; i < 8; ++i) mbar_init(&tbar[i], 1);
        for (int i = 0; i < B_MAXC; ++i) gseen[i] = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) tmem_alloc_pair(tslot, 512);
    tc_fence_before();
    __syncthreads();
    cluster_sync();            // the even CTA's barriers exist before the odd CTA's copies count on them
    tc_fence_after();
    const uint32_t tmem = *tslot;
    constexpr uint32_t ACC_COL = 256;
    const int nk = (a.d + TC_BK - 1) / TC_BK;

    if (warp == 0 && lane == 0) {
        // ================= TMA producer =================
        tma_prefetch_desc(&a.map_fix);
        tma_prefetch_desc(&a.map_loop);
        tma_prefetch_desc(&a.map_ys);
        tma_prefetch_desc(&a.map_g);
        int st = 0;
        uint32_t ph = 0, issued = 0, last_ph = 0;
        bool ok = true;
        int cnt[B_MAXC] = {};                  // tiles loaded so far, per writer
        // both CTAs' bytes of a stage count on the even CTA's barrier
        auto acquire = [&]() -> uint8_t * {
            if (!mbar_wait(&empty[st], ph ^ 1, err)) return nullptr;
            if (lead) {
                mbar_arrive_expect_tx(&full[st], 2 * B_STAGE);
                issued |= 1u << st;
                last_ph = (last_ph & ~(1u << st)) | (ph << st);
            }
            return ring + st * B_STAGE;
        };
        auto fbar = [&]() { return mapa_shared(smem_u32(&full[st]), 0); };
        auto advance = [&]() {
            if (++st == B_NST) { st = 0; ph ^= 1; }
        };
        BwdCursor cur, prev;
        cursor_set(cur, group, 0);
        bool have_prev = false;
        while (ok && (cur.u < n_units || have_prev)) {
            if (!ROWS && cur.u < n_units && cur.r == 0 && cur.u + n_groups < n_units) {
                // d_weight: the group's next unit has a new fixed tile (128 weight rows
                // over the whole d_model, read from HBM for the first time); bring it into
                // L2 now, the CTAs splitting its K steps
                const int fixn = bwd_unit(a, cur.u + n_groups).fixed * 256 + hh * 128;
                for (int kb = crank; kb < nk; kb += c) tma_prefetch_2d(&a.map_fix, kb * TC_BK, fixn);
            }
            if (cur.u < n_units) {
                const int y = cur.r * c + crank;
                if (y < cur.w.ny) {
                    // own 128 fixed rows of A, own 128 loop rows of B
                    const int fix0 = cur.w.fixed * 256 + hh * 128, loop0 = (cur.w.yt_begin + y) * BWD_BN + hh * 128;
                    for (int kb = 0; kb < nk; ++kb) {
                        uint8_t *sp = acquire();
                        if (!sp) { ok = false; break; }
                        const uint32_t fb = fbar();
                        tma_load_2d_pair(sp, &a.map_fix, fb, kb * TC_BK, fix0);
                        tma_load_2d_pair(sp + B_APART, &a.map_loop, fb, kb * TC_BK, loop0);
                        advance();
                    }
                    if (!ok) break;
                }
            }
            if (have_prev) {
                const int slice0 = (prev.w.dg * c + crank) * TC_SLICE + hh * 128;   // own half of the d-slice
                const int y0 = prev.r * c, y_end = min(y0 + c, prev.w.ny);
                for (int yy = y0; yy < y_end && ok; ++yy) {
                    const int wr = yy - y0;
                    const int cw = cnt_get(cnt, wr);
                    const int g = cw % G_SLOTS;
                    // the writer's cw-th tile is published (the poller has seen it; its
                    // acquire and this one order the tile's stores before the loads)
                    if (!scnt_wait(smem_u32(&gseen[wr]), static_cast<unsigned>(cw + 1), err)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_global();
                    const int loop0 = (prev.w.yt_begin + yy) * BWD_BN;
                    const int grow = slot_row(wcta(wr), g);
                    for (int sub = 0; sub < 2 && ok; ++sub)
                        for (int h = 0; h < 2; ++h) {
                            uint8_t *sp = acquire();
                            if (!sp) { ok = false; break; }
                            const uint32_t fb = fbar();
                            tma_load_2d_pair(sp, &a.map_g, fb, h * 64, grow + sub * 128);
                            if (a.ys3 && slice0 + 128 <= a.d)
                                // the half slice's two 64-column blocks in one box
                                tma_load_3d_pair(sp + B_APART, &a.map_ys3, fb, 0, loop0 + sub * 128 + h * 64,
                                                 slice0 / 64);
                            else
                                for (int q = 0; q < 2; ++q)
                                    tma_load_2d_pair(sp + B_APART + q * 8192, &a.map_ys, fb, slice0 + q * 64,
                                                     loop0 + sub * 128 + h * 64);
                            advance();
                        }
                    cnt_inc(cnt, wr);
                }
            }
            have_prev = cur.u < n_units;
            prev = cur;
            if (cur.u < n_units) cursor_next(cur);
        }
        for (int s = 0; s < B_NST; ++s)
            if (issued & (1u << s)) bw_wait_drain(&full[s], (last_ph >> s) & 1);
    } else if (warp == 1 && lane == 0 && lead) {
        // ================= MMA issuer (even CTA, for the pair) =================
        constexpr uint32_t ID_S = idesc_16_f32(256, BWD_BN, 0, 0, F16);
        constexpr uint32_t ID_ACC = idesc_16_f32(256, TC_SLICE, 0, 1, F16);
        int st = 0;
        uint32_t ph = 0;
        bool ok = true, first_acc = true;
        int m_all = 0;                         // own logit tiles issued so far
        int cnt[B_MAXC] = {};
        // Shared-memory descriptors of ring stage 0; stage s adds s * B_STAGE / 16 to the start
        // address field, a K step 32 B / 16 (K-major) or 2 KB / 16 (MN-major).  Every MMA then
        // costs one add per operand: work between MMAs holds the tensor pipe up.
        const uint32_t ring0 = smem_u32(ring);
        const uint64_t dA = sdesc_sw128(ring0, 16, 1024);                 // A: K-major, 128 rows per CTA
        const uint64_t dBs = sdesc_sw128(ring0 + B_APART, 16, 1024);      // logit B: K-major, 128 rows per CTA
        const uint64_t dBa = sdesc_sw128(ring0 + B_APART, 8192, 1024);    // accumulate B: MN-major
        constexpr uint64_t STEP = B_STAGE >> 4;
        BwdCursor cur, prev;
        cursor_set(cur, group, 0);
        bool have_prev = false;
        while (ok && (cur.u < n_units || have_prev)) {
            if (cur.u < n_units) {
                const int y = cur.r * c + crank;
                if (y < cur.w.ny) {
                    if (!mbar_wait(tempty, (m_all & 1) ^ 1, err)) { ok = false; break; }
                    tc_fence_after();
                    for (int kb = 0; kb < nk; ++kb) {
                        if (!mbar_wait(&full[st], ph, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t off = st * STEP;
                        const uint64_t a = dA + off, b = dBs + off;
                        tc_mma_bf16_pair(tmem, a, b, ID_S, kb != 0);
                        tc_mma_bf16_pair(tmem, a + 2, b + 2, ID_S, 1u);
                        tc_mma_bf16_pair(tmem, a + 4, b + 4, ID_S, 1u);
                        tc_mma_bf16_pair(tmem, a + 6, b + 6, ID_S, 1u);
                        tc_commit_pair_multicast(&empty[st], 3);
                        if (++st == B_NST) { st = 0; ph ^= 1; }
                    }
                    if (!ok) break;
                    tc_commit_pair_multicast(tfull, 3);
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
                const int y0 = prev.r * c, y_end = min(y0 + c, prev.w.ny);
                for (int yy = y0; yy < y_end && ok; ++yy) {
                    const int wr = yy - y0;
                    const int g = cnt_get(cnt, wr) % G_SLOTS;
                    for (int sidx = 0; sidx < 4; ++sidx) {
                        if (!mbar_wait(&full[st], ph, err)) { ok = false; break; }
                        tc_fence_after();
                        // all four quarters of both writer CTAs' halves have landed: their
                        // slots may be refilled (completed reads, nothing to publish: relaxed
                        // adds, which never hold the issuer)
                        if (sidx == 3) {
                            gsig_add_relaxed(&gfree[(2 * (pbase + wr)) * G_SLOTS + g], 1u);
                            gsig_add_relaxed(&gfree[(2 * (pbase + wr) + 1) * G_SLOTS + g], 1u);
                        }
                        const uint64_t off = st * STEP;
                        const uint64_t a = dA + off, b = dBa + off;
                        tc_mma_bf16_pair(tmem + ACC_COL, a, b, ID_ACC, first_acc ? 0u : 1u);
                        tc_mma_bf16_pair(tmem + ACC_COL, a + 2, b + 128, ID_ACC, 1u);
                        tc_mma_bf16_pair(tmem + ACC_COL, a + 4, b + 256, ID_ACC, 1u);
                        tc_mma_bf16_pair(tmem + ACC_COL, a + 6, b + 384, ID_ACC, 1u);
                        first_acc = false;
                        tc_commit_pair_multicast(&empty[st], 3);
                        if (++st == B_NST) { st = 0; ph ^= 1; }
                    }
                    cnt_inc(cnt, wr);
                }
                if (!ok) break;
                if (prev.r == prev.nr - 1) tc_commit_pair_multicast(accfull, 3);
            }
            have_prev = cur.u < n_units;
            prev = cur;
            if (cur.u < n_units) cursor_next(cur);
        }
        tc_commit_pair_multicast(drain, 1);
        bw_wait_drain(drain, 0);
    } else if (warp == 6 && lane == 0) {
        // ================= grad-tile poller =================
        // The loader's sequence of grad tiles (every round of every unit, the
        // round's writers in order): wait until the writer's tile is published
        // (its (cw / G_SLOTS)-th fill of slot cw % G_SLOTS: 4 warp adds per tile)
        // and pass the count on.  It runs ahead of the loader as far as the
        // writers allow, and a writer refills a slot only once this CTA has
        // loaded it, so the counts stay in step with what the loader reads.
        int cnt[B_MAXC] = {};
        bool ok = true;
        for (int u = group; u < n_units && ok; u += n_groups) {
            const BwdUnit w = bwd_unit(a, u);
            const int nr = (w.ny + c - 1) / c;
            for (int rr = 0; rr < nr && ok; ++rr) {
                const int y0 = rr * c, y_end = min(y0 + c, w.ny);
                for (int yy = y0; yy < y_end; ++yy) {
                    const int wr = yy - y0;
                    const int cw = cnt_get(cnt, wr);
                    if (!gsig_wait(&gready[wcta(wr) * G_SLOTS + cw % G_SLOTS],
                                   4u * static_cast<unsigned>(cw / G_SLOTS + 1), err)) {
                        ok = false;
                        break;
                    }
                    st_release_cta_shared(smem_u32(&gseen[wr]), static_cast<unsigned>(cw + 1));
                    cnt_inc(cnt, wr);
                }
            }
        }
    } else if (warp >= 2 && warp < 6) {
        // ================= epilogue =================
        const int quad = warp & 3;
        const int r = quad * 32 + lane;               // logit-tile row of this thread
        float4 *sP = sPall + quad * BWD_BN;           // this warp's copy
        // This warp's 4 KB staging block for TMA stores: the teacher-block region
        // in the d_weight pass, the (there unused) parameter region in the row passes.
        uint8_t *gblk = (ROWS ? reinterpret_cast<uint8_t *>(sPall) : tblk) + quad * B_STG;
        uint8_t *tw_s = tblk + quad * 2 * B_TBLK;     // TTMA: this warp's two teacher buffers
        uint64_t *tw_b = tbar + quad * 2;
        // TTMA: issued and waited fills of each buffer.  Chunk q always uses buffer
        // q & 1 and a supertile has an even number of chunks, so one count of
        // each kind serves both buffers: buffer b's k-th fill is the (2k+b)-th.
        int tiss_all = 0, tuse_all = 0;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const float L2E = static_cast<float>(LOG2E);
        const float kT = a.inv_t_l2e, kTln2 = kT * static_cast<float>(LN2);
        const float4 P0 = DISTILL ? make_float4(0.f, 0.f, 0.f, 0.f)
                                  : make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
        int m_all = 0;                                // own logit tiles consumed so far
        auto n_own_of = [&](const BwdUnit &w) { return crank < w.ny ? (w.ny - crank + c - 1) / c : 0; };
        // d_weight with the token range whole (one split): a CTA's own token
        // supertiles are the same in every unit, so their per-token parameters
        // are loaded once, into one copy the four warps share (four supertiles
        // at most: 16 KB).  The one barrier among the epilogue warps sits here,
        // before any wait a warp could unwind from.
        const int n_own_all = crank < a.n_loop ? (a.n_loop - crank + c - 1) / c : 0;
        const bool pcache = !ROWS && a.n_split == 1 && n_own_all <= 4;
        // Label-CE d_weight keeps a supertile's 256 token parameters (4 KB) as
        // {x_j, c_j, x_j+1, c_j+1} pairs in the first 2 KB (the exponent shift
        // and coefficient of two adjacent columns: one shared-memory load per two
        // elements), the targets (int) in the next 1 KB and the one-hot
        // coefficients a_j in the last; the other passes keep the float4 records.
        constexpr bool PAIRS = !ROWS && !DISTILL;
        auto put_param = [&](float4 *blk, int j, const float4 &p) {
            if (PAIRS) {
                float *f = reinterpret_cast<float *>(blk);
                f[(j >> 1) * 4 + (j & 1) * 2] = p.x;
                f[(j >> 1) * 4 + (j & 1) * 2 + 1] = p.y;
                reinterpret_cast<int *>(f + 512)[j] = __float_as_int(p.w);
                f[768 + j] = p.z;
            } else {
                blk[j] = p;
            }
        };
        if (pcache) {
            for (int i = r; i < n_own_all * BWD_BN; i += 128) {
                const int t = ((i / BWD_BN) * c + crank) * BWD_BN + i % BWD_BN;
                put_param(sPall + (i / BWD_BN) * BWD_BN, i % BWD_BN, t < a.n_tok ? a.tokp[t] : P0);
            }
            named_bar_sync(1, 128);
        }
        auto params_of = [&](const BwdUnit &w) {      // d_hidden: the fixed token row's parameters
            const int fixrow = w.fixed * 256 + hh * 128 + r;
            return (ROWS && fixrow < a.n_tok) ? a.tokp[fixrow] : P0;
        };
        // The first row of the teacher block of own supertile m of unit w, for
        // an L2 prefetch one supertile ahead of its use.
        auto teacher_prefetch = [&](const BwdUnit &w, int m) {
            const int fixrow = w.fixed * 256 + hh * 128 + r;
            const int loop0 = (w.yt_begin + m * c + crank) * BWD_BN;
            if (ROWS) {
                if (fixrow >= a.n_tok) return;
                const uint16_t *p = a.teacher + static_cast<int64_t>(fixrow) * a.vocab + loop0;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (loop0 + i * 64 < a.vocab) prefetch_l2(p + i * 64);
            } else {
                const int fix0 = w.fixed * 256 + hh * 128;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = loop0 + r + h * 128;
                    if (t >= a.n_tok) continue;
                    const uint16_t *p = a.teacher + static_cast<int64_t>(t) * a.vocab + fix0;
                    prefetch_l2(p);
                    if (fix0 + 64 < a.vocab) prefetch_l2(p + 64);
                }
            }
        };
        // One own logit tile (the m-th of unit w): wait for its ring slot and
        // its logits, form G in registers, store it into the slot, publish.
        auto tile = [&](const BwdUnit &w, int m, const float4 &P, double &zsum) -> bool {
            const int fixrow = w.fixed * 256 + hh * 128 + r;     // token (d_hidden) or vocabulary (d_weight) row
            const int y = m * c + crank;
            const int loop0 = (w.yt_begin + y) * BWD_BN;
            const int g = m_all % G_SLOTS;
            // the slot's previous tile has been loaded by every CTA of the group (one
            // lane polls; the warp's writes below follow its acquire)
            bool ok = true;
            if (lane == 0)
                ok = gsig_wait(&gfree[blockIdx.x * G_SLOTS + g], static_cast<unsigned>(c * (m_all / G_SLOTS)), err);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ROWS && !pcache) {
                // per-token parameters of this supertile's 256 token columns (each warp
                // keeps its own copy, so no barrier spans warps that may unwind apart)
                __syncwarp();
#pragma unroll
                for (int i = 0; i < BWD_BN / 32; ++i) {
                    const int t = loop0 + lane + i * 32;
                    put_param(sP, lane + i * 32, t < a.n_tok ? a.tokp[t] : P0);
                }
                __syncwarp();
            }
            const float4 *sPt = pcache ? sPall + m * BWD_BN : sP;   // d_weight: the tile's token parameters
            if (DISTILL && m + 1 < n_own_of(w)) teacher_prefetch(w, m + 1);
            ok = ok && mbar_wait(tfull, m_all & 1, err);
            if (!__all_sync(0xffffffffu, ok)) return false;
            tc_fence_after();
            const int ncols = min(BWD_BN, (ROWS ? a.vocab : a.n_tok) - loop0);   // valid loop columns
            const int rel = ROWS && !DISTILL ? __float_as_int(P.w) - loop0 : 0;
            // teacher logits of this thread's row and the supertile's columns
            const bool t_ok = DISTILL && (ROWS ? fixrow < a.n_tok : fixrow < a.vocab);
            const uint16_t *tbase =
                DISTILL ? a.teacher + (ROWS ? static_cast<int64_t>(t_ok ? fixrow : 0) * a.vocab + loop0
                                            : static_cast<int64_t>(loop0) * a.vocab + (t_ok ? fixrow : 0))
                        : nullptr;
            uint32_t tw[16];                          // a chunk's 32 teacher values (bf16 pairs)
            // TTMA: warp-local TMA of the teacher block [32 tokens][this warp's 32
            // vocabulary rows] of chunk q into buffer q & 1 (lane 0 issues; the
            // lanes' earlier reads of that buffer are ordered before it).
            auto tissue = [&](int q) {
                fence_proxy_async_smem();
                __syncwarp();
                ++tiss_all;
                if (lane == 0) {
                    uint64_t *bar = &tw_b[q & 1];
                    mbar_arrive_expect_tx(bar, B_TBLK);
                    tma_load_2d(tw_s + (q & 1) * B_TBLK, &a.map_teach, bar, w.fixed * 256 + hh * 128 + quad * 32,
                                loop0 + q * 32);
                }
            };
            bool tok_all = true;
            auto tload = [&](int q) {
                if (TTMA) {
                    const int b = q & 1;
                    const bool okw = mbar_wait(&tw_b[b], (tuse_all >> 1) & 1, err);
                    tok_all = tok_all && okw;
                    ++tuse_all;
                    const uint16_t *src = reinterpret_cast<const uint16_t *>(tw_s + b * B_TBLK) + lane;
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        tw[i >> 1] = static_cast<uint32_t>(src[i * 32]) | (static_cast<uint32_t>(src[(i + 1) * 32]) << 16);
                    return;
                }
                if (ROWS) {
                    // one contiguous 64-byte row segment: four 16-byte loads
                    const uint4 *src = reinterpret_cast<const uint4 *>(tbase + q * 32);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const uint4 v4 = (t_ok && q * 32 + c4 * 8 < ncols) ? __ldg(src + c4)
                                                                            : make_uint4(0, 0, 0, 0);
                        tw[c4 * 4 + 0] = v4.x; tw[c4 * 4 + 1] = v4.y;
                        tw[c4 * 4 + 2] = v4.z; tw[c4 * 4 + 3] = v4.w;
                    }
                } else {
                    // one element per token row; a warp reads 64 contiguous bytes per token
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const int j = q * 32 + i;
                        const uint32_t lo = (t_ok && j < ncols)
                                                ? __ldg(tbase + static_cast<int64_t>(j) * a.vocab) : 0u;
                        const uint32_t hi = (t_ok && j + 1 < ncols)
                                                ? __ldg(tbase + static_cast<int64_t>(j + 1) * a.vocab) : 0u;
                        tw[i >> 1] = lo | (hi << 16);
                    }
                }
            };
            if (TTMA) {
                tissue(0);
                tissue(1);
            }
            if (DISTILL) tload(0);
            if (TTMA) tissue(2);
            uint16_t *gdst = a.gscr + static_cast<int64_t>(((blockIdx.x * G_SLOTS + g) * 2) * 128 + r) * 128;
            const int grow0 = ((blockIdx.x * G_SLOTS + g) * 2) * 128 + quad * 32;   // this warp's first ring row
            float zt = 0.f;
#pragma unroll 1
            for (int q = 0; q < BWD_BN / 32; ++q) {
                uint32_t v[32];
                tmem_ld32(trow + q * 32, v);
                uint32_t tcur[16];
                if (DISTILL) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) tcur[i] = tw[i];
                    if (q + 1 < BWD_BN / 32) {
                        tload(q + 1);
                        if (TTMA && q + 3 < BWD_BN / 32) tissue(q + 3);
                    }
                }
                tmem_ld_wait();
                uint32_t pk[16];
                if (FUSED) {
                    // G' = 2^(s log2e - r_t); the chunk's sum of G' over the valid vocabulary
                    // columns in two partial sums (a chunk past the vocabulary's end tests
                    // each column)
                    float gf[32], z0 = 0.f, z1 = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) gf[i] = ex2_approx(fmaf(__uint_as_float(v[i]), L2E, -P.x));
                    if (q * 32 + 32 <= ncols) {
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            z0 += gf[i];
                            z1 += gf[i + 1];
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            z0 += q * 32 + i < ncols ? gf[i] : 0.f;
                            z1 += q * 32 + i + 1 < ncols ? gf[i + 1] : 0.f;
                        }
                    }
                    zt += z0 + z1;
#pragma unroll
                    for (int i = 0; i < 32; i += 2) pk[i >> 1] = pack_16x2<F16>(gf[i], gf[i + 1]);
                } else if (!DISTILL) {
                    // label CE: G = c p - a [v = y].  The one-hot term is added only in
                    // the chunks that hold one: this row's target column (d_hidden),
                    // or a column whose target is one of this warp's 32 rows (d_weight,
                    // found with one load and one vote per chunk).
                    float gf[32];
                    if (ROWS) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            gf[i] = P.y * ex2_approx(fmaf(__uint_as_float(v[i]), L2E, -P.x));
                        const int jr = rel - q * 32;
                        if (static_cast<unsigned>(jr) < 32u) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (i == jr) gf[i] -= P.z;
                        }
                    } else {
                        const float4 *pp = sPt + q * 16;             // the chunk's 16 column pairs
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float4 PP = pp[i >> 1];
                            gf[i] = PP.y * ex2_approx(fmaf(__uint_as_float(v[i]), L2E, -PP.x));
                            gf[i + 1] = PP.w * ex2_approx(fmaf(__uint_as_float(v[i + 1]), L2E, -PP.z));
                        }
                        const int *tg = reinterpret_cast<const int *>(sPt) + 512 + q * 32;
                        const float *sa = reinterpret_cast<const float *>(sPt) + 768 + q * 32;
                        const int row0w = w.fixed * 256 + hh * 128 + quad * 32;
                        const uint32_t hit =
                            __ballot_sync(0xffffffffu, static_cast<unsigned>(tg[lane] - row0w) < 32u);
                        if (hit) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (((hit >> i) & 1u) && tg[i] == fixrow) gf[i] -= sa[i];
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 2) pk[i >> 1] = pack_16x2<F16>(gf[i], gf[i + 1]);
                } else {
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float gg[2];
#pragma unroll
                    for (int uu = 0; uu < 2; ++uu) {
                        const int j = q * 32 + i + uu;           // loop column within the supertile
                        const float s = __uint_as_float(v[i + uu]);
                        const float4 Pq = ROWS ? P : sPt[j];
                        // distillation: the student's and teacher's logits scaled by log2e / T
                        // inside one FFMA each
                        const float tv = uu ? h16_hi<F16>(tcur[i >> 1]) : h16_lo<F16>(tcur[i >> 1]);
                        const float qv = ex2_approx(fmaf(s, kT, -Pq.x));
                        if (a.direction == DIR_RKL)
                            gg[uu] = Pq.z * qv * fmaf(s - tv, kTln2, Pq.w);
                        else
                            gg[uu] = Pq.z * qv - Pq.w * ex2_approx(fmaf(tv, kT, -Pq.y));
                    }
                    pk[i >> 1] = pack_16x2<F16>(gg[0], gg[1]);
                }
                }
                // columns q*32 .. q*32+31: sub-tile q/4, 64 bytes at column (q%4)*32
                if (GSTG && a.g_tma) {
                    // through this warp's staging block: chunk q in half q % 2 (64-byte
                    // swizzle: the 16-byte piece k of row r sits at piece k ^ ((r / 2) % 4)),
                    // stored by lane 0 with TMA once the half's previous store has read it
                    uint8_t *h = gblk + (q & 1) * (B_STG / 2);
                    if (lane == 0) {
                        if (q == 0) bulk_wait_read_all();
                        else if (q >= 2) bulk_wait_read_but1();
                    }
                    __syncwarp();
                    const uint32_t hb = smem_u32(h) + static_cast<uint32_t>(lane) * 64;
                    const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3;
#pragma unroll
                    for (int kq = 0; kq < 4; ++kq)
                        st_shared_v4(hb + ((static_cast<uint32_t>(kq) ^ sw) << 4), pk[4 * kq], pk[4 * kq + 1],
                                     pk[4 * kq + 2], pk[4 * kq + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&a.map_gst, h, (q & 3) * 32, grow0 + (q >> 2) * 128);
                        bulk_commit_group();
                    }
                } else {
                    uint16_t *dst = gdst + (q >> 2) * (128 * 128) + (q & 3) * 32;
                    st_global_v8(dst, pk);
                    st_global_v8(dst + 16, pk + 8);
                }
            }
            if (FUSED) zsum += static_cast<double>(zt);
            if (TTMA && !__all_sync(0xffffffffu, tok_all)) return false;
            // the staged stores have landed in global memory before the slot is published
            if (GSTG && a.g_tma && lane == 0) bulk_wait_all();
            // the tile is out of TMEM: give the pair's buffer back (one arrival per
            // warp on the even CTA's barrier; a buffer release publishes no data),
            // then publish the slot
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (lead) mbar_arrive(tempty);
                else mbar_arrive_remote_cta(mapa_shared(smem_u32(tempty), 0));
            }
            fence_proxy_async_global();
            __threadfence();
            __syncwarp();
            // publish: one release add per warp (4 per tile)
            if (lane == 0) gsig_add_release(&gready[blockIdx.x * G_SLOTS + g], 1u);
            ++m_all;
            return true;
        };
        // Units in order.  The next unit's first own tile is formed before this
        // unit's accumulator is stored: its logits are ready earlier (the MMA
        // issues them before this unit's last accumulates), and the MMA can
        // then start the next logit tile while the store runs.
        int u = group;
        BwdUnit w;
        float4 P = P0;
        double zsum = 0.0;
        int m0 = 0;                                   // own tiles of unit w already formed
        if (u < n_units) {
            w = bwd_unit(a, u);
            P = params_of(w);
        }
        bool ok = true;
        for (int k = 0; u < n_units && ok; ++k) {
            const int n_own = n_own_of(w);
            for (int m = m0; m < n_own && ok; ++m) ok = tile(w, m, P, zsum);
            if (!ok) break;
            const int u2 = u + n_groups;
            BwdUnit w2;
            float4 P2 = P0;
            double zsum2 = 0.0;
            int m02 = 0;
            if (u2 < n_units) {
                w2 = bwd_unit(a, u2);
                P2 = params_of(w2);
                if (n_own_of(w2) > 0) {
                    ok = tile(w2, 0, P2, zsum2);
                    if (!ok) break;
                    m02 = 1;
                }
            }
            const int fixrow = w.fixed * 256 + hh * 128 + r;
            const int split = u / (a.n_fixed * a.n_dg);
            if (FUSED && w.dg == 0 && fixrow < a.n_tok)
                // every d-group recomputes the same logits; the first one reports the sums
                a.zpart[(static_cast<int64_t>(split) * c + crank) * a.zpart_stride + fixrow] =
                    static_cast<float>(zsum);
            // the unit's accumulator: store this CTA's rows of its d-slice
            ok = mbar_wait(accfull, k & 1, err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const int slice0 = (w.dg * c + crank) * TC_SLICE;
            const int n_rows = ROWS ? a.n_tok : a.vocab;
            float *dst = a.out + static_cast<int64_t>(split) * a.out_split_stride +
                         static_cast<int64_t>(fixrow) * a.d;
            if (STG && a.out_tma) {
                // d_weight: per 16-column half chunk, each warp writes its 32 rows
                // into one of the two 2 KB halves of its block, alternately (64-byte
                // swizzle: the 16-byte piece k of row r sits at piece k ^ ((r / 2) % 4),
                // so a warp's stores hit every bank), and lane 0 stores the half with
                // TMA, which also clips the vocabulary tail and d_model.  A half is
                // refilled once the store issued from it two half chunks before has
                // read it: the TMA unit, busy with the operand loads, takes a while to
                // get to a store, and with one buffer the warp waited for each.  Only
                // this warp waits on its block, so no barrier spans warps that may
                // unwind apart.
                uint8_t *stg = gblk;
                const int row0 = w.fixed * 256 + hh * 128 + quad * 32;
                const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3;
#pragma unroll 1
                for (int q = 0; q < TC_SLICE / 32; ++q) {
                    const int col = slice0 + q * 32;
                    if (col >= a.d || row0 >= a.vocab) break;
                    uint32_t v[32];
                    tmem_ld32(trow + ACC_COL + q * 32, v);
                    tmem_ld_wait();
                    if (F16) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a.out_scale);
                    }
#pragma unroll
                    for (int hq = 0; hq < 2; ++hq) {
                        if (col + hq * 16 >= a.d) break;
                        const int hc = 2 * q + hq;
                        uint8_t *h = stg + (hc & 1) * (B_STG / 2);
                        if (lane == 0) {
                            if (hc == 0) bulk_wait_read_all();
                            else if (hc >= 2) bulk_wait_read_but1();
                        }
                        __syncwarp();
                        const uint32_t hb = smem_u32(h) + static_cast<uint32_t>(lane) * 64;
#pragma unroll
                        for (int kq = 0; kq < 4; ++kq)
                            st_shared_v4(hb + ((static_cast<uint32_t>(kq) ^ sw) << 4), v[hq * 16 + 4 * kq],
                                         v[hq * 16 + 4 * kq + 1], v[hq * 16 + 4 * kq + 2], v[hq * 16 + 4 * kq + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            // gradient accumulation: out += the accumulator, one add per element
                            if (a.accumulate) tma_reduce_add_2d(&a.map_out, h, col + hq * 16, row0);
                            else tma_store_2d(&a.map_out, h, col + hq * 16, row0);
                            bulk_commit_group();
                        }
                    }
                }
                // the teacher blocks of the next tile land in the same buffers: the
                // stores have read them first
                if (TTMA) {
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                }
            } else if (ROWS && a.out3_tma) {
                // d_hidden (or its split partial): the same staging, stored (or added)
                // as boxes of this split's plane, which clip at n_tok
                uint8_t *stg = gblk;
                const int row0 = w.fixed * 256 + hh * 128 + quad * 32;
                const uint32_t sb = smem_u32(stg) + static_cast<uint32_t>(lane) * 128;
#pragma unroll 1
                for (int q = 0; q < TC_SLICE / 32; ++q) {
                    const int col = slice0 + q * 32;
                    if (col >= a.d || row0 >= a.n_tok) break;
                    uint32_t v[32];
                    tmem_ld32(trow + ACC_COL + q * 32, v);
                    tmem_ld_wait();
                    if (F16) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a.out_scale);
                    }
                    if (lane == 0) bulk_wait_read_all();            // the block's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int kq = 0; kq < 8; ++kq)
                        st_shared_v4(sb + ((static_cast<uint32_t>(kq) ^ (lane & 7)) << 4), v[4 * kq], v[4 * kq + 1],
                                     v[4 * kq + 2], v[4 * kq + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (a.accumulate) tma_reduce_add_3d(&a.map_out3, stg, col, row0, split);
                        else tma_store_3d(&a.map_out3, stg, col, row0, split);
                        bulk_commit_group();
                    }
                }
            } else {
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
                        if (fixrow < n_rows && col < a.d) {
                            if (F16) {
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    v[h][i] = __float_as_uint(__uint_as_float(v[h][i]) * a.out_scale);
                            }
                            if (a.accumulate) {
                                // gradient accumulation: out += this unit's accumulator
                                for (int i = 0; i < 32; ++i)
                                    if (col + i < a.d)
                                        v[h][i] = __float_as_uint(__uint_as_float(v[h][i]) + dst[col + i]);
                            }
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
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (lead) mbar_arrive(accempty);
                else mbar_arrive_remote_cta(mapa_shared(smem_u32(accempty), 0));
            }
            u = u2;
            w = w2;
            P = P2;
            zsum = zsum2;
            m0 = m02;
        }
        if (TTMA)
            for (int k = tuse_all; k < tiss_all; ++k) bw_wait_drain(&tw_b[k & 1], (k >> 1) & 1);
        // this warp's TMA stores are complete before the CTA leaves
        if (GSTG && lane == 0) bulk_wait_all();
        tc_fence_before();
    }
    __syncthreads();
    // neither CTA of the pair leaves while the pair's MMAs, copies or arrivals may touch it
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

template <int MODE, bool DISTILL, bool F16>
static cudaError_t launch_bwp_one(const BwdArgs &a, int n_units, cudaStream_t st)
{
    auto k = bwp_kernel<MODE, DISTILL, F16>;
    constexpr int SMEM = bwd_smem<MODE, DISTILL>();
    // The function attribute and the resident-pair count are set up once per
    // device: the launch of the training step's first pass waits on the host
    // after the validation read-back, so host work here is GPU idle time.
    constexpr int MAX_DEV = 64;
    static std::atomic<int> resident[MAX_DEV];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cache = dev >= 0 && dev < MAX_DEV;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(B_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    int pairs = cache ? resident[dev].load(std::memory_order_acquire) : 0;
    if (pairs < 1) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(2 * G_MAX_CTAS, 1, 1);
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&pairs, k, &cfg) != cudaSuccess || pairs < 1) {
            (void)cudaGetLastError();
            return cudaErrorInvalidConfiguration;
        }
        if (cache) resident[dev].store(pairs, std::memory_order_release);
    }
    // As many groups of c pairs as are resident at once (and as the grad-tile
    // ring has slots for), each walking several units; the results do not
    // depend on the count, only the schedule does.  Every CTA of the grid
    // must be resident at the same time (the groups' pairs wait on each
    // other): the grid never holds more pairs than the occupancy query says
    // fit at once, one CTA per SM, so once no other kernel holds an SM every
    // pair is resident; a pair kept out longer than the waits' limit turns
    // into status 590, not a hang.  (A cooperative launch would state the same
    // guarantee, but the profiler cannot launch one.)
    int groups = pairs / a.n_cl;
    if (groups > n_units) groups = n_units;
    if (groups * 2 * a.n_cl > G_MAX_CTAS) groups = G_MAX_CTAS / (2 * a.n_cl);
    if (groups < 1) return cudaErrorInvalidConfiguration;
    // the ring's hand-off counters start from zero
    e = cudaMemsetAsync(a.gsig, 0, sizeof(unsigned) * 2 * G_MAX_CTAS * G_SLOTS, st);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(groups * 2 * a.n_cl, 1, 1);
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

cudaError_t launch_bwp(int mode, bool distill, bool f16, const BwdArgs &a, int n_units, cudaStream_t st)
{
    if (a.n_cl < 1 || a.n_cl > B_MAXC) return cudaErrorInvalidValue;
    if (mode == BWD_FUSED) return f16 ? cudaErrorInvalidValue : launch_bwp_one<BWD_FUSED, false, false>(a, n_units, st);
    if (f16) {
        if (mode == BWD_ROWS)
            return distill ? launch_bwp_one<BWD_ROWS, true, true>(a, n_units, st)
                           : launch_bwp_one<BWD_ROWS, false, true>(a, n_units, st);
        return distill ? launch_bwp_one<BWD_COLS, true, true>(a, n_units, st)
                       : launch_bwp_one<BWD_COLS, false, true>(a, n_units, st);
    }
    if (mode == BWD_ROWS)
        return distill ? launch_bwp_one<BWD_ROWS, true, false>(a, n_units, st)
                       : launch_bwp_one<BWD_ROWS, false, false>(a, n_units, st);
    return distill ? launch_bwp_one<BWD_COLS, true, false>(a, n_units, st)
                   : launch_bwp_one<BWD_COLS, false, false>(a, n_units, st);
}

} // namespace lossk
