// k_fwd2.cu -- forward statistics of the label cross-entropy on CTA pairs.
//
// The forward reduces each logit tile S = H_tile . W_tile^T to per-token
// (running max, sum of exp) pairs (the target logit comes from a separate kernel) -- the online
// log-sum-exp of "Loss functions and resident-context kernels" (lossk: a
// chunk's logits are reduced as soon as they exist).  Here two CTAs of a
// cluster act as one tcgen05 unit (cta_group::2): a 256-token x 256-vocabulary
// tile per MMA, each CTA holding its own 128 token rows of A and half (128
// rows) of the vocabulary operand B.  Per K step each SM then reads 8 KB of
// operands for 1 MFLOP instead of 12 KB (one CTA, N = 256), which is what
// bounds this contraction: shared-memory bytes per FLOP.
//
// The distillation forward (DISTILL) runs the same tiles on the student's
// logits a = s log2(e) / T and reads the teacher's row segment of each tile
// from global memory (16-byte loads, the next tile's segment prefetched into
// L2).  With the teacher's log-sum-exp already known per token (teacher_stats),
// each tile reports the student's (max, sum) and one cross term: sum p a with
// the teacher's probabilities exact (CE, forward KL), or sum 2^(a - max)(a - b)
// (reverse KL).
//
// Roles (192 threads per CTA): warp 0 of both CTAs loads its own halves with
// TMA, counting the bytes on the even CTA's stage barrier; warp 1 of both
// CTAs owns the pair's tensor memory, and the even CTA's issues the MMAs;
// warps 2-5 of each CTA reduce that CTA's 128 rows.  Every wait is bounded.
#include "lossk_internal.h"
#include "ptx.cuh"

#include <atomic>

namespace lossk {

namespace {

constexpr int F2_BN = 256;                      // vocabulary columns per tile
constexpr int F2_A_BYTES = 128 * 64 * 2;        // own 128 token rows x 64 K
constexpr int F2_B_BYTES = 128 * 64 * 2;        // own half: 128 vocabulary rows x 64 K
constexpr int F2_STAGE = F2_A_BYTES + F2_B_BYTES;
constexpr int F2_STAGES = 6;
constexpr int F2_NBARS = 2 * F2_STAGES + 2 + 2 + 1;
constexpr int F2_SMEM = 1024 + F2_STAGES * F2_STAGE + F2_NBARS * 8 + 16;
static_assert(F2_SMEM <= 232448, "fits the 227 KB per-CTA shared memory limit");

__device__ __forceinline__ void f2_wait_drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 200000000ull) return;
}

} // namespace

// F16: fp16 operands and teacher logits instead of bf16.
template <bool DISTILL, bool F16>
__global__ void __launch_bounds__(192, 1) fwd2_kernel(const __grid_constant__ TcArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + F2_STAGES * F2_STAGE);
    uint64_t *full = bars;                  // [S] even CTA's: both CTAs' bytes landed
    uint64_t *empty = full + F2_STAGES;     // [S] each CTA's: the pair's MMA is done with the stage
    uint64_t *tfull = empty + F2_STAGES;    // [2] each CTA's: its logit rows are in TMEM
    uint64_t *tempty = tfull + 2;           // [2] even CTA's: both epilogues done (8 warps)
    uint64_t *drain = tempty + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *err = a.err;
    const uint32_t crank = cluster_ctarank();        // 0: even (MMA issuer), 1: odd
    const bool lead = crank == 0;
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    const int n_pt = (a.n_xt + 1) / 2;               // 256-token pair tiles
    const int it_begin = static_cast<int>((static_cast<int64_t>(pair) * a.n_items) / n_pairs);
    const int it_end = static_cast<int>((static_cast<int64_t>(pair + 1) * a.n_items) / n_pairs);
    const int n_it = it_end - it_begin;
    auto coords = [&](int j, int &tok0, int &voc0, int &vt) {
        const int i = it_begin + j;
        vt = i / n_pt;
        const int pt = i - vt * n_pt;
        tok0 = pt * 256 + static_cast<int>(crank) * 128;
        voc0 = vt * F2_BN;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < F2_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);
        }
        mbar_init(drain, 1);
        fence_mbarrier_init();
    }
    if (warp == 1) tmem_alloc_pair(tslot, 512);
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int nk = (a.d + TC_BK - 1) / TC_BK;

    if (warp == 0 && lane == 0) {
        // ================= TMA producer (both CTAs) =================
        tma_prefetch_desc(&a.map_x);
        tma_prefetch_desc(&a.map_y);
        int st = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int j = 0; j < n_it && ok; ++j) {
            int tok0, voc0, vt;
            coords(j, tok0, voc0, vt);
            for (int kb = 0; kb < nk; ++kb) {
                if (!mbar_wait(&empty[st], ph ^ 1, err)) { ok = false; break; }
                if (lead) mbar_arrive_expect_tx(&full[st], 2 * F2_STAGE);
                const uint32_t fbar = mapa_shared(smem_u32(&full[st]), 0);
                uint8_t *sp = ring + st * F2_STAGE;
                tma_load_2d_pair(sp, &a.map_x, fbar, kb * TC_BK, tok0);
                tma_load_2d_pair(sp + F2_A_BYTES, &a.map_y, fbar, kb * TC_BK,
                                 voc0 + static_cast<int>(crank) * 128);
                if (++st == F2_STAGES) { st = 0; ph ^= 1; }
            }
        }
    } else if (warp == 1 && lane == 0 && lead) {
        // ================= MMA issuer (even CTA) =================
        constexpr uint32_t ID = idesc_16_f32(256, F2_BN, 0, 0, F16);
        static_assert(TC_BK == 64, "a ring stage holds four K steps of 16");
        const uint64_t dA = sdesc_sw128(smem_u32(ring), 16, 1024);
        const uint64_t dB = sdesc_sw128(smem_u32(ring) + F2_A_BYTES, 16, 1024);
        int st = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int j = 0; j < n_it && ok; ++j) {
            const int b = j & 1;
            if (!mbar_wait(&tempty[b], ((j >> 1) & 1) ^ 1, err)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem + b * F2_BN;
            for (int kb = 0; kb < nk; ++kb) {
                if (!mbar_wait(&full[st], ph, err)) { ok = false; break; }
                tc_fence_after();
                // descriptors of stage 0 plus the stage and K-step offsets (16-byte units):
                // one add per operand between MMAs
                const uint64_t off = st * (F2_STAGE >> 4);
                const uint64_t da = dA + off, db = dB + off;
                tc_mma_bf16_pair(d, da, db, ID, kb != 0);
                tc_mma_bf16_pair(d, da + 2, db + 2, ID, 1u);
                tc_mma_bf16_pair(d, da + 4, db + 4, ID, 1u);
                tc_mma_bf16_pair(d, da + 6, db + 6, ID, 1u);
                tc_commit_pair_multicast(&empty[st], 3);
                if (++st == F2_STAGES) { st = 0; ph ^= 1; }
            }
            if (!ok) break;
            tc_commit_pair_multicast(&tfull[b], 3);
        }
        tc_commit_pair_multicast(drain, 1);
        f2_wait_drain(drain, 0);
    } else if (warp >= 2) {
        // ================= epilogue (both CTAs, own 128 rows) =================
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const float kS = DISTILL ? a.inv_t_l2e : static_cast<float>(LOG2E);
        const uint32_t tempty_lead = mapa_shared(smem_u32(tempty), 0);
        bool ok = true;
        for (int j = 0; j < n_it && ok; ++j) {
            int tok0, voc0, vt;
            coords(j, tok0, voc0, vt);
            const int b = j & 1;
            const int t = tok0 + r;
            const bool row_ok = t < a.n_tok;
            const int ncols = min(F2_BN, a.vocab - voc0);
            const uint16_t *trow_g = nullptr;
            float lt2 = 0.f;
            if (DISTILL) {
                trow_g = a.teacher + static_cast<int64_t>(row_ok ? t : 0) * a.vocab + voc0;
                lt2 = row_ok ? static_cast<float>(a.tstat[t].x) : 0.f;
                if (j + 1 < n_it) {
                    // the next tile's teacher row segment (512 bytes) into L2
                    int tk1, vc1, vt1;
                    coords(j + 1, tk1, vc1, vt1);
                    if (tk1 + r < a.n_tok) {
                        const uint16_t *p = a.teacher + static_cast<int64_t>(tk1 + r) * a.vocab + vc1;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (vc1 + i * 64 < a.vocab) prefetch_l2(p + i * 64);
                    }
                }
            }
            ok = mbar_wait(&tfull[b], (j >> 1) & 1, err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const uint32_t tbuf = trow + b * F2_BN;
            float m2 = -INFINITY, z = 0.f, x = 0.f;
#pragma unroll 1
            for (int q = 0; q < F2_BN / 32; ++q) {
                if (q * 32 >= ncols) break;
                uint32_t v[32];
                tmem_ld32(tbuf + q * 32, v);
                float bt[32];                                  // raw teacher logits of the chunk
                if (DISTILL) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(trow_g + q * 32);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const uint4 w4 = (row_ok && q * 32 + c4 * 8 < ncols) ? __ldg(src + c4) : make_uint4(0, 0, 0, 0);
                        const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            bt[c4 * 8 + 2 * e] = h16_lo<F16>(ww[e]);
                            bt[c4 * 8 + 2 * e + 1] = h16_hi<F16>(ww[e]);
                        }
                    }
                }
                tmem_ld_wait();
                // The chunk's terms from the raw logits: its maximum first (kS > 0
                // commutes with it), each exponent argument one FFMA, the cross sum in
                // raw logits scaled once.  Only the vocabulary's last chunk tests its
                // columns.
                const bool full = q * 32 + 32 <= ncols;
                float cr = -INFINITY;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (full || q * 32 + i < ncols) cr = fmaxf(cr, __uint_as_float(v[i]));
                const float cm = cr * kS;
                if (cm > m2) {
                    const float sc = ex2_approx(m2 - cm);
                    z *= sc;
                    if (DISTILL && a.direction == DIR_RKL) x *= sc;
                    m2 = cm;
                }
                float acc = 0.f, xa = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const bool in = full || q * 32 + i < ncols;
                    const float sv = __uint_as_float(v[i]);
                    const float e = in ? ex2_approx(fmaf(sv, kS, -m2)) : 0.f;
                    acc += e;
                    if (DISTILL) {
                        if (a.direction == DIR_RKL) xa = fmaf(e, sv - bt[i], xa);
                        else xa = fmaf(in ? ex2_approx(fmaf(bt[i], kS, -lt2)) : 0.f, sv, xa);
                    }
                }
                z += acc;
                x += xa * kS;
            }
            if (row_ok) {
                const int64_t o = static_cast<int64_t>(vt) * a.part_stride + t;
                a.part[o] = m2;
                a.part[a.part_plane + o] = z;
                if (DISTILL) a.part[2 * a.part_plane + o] = x;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (lead) mbar_arrive(&tempty[b]);
                else mbar_arrive_remote_cta(tempty_lead + b * 8);   // a buffer release: no data to publish
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    cluster_sync();       // neither CTA leaves while the pair's MMAs or copies may touch it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

template <bool DISTILL, bool F16> static cudaError_t launch_fwd2_one(const TcArgs &a, int grid, cudaStream_t st)
{
    auto k = fwd2_kernel<DISTILL, F16>;
    // the shared-memory attribute is set once per device
    static std::atomic<int> attr_done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, F2_SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev].store(1, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = F2_SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

cudaError_t launch_fwd2(const TcArgs &a, bool distill, bool f16, int grid, cudaStream_t st)
{
    if (f16) return distill ? launch_fwd2_one<true, true>(a, grid, st) : launch_fwd2_one<false, true>(a, grid, st);
    return distill ? launch_fwd2_one<true, false>(a, grid, st) : launch_fwd2_one<false, false>(a, grid, st);
}

} // namespace lossk
