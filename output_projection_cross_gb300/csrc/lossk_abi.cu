// lossk_abi.cu -- the extern "C" entry points of liblossk.so (declared in
// include/lossk.h): the host contract arithmetic, argument checks in the
// documented order, workspace layout, tensor-map encoding and the launch
// sequence of each call.  No device memory is allocated here.
#include "../../include/lossk.h"
#include "lossk_internal.h"

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

using namespace lossk;

namespace {

// Ceilings: 2^46 work cells and 2^27 logit cells are the pages' constants
// ("Loss functions and resident-context kernels", lossk function table); the
// per-dimension ceiling 2^24 is this library's reading of the unprinted one.
constexpr int64_t MAX_WORK_CELLS = int64_t(1) << 46;
constexpr int64_t MAX_LOGIT_CELLS = int64_t(1) << 27;
constexpr int64_t MAX_DIM = int64_t(1) << 24;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A 2-D bf16 tensor [outer][inner] read in boxes of {box_inner, box_outer}
// without swizzle (row-major in shared memory); out-of-range elements read as zero.
bool make_map_plain(CUtensorMap *m, const void *base, int64_t inner, int64_t outer, uint32_t box_inner,
                    uint32_t box_outer)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 2-D bf16 tensor [outer][inner] (row pitch inner*2 bytes) read in boxes of
// {box_inner, box_outer} with the 128-byte swizzle; out-of-range elements
// read as zero.
bool make_map(CUtensorMap *m, const void *base, int64_t inner, int64_t outer, uint32_t box_inner,
              uint32_t box_outer)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same tensor seen as [inner/64 blocks][outer][64] -- dims {64, outer,
// inner/64}, block stride 128 B -- so one box {64, box_outer, nblk} lands nblk
// 64-column blocks one after another (the MN-major operand layout, 128-byte
// swizzle).  Needs inner % 64 == 0.
// The grad-tile ring [rows][128] bf16 written by 32 x 32 boxes from 64-byte-
// swizzled shared memory.
bool make_map_ring_store(CUtensorMap *m, void *base, int64_t rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {128 * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An fp32 [outer][inner] output written by 32 x 32 boxes from 128-byte-
// swizzled shared memory (inner % 4 == 0, so rows are 16-byte multiples).
bool make_map_out_f32(CUtensorMap *m, void *base, int64_t inner, int64_t outer)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || inner % 4 != 0) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 4};
    const cuuint32_t box[2] = {16, 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [planes][rows][inner] (a d_hidden pass's partial slabs, or d_hidden itself),
// 32 x 32 boxes of one plane: a box's rows past `rows` are clipped, never
// written into the next plane.
bool make_map_out3_f32(CUtensorMap *m, void *base, int64_t inner, int64_t rows, int64_t planes)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || inner % 4 != 0) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(planes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 4, static_cast<cuuint64_t>(inner * rows) * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_blocks(CUtensorMap *m, const void *base, int64_t inner, int64_t outer, uint32_t box_outer,
                     uint32_t nblk)
{
    if (inner % 64 != 0) return false;
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(outer), static_cast<cuuint64_t>(inner / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 2, 128};
    const cuuint32_t box[3] = {64, box_outer, nblk};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- tracing: launch counter and optional per-kernel event timing ------------
std::atomic<int64_t> g_launches{0};

struct Profiler {
    std::mutex mu;
    std::atomic<bool> on{false};
    struct Pending {
        int kind;
        cudaEvent_t a, b;
    };
    std::vector<Pending> pending;
    std::vector<cudaEvent_t> pool;
    double ms[KK_N] = {};
    int64_t count[KK_N] = {};
    cudaEvent_t get()
    {
        if (!pool.empty()) {
            cudaEvent_t e = pool.back();
            pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        return e;
    }
};

Profiler &profiler()
{
    static Profiler p;
    return p;
}

struct Hdr {
    int err, bad, n_valid;
};

// ---- read-backs ------------------------------------------------------------------
// A call reads a few words of its workspace header on the host: the validation
// counts, the device error word, the fused pass's range flag.  A copy engine
// would queue that 16-byte copy behind the large copies other streams may
// have in flight (a training loop moving gradients to the host), stalling the
// call for their whole duration, so a one-warp kernel writes the words into
// mapped pinned host memory instead: one 64-byte buffer per calling host
// thread, allocated on first use and kept for the thread's life.
int *readback_buffer()
{
    thread_local int *h = nullptr;
    if (!h) {
        void *p = nullptr;
        if (cudaHostAlloc(&p, 64, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        h = static_cast<int *>(p);
    }
    return h;
}

// The header's first four words (err, bad_targets, n_valid, redo) after all
// work queued on `st`.  begin() enqueues the read-back; end() synchronises `st`
// and returns the words (host work placed between the two overlaps the GPU).
struct HeaderRead {
    int *h = nullptr;
    int words[4] = {0, 0, 0, 0};
    bool begin(const WsHeader *hdr, cudaStream_t st)
    {
        h = readback_buffer();
        int *dptr = nullptr;
        if (h && cudaHostGetDevicePointer(reinterpret_cast<void **>(&dptr), h, 0) == cudaSuccess) {
            Launch k(KK_READBACK, st);
            return launch_publish_header(hdr, dptr, st) == cudaSuccess;
        }
        (void)cudaGetLastError();
        h = nullptr;
        // no mapped host memory: a plain copy
        return cudaMemcpyAsync(words, hdr, sizeof(words), cudaMemcpyDeviceToHost, st) == cudaSuccess;
    }
    bool end(cudaStream_t st, int out[4])
    {
        if (cudaStreamSynchronize(st) != cudaSuccess) return false;
        if (h) {
            const volatile int *v = h;
            for (int i = 0; i < 4; ++i) words[i] = v[i];
        }
        for (int i = 0; i < 4; ++i) out[i] = words[i];
        return true;
    }
};

bool read_header(const WsHeader *hdr, cudaStream_t st, int out[4])
{
    HeaderRead r;
    return r.begin(hdr, st) && r.end(st, out);
}

int32_t status_of(cudaError_t e) { return e == cudaSuccess ? LOSSK_OK : LOSSK_DEVICE_ERROR; }

// Run the validation kernel and read its result back (the one sync of a call;
// the bf16 training step validates without waiting, see ce_common).
int32_t validate(const int64_t *targets, const uint8_t *mask, int64_t n, int64_t V, WsHeader *hdr,
                 cudaStream_t st, Hdr *h)
{
    {
        Launch k(KK_VALIDATE, st);
        if (launch_validate(targets, mask, n, V, hdr, st) != cudaSuccess) return LOSSK_DEVICE_ERROR;
    }
    int buf[4] = {0, 0, 0, 0};
    if (!read_header(hdr, st, buf)) return LOSSK_DEVICE_ERROR;
    h->err = buf[0];
    h->bad = buf[1];
    h->n_valid = buf[2];
    if (h->err) return LOSSK_DEVICE_TIMEOUT;
    if (h->bad) return LOSSK_TARGET_OUT_OF_RANGE;
    return LOSSK_OK;
}

bool is_finite(double x) { return std::isfinite(x); }

// 16-bit inputs (bf16 or fp16): the tensor-core path.
bool is16(int32_t dtype) { return dtype == LOSSK_BF16 || dtype == LOSSK_F16; }
bool dtype_ok(int32_t dtype) { return dtype == LOSSK_F32 || is16(dtype); }

struct Ws {
    WsLayout L;
    uint8_t *base;
    WsHeader *hdr() const { return reinterpret_cast<WsHeader *>(base); }
    float4 *tokp() const { return reinterpret_cast<float4 *>(base + L.off_tokp); }
    float *tgt() const { return reinterpret_cast<float *>(base + L.off_tgt); }
    double *tokacc() const { return reinterpret_cast<double *>(base + L.off_tokacc); }
    float *part() const { return reinterpret_cast<float *>(base + L.off_part); }
    float *dhpart() const { return reinterpret_cast<float *>(base + L.off_dhpart); }
    float *zpart() const { return reinterpret_cast<float *>(base + L.off_zpart); }
    float2 *dhc() const { return reinterpret_cast<float2 *>(base + L.off_dhc); }
    uint16_t *gring() const { return reinterpret_cast<uint16_t *>(base + L.off_gring); }
    unsigned *gsig() const { return reinterpret_cast<unsigned *>(base + L.off_gsig); }
    float *dhacc() const { return reinterpret_cast<float *>(base + L.off_dhacc); }
};

// Tensor maps and shape fields of a cluster pass.  rows: d_hidden / fused
// (fixed = hidden token tiles, loop = vocabulary); otherwise d_weight (fixed =
// weight vocabulary tiles, loop = tokens).
bool bwd_args(const Ws &w, bool rows, int64_t n, int64_t d, int64_t V, const void *H, const void *W,
              BwdArgs *a)
{
    std::memset(a, 0, sizeof(*a));
    const void *Fx = rows ? H : W, *Lp = rows ? W : H;
    const int64_t nf = rows ? n : V, nl = rows ? V : n;
    const BwdGeom g = bwd_geometry(d, false);
    // a CTA of a pair loads its 128 fixed rows, half of the loop supertile and
    // half of the d-slice
    if (!make_map(&a->map_fix, Fx, d, nf, 64, 128) || !make_map(&a->map_loop, Lp, d, nl, 64, BWD_BN / 2) ||
        !make_map(&a->map_ys, Lp, d, nl, 64, 64) || !make_map(&a->map_g, w.gring(), 128, G_RING_ROWS, 64, 128))
        return false;
    a->ys3 = make_map_blocks(&a->map_ys3, Lp, d, nl, 64, 2) ? 1 : 0;
    a->g_tma = make_map_ring_store(&a->map_gst, w.gring(), G_RING_ROWS) ? 1 : 0;
    a->gscr = w.gring();
    a->gsig = w.gsig();
    a->n_tok = static_cast<int>(n);
    a->vocab = static_cast<int>(V);
    a->d = static_cast<int>(d);
    a->n_fixed = static_cast<int>(cdiv(nf, 256));
    a->n_loop = static_cast<int>(cdiv(nl, BWD_BN));
    a->n_split = 1;
    a->n_cl = g.n_cl;
    a->n_dg = g.n_dg;
    a->tokp = w.tokp();
    a->out_split_stride = n * d;
    a->err = &w.hdr()->err;
    a->refused = &w.hdr()->bad_targets;
    return true;
}

// ---- the forward statistics pass + merge + reduction (label CE) ------------
int32_t run_ce_fwd(const Ws &w, int64_t n, int64_t d, int64_t V, int32_t dtype, const void *H,
                   const void *W, const int64_t *targets, const uint8_t *mask, double wz,
                   float *lse_out, float *ce_out, double *scalars, cudaStream_t st, bool sum = false)
{
    const WsLayout &L = w.L;
    cudaError_t e;
    if (is16(dtype)) {
        {
            Launch k(KK_TGT_LOGIT, st);
            e = launch_tgt_logit(dtype == LOSSK_F16, static_cast<const uint16_t *>(H),
                                 static_cast<const uint16_t *>(W), targets, n, d, L.n_pad, w.tgt(), w.tokp(), st);
        }
        if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
        // CTA pairs: 256 tokens x 256 vocabulary per MMA, each CTA loading its
        // own 128 token rows and half (128 rows) of each vocabulary tile.
        TcArgs a;
        std::memset(&a, 0, sizeof(a));
        if (!make_map(&a.map_x, H, d, n, 64, TC_BM) || !make_map(&a.map_y, W, d, V, 64, 128))
            return LOSSK_DEVICE_ERROR;
        a.n_x = static_cast<int>(n);
        a.n_y = static_cast<int>(V);
        a.d = static_cast<int>(d);
        a.n_tok = static_cast<int>(n);
        a.vocab = static_cast<int>(V);
        a.n_xt = static_cast<int>(cdiv(n, TC_BM));
        a.n_yt = static_cast<int>(L.n_ct);
        a.n_items = static_cast<int>(cdiv(a.n_xt, 2)) * a.n_yt;
        a.targets = targets;
        a.part = w.part();
        a.tgt = w.tgt();
        a.part_stride = L.n_pad;
        a.part_plane = L.n_ct * L.n_pad;
        a.err = &w.hdr()->err;
        const int pairs = a.n_items < sm_count() / 2 ? a.n_items : sm_count() / 2;
        Launch k(KK_TC_STATS, st);
        e = launch_fwd2(a, false, dtype == LOSSK_F16, 2 * pairs, st);
    } else {
        Launch k(KK_FP_STATS, st);
        e = launch_fp(TC_STATS, false, H, W, nullptr, static_cast<int>(n), static_cast<int>(V),
                      static_cast<int>(d), static_cast<int>(n), static_cast<int>(V), 1, 0, 1.f,
                      targets, nullptr, nullptr, w.part(), w.tgt(), L.n_pad, L.n_ct * L.n_pad, nullptr, 0, st);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    {
        Launch k(KK_MERGE_CE, st);
        e = launch_merge_ce(w.part(), w.tgt(), targets, mask, n, L.n_ct, L.n_pad, wz, lse_out,
                            ce_out, w.tokacc(), st, !is16(dtype));
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    Launch k(KK_REDUCE, st);
    return status_of(launch_reduce(w.tokacc(), n, L.n_pad, w.hdr(), wz, scalars, st, sum));
}

// ---- the two accumulate passes (d_hidden, d_weight), label CE or distill ----
// out_scale: fp16 grad tiles carry G / out_scale (the per-token parameters were
// formed without the common factor), which the stored accumulators get back.
int32_t run_acc(const Ws &w, int64_t n, int64_t d, int64_t V, int32_t dtype, const void *H,
                const void *W, const void *teacher, bool distill, int direction, double temperature,
                float *d_hidden, float *d_weight, cudaStream_t st, bool accumulate = false,
                double out_scale = 1.0, const BwdArgs *pre_cols = nullptr)
{
    const WsLayout &L = w.L;
    cudaError_t e = cudaSuccess;
    const float inv_t = static_cast<float>(1.0 / temperature);
    if (is16(dtype)) {
        for (int pass = 0; pass < 2; ++pass) {
            float *dst = pass == 0 ? d_hidden : d_weight;
            if (!dst) continue;
            const bool rows = pass == 0;
            BwdArgs a;
            if (!rows && pre_cols) a = *pre_cols;
            else if (!bwd_args(w, rows, n, d, V, H, W, &a)) return LOSSK_DEVICE_ERROR;
            a.teacher = distill ? static_cast<const uint16_t *>(teacher) : nullptr;
            if (distill && !rows && !make_map_plain(&a.map_teach, teacher, V, n, 32, 32))
                return LOSSK_DEVICE_ERROR;
            a.n_split = rows ? static_cast<int>(L.nsplit) : 1;
            a.direction = direction;
            a.inv_t_l2e = static_cast<float>(LOG2E / temperature);
            a.out = (rows && L.nsplit > 1) ? w.dhpart() : dst;
            a.accumulate = (accumulate && a.out == dst) ? 1 : 0;
            a.out_scale = static_cast<float>(out_scale);
            // d_weight leaves TMEM through shared memory and TMA stores (row-per-
            // thread global stores would touch 32 lines per warp instruction)
            a.out_tma = (!rows && make_map_out_f32(&a.map_out, dst, d, V)) ? 1 : 0;
            // d_hidden: the accumulators leave through TMA stores too (per split plane)
            a.out3_tma = (rows && make_map_out3_f32(&a.map_out3, a.out, d, n, a.out == dst ? 1 : L.nsplit)) ? 1 : 0;
            const int n_units = a.n_fixed * a.n_split * a.n_dg;
            {
                Launch k(rows ? KK_TC_ROWS : KK_TC_COLS, st);
                e = launch_bwp(rows ? BWD_ROWS : BWD_COLS, distill, dtype == LOSSK_F16, a, n_units, st);
            }
            if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
            if (rows && L.nsplit > 1) {
                Launch k(KK_SUM_SPLITS, st);
                e = launch_sum_splits(w.dhpart(), L.nsplit, n * d, d_hidden, st, accumulate);
                if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
            }
        }
    } else {
        for (int pass = 0; pass < 2; ++pass) {
            float *dst = pass == 0 ? d_hidden : d_weight;
            if (!dst) continue;
            const bool rows = pass == 0;
            const void *X = rows ? H : W, *Y = rows ? W : H;
            const int64_t nx = rows ? n : V, ny = rows ? V : n;
            const int64_t nsplit = rows ? L.nsplit : 1;
            float *out = (rows && nsplit > 1) ? w.dhpart() : dst;
            {
                Launch k(rows ? KK_FP_ROWS : KK_FP_COLS, st);
                e = launch_fp(rows ? TC_ROWS : TC_COLS, distill, X, Y, static_cast<const float *>(teacher),
                          static_cast<int>(nx), static_cast<int>(ny), static_cast<int>(d),
                          static_cast<int>(n), static_cast<int>(V), static_cast<int>(nsplit),
                          direction, inv_t, nullptr, w.tokp(), nullptr, nullptr, nullptr, 0, 0, out, n * d, st,
                          accumulate && out == dst);
            }
            if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
            if (rows && nsplit > 1) {
                Launch k(KK_SUM_SPLITS, st);
                e = launch_sum_splits(w.dhpart(), nsplit, n * d, d_hidden, st, accumulate);
                if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
            }
        }
    }
    return LOSSK_OK;
}

// ---- forward + d_hidden in one pass (label CE, bf16) ---------------------------
// The d_hidden schedule of the backward run before any lse exists: every logit
// is exponentiated against the per-token shift r_t = s[t][y_t] log2e + 64
// (computed with the validation), the pass accumulates D = G' W and reports the sums of G'
// (BWD_FUSED in k_bwp.cu), merge_fused turns the sums into lse, ce, z and the
// d_weight parameters, and combine_dh scales D into d_hidden.  One logit pass
// less than the separate forward and d_hidden passes.  A row whose shifted
// terms left the trusted range raises the workspace's redo word; the caller
// then recomputes everything on the separate passes.
// A helper stream per (device, caller stream): the training step's small
// kernels that nothing after them waits for (the token mean, d_hidden's
// combine) run on it beside the d_weight pass, on the SMs its groups leave
// free; the call joins it back into the caller's stream before it returns.
// Calls on different caller streams get different helper streams, so neither
// waits for the other's helper work.  Up to SIDE_PER_DEV caller streams per
// device get one; a call on a further stream runs those kernels on its own
// stream (the same results, without the overlap).
struct SideStream {
    std::mutex mu;
    cudaStream_t owner = nullptr;      // the caller stream this helper serves
    bool used = false;
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool ready()
    {
        if (s) return true;
        if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            s = nullptr;
            return false;
        }
        return true;
    }
};

constexpr int SIDE_PER_DEV = 8;

SideStream *side_stream(cudaStream_t caller)
{
    static SideStream sides[64][SIDE_PER_DEV];
    static std::mutex table_mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> g(table_mu);
    for (int i = 0; i < SIDE_PER_DEV; ++i)
        if (sides[dev][i].used && sides[dev][i].owner == caller) return &sides[dev][i];
    for (int i = 0; i < SIDE_PER_DEV; ++i)
        if (!sides[dev][i].used) {
            sides[dev][i].used = true;
            sides[dev][i].owner = caller;
            return &sides[dev][i];
        }
    return nullptr;
}

int32_t run_fused(const Ws &w, int64_t n, int64_t d, int64_t V, const void *H, const void *W,
                  const int64_t *targets, const uint8_t *mask, double wz, double gs,
                  float *lse_out, float *ce_out, double *scalars, float *d_hidden, cudaStream_t st,
                  cudaStream_t aux, cudaEvent_t fork, bool sum, const BwdArgs *pre = nullptr)
{
    // the target logits and reference shifts came with the validation launch
    const WsLayout &L = w.L;
    const uint16_t *Wb = static_cast<const uint16_t *>(W);
    cudaError_t e;
    const BwdGeom g = bwd_geometry(d, false);
    BwdArgs a;
    if (pre) a = *pre;
    else if (!bwd_args(w, true, n, d, V, H, W, &a)) return LOSSK_DEVICE_ERROR;
    a.n_split = static_cast<int>(L.nsplit);
    a.inv_t_l2e = static_cast<float>(LOG2E);
    float *part = L.nsplit > 1 ? w.dhpart() : d_hidden;
    a.out = part;
    a.out3_tma = make_map_out3_f32(&a.map_out3, part, d, n, L.nsplit > 1 ? L.nsplit : 1) ? 1 : 0;
    a.out_split_stride = n * d;
    a.zpart = w.zpart();
    a.zpart_stride = L.n_pad;
    a.err = &w.hdr()->err;
    {
        Launch k(KK_TC_FUSED, st);
        e = launch_bwp(BWD_FUSED, false, false, a, a.n_fixed * a.n_split * a.n_dg, st);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    {
        Launch k(KK_MERGE_FUSED, st);
        e = launch_merge_fused(w.zpart(), L.nsplit * g.n_cl, w.tgt(), targets, mask, n, L.n_pad, gs, sum,
                               wz, lse_out, ce_out, w.tokacc(), w.tokp(), w.dhc(), w.hdr(), st);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    if (aux != st) {
        if (cudaEventRecord(fork, st) != cudaSuccess || cudaStreamWaitEvent(aux, fork, 0) != cudaSuccess)
            return LOSSK_DEVICE_ERROR;
    }
    {
        Launch k(KK_REDUCE, aux);
        e = launch_reduce(w.tokacc(), n, L.n_pad, w.hdr(), wz, scalars, aux, sum);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    Launch k(KK_COMBINE_DH, aux);
    return status_of(launch_combine_dh(part, L.nsplit, n, d, Wb, targets, w.dhc(), d_hidden, w.hdr(), aux));
}

// Checks shared by the fused calls, in the documented order up to 585.
int32_t check_fused(int64_t n, int64_t d, int64_t V, int64_t chunk, bool has_chunk, int32_t dtype,
                    const void *H, int64_t hl, const void *W, int64_t wl, const void *workspace,
                    int64_t wsb, int kind, WsLayout *L)
{
    int32_t s = lossk_dims_check(n, d, V);
    if (s != LOSSK_OK) return s;
    if (has_chunk) {
        s = lossk_chunk_check(chunk, V);
        if (s != LOSSK_OK) return s;
    }
    if (!dtype_ok(dtype)) return LOSSK_LENGTH_MISMATCH;
    if (!H || !W || !workspace) return LOSSK_LENGTH_MISMATCH;
    if (hl < n * d || wl < V * d) return LOSSK_LENGTH_MISMATCH;
    if (!ws_layout(kind, n, d, V, dtype, L) || wsb < static_cast<int64_t>(L->total))
        return LOSSK_LENGTH_MISMATCH;
    if (!aligned16(H) || !aligned16(W) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return LOSSK_UNALIGNED;
    if (is16(dtype) && d % 8 != 0) return LOSSK_UNALIGNED;
    return LOSSK_OK;
}

bool scalars_ok(double wz, double gs) { return is_finite(wz) && wz >= 0.0 && is_finite(gs); }

} // namespace

// ===========================================================================
namespace lossk {

Launch::Launch(int kind, cudaStream_t st) : kind_(kind), st_(st)
{
    g_launches.fetch_add(1, std::memory_order_relaxed);
    Profiler &p = profiler();
    if (!p.on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> g(p.mu);
    a_ = p.get();
    b_ = p.get();
    if (a_ && b_ && cudaEventRecord(a_, st_) == cudaSuccess) active_ = true;
}

Launch::~Launch()
{
    if (!active_) return;
    Profiler &p = profiler();
    std::lock_guard<std::mutex> g(p.mu);
    if (cudaEventRecord(b_, st_) == cudaSuccess) p.pending.push_back({kind_, a_, b_});
}

int32_t check_from_logits(int64_t n, int64_t V, int32_t dtype, const void *logits, int64_t logits_len,
                          const int64_t *targets, int64_t targets_len, const float *lse_out,
                          const double *scalars_out, const void *grad, int64_t grad_len, double wz,
                          double gs, const void *workspace, int64_t workspace_bytes, int64_t max_tok,
                          WsLayout *L)
{
    const bool ws = max_tok <= 0;
    if (n < 1 || V < 1) return LOSSK_EMPTY_DIMENSION;
    if (n > (ws ? MAX_DIM : max_tok) || V > MAX_DIM) return LOSSK_DIMENSION_TOO_LARGE;
    if (!dtype_ok(dtype)) return LOSSK_LENGTH_MISMATCH;
    if (ws && !ws_layout(LOSSK_KIND_FROM_LOGITS, n, 1, V, dtype, L)) return LOSSK_DIMENSION_TOO_LARGE;
    if (!logits || !targets || !lse_out || !scalars_out || (ws && !workspace)) return LOSSK_LENGTH_MISMATCH;
    if (logits_len < n * V || targets_len < n || (grad && grad_len < n * V) ||
        (ws && workspace_bytes < static_cast<int64_t>(L->total)))
        return LOSSK_LENGTH_MISMATCH;
    if (!aligned16(logits) || (grad && !aligned16(grad)) ||
        (ws && (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return LOSSK_UNALIGNED;
    if (!scalars_ok(wz, gs)) return LOSSK_NON_FINITE_SCALAR;
    return LOSSK_OK;
}

int32_t run_from_logits(int64_t n, int64_t V, int32_t dtype, const void *logits, const int64_t *targets,
                        const uint8_t *mask, double wz, double gs, float *lse_out, float *ce_out,
                        double *scalars_out, void *grad, WsHeader *hdr, double *tokacc, int64_t n_pad,
                        cudaStream_t st)
{
    Hdr h;
    int32_t s = validate(targets, mask, n, V, hdr, st, &h);
    if (s != LOSSK_OK) return s;
    const double alpha = h.n_valid > 0 ? gs / h.n_valid : 0.0;
    {
        Launch k(KK_FROM_LOGITS, st);
        if (launch_from_logits(dtype, logits, targets, mask, n, V, wz, alpha, lse_out, ce_out, tokacc, grad,
                               st) != cudaSuccess)
            return LOSSK_DEVICE_ERROR;
    }
    Launch k(KK_REDUCE, st);
    return status_of(launch_reduce(tokacc, n, n_pad, hdr, wz, scalars_out, st));
}

// Groups of c CTA pairs a 152-SM GB300 holds at once (one CTA per SM, at
// most G_MAX_CTAS CTAs for the grad-tile ring).  A fixed table, so the
// geometry -- and with it every rounding order -- is a function of the shape
// alone.
static int64_t resident_groups(int64_t c)
{
    const int64_t by_sm = 152 / (2 * c), by_ring = G_MAX_CTAS / (2 * c);
    return by_sm < by_ring ? by_sm : by_ring;
}

BwdGeom bwd_geometry(int64_t d, bool distill)
{
    // Per loop supertile and d-group a group spends nk + 4c stages per CTA
    // (the logit tile over the whole d_model, then c grad tiles in four
    // quarters), so the pass costs about n_dg (nk + 4c) / (CTAs resident).
    const int64_t ns = cdiv(d, TC_SLICE);               // 256-column slices
    const int64_t nk = cdiv(d, TC_BK);
    BwdGeom g{0, 0};
    double best = 0.0;
    for (int64_t dg = cdiv(ns, BWD_MAX_CL); dg <= ns; ++dg) {
        const int64_t c = cdiv(ns, dg);
        if (cdiv(ns, c) != dg) continue;                // the same groups with idle d-groups
        const int64_t ctas = 2 * c * resident_groups(c);
        if (ctas < 1) continue;
        const double cost = static_cast<double>(dg * (nk + 4 * c)) / static_cast<double>(ctas);
        if (g.n_cl == 0 || cost < best) {
            best = cost;
            g.n_cl = static_cast<int>(c);
            g.n_dg = static_cast<int>(dg);
        }
    }
    (void)distill;
    return g;
}

int64_t dh_splits(int64_t n, int64_t d, int64_t V, int dtype)
{
    // The d_hidden pass has one unit per (token tile, d-group, vocabulary
    // split), walked by the resident groups.  On the tensor-core path the
    // split count minimises the pass's estimated time: the rounds the busiest
    // group walks (its units times each unit's rounds of c supertiles, one
    // round = nk + 4c ring stages at about 512 clocks each) plus reading back
    // the splits' partial slabs (4 n d bytes each; writing them hides under
    // the pass's arithmetic).  At most 256 splits.  On the FFMA
    // path, about two CTAs per SM.  Shape-only, so results never depend on
    // the device.
    const bool tc = is16(dtype);
    if (tc) {
        const BwdGeom g = bwd_geometry(d, false);
        const int64_t c = g.n_cl, groups = resident_groups(c);
        const int64_t tiles = cdiv(n, 2 * TC_BM) * g.n_dg, n_loop = cdiv(V, BWD_BN),
                      nk = cdiv(d, TC_BK);
        const double round_s = static_cast<double>(nk + 4 * c) * 512.0 / 1.9e9;
        const double slab_s = 4.0 * static_cast<double>(n) * static_cast<double>(d) / 6.8e12;
        int64_t best_s = 1;
        double best = 0.0;
        for (int64_t s = 1; s <= n_loop && s <= 256; ++s) {
            const int64_t per_group = cdiv(tiles * s, groups), rounds = cdiv(cdiv(n_loop, s), c);
            const double cost = static_cast<double>(per_group * rounds) * round_s + (s > 1 ? s * slab_s : 0.0);
            if (s == 1 || cost < best) {
                best = cost;
                best_s = s;
            }
        }
        return best_s;
    }
    const int64_t n_yt = cdiv(V, FP_BN);
    const int64_t cap = n_yt / 8 > 1 ? n_yt / 8 : 1;
    const int64_t base = cdiv(n, FP_BM) * cdiv(d, FP_SLICE);
    int64_t s = base >= 296 ? 1 : cdiv(296, base);
    if (s < 1) s = 1;
    return s < cap ? s : cap;
}

bool ws_layout(int kind, int64_t n, int64_t d, int64_t V, int dtype, WsLayout *L)
{
    // the vocabulary-shard calls use the unsharded layouts at the shard's size
    if (kind == LOSSK_KIND_SHARD_FWD) kind = LOSSK_KIND_CE_FWD;
    else if (kind == LOSSK_KIND_SHARD_BWD) kind = LOSSK_KIND_CE_BWD;
    else if (kind == LOSSK_KIND_SHARD_COMBINE) kind = LOSSK_KIND_FROM_LOGITS;
    if (lossk_dims_check(n, d, V) != LOSSK_OK) return false;
    *L = WsLayout();
    const bool tc = is16(dtype);
    L->n_pad = cdiv(n, TC_BM) * TC_BM;
    const bool distill = kind == LOSSK_KIND_DISTILL;
    const bool chk = kind == LOSSK_KIND_CE_CHUNK_CHECK;   // a forward's layout, then the two runs' outputs
    L->bn = tc ? TC_BN_FWD : FP_BN;
    L->n_ct = cdiv(V, L->bn);
    L->nstat = distill ? NSTAT_DISTILL : NSTAT_CE;
    const bool fwd = kind == LOSSK_KIND_CE_FWD || kind == LOSSK_KIND_CE_FWD_BWD || distill || chk;
    const bool bwd = kind == LOSSK_KIND_CE_BWD || kind == LOSSK_KIND_CE_FWD_BWD || distill;
    L->nsplit = bwd ? dh_splits(n, d, V, dtype) : 1;
    size_t off = 256;
    L->off_tokp = off;
    off = align256(off + sizeof(float4) * L->n_pad);
    L->off_tgt = off;
    off = align256(off + sizeof(float) * L->n_pad);
    L->off_tokacc = off;
    off = align256(off + sizeof(double) * 3 * L->n_pad);
    L->off_part = off;
    if (fwd) off = align256(off + sizeof(float) * L->nstat * L->n_ct * L->n_pad);
    L->off_dhpart = off;
    if (bwd && L->nsplit > 1) off = align256(off + sizeof(float) * L->nsplit * n * d);
    // The training-step call on the tensor-core path folds d_hidden into the
    // forward (run_fused); it keeps the separate passes' space for its fallback.
    const bool fused = kind == LOSSK_KIND_CE_FWD_BWD && dtype == LOSSK_BF16;
    L->off_zpart = off;
    if (fused) off = align256(off + sizeof(float) * L->nsplit * BWD_MAX_CL * L->n_pad);
    L->off_dhc = off;
    if (fused) off = align256(off + sizeof(float2) * L->n_pad);
    L->off_gring = off;
    if (bwd && tc) off = align256(off + sizeof(uint16_t) * 128 * static_cast<size_t>(G_RING_ROWS));
    L->off_gsig = off;
    if (bwd && tc) off = align256(off + sizeof(unsigned) * 2 * G_MAX_CTAS * G_SLOTS);
    L->off_tstat = off;
    if (distill) off = align256(off + sizeof(double2) * L->n_pad);
    L->off_dhacc = off;
    if (fused) off = align256(off + sizeof(float) * static_cast<size_t>(n) * static_cast<size_t>(d));
    L->off_red = off;
    off = align256(off + 64);
    L->off_chk = off;      // = the total of a forward's layout
    if (chk) off = align256(off + sizeof(float) * 4 * L->n_pad + sizeof(double) * 8);
    L->total = off;
    return true;
}

} // namespace lossk

// ===========================================================================
extern "C" {

const char *lossk_status_name(int32_t code)
{
    switch (code) {
    case 580: return "ok";
    case 581: return "empty_dimension";
    case 582: return "length_mismatch";
    case 583: return "dimension_too_large";
    case 584: return "work_budget_exceeded";
    case 585: return "non_finite_scalar";
    case 586: return "target_id_out_of_range";
    case 587: return "chunk_exceeds_logit_budget";
    case 588: return "unknown_objective";
    case 589: return "device_error";
    case 590: return "device_timeout";
    case 591: return "unaligned";
    case 592: return "unknown_flags";
    default: return "unknown_status";
    }
}

int32_t lossk_work_fits(int64_t n, int64_t d, int64_t V, int64_t ceiling)
{
    if (n < 1 || d < 1 || V < 1 || ceiling < 0) return 0;
    return n <= (ceiling / d) / V ? 1 : 0;
}

int32_t lossk_dims_check(int64_t n, int64_t d, int64_t V)
{
    if (n < 1 || d < 1 || V < 1) return LOSSK_EMPTY_DIMENSION;
    if (n > MAX_DIM || d > MAX_DIM || V > MAX_DIM) return LOSSK_DIMENSION_TOO_LARGE;
    if (!lossk_work_fits(n, d, V, MAX_WORK_CELLS)) return LOSSK_WORK_BUDGET_EXCEEDED;
    return LOSSK_OK;
}

int32_t lossk_chunk_check(int64_t chunk, int64_t V)
{
    if (chunk < 1 || V < 1) return LOSSK_EMPTY_DIMENSION;
    if (chunk > MAX_LOGIT_CELLS / V) return LOSSK_CHUNK_EXCEEDS_LOGIT_BUDGET;
    return LOSSK_OK;
}

double lossk_logit_cells(int64_t chunk, int64_t V)
{
    if (chunk < 1 || V < 1) return -1.0;
    return static_cast<double>(chunk) * static_cast<double>(V);
}

int32_t lossk_peak_logit_cells(int64_t n, int64_t V, int64_t chunk, lossk_peak_cells *out)
{
    if (!out) return LOSSK_LENGTH_MISMATCH;
    if (n < 1 || V < 1 || chunk < 1) {
        out->chunked_cells = -1.0;
        out->materialized_cells = -1.0;
        out->ratio = 0.0;
        out->n_chunks = 0;
        out->status = LOSSK_EMPTY_DIMENSION;
        return out->status;
    }
    const int64_t held = chunk < n ? chunk : n;
    out->chunked_cells = static_cast<double>(held) * static_cast<double>(V);
    out->materialized_cells = static_cast<double>(n) * static_cast<double>(V);
    out->ratio = out->materialized_cells / out->chunked_cells;
    out->n_chunks = cdiv(n, chunk);
    out->status = lossk_chunk_check(chunk, V);
    return out->status;
}

int64_t lossk_workspace_bytes(int32_t kind, int64_t n, int64_t d, int64_t V, int32_t dtype)
{
    WsLayout L;
    if (!ws_layout(kind, n, d, V, dtype, &L)) return -1;
    return static_cast<int64_t>(L.total);
}

int32_t lossk_targets_check(int64_t n, int64_t V, const int64_t *targets, int64_t targets_len,
                            void *workspace, int64_t workspace_bytes, lossk_stream_t stream)
{
    if (n < 1 || V < 1) return LOSSK_EMPTY_DIMENSION;
    if (!targets || !workspace || targets_len < n || workspace_bytes < 256) return LOSSK_LENGTH_MISMATCH;
    Hdr h;
    return validate(targets, nullptr, n, V, static_cast<WsHeader *>(workspace),
                    reinterpret_cast<cudaStream_t>(stream), &h);
}

static int32_t ce_common(bool do_fwd, bool do_bwd, int64_t n, int64_t d, int64_t V, int64_t chunk,
                         bool has_chunk, int32_t dtype, const void *H, int64_t hl, const void *W,
                         int64_t wl, const int64_t *targets, int64_t tl, const uint8_t *mask,
                         double wz, double gs, float *lse_io, int64_t lse_len, float *ce_out,
                         double *scalars, float *dH, float *dW, void *workspace, int64_t wsb,
                         lossk_stream_t stream, uint32_t flags = 0)
{
    const int kind = do_fwd && do_bwd ? LOSSK_KIND_CE_FWD_BWD : (do_fwd ? LOSSK_KIND_CE_FWD : LOSSK_KIND_CE_BWD);
    Ws w;
    int32_t s = check_fused(n, d, V, chunk, has_chunk, dtype, H, hl, W, wl, workspace, wsb, kind, &w.L);
    if (s != LOSSK_OK) return s;
    if (!targets || tl < n || !lse_io || lse_len < n) return LOSSK_LENGTH_MISMATCH;
    if (do_fwd && !scalars) return LOSSK_LENGTH_MISMATCH;
    if (!scalars_ok(wz, gs)) return LOSSK_NON_FINITE_SCALAR;
    if (flags & ~static_cast<uint32_t>(LOSSK_ACCUMULATE_GRADS | LOSSK_REDUCE_SUM)) return LOSSK_UNKNOWN_FLAGS;
    const bool acc = (flags & LOSSK_ACCUMULATE_GRADS) != 0, sum = (flags & LOSSK_REDUCE_SUM) != 0;
    w.base = static_cast<uint8_t *>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool fused_path = do_fwd && do_bwd && dH && dtype == LOSSK_BF16;
    // gradient of grad_scale * total: a_t = grad_scale m_t / N_valid (mean) or grad_scale m_t (sum)
    double alpha = 0.0;
    if (fused_path) {
        // The training step reads the header back once, at its end.  The
        // validation (with the target logits) is queued first; every kernel
        // after it returns at once if it found a target out of range, so a
        // refused call still touches no output, and N_valid reaches the
        // merge on the device.  With accumulation, d_hidden is formed in the
        // workspace and the caller's gradients are touched only once the
        // read-back has come back clean.
        {
            Launch k(KK_VALIDATE, st);
            if (launch_validate_tgt(static_cast<const uint16_t *>(H), static_cast<const uint16_t *>(W), targets,
                                    mask, n, d, V, w.L.n_pad, w.hdr(), w.tgt(), w.tokp(), st) != cudaSuccess)
                return LOSSK_DEVICE_ERROR;
        }
        BwdArgs fa, ca;
        if (!bwd_args(w, true, n, d, V, H, W, &fa) || (dW && !bwd_args(w, false, n, d, V, H, W, &ca)))
            return LOSSK_DEVICE_ERROR;
        float *dh_fused = acc ? w.dhacc() : dH;
        SideStream *sd = acc ? nullptr : side_stream(st);
        std::unique_lock<std::mutex> lk;
        cudaStream_t aux = st;
        if (sd) {
            lk = std::unique_lock<std::mutex>(sd->mu);
            if (sd->ready()) aux = sd->s;
        }
        s = run_fused(w, n, d, V, H, W, targets, mask, wz, gs, lse_io, ce_out, scalars, dh_fused, st, aux,
                      aux != st ? sd->fork : nullptr, sum, &fa);
        if (s == LOSSK_OK && dW && !acc)
            s = run_acc(w, n, d, V, dtype, H, W, nullptr, false, 0, 1.0, nullptr, dW, st, false, 1.0, &ca);
        if (aux != st &&
            (cudaEventRecord(sd->join, aux) != cudaSuccess || cudaStreamWaitEvent(st, sd->join, 0) != cudaSuccess))
            return LOSSK_DEVICE_ERROR;
        if (s != LOSSK_OK) return s;
        // The read-back: a device timeout, a target out of range (nothing was
        // written), or a row the shifted pass could not represent (then every
        // output is recomputed by the separate passes below, which need no shift).
        int flags_d[4] = {0, 0, 0, 0};
        if (!read_header(w.hdr(), st, flags_d)) return LOSSK_DEVICE_ERROR;
        if (flags_d[0]) return LOSSK_DEVICE_TIMEOUT;
        if (flags_d[1]) return LOSSK_TARGET_OUT_OF_RANGE;
        alpha = sum ? gs : (flags_d[2] > 0 ? gs / flags_d[2] : 0.0);
        if (!flags_d[3]) {
            if (!acc) return LOSSK_OK;
            {
                Launch k(KK_SUM_SPLITS, st);
                if (launch_sum_splits(w.dhacc(), 1, n * d, dH, st, true) != cudaSuccess) return LOSSK_DEVICE_ERROR;
            }
            if (dW) return run_acc(w, n, d, V, dtype, H, W, nullptr, false, 0, 1.0, nullptr, dW, st, true);
            return LOSSK_OK;
        }
    } else {
        Hdr h;
        s = validate(targets, mask, n, V, w.hdr(), st, &h);
        if (s != LOSSK_OK) return s;
        alpha = sum ? gs : (h.n_valid > 0 ? gs / h.n_valid : 0.0);
    }
    if (do_fwd) {
        s = run_ce_fwd(w, n, d, V, dtype, H, W, targets, mask, wz, lse_io, ce_out, scalars, st, sum);
        if (s != LOSSK_OK) return s;
    }
    if (do_bwd && (dH || dW)) {
        // fp16: the grad tiles leave out the common factor alpha, which the
        // stored accumulators get back
        const bool f16 = dtype == LOSSK_F16;
        const double a_tok = f16 ? (alpha != 0.0 ? 1.0 : 0.0) : alpha;
        {
            Launch k(KK_TOKP, st);
            if (launch_tokp_ce(lse_io, targets, mask, n, w.L.n_pad, a_tok, wz, w.tokp(), st, 0, V) != cudaSuccess)
                return LOSSK_DEVICE_ERROR;
        }
        s = run_acc(w, n, d, V, dtype, H, W, nullptr, false, 0, 1.0, dH, dW, st, acc, f16 ? alpha : 1.0);
    }
    return s;
}

int32_t lossk_ce_fwd(int64_t n, int64_t d, int64_t V, int64_t chunk, int32_t dtype, const void *hidden,
                     int64_t hidden_len, const void *weight, int64_t weight_len, const int64_t *targets,
                     int64_t targets_len, const uint8_t *loss_mask, double z_weight, float *lse_out,
                     float *ce_out, double *scalars_out, void *workspace, int64_t workspace_bytes,
                     lossk_stream_t stream)
{
    return ce_common(true, false, n, d, V, chunk, true, dtype, hidden, hidden_len, weight, weight_len,
                     targets, targets_len, loss_mask, z_weight, 1.0, lse_out, n, ce_out, scalars_out,
                     nullptr, nullptr, workspace, workspace_bytes, stream);
}

int32_t lossk_ce_bwd(int64_t n, int64_t d, int64_t V, int32_t dtype, const void *hidden,
                     int64_t hidden_len, const void *weight, int64_t weight_len, const int64_t *targets,
                     int64_t targets_len, const uint8_t *loss_mask, double z_weight, double grad_scale,
                     const float *lse, int64_t lse_len, float *d_hidden, float *d_weight,
                     void *workspace, int64_t workspace_bytes, lossk_stream_t stream)
{
    return ce_common(false, true, n, d, V, 0, false, dtype, hidden, hidden_len, weight, weight_len,
                     targets, targets_len, loss_mask, z_weight, grad_scale, const_cast<float *>(lse),
                     lse_len, nullptr, nullptr, d_hidden, d_weight, workspace, workspace_bytes, stream);
}

int32_t lossk_ce_fwd_bwd(int64_t n, int64_t d, int64_t V, int64_t chunk, int32_t dtype,
                         const void *hidden, int64_t hidden_len, const void *weight, int64_t weight_len,
                         const int64_t *targets, int64_t targets_len, const uint8_t *loss_mask,
                         double z_weight, double grad_scale, float *lse_out, float *ce_out,
                         double *scalars_out, float *d_hidden, float *d_weight, void *workspace,
                         int64_t workspace_bytes, lossk_stream_t stream)
{
    return ce_common(true, true, n, d, V, chunk, true, dtype, hidden, hidden_len, weight, weight_len,
                     targets, targets_len, loss_mask, z_weight, grad_scale, lse_out, n, ce_out,
                     scalars_out, d_hidden, d_weight, workspace, workspace_bytes, stream);
}

int32_t lossk_ce_fwd_bwd_ex(int64_t n, int64_t d, int64_t V, int64_t chunk, int32_t dtype,
                            const void *hidden, int64_t hidden_len, const void *weight, int64_t weight_len,
                            const int64_t *targets, int64_t targets_len, const uint8_t *loss_mask,
                            double z_weight, double grad_scale, uint32_t flags, float *lse_out, float *ce_out,
                            double *scalars_out, float *d_hidden, float *d_weight, void *workspace,
                            int64_t workspace_bytes, lossk_stream_t stream)
{
    return ce_common(true, true, n, d, V, chunk, true, dtype, hidden, hidden_len, weight, weight_len,
                     targets, targets_len, loss_mask, z_weight, grad_scale, lse_out, n, ce_out,
                     scalars_out, d_hidden, d_weight, workspace, workspace_bytes, stream, flags);
}

int32_t lossk_ce_from_logits(int64_t n, int64_t V, int32_t dtype, const void *logits, int64_t logits_len,
                             const int64_t *targets, int64_t targets_len, const uint8_t *loss_mask,
                             double z_weight, double grad_scale, float *lse_out, float *ce_out,
                             double *scalars_out, void *grad_logits, int64_t grad_len, void *workspace,
                             int64_t workspace_bytes, lossk_stream_t stream)
{
    Ws w;
    int32_t s = check_from_logits(n, V, dtype, logits, logits_len, targets, targets_len, lse_out, scalars_out,
                                  grad_logits, grad_len, z_weight, grad_scale, workspace, workspace_bytes, 0, &w.L);
    if (s != LOSSK_OK) return s;
    w.base = static_cast<uint8_t *>(workspace);
    return run_from_logits(n, V, dtype, logits, targets, loss_mask, z_weight, grad_scale, lse_out, ce_out,
                           scalars_out, grad_logits, w.hdr(), w.tokacc(), w.L.n_pad,
                           reinterpret_cast<cudaStream_t>(stream));
}

int32_t lossk_distill_fwd_bwd_ex(int64_t n, int64_t d, int64_t V, int64_t chunk, int32_t dtype,
                                 const void *hidden, int64_t hidden_len, const void *weight,
                                 int64_t weight_len, const void *teacher, int64_t teacher_len,
                                 const uint8_t *loss_mask, int32_t direction, double temperature,
                                 double z_weight, double grad_scale, uint32_t flags, double *scalars_out,
                                 float *per_token_out, float *lse_out, float *d_hidden, float *d_weight,
                                 void *workspace, int64_t workspace_bytes, lossk_stream_t stream)
{
    Ws w;
    int32_t s = check_fused(n, d, V, chunk, true, dtype, hidden, hidden_len, weight, weight_len,
                            workspace, workspace_bytes, LOSSK_KIND_DISTILL, &w.L);
    if (s != LOSSK_OK) return s;
    if (!teacher || teacher_len < n * V || !scalars_out) return LOSSK_LENGTH_MISMATCH;
    if (!aligned16(teacher) || (is16(dtype) && V % 8 != 0)) return LOSSK_UNALIGNED;
    if (!scalars_ok(z_weight, grad_scale) || !is_finite(temperature) || temperature <= 0.0)
        return LOSSK_NON_FINITE_SCALAR;
    if (direction < LOSSK_DISTILL_CE || direction > LOSSK_DISTILL_REV_KL) return LOSSK_UNKNOWN_OBJECTIVE;
    if (flags & ~static_cast<uint32_t>(LOSSK_ACCUMULATE_GRADS | LOSSK_REDUCE_SUM)) return LOSSK_UNKNOWN_FLAGS;
    const bool acc = (flags & LOSSK_ACCUMULATE_GRADS) != 0, sum = (flags & LOSSK_REDUCE_SUM) != 0;
    w.base = static_cast<uint8_t *>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Hdr h;
    s = validate(nullptr, loss_mask, n, V, w.hdr(), st, &h);
    if (s != LOSSK_OK) return s;
    const WsLayout &L = w.L;
    cudaError_t e;
    double2 *tstat = reinterpret_cast<double2 *>(w.base + L.off_tstat);
    {
        // the teacher's own statistics: one HBM stream over the teacher logits
        Launch k(KK_TEACHER_STATS, st);
        e = launch_teacher_stats(dtype, teacher, n, V, temperature, tstat, st);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    if (is16(dtype)) {
        // CTA pairs, 256 tokens x 256 vocabulary per MMA, the teacher read in the epilogue
        TcArgs a;
        std::memset(&a, 0, sizeof(a));
        if (!make_map(&a.map_x, hidden, d, n, 64, TC_BM) || !make_map(&a.map_y, weight, d, V, 64, 128))
            return LOSSK_DEVICE_ERROR;
        a.n_x = static_cast<int>(n);
        a.n_y = static_cast<int>(V);
        a.d = static_cast<int>(d);
        a.n_tok = static_cast<int>(n);
        a.vocab = static_cast<int>(V);
        a.n_xt = static_cast<int>(cdiv(n, TC_BM));
        a.n_yt = static_cast<int>(L.n_ct);
        a.n_items = static_cast<int>(cdiv(a.n_xt, 2)) * a.n_yt;
        a.direction = direction;
        a.inv_t_l2e = static_cast<float>(LOG2E / temperature);
        a.teacher = static_cast<const uint16_t *>(teacher);
        a.tstat = tstat;
        a.part = w.part();
        a.part_stride = L.n_pad;
        a.part_plane = L.n_ct * L.n_pad;
        a.err = &w.hdr()->err;
        const int pairs = a.n_items < sm_count() / 2 ? a.n_items : sm_count() / 2;
        Launch k(KK_TC_STATS, st);
        e = launch_fwd2(a, true, dtype == LOSSK_F16, 2 * pairs, st);
    } else {
        Launch k(KK_FP_STATS, st);
        e = launch_fp(TC_STATS, true, hidden, weight, static_cast<const float *>(teacher),
                      static_cast<int>(n), static_cast<int>(V), static_cast<int>(d), static_cast<int>(n),
                      static_cast<int>(V), 1, direction, static_cast<float>(1.0 / temperature), nullptr,
                      nullptr, tstat, w.part(), nullptr, L.n_pad, L.n_ct * L.n_pad, nullptr, 0, st);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    const double alpha = sum ? grad_scale : (h.n_valid > 0 ? grad_scale / h.n_valid : 0.0);
    // fp16: the grad tiles leave out the common factor alpha (as in the label loss)
    const bool f16 = dtype == LOSSK_F16;
    const double a_tok = f16 ? (alpha != 0.0 ? 1.0 : 0.0) : alpha;
    {
        Launch k(KK_MERGE_DISTILL, st);
        e = launch_merge_distill(w.part(), tstat, loss_mask, n, L.n_ct, L.n_pad, direction, z_weight,
                                 lse_out, per_token_out, w.tokacc(), w.tokp(), a_tok, temperature, st);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    {
        Launch k(KK_REDUCE, st);
        e = launch_reduce(w.tokacc(), n, L.n_pad, w.hdr(), z_weight, scalars_out, st, sum);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    if (!d_hidden && !d_weight) return LOSSK_OK;
    return run_acc(w, n, d, V, dtype, hidden, weight, teacher, true, direction, temperature, d_hidden,
                   d_weight, st, acc, f16 ? alpha : 1.0);
}

int32_t lossk_distill_fwd_bwd(int64_t n, int64_t d, int64_t V, int64_t chunk, int32_t dtype,
                              const void *hidden, int64_t hidden_len, const void *weight,
                              int64_t weight_len, const void *teacher, int64_t teacher_len,
                              const uint8_t *loss_mask, int32_t direction, double temperature,
                              double z_weight, double grad_scale, double *scalars_out,
                              float *per_token_out, float *lse_out, float *d_hidden, float *d_weight,
                              void *workspace, int64_t workspace_bytes, lossk_stream_t stream)
{
    return lossk_distill_fwd_bwd_ex(n, d, V, chunk, dtype, hidden, hidden_len, weight, weight_len, teacher,
                                    teacher_len, loss_mask, direction, temperature, z_weight, grad_scale, 0,
                                    scalars_out, per_token_out, lse_out, d_hidden, d_weight, workspace,
                                    workspace_bytes, stream);
}

int32_t lossk_distill_from_logits(int64_t n, int64_t V, int32_t dtype, const void *logits, int64_t logits_len,
                                  const void *teacher, int64_t teacher_len, const uint8_t *loss_mask,
                                  int32_t direction, double temperature, double z_weight, double grad_scale,
                                  uint32_t flags, double *scalars_out, float *per_token_out, float *lse_out,
                                  void *grad_logits, int64_t grad_len, void *workspace, int64_t workspace_bytes,
                                  lossk_stream_t stream)
{
    int32_t s = lossk_dims_check(n, 1, V);
    if (s != LOSSK_OK) return s;
    if (!dtype_ok(dtype)) return LOSSK_LENGTH_MISMATCH;
    if (!logits || !teacher || !scalars_out || !workspace) return LOSSK_LENGTH_MISMATCH;
    if (logits_len < n * V || teacher_len < n * V || (grad_logits && grad_len < n * V))
        return LOSSK_LENGTH_MISMATCH;
    Ws w;
    if (!ws_layout(LOSSK_KIND_FROM_LOGITS, n, 1, V, dtype, &w.L) || workspace_bytes < static_cast<int64_t>(w.L.total))
        return LOSSK_LENGTH_MISMATCH;
    if (!aligned16(logits) || !aligned16(teacher) || (grad_logits && !aligned16(grad_logits)) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return LOSSK_UNALIGNED;
    if (!scalars_ok(z_weight, grad_scale) || !is_finite(temperature) || temperature <= 0.0)
        return LOSSK_NON_FINITE_SCALAR;
    if (direction < LOSSK_DISTILL_CE || direction > LOSSK_DISTILL_REV_KL) return LOSSK_UNKNOWN_OBJECTIVE;
    if (flags & ~static_cast<uint32_t>(LOSSK_ACCUMULATE_GRADS | LOSSK_REDUCE_SUM)) return LOSSK_UNKNOWN_FLAGS;
    const bool acc = (flags & LOSSK_ACCUMULATE_GRADS) != 0, sum = (flags & LOSSK_REDUCE_SUM) != 0;
    w.base = static_cast<uint8_t *>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Hdr h;
    s = validate(nullptr, loss_mask, n, V, w.hdr(), st, &h);
    if (s != LOSSK_OK) return s;
    const double at_on = sum ? grad_scale : (h.n_valid > 0 ? grad_scale / h.n_valid : 0.0);
    cudaError_t e;
    {
        Launch k(KK_DISTILL_LOGITS, st);
        e = launch_distill_logits(dtype, logits, teacher, loss_mask, n, V, direction, temperature,
                                  z_weight, at_on, lse_out, per_token_out, w.tokacc(), w.L.n_pad, grad_logits,
                                  acc, st);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    Launch k(KK_REDUCE, st);
    return status_of(launch_reduce(w.tokacc(), n, w.L.n_pad, w.hdr(), z_weight, scalars_out, st, sum));
}

int32_t lossk_ce_chunk_invariance(int64_t n, int64_t d, int64_t V, int32_t dtype, const void *hidden,
                                  int64_t hidden_len, const void *weight, int64_t weight_len,
                                  const int64_t *targets, int64_t targets_len, const uint8_t *loss_mask,
                                  double z_weight, double *max_abs_delta, void *workspace,
                                  int64_t workspace_bytes, lossk_stream_t stream)
{
    int32_t s = lossk_dims_check(n, d, V);
    if (s != LOSSK_OK) return s;
    if (!max_abs_delta) return LOSSK_LENGTH_MISMATCH;
    WsLayout L;
    if (!ws_layout(LOSSK_KIND_CE_CHUNK_CHECK, n, d, V, dtype, &L) || workspace_bytes < static_cast<int64_t>(L.total) ||
        !workspace)
        return LOSSK_LENGTH_MISMATCH;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return LOSSK_UNALIGNED;
    // chunk = 1 and chunk = n_tok, or the largest chunk the logit budget allows
    const int64_t c_max = MAX_LOGIT_CELLS / V;
    const int64_t chunks[2] = {1, n < c_max ? n : c_max};
    uint8_t *base = static_cast<uint8_t *>(workspace);
    float *runs = reinterpret_cast<float *>(base + L.off_chk);             // lse_a, ce_a, lse_b, ce_b
    double *scal = reinterpret_cast<double *>(base + L.off_chk + sizeof(float) * 4 * L.n_pad);   // 2 x 3
    for (int r = 0; r < 2; ++r) {
        s = lossk_ce_fwd(n, d, V, chunks[r], dtype, hidden, hidden_len, weight, weight_len, targets, targets_len,
                         loss_mask, z_weight, runs + (2 * r) * L.n_pad, runs + (2 * r + 1) * L.n_pad, scal + 3 * r,
                         workspace, static_cast<int64_t>(L.off_chk), stream);
        if (s != LOSSK_OK) return s;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    std::vector<float> hr(static_cast<size_t>(4 * L.n_pad));
    double hs[6];
    if (cudaMemcpyAsync(hr.data(), runs, sizeof(float) * hr.size(), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(hs, scal, sizeof(hs), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return LOSSK_DEVICE_ERROR;
    double m = 0.0;
    for (int i = 0; i < 3; ++i) m = std::fmax(m, std::fabs(hs[i] - hs[3 + i]));
    for (int64_t t = 0; t < n; ++t)
        for (int q = 0; q < 2; ++q)
            m = std::fmax(m, std::fabs(static_cast<double>(hr[q * L.n_pad + t]) -
                                       static_cast<double>(hr[(2 + q) * L.n_pad + t])));
    *max_abs_delta = m;
    return LOSSK_OK;
}

int32_t lossk_device_status(void *workspace, int64_t workspace_bytes, lossk_stream_t stream)
{
    if (!workspace || workspace_bytes < 256) return LOSSK_LENGTH_MISMATCH;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return LOSSK_DEVICE_ERROR;
    int err = 0;
    if (cudaMemcpy(&err, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LOSSK_DEVICE_ERROR;
    if (err == 0) return LOSSK_OK;
    const int zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return LOSSK_DEVICE_ERROR;
    return LOSSK_DEVICE_TIMEOUT;
}

// ---- vocabulary-parallel cross-entropy ---------------------------------------
// Checks shared by the two shard calls, in the documented order: the fused
// calls' checks at the shard's size (581, 583, 584, 582, 591), the whole
// vocabulary's size (581, 583) and the shard's place in it (582).
static int32_t check_shard(int64_t n, int64_t d, int64_t Vs, int64_t v0, int64_t V_total, int32_t dtype,
                           const void *H, int64_t hl, const void *Ws, int64_t wl, const int64_t *targets,
                           int64_t tl, const void *workspace, int64_t wsb, int kind, WsLayout *L)
{
    if (V_total < 1) return LOSSK_EMPTY_DIMENSION;
    int32_t s = check_fused(n, d, Vs, 0, false, dtype, H, hl, Ws, wl, workspace, wsb, kind, L);
    if (s != LOSSK_OK) return s;
    if (V_total > MAX_DIM) return LOSSK_DIMENSION_TOO_LARGE;
    if (v0 < 0 || v0 > V_total - Vs) return LOSSK_LENGTH_MISMATCH;
    if (!targets || tl < n) return LOSSK_LENGTH_MISMATCH;
    return LOSSK_OK;
}

int32_t lossk_ce_shard_fwd(int64_t n, int64_t d, int64_t Vs, int64_t v0, int64_t V_total, int32_t dtype,
                           const void *hidden, int64_t hidden_len, const void *weight_shard, int64_t weight_len,
                           const int64_t *targets, int64_t targets_len, float *partials, int64_t partials_len,
                           void *workspace, int64_t workspace_bytes, lossk_stream_t stream)
{
    Ws w;
    int32_t s = check_shard(n, d, Vs, v0, V_total, dtype, hidden, hidden_len, weight_shard, weight_len, targets,
                            targets_len, workspace, workspace_bytes, LOSSK_KIND_SHARD_FWD, &w.L);
    if (s != LOSSK_OK) return s;
    if (!partials || partials_len < 3 * n) return LOSSK_LENGTH_MISMATCH;
    if (!aligned16(partials)) return LOSSK_UNALIGNED;
    w.base = static_cast<uint8_t *>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Hdr h;
    s = validate(targets, nullptr, n, V_total, w.hdr(), st, &h);
    if (s != LOSSK_OK) return s;
    const WsLayout &L = w.L;
    {
        Launch k(KK_SHARD_TGT, st);
        if (launch_shard_tgt(dtype, hidden, weight_shard, targets, n, d, v0, Vs, partials + n, partials + 2 * n,
                             st) != cudaSuccess)
            return LOSSK_DEVICE_ERROR;
    }
    cudaError_t e;
    if (is16(dtype)) {
        TcArgs a;
        std::memset(&a, 0, sizeof(a));
        if (!make_map(&a.map_x, hidden, d, n, 64, TC_BM) || !make_map(&a.map_y, weight_shard, d, Vs, 64, 128))
            return LOSSK_DEVICE_ERROR;
        a.n_x = static_cast<int>(n);
        a.n_y = static_cast<int>(Vs);
        a.d = static_cast<int>(d);
        a.n_tok = static_cast<int>(n);
        a.vocab = static_cast<int>(Vs);
        a.n_xt = static_cast<int>(cdiv(n, TC_BM));
        a.n_yt = static_cast<int>(L.n_ct);
        a.n_items = static_cast<int>(cdiv(a.n_xt, 2)) * a.n_yt;
        a.part = w.part();
        a.part_stride = L.n_pad;
        a.part_plane = L.n_ct * L.n_pad;
        a.err = &w.hdr()->err;
        const int pairs = a.n_items < sm_count() / 2 ? a.n_items : sm_count() / 2;
        Launch k(KK_TC_STATS, st);
        e = launch_fwd2(a, false, dtype == LOSSK_F16, 2 * pairs, st);
    } else {
        Launch k(KK_FP_STATS, st);
        e = launch_fp(TC_STATS, false, hidden, weight_shard, nullptr, static_cast<int>(n), static_cast<int>(Vs),
                      static_cast<int>(d), static_cast<int>(n), static_cast<int>(Vs), 1, 0, 1.f, nullptr, nullptr,
                      nullptr, w.part(), w.tgt(), L.n_pad, L.n_ct * L.n_pad, nullptr, 0, st);
    }
    if (e != cudaSuccess) return LOSSK_DEVICE_ERROR;
    // the shard's log-sum-exp per token into row 0 (merge_ce's other outputs
    // land in the workspace)
    Launch k(KK_MERGE_CE, st);
    return status_of(launch_merge_ce(w.part(), partials + n, nullptr, nullptr, n, L.n_ct, L.n_pad, 0.0, partials,
                                     nullptr, w.tokacc(), st, !is16(dtype)));
}

int32_t lossk_ce_shard_combine(int64_t n, int64_t n_shards, const float *partials_all, int64_t partials_len,
                               const uint8_t *loss_mask, double z_weight, float *lse_out, float *ce_out,
                               double *scalars_out, void *workspace, int64_t workspace_bytes, lossk_stream_t stream)
{
    if (n < 1 || n_shards < 1) return LOSSK_EMPTY_DIMENSION;
    if (n > MAX_DIM || n_shards > MAX_DIM) return LOSSK_DIMENSION_TOO_LARGE;
    Ws w;
    if (!ws_layout(LOSSK_KIND_SHARD_COMBINE, n, 1, 1, LOSSK_F32, &w.L)) return LOSSK_DIMENSION_TOO_LARGE;
    if (!partials_all || !lse_out || !scalars_out || !workspace) return LOSSK_LENGTH_MISMATCH;
    if (partials_len < 3 * n * n_shards || workspace_bytes < static_cast<int64_t>(w.L.total))
        return LOSSK_LENGTH_MISMATCH;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return LOSSK_UNALIGNED;
    if (!scalars_ok(z_weight, 1.0)) return LOSSK_NON_FINITE_SCALAR;
    w.base = static_cast<uint8_t *>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    {
        Launch k(KK_VALIDATE, st);
        if (launch_shard_check(partials_all, n_shards, n, loss_mask, w.hdr(), st) != cudaSuccess)
            return LOSSK_DEVICE_ERROR;
    }
    int buf[4] = {0, 0, 0, 0};
    if (!read_header(w.hdr(), st, buf)) return LOSSK_DEVICE_ERROR;
    if (buf[0]) return LOSSK_DEVICE_TIMEOUT;
    if (buf[1]) return LOSSK_TARGET_OUT_OF_RANGE;
    {
        Launch k(KK_SHARD_COMBINE, st);
        if (launch_shard_combine(partials_all, n_shards, n, w.L.n_pad, loss_mask, z_weight, lse_out, ce_out,
                                 w.tokacc(), st) != cudaSuccess)
            return LOSSK_DEVICE_ERROR;
    }
    Launch k(KK_REDUCE, st);
    return status_of(launch_reduce(w.tokacc(), n, w.L.n_pad, w.hdr(), z_weight, scalars_out, st));
}

int32_t lossk_ce_shard_bwd(int64_t n, int64_t d, int64_t Vs, int64_t v0, int64_t V_total, int32_t dtype,
                           const void *hidden, int64_t hidden_len, const void *weight_shard, int64_t weight_len,
                           const int64_t *targets, int64_t targets_len, const uint8_t *loss_mask, double z_weight,
                           double grad_scale, const float *lse, int64_t lse_len, float *d_hidden_part,
                           float *d_weight_shard, void *workspace, int64_t workspace_bytes, lossk_stream_t stream)
{
    Ws w;
    int32_t s = check_shard(n, d, Vs, v0, V_total, dtype, hidden, hidden_len, weight_shard, weight_len, targets,
                            targets_len, workspace, workspace_bytes, LOSSK_KIND_SHARD_BWD, &w.L);
    if (s != LOSSK_OK) return s;
    if (!lse || lse_len < n) return LOSSK_LENGTH_MISMATCH;
    if ((d_hidden_part && !aligned16(d_hidden_part)) || (d_weight_shard && !aligned16(d_weight_shard)))
        return LOSSK_UNALIGNED;
    if (!scalars_ok(z_weight, grad_scale)) return LOSSK_NON_FINITE_SCALAR;
    w.base = static_cast<uint8_t *>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Hdr h;
    s = validate(targets, loss_mask, n, V_total, w.hdr(), st, &h);
    if (s != LOSSK_OK) return s;
    if (!d_hidden_part && !d_weight_shard) return LOSSK_OK;
    const double alpha = h.n_valid > 0 ? grad_scale / h.n_valid : 0.0;
    const bool f16 = dtype == LOSSK_F16;
    const double a_tok = f16 ? (alpha != 0.0 ? 1.0 : 0.0) : alpha;
    {
        Launch k(KK_TOKP, st);
        if (launch_tokp_ce(lse, targets, loss_mask, n, w.L.n_pad, a_tok, z_weight, w.tokp(), st, v0, Vs) !=
            cudaSuccess)
            return LOSSK_DEVICE_ERROR;
    }
    return run_acc(w, n, d, Vs, dtype, hidden, weight_shard, nullptr, false, 0, 1.0, d_hidden_part, d_weight_shard,
                   st, false, f16 ? alpha : 1.0);
}

int32_t lossk_selftest_wait(int32_t n_stages, int32_t n_arrive, int64_t limit_ns, int32_t *stages_seen,
                            void *workspace, int64_t workspace_bytes, lossk_stream_t stream)
{
    if (n_stages < 1 || n_stages > 8 || n_arrive < 0 || n_arrive > n_stages) return LOSSK_LENGTH_MISMATCH;
    if (!workspace || workspace_bytes < 256) return LOSSK_LENGTH_MISMATCH;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return LOSSK_UNALIGNED;
    if (limit_ns < 1000 || limit_ns > 1000000000) return LOSSK_NON_FINITE_SCALAR;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    WsHeader *hdr = static_cast<WsHeader *>(workspace);
    int *seen = &hdr->pad[0];
    {
        Launch k(KK_SELFTEST, st);
        if (launch_wait_selftest(n_stages, n_arrive, static_cast<uint64_t>(limit_ns), &hdr->err, seen, st) !=
            cudaSuccess)
            return LOSSK_DEVICE_ERROR;
    }
    int h[5] = {0, 0, 0, 0, 0};
    if (cudaMemcpyAsync(h, hdr, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return LOSSK_DEVICE_ERROR;
    if (stages_seen) *stages_seen = h[4];
    return h[0] ? LOSSK_DEVICE_TIMEOUT : LOSSK_OK;
}

const char *lossk_kernel_name(int32_t kind)
{
    static const char *names[KK_N] = {"validate",     "tc_stats",      "tc_rows",     "tc_cols",
                                      "fp_stats",     "fp_rows",       "fp_cols",     "merge_ce",
                                      "merge_distill", "reduce",        "tokp_ce",     "sum_splits",
                                      "from_logits",  "tc_fused",      "tgt_logit",   "merge_fused",
                                      "combine_dh",   "teacher_stats", "distill_logits", "readback",
                                      "wait_selftest", "shard_tgt",    "shard_combine"};
    return (kind >= 0 && kind < KK_N) ? names[kind] : "unknown_kernel";
}

int64_t lossk_launch_count(void) { return g_launches.load(); }

int32_t lossk_profile_enable(int32_t on)
{
    profiler().on.store(on != 0);
    return LOSSK_OK;
}

int32_t lossk_profile_read(double *total_ms, int64_t *launches, int32_t cap, int32_t reset)
{
    Profiler &p = profiler();
    std::lock_guard<std::mutex> g(p.mu);
    int32_t rc = 0;
    for (auto &q : p.pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(q.b) != cudaSuccess || cudaEventElapsedTime(&ms, q.a, q.b) != cudaSuccess)
            rc = -1;
        else {
            p.ms[q.kind] += ms;
            p.count[q.kind] += 1;
        }
        p.pool.push_back(q.a);
        p.pool.push_back(q.b);
    }
    p.pending.clear();
    const int32_t k = cap < KK_N ? cap : KK_N;
    for (int32_t i = 0; i < k; ++i) {
        if (total_ms) total_ms[i] = p.ms[i];
        if (launches) launches[i] = p.count[i];
    }
    if (reset)
        for (int i = 0; i < KK_N; ++i) {
            p.ms[i] = 0.0;
            p.count[i] = 0;
        }
    return rc < 0 ? rc : k;
}

} // extern "C"
