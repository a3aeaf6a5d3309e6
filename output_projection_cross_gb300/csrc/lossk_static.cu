// lossk_static.cu -- lossk_ce_from_logits_static: cross-entropy from logits for
// callers that cannot allocate device memory at all.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: a
// plug-in running inside another framework that owns every byte of device
// memory through its own pre-planned arena, or a runtime whose memory plan is
// fixed at start-up and which treats any allocation during a step as an
// error.  For them this entry point keeps its scratch (the 256-byte header and
// the per-token reduction terms) in a file-scope device array that the
// library carries in its image, so the call itself allocates nothing: no
// cudaMalloc, no cudaFree, no allocating library routine.
//
// The kernels are the same ones lossk_ce_from_logits launches; only the
// source of their scratch pointer differs.
#include "../../include/lossk.h"
#include "lossk_internal.h"

#include <cmath>
#include <mutex>

namespace {

using namespace lossk;

// Header (256 B) + three doubles per token, tokens rounded up to 128.
constexpr int64_t STATIC_MAX_TOKENS = 16384;
constexpr size_t STATIC_SCRATCH_BYTES = 256 + 3 * sizeof(double) * STATIC_MAX_TOKENS;

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[STATIC_SCRATCH_BYTES];

// The array's device address, looked up once per device with that device
// current.  In host code the symbol itself is only a host-side stand-in, never
// a device address, so it is never passed to a kernel directly.
constexpr int MAX_DEVICES = 64;
void *g_scratch_addr[MAX_DEVICES] = {nullptr};
std::mutex g_scratch_mu;

cudaError_t scratch_for_current_device(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

} // namespace

extern "C" int32_t lossk_ce_from_logits_static(int64_t n, int64_t V, int32_t dtype,
                                               const void *logits, int64_t logits_len,
                                               const int64_t *targets, int64_t targets_len,
                                               const uint8_t *loss_mask, double z_weight,
                                               double grad_scale, float *lse_out, float *ce_out,
                                               double *scalars_out, void *grad_logits,
                                               int64_t grad_len, lossk_stream_t stream)
{
    if (n < 1 || V < 1) return LOSSK_EMPTY_DIMENSION;
    if (n > STATIC_MAX_TOKENS || V > (int64_t(1) << 24)) return LOSSK_DIMENSION_TOO_LARGE;
    if (dtype != LOSSK_F32 && dtype != LOSSK_BF16 && dtype != LOSSK_F16) return LOSSK_LENGTH_MISMATCH;
    if (!logits || !targets || !lse_out || !scalars_out) return LOSSK_LENGTH_MISMATCH;
    if (logits_len < n * V || targets_len < n || (grad_logits && grad_len < n * V))
        return LOSSK_LENGTH_MISMATCH;
    if ((reinterpret_cast<uintptr_t>(logits) & 15u) ||
        (grad_logits && (reinterpret_cast<uintptr_t>(grad_logits) & 15u)))
        return LOSSK_UNALIGNED;
    if (!std::isfinite(z_weight) || z_weight < 0.0 || !std::isfinite(grad_scale))
        return LOSSK_NON_FINITE_SCALAR;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return LOSSK_DEVICE_ERROR;
    WsHeader *hdr = static_cast<WsHeader *>(scratch);
    double *tokacc = reinterpret_cast<double *>(static_cast<unsigned char *>(scratch) + 256);
    const int64_t n_pad = (n + TC_BM - 1) / TC_BM * TC_BM;

    // The array keeps the previous call's contents: clear the header (error
    // word and counters).  The per-token terms are fully rewritten before use.
    if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st) != cudaSuccess) return LOSSK_DEVICE_ERROR;
    if (launch_validate(targets, loss_mask, n, V, hdr, st) != cudaSuccess) return LOSSK_DEVICE_ERROR;
    int h[3] = {0, 0, 0};
    if (cudaMemcpyAsync(h, hdr, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return LOSSK_DEVICE_ERROR;
    if (h[1]) return LOSSK_TARGET_OUT_OF_RANGE;
    const double alpha = h[2] > 0 ? grad_scale / h[2] : 0.0;
    if (launch_from_logits(dtype, logits, targets, loss_mask, n, V, z_weight, alpha, lse_out, ce_out,
                           tokacc, grad_logits, st) != cudaSuccess)
        return LOSSK_DEVICE_ERROR;
    if (launch_reduce(tokacc, n, n_pad, hdr, z_weight, scalars_out, st) != cudaSuccess)
        return LOSSK_DEVICE_ERROR;
    return LOSSK_OK;
}
