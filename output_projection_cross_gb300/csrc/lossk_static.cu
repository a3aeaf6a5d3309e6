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
// a device address, so it is never passed to a kernel directly.  The address
// belongs to the device's primary context: a cudaDeviceReset on that device
// makes the cached value stale, so this library must not be called on a
// device after it has been reset.
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
    // The same checks, in the same order, as the workspace entry point; only
    // the token limit differs (the array's size, 583 beyond it).
    int32_t s = check_from_logits(n, V, dtype, logits, logits_len, targets, targets_len, lse_out, scalars_out,
                                  grad_logits, grad_len, z_weight, grad_scale, nullptr, 0, STATIC_MAX_TOKENS,
                                  nullptr);
    if (s != LOSSK_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return LOSSK_DEVICE_ERROR;
    WsHeader *hdr = static_cast<WsHeader *>(scratch);
    double *tokacc = reinterpret_cast<double *>(static_cast<unsigned char *>(scratch) + 256);
    const int64_t n_pad = (n + TC_BM - 1) / TC_BM * TC_BM;
    // The array keeps the previous call's contents: clear the header (error
    // word and counters).  The per-token terms are fully rewritten before use.
    if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st) != cudaSuccess) return LOSSK_DEVICE_ERROR;
    // The same launches as the workspace entry point (validation read-back,
    // row stream, token mean), each counted and traced like every other launch.
    return run_from_logits(n, V, dtype, logits, targets, loss_mask, z_weight, grad_scale, lse_out, ce_out,
                           scalars_out, grad_logits, hdr, tokacc, n_pad, st);
}
