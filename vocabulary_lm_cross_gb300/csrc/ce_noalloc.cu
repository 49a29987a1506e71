// ce_noalloc.cu -- ce_fwd_bwd_noalloc: ce_fwd_bwd for callers that cannot
// allocate device memory, with its scratch in a fixed device array.
//
// ce_fwd_bwd needs a caller-provided workspace (label census, error word and,
// when the caller passes no output for them, per-row losses and argmaxes).
// Some callers cannot obtain one: code that runs inside a framework whose
// allocator owns all device memory and forbids side allocations, or
// latency-critical code for which cudaMalloc's implicit device
// synchronisation is unacceptable.  This entry point takes the workspace from
// the file-scope array below instead and otherwise runs exactly ce_fwd_bwd.
#include <cuda_runtime.h>

#include <mutex>

#include "host_util.h"
#include "vlmce.h"

namespace vlmce {
namespace {

// Rows the array can serve: 256 B of header + 4 B of loss + 8 B of argmax per
// row (the same layout as ce_fwd_bwd's workspace), 768.25 KiB in all.
constexpr int64_t kNoAllocMaxRows = 65536;
constexpr size_t kNoAllocScratchBytes =
    256 + 4 * static_cast<size_t>(kNoAllocMaxRows) + 8 * static_cast<size_t>(kNoAllocMaxRows);

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_ce_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch[kMaxDevices] = {};

// Device address of g_ce_scratch on the current device.  The first call on a
// device looks it up (the host-side name is only a stand-in, not a device
// address) and caches it for the life of the process, which assumes the
// runtime's primary context: after cudaDeviceReset, or under another context,
// the module is loaded again and the cached address would be stale.
vlmce_status scratch_address(void **out) {
    int dev = -1;
    if (record_cuda(cudaGetDevice(&dev), "cudaGetDevice") != cudaSuccess || dev < 0 ||
        dev >= kMaxDevices)
        return VLMCE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        if (record_cuda(cudaGetSymbolAddress(&p, g_ce_scratch), "cudaGetSymbolAddress(g_ce_scratch)") !=
                cudaSuccess ||
            !p)
            return VLMCE_ERR_CUDA;
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return VLMCE_OK;
}

}  // namespace
}  // namespace vlmce

extern "C" int64_t vlmce_ce_noalloc_max_rows(void) { return vlmce::kNoAllocMaxRows; }

extern "C" vlmce_status ce_fwd_bwd_noalloc(void *logits, int32_t dtype, const int64_t *labels,
                                           int64_t N, int64_t V, int64_t row_stride,
                                           int64_t ignore_index, float label_smoothing,
                                           float softcap, int32_t reduction, float grad_scale,
                                           float *out_loss, int64_t *out_argmax, float *out_reduced,
                                           int64_t *out_counts, vlmce_stream_t stream) {
    if (N < 0) return VLMCE_ERR_INVALID_ARG;
    if (N > vlmce::kNoAllocMaxRows) return VLMCE_ERR_TOO_LARGE;
    void *scratch = nullptr;
    const vlmce_status st = vlmce::scratch_address(&scratch);
    if (st != VLMCE_OK) return st;
    return ce_fwd_bwd(logits, dtype, labels, N, V, row_stride, ignore_index, label_smoothing,
                      softcap, reduction, grad_scale, out_loss, out_argmax, out_reduced,
                      out_counts, scratch, vlmce::kNoAllocScratchBytes, stream);
}
