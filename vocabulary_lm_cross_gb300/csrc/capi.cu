// capi.cu -- status strings and the per-device properties cache.
#include <cstdio>
#include <mutex>

#include "host_util.h"

namespace vlmce {

namespace {
thread_local char t_last_error[256] = "";
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices] = {};
std::mutex g_mu;
}  // namespace

cudaError_t record_cuda(cudaError_t e, const char *where) {
    if (e != cudaSuccess) {
        snprintf(t_last_error, sizeof(t_last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
                 cudaGetErrorString(e));
        cudaGetLastError();
    }
    return e;
}

vlmce_status current_device(DeviceInfo *out) {
    int dev = -1;
    if (record_cuda(cudaGetDevice(&dev), "cudaGetDevice") != cudaSuccess || dev < 0 ||
        dev >= kMaxDevices)
        return VLMCE_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_have[dev]) {
            DeviceInfo d;
            d.device = dev;
            if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                       dev) != cudaSuccess) {
                record_cuda(cudaGetLastError(), "cudaDeviceGetAttribute");
                return VLMCE_ERR_CUDA;
            }
            g_info[dev] = d;
            g_have[dev] = true;
        }
        *out = g_info[dev];
    }
    // The kernels are built for sm_103a only.
    if (out->cc_major != 10 || out->cc_minor != 3) return VLMCE_ERR_UNSUPPORTED_DEVICE;
    return VLMCE_OK;
}

}  // namespace vlmce

extern "C" const char *vlmce_last_error(void) { return vlmce::t_last_error; }

extern "C" const char *vlmce_status_string(int32_t status) {
    switch (status) {
        case VLMCE_OK: return "VLMCE_OK";
        case VLMCE_ERR_INVALID_ARG: return "VLMCE_ERR_INVALID_ARG: invalid argument";
        case VLMCE_ERR_UNSUPPORTED_DTYPE: return "VLMCE_ERR_UNSUPPORTED_DTYPE: unsupported dtype";
        case VLMCE_ERR_MISALIGNED: return "VLMCE_ERR_MISALIGNED: pointer not aligned as required";
        case VLMCE_ERR_UNSUPPORTED_DEVICE:
            return "VLMCE_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 (sm_103a) GPU";
        case VLMCE_ERR_WORKSPACE_TOO_SMALL:
            return "VLMCE_ERR_WORKSPACE_TOO_SMALL: workspace missing or too small";
        case VLMCE_ERR_CUDA: return "VLMCE_ERR_CUDA: CUDA runtime call or kernel launch failed";
        case VLMCE_ERR_TOO_LARGE: return "VLMCE_ERR_TOO_LARGE: size beyond what the kernels support";
        default: return "VLMCE: unknown status";
    }
}
