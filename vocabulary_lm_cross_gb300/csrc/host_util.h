// host_util.h -- host-side helpers shared by the entry points: device
// properties cache, alignment checks, launch-error mapping.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "vlmce.h"

namespace vlmce {

struct DeviceInfo {
    int device = -1;
    int cc_major = 0, cc_minor = 0;
    int sm_count = 0;
    int smem_optin = 0;  // max dynamic shared memory per block (bytes)
};

// Properties of the current device, cached per device.  Returns VLMCE_OK,
// VLMCE_ERR_CUDA (no device / runtime error) or VLMCE_ERR_UNSUPPORTED_DEVICE.
vlmce_status current_device(DeviceInfo *out);

inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Remember a failed CUDA call (per host thread) for vlmce_last_error(), and
// clear the runtime's error state.  Returns `e`.
cudaError_t record_cuda(cudaError_t e, const char *where);

// Status of a launch: `e` from the launch API, else the runtime's last error.
inline vlmce_status launch_status(cudaError_t e, const char *where) {
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) return VLMCE_OK;
    record_cuda(e, where);
    return VLMCE_ERR_CUDA;
}

}  // namespace vlmce
