// gemm_mm.cu -- tcgen05 GEMM instantiations: A MN-major, B MN-major.
#include "gemm_launch.h"

namespace vlmce {
namespace gemm {
namespace {
template <int MODE>
cudaError_t launch_one(const CUtensorMap &a, const CUtensorMap &b, const Args &args, int grid,
                       cudaStream_t s) {
    auto kern = vlmce_gemm_kernel<MODE, true, true>;
    static bool attr_set = false;  // per process; the attribute is per function
    if (!attr_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    kern<<<grid, kThreads, kSmemBytes, s>>>(a, b, args);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_mm(int mode, const CUtensorMap &a, const CUtensorMap &b, const Args &args,
                      int grid, cudaStream_t s) {
    switch (mode) {
        case kStoreF32: return launch_one<kStoreF32>(a, b, args, grid, s);
        case kAccF32: return launch_one<kAccF32>(a, b, args, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gemm
}  // namespace vlmce
