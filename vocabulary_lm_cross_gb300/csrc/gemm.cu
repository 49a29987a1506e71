// gemm.cu -- host side of the tcgen05 GEMM: operand tensor maps, the
// co-resident cluster count of the device and the cluster launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gemm.cuh"
#include "gemm_launch.h"

namespace vlmce {
namespace gemm {
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static std::once_flag once;
    static EncodeTiled fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// A bf16 matrix of `outer` rows of `inner` elements (row stride `stride`
// elements), read in boxes of box_inner x box_outer with 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t stride,
              uint32_t box_inner, uint32_t box_outer, bool f16) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;

// Clusters of `csize` CTAs that fit on the device at once (SMs of a GPC
// that cannot complete a cluster stay idle); cached per device.
int co_resident_clusters(int device, int csize, cudaError_t *err) {
    static std::mutex mu;
    static int cached[kMaxDevices] = {};
    static bool attr_done = false;
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(vlmce_gemm_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) {
            *err = e;
            return 0;
        }
        attr_done = true;
    }
    if (device >= 0 && device < kMaxDevices && cached[device] > 0) return cached[device];
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(csize, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, vlmce_gemm_kernel, &cfg);
    if (e != cudaSuccess || n < 1) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
        return 0;
    }
    if (device >= 0 && device < kMaxDevices) cached[device] = n;
    return n;
}

}  // namespace

bool make_operand_map(CUtensorMap *m, const void *base, bool mn, int64_t rows, int64_t K,
                      int64_t ld, bool f16) {
    if (mn) return make_map(m, base, rows, K, ld, 64, 64, f16);
    return make_map(m, base, K, rows, ld, 64, kHalf, f16);
}

cudaError_t launch_group(const Maps &maps, Params &a, cudaStream_t s) {
    int tiles = 0;
    for (int i = 0; i < a.nprob; ++i) {
        Problem &p = a.p[i];
        p.mt = (p.M + BM - 1) / BM;
        p.tile0 = tiles;
        tiles += p.mt * ((p.N + BN - 1) / BN);
    }
    a.tiles = tiles;
    if (tiles < 1) return cudaSuccess;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    e = cudaSuccess;
    constexpr int csize = 2;  // one CTA pair
    const int clusters_max = co_resident_clusters(device, csize, &e);
    if (clusters_max < 1) return e;
    const int clusters = tiles < clusters_max ? tiles : clusters_max;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(csize * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, vlmce_gemm_kernel, maps, static_cast<const Params>(a));
}

}  // namespace gemm
}  // namespace vlmce
