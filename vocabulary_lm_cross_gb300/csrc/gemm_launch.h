// gemm_launch.h -- host-side launchers of the tcgen05 GEMM instantiations
// (gemm_kk.cu, gemm_km.cu, gemm_mk.cu, gemm_mm.cu: K- or MN-major A and B).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm.cuh"

namespace vlmce {
namespace gemm {

// Launch mode `mode` (gemm::Mode) on `grid` CTAs; returns the launch error.
cudaError_t launch_kk(int mode, const CUtensorMap &a, const CUtensorMap &b, const Args &args,
                      int grid, cudaStream_t s);
cudaError_t launch_km(int mode, const CUtensorMap &a, const CUtensorMap &b, const Args &args,
                      int grid, cudaStream_t s);
cudaError_t launch_mk(int mode, const CUtensorMap &a, const CUtensorMap &b, const Args &args,
                      int grid, cudaStream_t s);
cudaError_t launch_mm(int mode, const CUtensorMap &a, const CUtensorMap &b, const Args &args,
                      int grid, cudaStream_t s);

}  // namespace gemm
}  // namespace vlmce
