// gemm_launch.h -- host side of the tcgen05 GEMM (gemm.cuh): tensor maps of
// the operands and the launch of a group of up to kMaxProblems products.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_types.h"

namespace vlmce {
namespace gemm {

// Tensor map of operand A (rows = M) or B (rows = N) of C = A B^T, bf16
// (fp16 with f16): K-major ([rows, ld], K contiguous; boxes of 64 K x 128
// rows) or MN-major ([K, ld], rows contiguous; boxes of 64 x 64).
// Out-of-range elements read as zero.  False if the driver refuses it.
bool make_operand_map(CUtensorMap *m, const void *base, bool mn, int64_t rows, int64_t K,
                      int64_t ld, bool f16 = false);

// Fill p.mt / p.tile0 / a.tiles from the problems' shapes and launch them on
// `s` as one persistent grid of clusters of one CTA pair (a.nprob
// problems, maps.a/b[i] for problem i).  Returns the launch error.
cudaError_t launch_group(const Maps &maps, Params &a, cudaStream_t s);

}  // namespace gemm
}  // namespace vlmce
