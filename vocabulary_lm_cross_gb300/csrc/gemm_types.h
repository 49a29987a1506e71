// gemm_types.h -- shapes, modes and launch parameters of the tcgen05 GEMM
// (the kernel is in gemm.cuh, its host side in gemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "ce_common.cuh"

namespace vlmce {
namespace gemm {

constexpr int BM = 256, BN = 256, BK = 128;  // pair tile
constexpr int kHalf = 128;                  // rows of A and of B held by one CTA
constexpr int kStages = 3;
constexpr int kOpBytes = kHalf * BK * 2;    // 32 KB per operand per stage
constexpr int kStageBytes = 2 * kOpBytes;   // 64 KB per CTA
constexpr int kThreads = 224;
constexpr int kTmemCols = 2 * BN;
// Dynamic tile order: a scheduler warp of the pair leader takes the next tile
// number from a counter in global memory and publishes it to both CTAs'
// roles through a queue of kTileQ slots.
constexpr int kTileQ = 4;
constexpr int kTileQConsumers = 11;  // leader: producer, MMA issuer, 4 epilogue warps; peer: producer, 4
// full, empty, tmem full x2, tmem empty x2, drain, tile queue full / empty
constexpr int kBarriers = 2 * kStages + 5 + 2 * kTileQ;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 8 * kBarriers + 16 + 4 * kTileQ;
constexpr int kMaxProblems = 3;
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

enum Mode : int {
    kStoreF32 = 0,   // C = acc (fp32)
    kAccF32 = 1,     // C += acc (fp32)
    kStats = 2,      // row statistics of the logits tile (fused linear CE, pass 1)
    kGrad = 3,       // gradient tile (p - q) (1 - t^2) grad_mul -> 16-bit (pass 2)
    kStoreBF16 = 4,  // C16 = 16-bit(acc)
    kAccToBF16 = 5,  // C16 = 16-bit(C + acc)
};

// One product of a launch.
struct Problem {
    int M, N, K;
    int mode;                  // Mode
    int a_mn, b_mn;            // operand stored MN-major
    int mt;                    // tiles along M
    int tile0;                 // number of the problem's first tile in the launch
    float *C;                  // fp32 [M, ldc]
    int64_t ldc;
    uint16_t *C16;             // bf16 or fp16 (Params::f16) [M, ldc16]
    int64_t ldc16;
    int col0;                  // kStats / kGrad: vocabulary column of n = 0
    ce::RowPart *part;         // kStats: part[n_tile * part_ld + row]
    int64_t part_ld;
};

struct Params {
    Problem p[kMaxProblems];
    int nprob;
    int tiles;                 // all problems' tiles
    // cross-entropy epilogues (shared by the problems of a launch)
    const int64_t *labels;     // [M]
    int64_t ignore_index;
    int V;                     // vocabulary size
    float eps, T, k2;          // smoothing, softcap (0 = off), -2 log2e / T
    const float *lse;          // kGrad: [M]
    const float *row_scale;    // kGrad: [M] nonzero for a valid row, 0 otherwise
    float grad_mul;            // kGrad: power of two the stored tile is multiplied by
    const float *out_scale;    // store modes: the accumulator is multiplied by *out_scale (null: 1)
    int f16;                   // operands and 16-bit outputs are fp16 (else bf16)
    int *err;                  // device error word (may be null)
    // null: cluster c runs tiles c, c + #clusters, ...; else the tiles are
    // taken in order from this counter (zero before the launch), so the
    // tiles in flight stay a window of consecutive numbers
    unsigned int *tile_ctr;
};

struct Maps {
    CUtensorMap a[kMaxProblems];  // K-major: box 64 K x 128 rows; MN-major: 64 x 64
    CUtensorMap b[kMaxProblems];
};

}  // namespace gemm
}  // namespace vlmce
