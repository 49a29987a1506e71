// ce_census.cuh -- the label census and the final reduction of the
// cross-entropy entry points (ce.cu, ce_shard.cu): one CTA each.
//   ce_count_kernel    -- n_valid (labels in [0, V)) and bad labels (neither
//                         ignore_index nor in range); clears the error word.
//   ce_finalize_kernel -- fixed-order fp64 sum of the per-row losses (mean or
//                         sum), token accuracy, the counts and error bits.
// Internal linkage: each translation unit that launches them has its own copy.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"
#include "vlmce.h"

namespace vlmce {
namespace ce {
namespace {

__global__ void __launch_bounds__(1024) ce_count_kernel(const int64_t *__restrict__ labels, int64_t N,
                                                     int64_t V, int64_t ignore_index,
                                                     int64_t *counts, int *err) {
    ptx::griddep_launch_dependents();
    long long nv = 0, nb = 0;
    const int64_t st = blockDim.x;
    // four labels in flight per thread (the loop is load-latency bound)
    for (int64_t r0 = threadIdx.x; r0 < N; r0 += 4 * st) {
        int64_t y[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) y[u] = r0 + u * st < N ? labels[r0 + u * st] : ignore_index;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (y[u] == ignore_index) continue;
            if (y[u] >= 0 && y[u] < V)
                ++nv;
            else
                ++nb;
        }
    }
    __shared__ long long sv[32], sb[32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        nv += __shfl_xor_sync(0xffffffffu, nv, off);
        nb += __shfl_xor_sync(0xffffffffu, nb, off);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sv[warp] = nv;
        sb[warp] = nb;
    }
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        nv = lane < nw ? sv[lane] : 0;
        nb = lane < nw ? sb[lane] : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            nv += __shfl_xor_sync(0xffffffffu, nv, off);
            nb += __shfl_xor_sync(0xffffffffu, nb, off);
        }
        if (lane == 0) {
            counts[0] = nv;
            counts[1] = nb;
            *err = 0;
        }
    }
}

__global__ void __launch_bounds__(1024) ce_finalize_kernel(
    const float *__restrict__ loss, const int64_t *__restrict__ argmax,
    const int64_t *__restrict__ labels, int64_t N, int64_t V, int64_t ignore_index, int reduction,
    const int64_t *counts, const int *err, float *out_reduced, int64_t *out_counts) {
    ptx::griddep_wait();
    double acc = 0.0;
    long long nc = 0;
    const int64_t st = blockDim.x;
    // four rows' values in flight per thread (the loop is load-latency bound);
    // each thread still adds its rows r, r + st, r + 2 st, ... in that order
    for (int64_t r0 = threadIdx.x; r0 < N; r0 += 4 * st) {
        int64_t y[4], am[4];
        float l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t r = r0 + u * st;
            y[u] = r < N ? labels[r] : ignore_index;
            l[u] = r < N ? loss[r] : 0.f;
            am[u] = r < N ? argmax[r] : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (y[u] == ignore_index) continue;
            acc += static_cast<double>(l[u]);
            if (y[u] >= 0 && y[u] < V && am[u] == y[u]) ++nc;
        }
    }
    __shared__ double sa[32];
    __shared__ long long sc[32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
        nc += __shfl_xor_sync(0xffffffffu, nc, off);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sa[warp] = acc;
        sc[warp] = nc;
    }
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        acc = lane < nw ? sa[lane] : 0.0;
        nc = lane < nw ? sc[lane] : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
            nc += __shfl_xor_sync(0xffffffffu, nc, off);
        }
        if (lane == 0) {
            const long long nv = counts[0];
            double red = acc;
            if (reduction == VLMCE_MEAN) red = nv > 0 ? acc / static_cast<double>(nv) : 0.0;
            const double accuracy = nv > 0 ? static_cast<double>(nc) / static_cast<double>(nv) : 0.0;
            if (out_reduced) {
                out_reduced[0] = static_cast<float>(red);
                out_reduced[1] = static_cast<float>(accuracy);
            }
            if (out_counts) {
                out_counts[0] = nv;
                out_counts[1] = nc;
                out_counts[2] = counts[1];
                out_counts[3] = *err;
            }
        }
    }
}

}  // namespace
}  // namespace ce
}  // namespace vlmce
