// ce_census.cuh -- the label census and the final reduction of the
// cross-entropy entry points (ce.cu, ce_shard.cu): one CTA each.
//   ce_count_kernel    -- n_valid (labels in [0, V)) and bad labels (neither
//                         ignore_index nor in range); clears the error word.
//   ce_finalize_kernel -- fixed-order float-float sum of the per-row losses
//                         (mean or sum), token accuracy, the counts and error
//                         bits.
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
    // Launched dependent on whatever precedes it on the stream: it waits for
    // that work (whose results the row work may read), then lets the row
    // work start while it counts.
    ptx::griddep_wait();
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

// Float-float sum hi + lo: each addend goes through Knuth's TwoSum with hi
// and its rounding error is gathered in lo, so fixed-order sums of the
// per-row losses keep about 44 bits with fp32 arithmetic only (this GPU's
// fp64 rate is a small fraction of its fp32 rate).
struct FloatFloat {
    float hi, lo;
};
__device__ __forceinline__ void ff_add(FloatFloat &a, float b) {
    const float s = a.hi + b;
    const float bb = s - a.hi;
    const float e = (a.hi - (s - bb)) + (b - bb);
    a.hi = s;
    a.lo += e;
}
__device__ __forceinline__ void ff_add(FloatFloat &a, const FloatFloat &b) {
    ff_add(a, b.hi);
    a.lo += b.lo;
}

__global__ void __launch_bounds__(1024) ce_finalize_kernel(
    const float *__restrict__ loss, const int64_t *__restrict__ argmax,
    const int64_t *__restrict__ labels, int64_t N, int64_t V, int64_t ignore_index, int reduction,
    const int64_t *counts, const int *err, float *out_reduced, int64_t *out_counts) {
    // the next call's census may be scheduled now (it waits for this kernel
    // before it reads anything); this kernel waits for the row work
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    FloatFloat acc = {0.f, 0.f};
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
            ff_add(acc, l[u]);
            if (y[u] >= 0 && y[u] < V && am[u] == y[u]) ++nc;
        }
    }
    __shared__ FloatFloat sa[32];
    __shared__ long long sc[32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const FloatFloat o = {__shfl_xor_sync(0xffffffffu, acc.hi, off),
                              __shfl_xor_sync(0xffffffffu, acc.lo, off)};
        ff_add(acc, o);
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
        acc = lane < nw ? sa[lane] : FloatFloat{0.f, 0.f};
        nc = lane < nw ? sc[lane] : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const FloatFloat o = {__shfl_xor_sync(0xffffffffu, acc.hi, off),
                                  __shfl_xor_sync(0xffffffffu, acc.lo, off)};
            ff_add(acc, o);
            nc += __shfl_xor_sync(0xffffffffu, nc, off);
        }
        if (lane == 0) {
            const long long nv = counts[0];
            double red = static_cast<double>(acc.hi) + static_cast<double>(acc.lo);
            if (reduction == VLMCE_MEAN) red = nv > 0 ? red / static_cast<double>(nv) : 0.0;
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
