// swiglu.cu -- the fused gate-up SwiGLU of a Megatron MLP ("[Megatron] Add
// SwiGLU integration", Summary and Background): the first linear layer writes
// one [tokens, 2n] tensor, gate in columns [0, n) and up in [n, 2n); the
// activation reads both halves of each row in place (no split copies):
//
//   forward   y       = silu(gate) up                     ([tokens, n])
//   backward  d_gate  = dy up sigma(gate) (1 + gate (1 - sigma(gate)))
//             d_up    = dy silu(gate)                      ([tokens, 2n], may be x itself)
//
// with silu(a) = a sigma(a), sigma(a) = 1 / (1 + exp(-a)), all in fp32 and
// rounded to the storage dtype (round to nearest even).  Memory-bound: each
// thread moves 16-byte granules (8 bf16 or 4 fp32 elements) of the gate and
// up halves of a row; rows of a CTA's grid column are visited in a stride
// loop.  A scalar variant handles rows that are not 16-byte aligned.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ce_common.cuh"
#include "host_util.h"
#include "ptx.cuh"
#include "vlmce.h"

namespace vlmce {
namespace swiglu {
namespace {

constexpr int kThreads = 256;

struct Params {
    const unsigned char *x;   // [T, x_stride]: gate | up
    const unsigned char *dy;  // backward: [T, dy_stride]
    unsigned char *out;       // forward: y [T, out_stride]; backward: dx [T, out_stride]
    int64_t T, n;
    int64_t x_stride, dy_stride, out_stride;  // bytes
};

// sigma(a) on the MUFU unit: 1 / (1 + 2^(-a log2 e)); 0 and 1 at the extremes.
__device__ __forceinline__ float sigmoid(float a) {
    return ptx::rcp(1.f + ptx::ex2(-a * ce::kLog2e));
}

template <bool BF16>
__device__ __forceinline__ void load8(const unsigned char *p, float (&v)[ce::Elem<BF16>::kPerGranule]) {
    uint4 w;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                 : "l"(p));
    ce::unpack<BF16>(w, v);
}

template <bool BF16>
__device__ __forceinline__ uint4 pack(const float (&v)[ce::Elem<BF16>::kPerGranule]) {
    if constexpr (BF16)
        return make_uint4(ce::pack_bf16x2(v[0], v[1]), ce::pack_bf16x2(v[2], v[3]),
                          ce::pack_bf16x2(v[4], v[5]), ce::pack_bf16x2(v[6], v[7]));
    else
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
}

// Vector path: n, the strides and the bases are multiples of 16 bytes.
template <bool BF16, bool BWD>
__global__ void __launch_bounds__(kThreads) swiglu_vec_kernel(const Params p) {
    constexpr int EPG = ce::Elem<BF16>::kPerGranule;
    const int64_t ng = p.n / EPG;  // granules per half row
    const int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (g >= ng) return;
    const int64_t off = 16 * g;
    const int64_t half = p.n * (BF16 ? 2 : 4);
    for (int64_t r = blockIdx.y; r < p.T; r += gridDim.y) {
        const unsigned char *xr = p.x + r * p.x_stride;
        float a[EPG], b[EPG];
        load8<BF16>(xr + off, a);
        load8<BF16>(xr + half + off, b);
        if constexpr (!BWD) {
            float y[EPG];
#pragma unroll
            for (int l = 0; l < EPG; ++l) y[l] = a[l] * sigmoid(a[l]) * b[l];
            ptx::st_global_cs_v4(p.out + r * p.out_stride + off, pack<BF16>(y));
        } else {
            float d[EPG], dg[EPG], du[EPG];
            load8<BF16>(p.dy + r * p.dy_stride + off, d);
#pragma unroll
            for (int l = 0; l < EPG; ++l) {
                const float s = sigmoid(a[l]);
                const float silu = a[l] * s;
                du[l] = d[l] * silu;
                dg[l] = d[l] * b[l] * fmaf(silu, 1.f - s, s);  // sigma (1 + a (1 - sigma))
            }
            unsigned char *orow = p.out + r * p.out_stride;
            ptx::st_global_cs_v4(orow + off, pack<BF16>(dg));
            ptx::st_global_cs_v4(orow + half + off, pack<BF16>(du));
        }
    }
}

template <bool BF16>
__device__ __forceinline__ float ld1(const unsigned char *p) {
    if constexpr (BF16)
        return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(p)) << 16);
    else
        return *reinterpret_cast<const float *>(p);
}

// Scalar path: one element per thread and row.
template <bool BF16, bool BWD>
__global__ void __launch_bounds__(kThreads) swiglu_scalar_kernel(const Params p) {
    constexpr int ELT = BF16 ? 2 : 4;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (j >= p.n) return;
    const int64_t half = p.n * ELT;
    for (int64_t r = blockIdx.y; r < p.T; r += gridDim.y) {
        const unsigned char *xr = p.x + r * p.x_stride + ELT * j;
        const float a = ld1<BF16>(xr), b = ld1<BF16>(xr + half);
        unsigned char *orow = p.out + r * p.out_stride + ELT * j;
        if constexpr (!BWD) {
            ce::store_elem<BF16>(orow, a * sigmoid(a) * b);
        } else {
            const float d = ld1<BF16>(p.dy + r * p.dy_stride + ELT * j);
            const float s = sigmoid(a);
            const float silu = a * s;
            ce::store_elem<BF16>(orow, d * b * fmaf(silu, 1.f - s, s));
            ce::store_elem<BF16>(orow + half, d * silu);
        }
    }
}

using Kernel = void (*)(Params);

vlmce_status run(const void *x, const void *dy, void *out, int32_t dtype, int64_t T, int64_t n,
                 int64_t x_stride, int64_t dy_stride, int64_t out_stride, bool bwd,
                 cudaStream_t s) {
    if (dtype != VLMCE_F32 && dtype != VLMCE_BF16) return VLMCE_ERR_UNSUPPORTED_DTYPE;
    if (T < 0 || n < 1 || x_stride < 2 * n || out_stride < (bwd ? 2 * n : n) ||
        (bwd && dy_stride < n))
        return VLMCE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !out || (bwd && !dy))) return VLMCE_ERR_INVALID_ARG;
    const int64_t elt = dtype == VLMCE_BF16 ? 2 : 4;
    if (n > (INT64_MAX / 4) / elt || (T > 0 && (x_stride > (INT64_MAX / elt) / T ||
                                                out_stride > (INT64_MAX / elt) / T ||
                                                dy_stride > (INT64_MAX / elt) / T)))
        return VLMCE_ERR_TOO_LARGE;
    if (!aligned(x, static_cast<uintptr_t>(elt)) || !aligned(out, static_cast<uintptr_t>(elt)) ||
        (bwd && !aligned(dy, static_cast<uintptr_t>(elt))))
        return VLMCE_ERR_MISALIGNED;
    if (!bwd && out && x) {
        // y must not overlap the input rows it is computed from (dx may be x itself)
        const uintptr_t xb = reinterpret_cast<uintptr_t>(x), ob = reinterpret_cast<uintptr_t>(out);
        if (T > 0 && ob < xb + static_cast<uintptr_t>((T - 1) * x_stride + 2 * n) * elt &&
            xb < ob + static_cast<uintptr_t>((T - 1) * out_stride + n) * elt)
            return VLMCE_ERR_INVALID_ARG;
    }
    if (T == 0) return VLMCE_OK;
    DeviceInfo dev;
    vlmce_status st = current_device(&dev);
    if (st != VLMCE_OK) return st;
    const int64_t epg = 16 / elt;
    const bool vec = (n % epg) == 0 && (x_stride % epg) == 0 && (out_stride % epg) == 0 &&
                     (!bwd || (dy_stride % epg) == 0) && aligned(x, 16) && aligned(out, 16) &&
                     (!bwd || aligned(dy, 16));
    Params p;
    p.x = static_cast<const unsigned char *>(x);
    p.dy = static_cast<const unsigned char *>(dy);
    p.out = static_cast<unsigned char *>(out);
    p.T = T;
    p.n = n;
    p.x_stride = x_stride * elt;
    p.dy_stride = dy_stride * elt;
    p.out_stride = out_stride * elt;
    const int64_t cols = vec ? n / epg : n;
    const int64_t gx = (cols + kThreads - 1) / kThreads;
    if (gx > INT_MAX) return VLMCE_ERR_TOO_LARGE;
    // enough CTAs to fill every SM several times over; rows strided over grid.y
    int64_t want_y = (static_cast<int64_t>(dev.sm_count) * 8 * 4 + gx - 1) / gx;
    if (want_y > T) want_y = T;
    if (want_y > 65535) want_y = 65535;
    if (want_y < 1) want_y = 1;
    const bool bf16 = dtype == VLMCE_BF16;
    Kernel k;
    if (vec)
        k = bf16 ? (bwd ? swiglu_vec_kernel<true, true> : swiglu_vec_kernel<true, false>)
                 : (bwd ? swiglu_vec_kernel<false, true> : swiglu_vec_kernel<false, false>);
    else
        k = bf16 ? (bwd ? swiglu_scalar_kernel<true, true> : swiglu_scalar_kernel<true, false>)
                 : (bwd ? swiglu_scalar_kernel<false, true> : swiglu_scalar_kernel<false, false>);
    k<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(want_y), 1), kThreads, 0, s>>>(p);
    return launch_status(cudaSuccess, bwd ? "swiglu_bwd" : "swiglu_fwd");
}

}  // namespace
}  // namespace swiglu
}  // namespace vlmce

extern "C" vlmce_status swiglu_fwd(const void *x, int32_t dtype, int64_t T, int64_t n,
                                   int64_t x_stride, void *y, int64_t y_stride,
                                   vlmce_stream_t stream) {
    return vlmce::swiglu::run(x, nullptr, y, dtype, T, n, x_stride, 0, y_stride, false,
                              reinterpret_cast<cudaStream_t>(stream));
}

extern "C" vlmce_status swiglu_bwd(const void *x, int64_t x_stride, const void *dy,
                                   int64_t dy_stride, void *dx, int64_t dx_stride, int32_t dtype,
                                   int64_t T, int64_t n, vlmce_stream_t stream) {
    return vlmce::swiglu::run(x, dy, dx, dtype, T, n, x_stride, dy_stride, dx_stride, true,
                              reinterpret_cast<cudaStream_t>(stream));
}
