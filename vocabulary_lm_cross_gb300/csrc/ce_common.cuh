// ce_common.cuh -- device helpers shared by the cross-entropy kernels: row
// statistics and their merge, the softcap, packed fp32x2 arithmetic, bf16/fp32
// granule (16-byte) unpacking, packing and stores.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ptx.cuh"
#include "vlmce.h"

namespace vlmce {
namespace ce {

constexpr float kLog2e = 1.4426950408889634f;

// One CTA's (or warp's, or thread's) statistics of one row.
struct __align__(16) RowPart {
    float mx;   // max of the raw logits x
    int idx;    // smallest column holding mx
    float mz;   // reference of s (z space), >= every z folded
    float s;    // sum exp(z - mz)
    float sz;   // sum z
    float zy;   // z at the label column (only its owner adds it)
    float pad0, pad1;
};

template <bool BF16>
struct Elem {
    static constexpr int kBytes = BF16 ? 2 : 4;
    static constexpr int kPerGranule = 16 / kBytes;
};

// ----------------------------------------------------------- packed fp32x2
__device__ __forceinline__ uint64_t pk(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t ex2x2(uint64_t a) {
    float x, y;
    upk(a, x, y);
    return pk(ptx::ex2(x), ptx::ex2(y));
}

__device__ __forceinline__ RowPart part_identity() {
    RowPart p;
    p.mx = -INFINITY;
    p.idx = INT_MAX;
    p.mz = -INFINITY;
    p.s = 0.f;
    p.sz = 0.f;
    p.zy = 0.f;
    p.pad0 = p.pad1 = 0.f;
    return p;
}

// a <- merge(a, b).  Commutative, so a butterfly leaves every lane identical.
__device__ __forceinline__ void part_merge(RowPart &a, float mx, int idx, float mz, float s,
                                           float sz, float zy) {
    if (mx > a.mx || (mx == a.mx && idx < a.idx)) {
        a.mx = mx;
        a.idx = idx;
    }
    const float M = fmaxf(a.mz, mz);
    const float u = (a.s == 0.f) ? 0.f : a.s * ptx::ex2((a.mz - M) * kLog2e);
    const float v = (s == 0.f) ? 0.f : s * ptx::ex2((mz - M) * kLog2e);
    a.mz = M;
    a.s = u + v;
    a.sz = a.sz + sz;
    a.zy = a.zy + zy;
}

__device__ __forceinline__ void warp_allreduce(RowPart &p) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float mx = __shfl_xor_sync(0xffffffffu, p.mx, off);
        const int idx = __shfl_xor_sync(0xffffffffu, p.idx, off);
        const float mz = __shfl_xor_sync(0xffffffffu, p.mz, off);
        const float s = __shfl_xor_sync(0xffffffffu, p.s, off);
        const float sz = __shfl_xor_sync(0xffffffffu, p.sz, off);
        const float zy = __shfl_xor_sync(0xffffffffu, p.zy, off);
        part_merge(p, mx, idx, mz, s, sz, zy);
    }
}

// z = T tanh(x/T) and dz/dx = 1 - tanh^2, from tanh(u) = sign(u) (1 - a) / (1 + a),
// a = exp(-2|u|), so that 1 - tanh^2 = 4 a / (1 + a)^2 needs no extra MUFU op.
struct Capped {
    float z, dz;
};
template <bool SOFTCAP>
__device__ __forceinline__ Capped softcap_z(float x, float T, float neg2_log2e_over_T) {
    if constexpr (!SOFTCAP) {
        return {x, 1.f};
    } else {
        const float a = ptx::ex2(fabsf(x) * neg2_log2e_over_T);
        const float r = ptx::rcp(1.f + a);
        const float t = copysignf((1.f - a) * r, x);
        return {T * t, 4.f * a * r * r};
    }
}

// The same softcap, two columns at a time, for the memory-bound row kernels,
// which are bound by instruction issue and the MUFU unit when a softcap is
// set.  a = exp(-2|x|/T) is the one MUFU op; r = 1/(1 + a) is formed in packed
// fp32x2 arithmetic on the FMA pipe (one issue slot per two columns) by
// Newton-type steps from the minimax line of 1/d on d = 1 + a in [1, 2]:
//   r0 = 16/17 - (8/17) a                   |1 - d r0| <= 1/17
//   r1 = r0 (1 + e + e^2),  e = 1 - d r0     |1 - d r1| = |e|^3 <= 2.1e-4
//   r2 = r1 (1 + e),        e = 1 - d r1     |1 - d r2| = e^2  <= 4.2e-8
// (plus the rounding of the last FMA): about one ulp, like the MUFU
// reciprocal.  tanh(|x|/T) = (1 - a) r = 2 r - 1 (absolute error about 1e-7,
// i.e. about 3e-6 in z at T = 30), and 1 - tanh^2 = 4 a r^2, which stays
// accurate where tanh is close to 1.
struct Cap2 {
    uint64_t t;    // tanh(x/T) of the two columns, with the sign of x
    uint64_t ar2;  // a r^2 of the two columns (dz/dx = 4 a r^2)
};
__device__ __forceinline__ Cap2 softcap2(float x0, float x1, float neg2_log2e_over_T) {
    const uint64_t a = pk(ptx::ex2(fabsf(x0) * neg2_log2e_over_T),
                          ptx::ex2(fabsf(x1) * neg2_log2e_over_T));
    const uint64_t one = pk(1.f, 1.f), m_one = pk(-1.f, -1.f);
    const uint64_t nd = fma2(a, m_one, m_one);  // -(1 + a)
    uint64_t r = fma2(a, pk(-8.f / 17.f, -8.f / 17.f), pk(16.f / 17.f, 16.f / 17.f));
    uint64_t e = fma2(nd, r, one);
    r = fma2(r, fma2(e, e, e), r);
    e = fma2(nd, r, one);
    r = fma2(r, e, r);
    float t0, t1;
    upk(fma2(r, pk(2.f, 2.f), m_one), t0, t1);  // 2 r - 1
    Cap2 c;
    c.t = pk(copysignf(t0, x0), copysignf(t1, x1));
    c.ar2 = mul2(mul2(a, r), r);
    return c;
}
// ---------------------------------------------------- polynomial softcap
// Where |x| <= 0.55 T (nearly every column at the softcaps the pages use),
// tanh(x/T) = u P(u^2) with u = x/T and P the degree-4 least-squares fit of
// tanh(u)/u on u in [0, 0.55] (relative error 3.3e-8 at 4000 Chebyshev nodes;
// measured fp32 error of t below 8e-8).  The row kernels evaluate it as
// x Q(x^2), Q's i-th coefficient P's divided by T^(2i+1) (ce_rows.cuh): six
// packed fp32x2 FMA-pipe ops per column pair and no MUFU op, against about
// twelve and two MUFU ops for softcap2.  There 1 - t^2 >= 0.75 is formed
// directly, with no cancellation.  Columns beyond 0.55 T keep softcap2.
constexpr float kPolyRange = 0.55f;
// P's coefficients, constant term first
constexpr float kTanhP0 = 0.9999999667018895f;
constexpr float kTanhP1 = -0.33332785337019116f;
constexpr float kTanhP2 = 0.13318718793849865f;
constexpr float kTanhP3 = -0.05258102516972439f;
constexpr float kTanhP4 = 0.016301813790173283f;

struct PolyCap {
    float rT;       // 1 / T
    float lim;      // 0.55 T
    uint32_t lim2;  // bf16x2: the largest bf16 at most 0.55 T, in both halves
};
__device__ __forceinline__ PolyCap poly_cap(float T) {
    PolyCap pc;
    pc.rT = 1.f / T;
    pc.lim = kPolyRange * T;
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rd(pc.lim));
    pc.lim2 = h | (h << 16);
    return pc;
}

// tanh(x/T) of one column, by the same arithmetic as softcap2.
__device__ __forceinline__ float softcap_t1(float x, float neg2_log2e_over_T) {
    float t0, t1;
    upk(softcap2(x, x, neg2_log2e_over_T).t, t0, t1);
    return t0;
}

template <bool BF16>
__device__ __forceinline__ void unpack(const uint4 w, float (&x)[Elem<BF16>::kPerGranule]) {
    if constexpr (BF16) {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            x[2 * q] = __uint_as_float(u[q] << 16);
            x[2 * q + 1] = __uint_as_float(u[q] & 0xffff0000u);
        }
    } else {
        x[0] = __uint_as_float(w.x);
        x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z);
        x[3] = __uint_as_float(w.w);
    }
}

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t u) {
    __nv_bfloat162 r;
    memcpy(&r, &u, 4);
    return r;
}

// Max of a full granule (packed bf16x2 max for bf16).
template <bool BF16>
__device__ __forceinline__ float granule_max(const uint4 w) {
    if constexpr (BF16) {
        const __nv_bfloat162 a = __hmax2(as_bf162(w.x), as_bf162(w.y));
        const __nv_bfloat162 b = __hmax2(as_bf162(w.z), as_bf162(w.w));
        const __nv_bfloat162 c = __hmax2(a, b);
        return fmaxf(__low2float(c), __high2float(c));
    } else {
        return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                     fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
}

// ------------------------------------------- gradients in the subnormal range
// ex2.approx.ftz returns 0 once its result would be subnormal (exponent e <
// -126), while scale p_j can still be a representable fp32 / bf16 subnormal
// gradient.  The gradient kernels therefore form 2^(e + 24) -- the 24 folded
// into the per-row constant -lse log2 e, at no extra instruction -- and move
// the 2^-24 into the coefficient that multiplies it: results down to 2^-150
// (below the smallest fp32 subnormal) are then rounded once, by the fused
// multiply-add that applies the coefficient.  The cost is the rounding of the
// biased exponent (magnitude up to 24 for the largest p_j: about 1e-6
// relative), far below a bf16 ulp and within the fp32 parity bound.  Rows
// whose scale is below 2^-100 keep the unbiased exponent (scale 2^-24 would
// itself be subnormal there, and their gradients underflow anyway).
constexpr float kGradExpBias = 24.f;
constexpr float kGradExpBiasScale = 5.9604644775390625e-8f;  // 2^-24
constexpr float kMinBiasedScale = 7.8886090522101181e-31f;   // 2^-100

// The per-row exponent constant (-lse log2 e, plus the bias) and the
// coefficient of 2^e (scale, times 2^-bias) of a row's gradient.
struct ExpCoef {
    float nlseL, scale;
};
__device__ __forceinline__ ExpCoef grad_exp_coef(float lse, float scale) {
    const bool bias = fabsf(scale) >= kMinBiasedScale;
    ExpCoef c;
    c.nlseL = fmaf(-lse, kLog2e, bias ? kGradExpBias : 0.f);
    c.scale = bias ? scale * kGradExpBiasScale : scale;
    return c;
}

// Whether every value of a whole granule lies within the polynomial
// softcap's range (|x| <= 0.55 T); NaN counts as outside.
template <bool BF16>
__device__ __forceinline__ bool granule_in_poly_range(const uint4 w, const PolyCap &pc) {
    if constexpr (BF16) {
        const __nv_bfloat162 mx =
            __hmax2(__hmax2(as_bf162(w.x), as_bf162(w.y)), __hmax2(as_bf162(w.z), as_bf162(w.w)));
        const __nv_bfloat162 mn =
            __hmin2(__hmin2(as_bf162(w.x), as_bf162(w.y)), __hmin2(as_bf162(w.z), as_bf162(w.w)));
        uint32_t nmn;
        memcpy(&nmn, &mn, 4);
        nmn ^= 0x80008000u;  // -min
        return __hble2(__hmax2(mx, as_bf162(nmn)), as_bf162(pc.lim2));
    } else {
        const float m = fmaxf(fmaxf(fabsf(__uint_as_float(w.x)), fabsf(__uint_as_float(w.y))),
                              fmaxf(fabsf(__uint_as_float(w.z)), fabsf(__uint_as_float(w.w))));
        return m <= pc.lim;
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    uint32_t u;
    memcpy(&u, &v, 4);
    return u;
}

template <bool BF16>
__device__ __forceinline__ void store_elem(unsigned char *p, float g) {
    if constexpr (BF16) {
        const __nv_bfloat16 b = __float2bfloat16_rn(g);
        uint16_t u;
        memcpy(&u, &b, 2);
        *reinterpret_cast<uint16_t *>(p) = u;
    } else {
        *reinterpret_cast<float *>(p) = g;
    }
}

}  // namespace ce
}  // namespace vlmce
