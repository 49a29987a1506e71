// ce_rows.cuh -- the cross-entropy row kernel (default path): one CTA of 1024
// threads per row, two CTAs per SM (64 warps: every SM is fully occupied).
//
//   pass 1: one thread asks the bulk-copy engine to prefetch the whole row
//           into L2; all threads stream it in 16-byte granules: max and first
//           argmax of the raw logits, online sum of exp(z - m) and sum of z;
//   merge:  warp shuffles, then the 32 warp partials (fixed order);
//   pass 2: read the row again -- it is still in the 129 MB L2, since at most
//           2 x 152 rows (78 MB for 256 KB rows) are in flight -- and store the
//           gradient scale (p - q) (1 - t^2), rounded to the storage dtype,
//           with 16-byte evict-first stores over the logits.
// HBM sees one read and one write of every byte; the second read is served by
// L2.  The label census of the call is only needed by pass 2, so the kernel
// waits for it (programmatic dependent launch) after pass 1.
#pragma once

#include "ce_common.cuh"

namespace vlmce {
namespace ce {
namespace rows {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kPrefetchBytes = 65536;  // bytes per L2 bulk-prefetch instruction

struct Params {
    unsigned char *logits;
    const int64_t *labels;
    int V;
    int64_t stride_bytes;
    int64_t ignore_index;
    float eps;
    float softcap;
    float grad_scale;
    int reduction;
    float *loss;
    int64_t *argmax;
    const int64_t *counts;  // [0] n_valid (written by the count kernel)
};

using Kernel = void (*)(Params);

__device__ __forceinline__ uint4 ld_v4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Pass-1 state of one thread.
struct Acc {
    float mv;   // max raw logit seen
    int midx;   // its first column
    float mz;   // z of mv: reference of s
    float nmL;  // -mz log2e
    float s0, s1, z0, z1;
};

// Fold one granule (first column jg; granules come in column order).
template <bool BF16, bool SOFTCAP>
__device__ __forceinline__ void fold(Acc &a, const uint4 w, int jg, int V, float T, float k2) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    float x[EPG];
    unpack<BF16>(w, x);
    const bool full = jg >= 0 && jg + EPG <= V;
    float gm;
    if (full) {
        gm = granule_max<BF16>(w);
    } else {
        gm = -INFINITY;
#pragma unroll
        for (int l = 0; l < EPG; ++l)
            if (jg + l >= 0 && jg + l < V) gm = fmaxf(gm, x[l]);
    }
    if (gm > a.mv) {  // new maximum (rare after the first granules): locate it, rescale
        int li = EPG - 1;
#pragma unroll
        for (int l = EPG - 1; l >= 0; --l)
            if (x[l] == gm && jg + l >= 0 && jg + l < V) li = l;
        const float nz = softcap_z<SOFTCAP>(gm, T, k2).z;
        const float f = ptx::ex2((a.mz - nz) * kLog2e);
        a.s0 = (a.s0 == 0.f) ? 0.f : a.s0 * f;
        a.s1 = (a.s1 == 0.f) ? 0.f : a.s1 * f;
        a.mv = gm;
        a.midx = jg + li;
        a.mz = nz;
        a.nmL = -nz * kLog2e;
    }
    if (full) {
#pragma unroll
        for (int l = 0; l < EPG; l += 2) {
            const float za = softcap_z<SOFTCAP>(x[l], T, k2).z;
            const float zb = softcap_z<SOFTCAP>(x[l + 1], T, k2).z;
            a.s0 += ptx::ex2(fmaf(za, kLog2e, a.nmL));
            a.s1 += ptx::ex2(fmaf(zb, kLog2e, a.nmL));
            a.z0 += za;
            a.z1 += zb;
        }
    } else {
#pragma unroll
        for (int l = 0; l < EPG; ++l) {
            if (jg + l >= 0 && jg + l < V) {
                const float z = softcap_z<SOFTCAP>(x[l], T, k2).z;
                a.s0 += ptx::ex2(fmaf(z, kLog2e, a.nmL));
                a.z0 += z;
            }
        }
    }
}

// Gradient of one granule, stored over the logits.
template <bool BF16, bool SOFTCAP>
__device__ __forceinline__ void grad_granule(const uint4 w, int jg, int V, unsigned char *dst,
                                             float T, float k2, float nlseL, float scale,
                                             float c_smooth, float c_label, int label_lane) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    constexpr int ELT = Elem<BF16>::kBytes;
    float x[EPG], g[EPG];
    unpack<BF16>(w, x);
#pragma unroll
    for (int l = 0; l < EPG; ++l) {
        const Capped c = softcap_z<SOFTCAP>(x[l], T, k2);
        const float pr = ptx::ex2(fmaf(c.z, kLog2e, nlseL));  // p_j
        g[l] = fmaf(pr, scale, (l == label_lane) ? -c_label : -c_smooth);
        if constexpr (SOFTCAP) g[l] *= c.dz;
    }
    if (jg >= 0 && jg + EPG <= V) {
        uint4 o;
        if constexpr (BF16) {
            o = make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]),
                           pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7]));
        } else {
            o = make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                           __float_as_uint(g[3]));
        }
        ptx::st_global_cs_v4(dst, o);
    } else {
#pragma unroll
        for (int l = 0; l < EPG; ++l)
            if (jg + l >= 0 && jg + l < V) store_elem<BF16>(dst + ELT * l, g[l]);
    }
}

template <bool BF16>
__device__ __forceinline__ void zero_granule(int jg, int V, unsigned char *dst) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    constexpr int ELT = Elem<BF16>::kBytes;
    if (jg >= 0 && jg + EPG <= V) {
        ptx::st_global_cs_v4(dst, make_uint4(0u, 0u, 0u, 0u));
    } else {
#pragma unroll
        for (int l = 0; l < EPG; ++l)
            if (jg + l >= 0 && jg + l < V) store_elem<BF16>(dst + ELT * l, 0.f);
    }
}

template <bool BF16, bool SOFTCAP>
__global__ void __launch_bounds__(kThreads, 2) ce_rows_kernel(const Params p) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    constexpr int ELT = Elem<BF16>::kBytes;
    __shared__ RowPart wpart[kWarps];
    __shared__ float bcast;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p.logits) + r * p.stride_bytes;
    unsigned char *gbase = reinterpret_cast<unsigned char *>(a0 & ~static_cast<uintptr_t>(15));
    const uint4 *row = reinterpret_cast<const uint4 *>(gbase);
    const int lead = static_cast<int>((a0 & 15) / ELT);
    const int G = (lead + p.V + EPG - 1) / EPG;
    const float T = p.softcap;
    const float k2 = SOFTCAP ? -2.f * kLog2e / T : 0.f;

    // ---- pass 1
    Acc a;
    a.mv = -INFINITY;
    a.midx = INT_MAX;
    a.mz = -INFINITY;
    a.nmL = INFINITY;
    a.s0 = a.s1 = a.z0 = a.z1 = 0.f;
    if (tid == 0) {  // pull the whole row towards L2 with the bulk-copy engine
        const uint32_t bytes = static_cast<uint32_t>(G) * 16u;
        for (uint32_t off = 0; off < bytes; off += kPrefetchBytes)
            ptx::bulk_prefetch_l2(gbase + off, min(kPrefetchBytes, bytes - off));
    }
    int gl;
    for (gl = tid; gl < G; gl += kThreads)
        fold<BF16, SOFTCAP>(a, ld_v4(row + gl), gl * EPG - lead, p.V, T, k2);

    RowPart pt = part_identity();
    pt.mx = a.mv;
    pt.idx = a.midx;
    pt.mz = a.mz;
    pt.s = a.s0 + a.s1;
    pt.sz = a.z0 + a.z1;
    warp_allreduce(pt);
    if (lane == 0) wpart[warp] = pt;

    const int64_t y = p.labels[r];
    const bool ignored = (y == p.ignore_index);
    const bool valid = !ignored && y >= 0 && y < p.V;
    __syncthreads();
    if (warp == 0) {
        RowPart q = wpart[lane];  // kWarps == 32
        warp_allreduce(q);
        if (lane == 0) {
            const float lse = q.mz + logf(q.s);
            float l = 0.f;
            if (valid) {
                const unsigned char *py = reinterpret_cast<const unsigned char *>(a0) + ELT * y;
                float xy;
                if constexpr (BF16)
                    xy = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(py)) << 16);
                else
                    xy = *reinterpret_cast<const float *>(py);
                const float zy = softcap_z<SOFTCAP>(xy, T, k2).z;
                l = lse - fmaf(1.f - p.eps, zy, (p.eps / static_cast<float>(p.V)) * q.sz);
            } else if (!ignored) {
                l = __int_as_float(0x7fc00000);  // bad label: NaN
            }
            p.loss[r] = l;
            p.argmax[r] = q.idx;
            bcast = lse;
        }
    }
    __syncthreads();

    // ---- pass 2
    if (valid) {
        ptx::griddep_wait();  // the label census of this call
        const int64_t n_valid = p.counts[0];
        float scale = p.grad_scale;
        if (p.reduction == VLMCE_MEAN)
            scale = n_valid > 0 ? p.grad_scale / static_cast<float>(n_valid) : 0.f;
        const float c_smooth = scale * (p.eps / static_cast<float>(p.V));  // scale eps / V
        const float c_label = c_smooth + scale * (1.f - p.eps);            // + scale (1 - eps)
        const float nlseL = -bcast * kLog2e;
        const int gy = static_cast<int>((y + lead) / EPG);
        const int ly = static_cast<int>((y + lead) % EPG);
        for (gl = tid; gl < G; gl += kThreads)
            grad_granule<BF16, SOFTCAP>(ld_v4(row + gl), gl * EPG - lead, p.V, gbase + 16 * gl, T, k2,
                                        nlseL, scale, c_smooth, c_label, gl == gy ? ly : -1);
    } else {
        for (gl = tid; gl < G; gl += kThreads) zero_granule<BF16>(gl * EPG - lead, p.V, gbase + 16 * gl);
    }
}

// The row kernel for the given softcap, per element type (ce_rows_bf16.cu,
// ce_rows_f32.cu).
Kernel kernel_bf16(bool softcap);
Kernel kernel_f32(bool softcap);

}  // namespace rows
}  // namespace ce
}  // namespace vlmce
