// ce.cu -- fused cross-entropy forward + backward over [N, V] logits, with
// the gradient written in place of the logits (entry point ce_fwd_bwd).
//
// Method (web pages on Liger-Kernel / Megatron-LM cross-entropy): per row, an
// online softmax (running max and sum-exp) over the vocabulary, the loss with
// ignore_index, label smoothing and an optional final-logit softcap
// T tanh(x/T), the argmax with smallest-index ties, and the gradient
// scale (softmax - smoothed one-hot) (1 - t^2) stored over the logits, so the
// softmax is never materialised.
//
// GB300 design.  Three launches on the caller's stream:
//   1. ce_count_kernel  -- label census (n_valid for the mean, bad labels).
//   2. ce_rows_kernel   -- persistent, one thread-block cluster of k CTAs per
//      row at a time.  Each CTA owns 1/k of the row's 16-byte granules; a
//      bulk (TMA) copy stages its slice in shared memory, several rows ahead,
//      so the row crosses HBM exactly once in and once out.  Pass A over the
//      slice: max / argmax of the raw logits and an online sum-exp and sum of
//      z.  The k partials are merged through distributed shared memory (one
//      release/acquire mbarrier exchange per row).  Pass B: the gradient,
//      rounded to the storage dtype, stored with 16-byte streaming stores.
//   3. ce_finalize_kernel -- fixed-order fp64 reduction of the per-row losses
//      and correct-prediction count.
// Kernels 2 and 3 use programmatic dependent launch so their prologues
// overlap the previous kernel's tail.  No floating-point atomics: results are
// bit-reproducible.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "host_util.h"
#include "ptx.cuh"
#include "vlmce.h"

namespace vlmce {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxStages = 4;
constexpr int kCtlBytes = 1024;       // control block at the start of shared memory
constexpr uint32_t kChunk = 16384;    // bytes per bulk copy instruction
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s per on-chip wait

// One CTA's (or warp's, or thread's) statistics of one row.
struct __align__(16) RowPart {
    float mx;   // max of the raw logits x
    int idx;    // smallest column holding mx
    float mz;   // reference maximum (z space) of s
    float s;    // sum exp(z - mz)
    float sz;   // sum z
    float zy;   // z at the label column (only its owner CTA adds it)
    float pad0, pad1;
};

struct Ctl {
    unsigned long long full[kMaxStages];  // stage landed (transaction bytes)
    unsigned long long stat[2];           // all k partials of a row written (k arrivals)
    RowPart slot[2];                      // this CTA's partial, read by the whole cluster
    RowPart warp[kWarps];                 // per-warp partials
    int abort;                            // an on-chip wait gave up
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block too large");

struct CeParams {
    unsigned char *logits;
    const int64_t *labels;
    int64_t N;
    int V;
    int64_t stride_bytes;
    int64_t ignore_index;
    float eps;
    float softcap;
    float grad_scale;
    int reduction;
    float *loss;
    int64_t *argmax;
    const int64_t *counts;  // [0] n_valid, [1] n_bad (from ce_count_kernel)
    int *err;
    int gran_per_cta;       // 16-byte granules of a row owned by one CTA
    int nstage;
    int stage_bytes;
};

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

template <bool BF16>
struct Elem {
    static constexpr int kBytes = BF16 ? 2 : 4;
    static constexpr int kPerGranule = 16 / kBytes;
};

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
__device__ __forceinline__ float granule_max(const uint4 w, const float (&x)[Elem<BF16>::kPerGranule]) {
    if constexpr (BF16) {
        const __nv_bfloat162 a = __hmax2(as_bf162(w.x), as_bf162(w.y));
        const __nv_bfloat162 b = __hmax2(as_bf162(w.z), as_bf162(w.w));
        const __nv_bfloat162 c = __hmax2(a, b);
        return fmaxf(__low2float(c), __high2float(c));
    } else {
        return fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    }
}

template <bool BF16>
__device__ __forceinline__ uint4 pack(const float (&g)[Elem<BF16>::kPerGranule]) {
    uint4 o;
    if constexpr (BF16) {
        uint32_t u[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(g[2 * q], g[2 * q + 1]);
            memcpy(&u[q], &b, 4);
        }
        o = make_uint4(u[0], u[1], u[2], u[3]);
    } else {
        o = make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                       __float_as_uint(g[3]));
    }
    return o;
}

template <bool BF16>
__device__ __forceinline__ float load_elem_smem(const unsigned char *p) {
    if constexpr (BF16) {
        return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(p)) << 16);
    } else {
        return *reinterpret_cast<const float *>(p);
    }
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

// Where row r's granules start and which of them this CTA owns.
struct RowGeo {
    uintptr_t gbase;  // 16-byte aligned address of the row's first granule
    int lead;         // elements of the first granule that precede column 0
    int g_beg;        // first granule owned by this CTA
    int n_my;         // granules owned by this CTA (may be 0)
};

template <bool BF16>
__device__ __forceinline__ RowGeo row_geo(const CeParams &p, int64_t r, uint32_t crank) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p.logits) + r * p.stride_bytes;
    RowGeo g;
    g.gbase = a0 & ~static_cast<uintptr_t>(15);
    g.lead = static_cast<int>((a0 & 15) / Elem<BF16>::kBytes);
    const int G = (g.lead + p.V + EPG - 1) / EPG;
    g.g_beg = static_cast<int>(crank) * p.gran_per_cta;
    g.n_my = min(G - g.g_beg, p.gran_per_cta);
    if (g.n_my < 0) g.n_my = 0;
    return g;
}

// Bounded wait on a stage's bulk-copy barrier.  Gives up (sets the abort flag
// and the device error bit) after kWaitLimitNs, or at once if aborted.
__device__ __noinline__ bool wait_stage(uint32_t bar, uint32_t parity, volatile int *abort,
                                        int *err) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = ptx::globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicOr(err, VLMCE_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait on the cluster exchange barrier (acquire, cluster scope).  Peers
// always arrive, so it is never skipped; once a wait has already given up the
// limit drops to 1 ms so a broken kernel still ends promptly.
__device__ __noinline__ bool wait_cluster(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int *err) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = ptx::globaltimer_ns();
    const unsigned long long limit = *abort ? 1000000ull : kWaitLimitNs;
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
        if (ptx::globaltimer_ns() - t0 > limit) {
            *abort = 1;
            atomicOr(err, VLMCE_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Thread 0: stage row iteration `it` of this cluster into stage `it % nstage`.
template <bool BF16>
__device__ __forceinline__ void issue_row(const CeParams &p, int64_t it, uint32_t cid,
                                          uint32_t ncl, uint32_t crank, uint32_t stage0,
                                          uint32_t full0) {
    const int s = static_cast<int>(it % p.nstage);
    const int64_t r = static_cast<int64_t>(cid) + it * ncl;
    const RowGeo g = row_geo<BF16>(p, r, crank);
    const uint32_t bytes = static_cast<uint32_t>(g.n_my) * 16u;
    const uint32_t bar = full0 + 8u * s;
    const uint32_t dst = stage0 + static_cast<uint32_t>(s) * p.stage_bytes;
    const unsigned char *src = reinterpret_cast<const unsigned char *>(g.gbase) + 16 * g.g_beg;
    ptx::mbar_arrive_expect_tx(bar, bytes);
    for (uint32_t off = 0; off < bytes; off += kChunk)
        ptx::bulk_g2s(dst + off, src + off, min(kChunk, bytes - off), bar);
}

// ------------------------------------------------------------------ kernels

__global__ void __launch_bounds__(1024) ce_count_kernel(const int64_t *__restrict__ labels,
                                                        int64_t N, int64_t V, int64_t ignore_index,
                                                        int64_t *counts, int *err) {
    ptx::griddep_launch_dependents();
    long long nv = 0, nb = 0;
    for (int64_t r = threadIdx.x; r < N; r += blockDim.x) {
        const int64_t y = labels[r];
        if (y == ignore_index) continue;
        if (y >= 0 && y < V)
            ++nv;
        else
            ++nb;
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

template <bool BF16, bool SOFTCAP>
__global__ void __launch_bounds__(kThreads, 1) ce_rows_kernel(const CeParams p) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    constexpr int ELT = Elem<BF16>::kBytes;
    extern __shared__ __align__(1024) unsigned char smem[];
    Ctl &ctl = *reinterpret_cast<Ctl *>(smem);
    unsigned char *stages = smem + kCtlBytes;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t k = ptx::cluster_nctarank();
    const uint32_t crank = ptx::cluster_ctarank();
    const uint32_t cid = ptx::cluster_id_x();
    const uint32_t ncl = ptx::ncluster_x();
    const uint32_t full0 = ptx::smem_addr(&ctl.full[0]);
    const uint32_t stage0 = ptx::smem_addr(stages);

    if (tid == 0) {
        for (int s = 0; s < p.nstage; ++s) ptx::mbar_init(full0 + 8u * s, 1);
        ptx::mbar_init(ptx::smem_addr(&ctl.stat[0]), k);
        ptx::mbar_init(ptx::smem_addr(&ctl.stat[1]), k);
        ctl.abort = 0;
        ptx::fence_mbar_init_cluster();
    }
    __syncthreads();
    ptx::cluster_sync();  // every CTA's barriers exist before anyone signals them

    const int64_t n_iter = (static_cast<int64_t>(cid) < p.N) ? (p.N - 1 - cid) / ncl + 1 : 0;
    int64_t issued = 0;  // thread 0 only
    if (tid == 0) {
        for (; issued < n_iter && issued < p.nstage; ++issued)
            issue_row<BF16>(p, issued, cid, ncl, crank, stage0, full0);
    }

    // The label census of this call must be complete before it is read.
    ptx::griddep_wait();
    const int64_t n_valid = p.counts[0];
    float scale = p.grad_scale;
    if (p.reduction == VLMCE_MEAN) scale = n_valid > 0 ? p.grad_scale / static_cast<float>(n_valid) : 0.f;
    const float c_smooth = scale * (p.eps / static_cast<float>(p.V));  // scale * eps / V
    const float c_label = c_smooth + scale * (1.f - p.eps);            // ... + scale (1 - eps)
    const float T = p.softcap;
    const float k2 = SOFTCAP ? -2.f * kLog2e / T : 0.f;
    volatile int *abort = &ctl.abort;

    for (int64_t it = 0; it < n_iter; ++it) {
        const int s = static_cast<int>(it % p.nstage);
        const int pp = static_cast<int>(it & 1);
        const int64_t r = static_cast<int64_t>(cid) + it * ncl;
        const int64_t y = p.labels[r];
        const bool ignored = (y == p.ignore_index);
        const bool valid = !ignored && y >= 0 && y < p.V;
        const RowGeo g = row_geo<BF16>(p, r, crank);
        const unsigned char *buf = stages + static_cast<size_t>(s) * p.stage_bytes;

        wait_stage(full0 + 8u * s, static_cast<uint32_t>((it / p.nstage) & 1), abort, p.err);

        // ---- pass A: max / argmax of x, online sum exp(z - mz), sum z
        float mv = -INFINITY, mz = -INFINITY, mzL = -INFINITY;
        int mgl = -1;
        float s0 = 0.f, s1 = 0.f, z0 = 0.f, z1 = 0.f;
        for (int gl = tid; gl < g.n_my; gl += kThreads) {
            const uint4 w = *reinterpret_cast<const uint4 *>(buf + 16 * gl);
            float x[EPG];
            unpack<BF16>(w, x);
            const int jg = (g.g_beg + gl) * EPG - g.lead;
            const bool full = jg >= 0 && jg + EPG <= p.V;
            if (full) {
                const float gm = granule_max<BF16>(w, x);
                if (gm > mv) {
                    const float nz = softcap_z<SOFTCAP>(gm, T, k2).z;
                    const float f = ptx::ex2((mz - nz) * kLog2e);
                    s0 = (s0 == 0.f) ? 0.f : s0 * f;
                    s1 = (s1 == 0.f) ? 0.f : s1 * f;
                    mv = gm;
                    mgl = gl;
                    mz = nz;
                    mzL = nz * kLog2e;
                }
#pragma unroll
                for (int l = 0; l < EPG; l += 2) {
                    const float za = softcap_z<SOFTCAP>(x[l], T, k2).z;
                    const float zb = softcap_z<SOFTCAP>(x[l + 1], T, k2).z;
                    s0 += ptx::ex2(fmaf(za, kLog2e, -mzL));
                    s1 += ptx::ex2(fmaf(zb, kLog2e, -mzL));
                    z0 += za;
                    z1 += zb;
                }
            } else {
                float gm = -INFINITY;
#pragma unroll
                for (int l = 0; l < EPG; ++l)
                    if (jg + l >= 0 && jg + l < p.V) gm = fmaxf(gm, x[l]);
                if (gm > mv) {
                    const float nz = softcap_z<SOFTCAP>(gm, T, k2).z;
                    const float f = ptx::ex2((mz - nz) * kLog2e);
                    s0 = (s0 == 0.f) ? 0.f : s0 * f;
                    s1 = (s1 == 0.f) ? 0.f : s1 * f;
                    mv = gm;
                    mgl = gl;
                    mz = nz;
                    mzL = nz * kLog2e;
                }
#pragma unroll
                for (int l = 0; l < EPG; ++l) {
                    if (jg + l >= 0 && jg + l < p.V) {
                        const float z = softcap_z<SOFTCAP>(x[l], T, k2).z;
                        s0 += ptx::ex2(fmaf(z, kLog2e, -mzL));
                        z0 += z;
                    }
                }
            }
        }
        RowPart part = part_identity();
        part.mx = mv;
        part.mz = mz;
        part.s = s0 + s1;
        part.sz = z0 + z1;
        if (mgl >= 0) {  // first column of this thread's first maximal granule that holds mv
            const uint4 w = *reinterpret_cast<const uint4 *>(buf + 16 * mgl);
            float x[EPG];
            unpack<BF16>(w, x);
            const int jg = (g.g_beg + mgl) * EPG - g.lead;
#pragma unroll
            for (int l = EPG - 1; l >= 0; --l)
                if (jg + l >= 0 && jg + l < p.V && x[l] == mv) part.idx = jg + l;
        }
        warp_allreduce(part);
        if (lane == 0) ctl.warp[warp] = part;
        __syncthreads();

        // ---- CTA partial -> cluster exchange
        if (warp == 0) {
            RowPart q = lane < kWarps ? ctl.warp[lane] : part_identity();
            warp_allreduce(q);
            if (lane == 0) {
                q.zy = 0.f;
                if (valid) {
                    const int gy = static_cast<int>((y + g.lead) / EPG) - g.g_beg;
                    const int ly = static_cast<int>((y + g.lead) % EPG);
                    if (gy >= 0 && gy < g.n_my)
                        q.zy = softcap_z<SOFTCAP>(load_elem_smem<BF16>(buf + 16 * gy + ELT * ly), T, k2).z;
                }
                ctl.slot[pp] = q;
                const uint32_t bar = ptx::smem_addr(&ctl.stat[pp]);
                for (uint32_t c = 0; c < k; ++c) ptx::mbar_remote_arrive_release(ptx::mapa(bar, c));
            }
        }
        wait_cluster(ptx::smem_addr(&ctl.stat[pp]), static_cast<uint32_t>((it >> 1) & 1), abort,
                     p.err);
        RowPart rp = part_identity();
        if (lane < static_cast<int>(k)) {
            const uint32_t a = ptx::mapa(ptx::smem_addr(&ctl.slot[pp]), lane);
            const uint4 v0 = ptx::ld_dsmem_v4(a);
            const uint4 v1 = ptx::ld_dsmem_v4(a + 16);
            rp.mx = __uint_as_float(v0.x);
            rp.idx = static_cast<int>(v0.y);
            rp.mz = __uint_as_float(v0.z);
            rp.s = __uint_as_float(v0.w);
            rp.sz = __uint_as_float(v1.x);
            rp.zy = __uint_as_float(v1.y);
        }
        warp_allreduce(rp);
        const float lse = rp.mz + logf(rp.s);

        if (crank == 0 && tid == 0) {
            float l = 0.f;
            if (valid)
                l = lse - fmaf(1.f - p.eps, rp.zy, (p.eps / static_cast<float>(p.V)) * rp.sz);
            else if (!ignored)
                l = __int_as_float(0x7fc00000);  // bad label: NaN
            p.loss[r] = l;
            p.argmax[r] = rp.idx;
        }

        // ---- pass B: gradient, in place
        unsigned char *grow = reinterpret_cast<unsigned char *>(g.gbase);
        if (valid) {
            const float lseL = lse * kLog2e;
            const int gly = static_cast<int>((y + g.lead) / EPG) - g.g_beg;
            const int lly = static_cast<int>((y + g.lead) % EPG);
            for (int gl = tid; gl < g.n_my; gl += kThreads) {
                const uint4 w = *reinterpret_cast<const uint4 *>(buf + 16 * gl);
                float x[EPG], pr[EPG], dz[EPG], gr[EPG];
                unpack<BF16>(w, x);
#pragma unroll
                for (int l = 0; l < EPG; ++l) {
                    const Capped c = softcap_z<SOFTCAP>(x[l], T, k2);
                    pr[l] = ptx::ex2(fmaf(c.z, kLog2e, -lseL));  // p_j
                    dz[l] = c.dz;
                    gr[l] = fmaf(pr[l], scale, -c_smooth);       // scale (p_j - eps/V)
                }
                if (gl == gly) {  // the label column: q_y = 1 - eps + eps/V
#pragma unroll
                    for (int l = 0; l < EPG; ++l)
                        if (l == lly) gr[l] = fmaf(pr[l], scale, -c_label);
                }
                if constexpr (SOFTCAP) {
#pragma unroll
                    for (int l = 0; l < EPG; ++l) gr[l] *= dz[l];
                }
                const int jg = (g.g_beg + gl) * EPG - g.lead;
                unsigned char *dst = grow + 16 * (g.g_beg + gl);
                if (jg >= 0 && jg + EPG <= p.V) {
                    ptx::st_global_cs_v4(dst, pack<BF16>(gr));
                } else {
#pragma unroll
                    for (int l = 0; l < EPG; ++l)
                        if (jg + l >= 0 && jg + l < p.V) store_elem<BF16>(dst + ELT * l, gr[l]);
                }
            }
        } else {
            for (int gl = tid; gl < g.n_my; gl += kThreads) {
                const int jg = (g.g_beg + gl) * EPG - g.lead;
                unsigned char *dst = grow + 16 * (g.g_beg + gl);
                if (jg >= 0 && jg + EPG <= p.V) {
                    ptx::st_global_cs_v4(dst, make_uint4(0u, 0u, 0u, 0u));
                } else {
#pragma unroll
                    for (int l = 0; l < EPG; ++l)
                        if (jg + l >= 0 && jg + l < p.V) store_elem<BF16>(dst + ELT * l, 0.f);
                }
            }
        }

        __syncthreads();  // stage s fully consumed
        if (tid == 0 && issued < n_iter && !*abort) {
            ptx::fence_proxy_async_smem();
            issue_row<BF16>(p, issued, cid, ncl, crank, stage0, full0);
            ++issued;
        }
    }

    ptx::griddep_launch_dependents();
    // Every issued bulk copy has landed before the CTA may exit.
    if (tid == 0) {
        for (int s = 0; s < p.nstage; ++s) {
            int64_t last = -1;
            for (int64_t it = issued - 1; it >= 0 && it >= issued - p.nstage; --it)
                if (it % p.nstage == s) {
                    last = it;
                    break;
                }
            if (last >= 0) {
                volatile int no_abort = 0;
                wait_stage(full0 + 8u * s, static_cast<uint32_t>((last / p.nstage) & 1), &no_abort,
                           p.err);
            }
        }
    }
    __syncthreads();
    ptx::cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

__global__ void __launch_bounds__(1024) ce_finalize_kernel(
    const float *__restrict__ loss, const int64_t *__restrict__ argmax,
    const int64_t *__restrict__ labels, int64_t N, int64_t V, int64_t ignore_index, int reduction,
    const int64_t *counts, const int *err, float *out_reduced, int64_t *out_counts) {
    ptx::griddep_wait();
    double acc = 0.0;
    long long nc = 0;
    for (int64_t r = threadIdx.x; r < N; r += blockDim.x) {
        const int64_t y = labels[r];
        if (y == ignore_index) continue;
        acc += static_cast<double>(loss[r]);
        if (y >= 0 && y < V && argmax[r] == y) ++nc;
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

// ------------------------------------------------------------------ host side

struct Workspace {
    int64_t *counts;  // [4]
    int *err;
    float *loss;      // [N]
    int64_t *argmax;  // [N]
};

constexpr int64_t kWsHeader = 256;

size_t workspace_bytes(int64_t N) {
    return static_cast<size_t>(kWsHeader + round_up(4 * N, 256) + round_up(8 * N, 256));
}

Workspace carve(void *ws, int64_t N) {
    unsigned char *b = static_cast<unsigned char *>(ws);
    Workspace w;
    w.counts = reinterpret_cast<int64_t *>(b);
    w.err = reinterpret_cast<int *>(b + 64);
    w.loss = reinterpret_cast<float *>(b + kWsHeader);
    w.argmax = reinterpret_cast<int64_t *>(b + kWsHeader + round_up(4 * N, 256));
    return w;
}

struct Plan {
    int k = 0, nstage = 0, gran_per_cta = 0, stage_bytes = 0, smem = 0, max_clusters = 0;
};

using RowKernel = void (*)(CeParams);

RowKernel pick_kernel(bool bf16, bool softcap) {
    if (bf16) return softcap ? ce_rows_kernel<true, true> : ce_rows_kernel<true, false>;
    return softcap ? ce_rows_kernel<false, true> : ce_rows_kernel<false, false>;
}

// Granules of the widest row (any alignment of its first element).
int64_t max_granules(bool bf16, int64_t V) {
    const int64_t epg = bf16 ? 8 : 4;
    return (epg - 1 + V + epg - 1) / epg;
}

// Smallest cluster whose per-CTA slice fits `want_stages` stages.
bool shape_plan(int64_t smem_optin, bool bf16, int64_t V, int force_k, int force_st, Plan *pl) {
    const int64_t G = max_granules(bf16, V);
    const int64_t budget = smem_optin - kCtlBytes;
    for (int k = 1; k <= kMaxCluster; ++k) {
        if (force_k && k != force_k) continue;
        const int64_t gc = (G + k - 1) / k;
        const int64_t stage = round_up(gc * 16, 128);
        int64_t nst = budget / stage;
        if (nst > kMaxStages) nst = kMaxStages;
        if (force_st) {
            if (force_st > nst) continue;
            nst = force_st;
        }
        const bool ok = force_k ? nst >= 2 : (nst >= 3 || (k == kMaxCluster && nst >= 2));
        if (!ok) continue;
        pl->k = k;
        pl->nstage = static_cast<int>(nst);
        pl->gran_per_cta = static_cast<int>(gc);
        pl->stage_bytes = static_cast<int>(stage);
        pl->smem = static_cast<int>(kCtlBytes + nst * stage);
        return true;
    }
    return false;
}

thread_local cudaEvent_t t_prof_begin = nullptr;
thread_local cudaEvent_t t_prof_end = nullptr;

std::mutex g_plan_mu;
std::map<std::tuple<int, bool, bool, int64_t, int, int>, Plan> g_plans;

// Optional tuning override "k,stages" (cluster size, pipeline depth).
void plan_override(int *k, int *st) {
    *k = 0;
    *st = 0;
    const char *e = getenv("VLMCE_CE_PLAN");
    if (e && *e) {
        int a = 0, b = 0;
        if (sscanf(e, "%d,%d", &a, &b) == 2 && a >= 1 && a <= kMaxCluster && b >= 2 &&
            b <= kMaxStages) {
            *k = a;
            *st = b;
        }
    }
}

vlmce_status get_plan(const DeviceInfo &d, bool bf16, bool softcap, int64_t V, Plan *out) {
    int fk, fs;
    plan_override(&fk, &fs);
    const auto key = std::make_tuple(d.device, bf16, softcap, V, fk, fs);
    std::lock_guard<std::mutex> lk(g_plan_mu);
    auto itp = g_plans.find(key);
    if (itp != g_plans.end()) {
        *out = itp->second;
        return VLMCE_OK;
    }
    Plan pl;
    if (!shape_plan(d.smem_optin, bf16, V, fk, fs, &pl)) return VLMCE_ERR_TOO_LARGE;
    RowKernel kern = pick_kernel(bf16, softcap);
    // The attribute belongs to the kernel, not to the plan: set it to the device
    // maximum so every plan of this kernel can launch.
    if (record_cuda(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         d.smem_optin),
                    "cudaFuncSetAttribute(ce_rows_kernel)") != cudaSuccess)
        return VLMCE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.k * d.sm_count, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pl.k;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int ncl = 0;
    if (record_cuda(cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg),
                    "cudaOccupancyMaxActiveClusters(ce_rows_kernel)") != cudaSuccess)
        return VLMCE_ERR_CUDA;
    if (ncl < 1) return VLMCE_ERR_TOO_LARGE;
    pl.max_clusters = ncl;
    g_plans[key] = pl;
    *out = pl;
    return VLMCE_OK;
}

}  // namespace
}  // namespace vlmce

using namespace vlmce;

extern "C" void vlmce_profile_events(void *ev_begin, void *ev_end) {
    t_prof_begin = static_cast<cudaEvent_t>(ev_begin);
    t_prof_end = static_cast<cudaEvent_t>(ev_end);
}

extern "C" int64_t vlmce_ce_max_vocab(int32_t dtype) {
    if (dtype != VLMCE_F32 && dtype != VLMCE_BF16) return 0;
    // sm_103: 227 KB of dynamic shared memory per block; 8 CTAs x 2 stages.
    const int64_t stage = (232448 - kCtlBytes) / 2 / 128 * 128;
    const int64_t epg = dtype == VLMCE_BF16 ? 8 : 4;
    const int64_t G = (stage / 16) * kMaxCluster;
    return G * epg - 2 * (epg - 1);
}

extern "C" size_t vlmce_ce_workspace_bytes(int64_t N, int64_t V, int32_t dtype) {
    (void)V;
    (void)dtype;
    if (N < 0) return 0;
    return workspace_bytes(N);
}

extern "C" vlmce_status ce_fwd_bwd(void *logits, int32_t dtype, const int64_t *labels, int64_t N,
                                   int64_t V, int64_t row_stride, int64_t ignore_index,
                                   float label_smoothing, float softcap, int32_t reduction,
                                   float grad_scale, float *out_loss, int64_t *out_argmax,
                                   float *out_reduced, int64_t *out_counts, void *workspace,
                                   size_t workspace_bytes_given, vlmce_stream_t stream) {
    // ---- host-side argument checks; nothing is enqueued on failure
    if (dtype != VLMCE_F32 && dtype != VLMCE_BF16) return VLMCE_ERR_UNSUPPORTED_DTYPE;
    if (N < 0 || V < 1 || row_stride < V) return VLMCE_ERR_INVALID_ARG;
    if (N > 0 && (!logits || !labels)) return VLMCE_ERR_INVALID_ARG;
    if (!(label_smoothing >= 0.f && label_smoothing <= 1.f)) return VLMCE_ERR_INVALID_ARG;
    if (!(softcap >= 0.f) || !std::isfinite(softcap)) return VLMCE_ERR_INVALID_ARG;
    if (!std::isfinite(grad_scale)) return VLMCE_ERR_INVALID_ARG;
    if (reduction != VLMCE_MEAN && reduction != VLMCE_SUM) return VLMCE_ERR_INVALID_ARG;
    if (V > vlmce_ce_max_vocab(dtype)) return VLMCE_ERR_TOO_LARGE;
    const int64_t elt = dtype == VLMCE_BF16 ? 2 : 4;
    if (N > 0 && row_stride > (INT64_MAX / elt) / N) return VLMCE_ERR_TOO_LARGE;
    if (!workspace || workspace_bytes_given < workspace_bytes(N)) return VLMCE_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return VLMCE_ERR_MISALIGNED;
    if (logits && !aligned(logits, static_cast<uintptr_t>(elt))) return VLMCE_ERR_MISALIGNED;
    if (labels && !aligned(labels, 8)) return VLMCE_ERR_MISALIGNED;
    if (out_loss && !aligned(out_loss, 4)) return VLMCE_ERR_MISALIGNED;
    if (out_argmax && !aligned(out_argmax, 8)) return VLMCE_ERR_MISALIGNED;
    if (out_reduced && !aligned(out_reduced, 4)) return VLMCE_ERR_MISALIGNED;
    if (out_counts && !aligned(out_counts, 8)) return VLMCE_ERR_MISALIGNED;

    DeviceInfo dev;
    vlmce_status st = current_device(&dev);
    if (st != VLMCE_OK) return st;

    const bool bf16 = dtype == VLMCE_BF16;
    const bool capped = softcap > 0.f;
    Plan pl;
    if (N > 0) {
        st = get_plan(dev, bf16, capped, V, &pl);
        if (st != VLMCE_OK) return st;
    }

    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    Workspace w = carve(workspace, N);
    float *loss = out_loss ? out_loss : w.loss;
    int64_t *amax = out_argmax ? out_argmax : w.argmax;

    ce_count_kernel<<<1, 1024, 0, cs>>>(labels, N, V, ignore_index, w.counts, w.err);
    st = launch_status(cudaSuccess, "ce_count_kernel");
    if (st != VLMCE_OK) return st;

    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    if (N > 0) {
        CeParams p;
        p.logits = static_cast<unsigned char *>(logits);
        p.labels = labels;
        p.N = N;
        p.V = static_cast<int>(V);
        p.stride_bytes = row_stride * elt;
        p.ignore_index = ignore_index;
        p.eps = label_smoothing;
        p.softcap = softcap;
        p.grad_scale = grad_scale;
        p.reduction = reduction;
        p.loss = loss;
        p.argmax = amax;
        p.counts = w.counts;
        p.err = w.err;
        p.gran_per_cta = pl.gran_per_cta;
        p.nstage = pl.nstage;
        p.stage_bytes = pl.stage_bytes;

        const int64_t ncl = N < pl.max_clusters ? N : pl.max_clusters;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ncl * pl.k), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = pl.smem;
        cfg.stream = cs;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = pl.k;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        cudaEvent_t eb = t_prof_begin, ee = t_prof_end;
        t_prof_begin = t_prof_end = nullptr;
        if (eb && (st = launch_status(cudaEventRecord(eb, cs), "cudaEventRecord")) != VLMCE_OK)
            return st;
        st = launch_status(cudaLaunchKernelEx(&cfg, pick_kernel(bf16, capped), p), "ce_rows_kernel");
        if (st != VLMCE_OK) return st;
        if (ee && (st = launch_status(cudaEventRecord(ee, cs), "cudaEventRecord")) != VLMCE_OK)
            return st;
    }

    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, 1);
        cfg.blockDim = dim3(1024, 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = cs;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        st = launch_status(cudaLaunchKernelEx(&cfg, ce_finalize_kernel,
                                              static_cast<const float *>(loss),
                                              static_cast<const int64_t *>(amax), labels, N, V,
                                              ignore_index, static_cast<int>(reduction),
                                              static_cast<const int64_t *>(w.counts),
                                              static_cast<const int *>(w.err), out_reduced,
                                              out_counts),
                           "ce_finalize_kernel");
    }
    return st;
}
