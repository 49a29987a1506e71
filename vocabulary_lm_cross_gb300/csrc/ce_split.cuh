// ce_split.cuh -- the cross-entropy V-split kernel for few, wide rows
// (forward + backward, in place).
//
// One thread-block cluster of k CTAs owns one row at a time; CTA c of the
// cluster owns the c-th 1/k of the row's 16-byte granules (its "slice").
// Two CTAs share each SM (16 warps each), so one CTA's per-row exchange
// bubble is filled by the other's arithmetic.
//
// Warp 15 of each CTA is a producer: one lane streams the slices of the
// cluster's rows, in order, through a ring of 7.5 KB shared-memory slots
// (480 granules: one per consumer thread) with bulk (TMA) copies, as far
// ahead as free slots allow.  A row's slots stay resident until its gradient
// has been written, then the 15 consumer warps release them.  Per row:
//   pass A: one pass over the slice in shared memory: max and first argmax of
//           the raw logits, online sum of exp(z - m) and sum of z (packed
//           f32x2 arithmetic);
//   merge:  warp shuffles, then the 15 warp partials (fixed order) into the
//           CTA's partial, which the first consumer warp writes into every CTA
//           of the cluster through distributed shared memory (lane c to CTA
//           c), release-arriving on each CTA's row barrier; after the
//           acquire-wait every warp merges the k CTA partials in the same
//           fixed order, so every CTA holds the same lse;
//   pass B: gradient scale (p - q) (1 - t^2), rounded to the storage dtype,
//           16-byte streaming stores over the logits.
// Each byte of the row crosses HBM once in and once out.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ce_common.cuh"
#include "ptx.cuh"
#include "vlmce.h"

namespace vlmce {
namespace ce {
namespace split {

constexpr int kConsumerWarps = 15;
constexpr int kConsumers = 32 * kConsumerWarps;   // 480 consumer threads
constexpr int kThreads = kConsumers + 32;         // + 1 producer warp
constexpr int kCtasPerSm = 2;
constexpr int kChunkGranules = kConsumers;        // one granule per consumer thread
constexpr int kChunkBytes = 16 * kChunkGranules;  // 7.5 KB per slot
constexpr int kSlots = 13;
constexpr int kCtlBytes = 8192;
constexpr int kSmemBytes = kCtlBytes + kSlots * kChunkBytes;  // 108,032 B: two CTAs per SM
constexpr int kMaxCluster = 8;
constexpr int kPreferredChunks = 6;  // slices of <= 6 slots keep two rows in the ring
constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s per on-chip wait

struct Ctl {
    unsigned long long full[kSlots];   // slot landed (transaction bytes)
    unsigned long long empty[kSlots];  // slot released by the 15 consumer warps
    unsigned long long stat[2];        // all partials of a row arrived (k arrivals)
    // This CTA's consumer-warp partials, and the CTA partials of the cluster
    // (written by their owners through distributed shared memory), indexed
    // by row parity.
    RowPart wslot[2][kConsumerWarps];
    RowPart xslot[2][kMaxCluster];
    int abort;                         // an on-chip wait gave up
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block too large");

struct SplitParams {
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
    const int64_t *counts;  // [0] n_valid (written by the count kernel)
    int *err;
    int gran_per_cta;       // granules of a row owned by one CTA (<= kSlots * kChunkGranules)
    const float *token_scale;  // [N] per-row factor of the gradient, or null
    int want_grad;             // 0: forward only, the logits are not written
};

using SplitKernel = void (*)(SplitParams);

// Where row r's granules start and which of them this CTA owns.
struct RowGeo {
    uintptr_t gbase;  // 16-byte aligned address of the row's first granule
    int lead;         // elements of the first granule that precede column 0
    int g_beg;        // first granule owned by this CTA
    int n_my;         // granules owned by this CTA (may be 0)
};

template <bool BF16>
__device__ __forceinline__ RowGeo row_geo(const SplitParams &p, int64_t r, uint32_t crank) {
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

// Bounded mbarrier wait (slow path).  CLUSTER: acquire at cluster scope (pairs
// with the peers' release-arrives).  Gives up after kWaitLimitNs (1 ms once
// another wait has already given up), setting the abort flag and the device
// error bit; SKIP_IF_ABORT returns at once when aborted (waits whose arrival
// may never come once the pipeline stopped).
template <bool CLUSTER, bool SKIP_IF_ABORT>
__device__ __noinline__ bool bounded_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort,
                                               int *err) {
    auto poll = [&]() {
        return CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (SKIP_IF_ABORT && *abort) return false;
    const unsigned long long t0 = ptx::globaltimer_ns();
    const unsigned long long limit = *abort ? 1000000ull : kWaitLimitNs;
    for (;;) {
        for (int i = 0; i < 16; ++i)
            if (poll()) return true;
        if (SKIP_IF_ABORT && *abort) return false;
        if (ptx::globaltimer_ns() - t0 > limit) {
            *abort = 1;
            atomicOr(err, VLMCE_DEVERR_TIMEOUT);
            return false;
        }
    }
}

template <bool CLUSTER, bool SKIP_IF_ABORT>
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                             int *err) {
    const bool ok =
        CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    if (ok) return true;
    return bounded_wait_slow<CLUSTER, SKIP_IF_ABORT>(bar, parity, abort, err);
}

// Barrier 1 over the kConsumers consumer threads (the producer warp does not
// take part).
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Per-thread pass-A accumulators.
struct Acc {
    float mv;      // max raw logit seen
    int midx;      // its first column
    float mz;      // z of mv: reference of s
    uint64_t nmL;  // (-mz log2e, -mz log2e)
    uint64_t s;    // sums of exp(z - mz), two lanes
    uint64_t sz;   // sums of z, two lanes
};

// Fold one granule into the pass-A accumulators (granules arrive in column order).
template <bool BF16, bool SOFTCAP>
__device__ __forceinline__ void pass_a_granule(Acc &a, const uint4 w, int jg, int V, float T,
                                               float k2) {
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
        float s0, s1;
        upk(a.s, s0, s1);
        s0 = (s0 == 0.f) ? 0.f : s0 * f;
        s1 = (s1 == 0.f) ? 0.f : s1 * f;
        a.s = pk(s0, s1);
        a.mv = gm;
        a.midx = jg + li;
        a.mz = nz;
        a.nmL = pk(-nz * kLog2e, -nz * kLog2e);
    }
    const uint64_t L2 = pk(kLog2e, kLog2e);
    if (full) {
#pragma unroll
        for (int l = 0; l < EPG; l += 2) {
            const float za = softcap_z<SOFTCAP>(x[l], T, k2).z;
            const float zb = softcap_z<SOFTCAP>(x[l + 1], T, k2).z;
            const uint64_t z2 = pk(za, zb);
            a.s = add2(a.s, ex2x2(fma2(z2, L2, a.nmL)));
            a.sz = add2(a.sz, z2);
        }
    } else {
        float s0, s1, z0, z1, nm, dummy;
        upk(a.s, s0, s1);
        upk(a.sz, z0, z1);
        upk(a.nmL, nm, dummy);
#pragma unroll
        for (int l = 0; l < EPG; ++l) {
            if (jg + l >= 0 && jg + l < V) {
                const float z = softcap_z<SOFTCAP>(x[l], T, k2).z;
                s0 += ptx::ex2(fmaf(z, kLog2e, nm));
                z0 += z;
            }
        }
        a.s = pk(s0, s1);
        a.sz = pk(z0, z1);
    }
}

// Gradient of one granule, stored over the logits.  nlseL2 / scale2: the
// row's exponent constant and the coefficient of 2^e (grad_exp_coef); scale_p
// multiplies 2^e at the label column, c_label its target term.
template <bool BF16, bool SOFTCAP>
__device__ __forceinline__ void pass_b_granule(const uint4 w, int jg, int V, unsigned char *dst,
                                               float T, float k2, uint64_t nlseL2, uint64_t scale2,
                                               uint64_t negc2, int label_lane, float scale_p,
                                               float c_label) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    constexpr int ELT = Elem<BF16>::kBytes;
    float x[EPG], g[EPG], dz[EPG];
    unpack<BF16>(w, x);
    const uint64_t L2 = pk(kLog2e, kLog2e);
#pragma unroll
    for (int l = 0; l < EPG; l += 2) {
        const Capped ca = softcap_z<SOFTCAP>(x[l], T, k2);
        const Capped cb = softcap_z<SOFTCAP>(x[l + 1], T, k2);
        dz[l] = ca.dz;
        dz[l + 1] = cb.dz;
        const uint64_t p2 = ex2x2(fma2(pk(ca.z, cb.z), L2, nlseL2));  // p_j (times 2^bias)
        const uint64_t g2 = fma2(p2, scale2, negc2);                  // scale (p_j - eps/V)
        upk(g2, g[l], g[l + 1]);
        if (label_lane >= 0) {  // the label column: q_y = 1 - eps + eps/V
            float pa, pb;
            upk(p2, pa, pb);
            if (label_lane == l) g[l] = fmaf(pa, scale_p, -c_label);
            if (label_lane == l + 1) g[l + 1] = fmaf(pb, scale_p, -c_label);
        }
    }
    if constexpr (SOFTCAP) {
#pragma unroll
        for (int l = 0; l < EPG; ++l) g[l] *= dz[l];
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
__device__ __forceinline__ void store_zero_granule(int jg, int V, unsigned char *dst) {
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

// Producer lane: stream this cluster's rows (this CTA's slices), one chunk per slot.
template <bool BF16>
__device__ __forceinline__ void produce(const SplitParams &p, Ctl &ctl, uint32_t ring0, uint32_t cid,
                                        uint32_t ncl, uint32_t crank, int64_t n_iter) {
    volatile int *abort = &ctl.abort;
    const uint32_t full0 = ptx::smem_addr(&ctl.full[0]);
    const uint32_t empty0 = ptx::smem_addr(&ctl.empty[0]);
    int64_t q = 0;
    for (int64_t it = 0; it < n_iter && !*abort; ++it) {
        const RowGeo g = row_geo<BF16>(p, static_cast<int64_t>(cid) + it * ncl, crank);
        const unsigned char *src = reinterpret_cast<const unsigned char *>(g.gbase) + 16 * g.g_beg;
        for (int c = 0; c * kChunkGranules < g.n_my; ++c, ++q) {
            const int slot = static_cast<int>(q % kSlots);
            const int64_t use = q / kSlots;
            if (use > 0 &&
                !bounded_wait<false, true>(empty0 + 8u * slot,
                                           static_cast<uint32_t>((use - 1) & 1), abort, p.err))
                break;
            const int gran = min(kChunkGranules, g.n_my - c * kChunkGranules);
            const uint32_t bytes = static_cast<uint32_t>(gran) * 16u;
            ptx::mbar_arrive_expect_tx(full0 + 8u * slot, bytes);
            ptx::bulk_g2s(ring0 + static_cast<uint32_t>(slot) * kChunkBytes,
                          src + static_cast<size_t>(c) * kChunkBytes, bytes, full0 + 8u * slot);
        }
    }
    // Every issued copy has landed before the CTA may exit.
    for (int slot = 0; slot < kSlots; ++slot) {
        if (q <= slot) break;
        const int64_t last = q - 1 - ((q - 1 - slot) % kSlots);
        volatile int no_abort = 0;
        bounded_wait<false, false>(full0 + 8u * slot, static_cast<uint32_t>((last / kSlots) & 1),
                                   &no_abort, p.err);
    }
}

template <bool BF16, bool SOFTCAP>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) ce_split_kernel(const SplitParams p) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    extern __shared__ __align__(1024) unsigned char smem[];
    Ctl &ctl = *reinterpret_cast<Ctl *>(smem);
    unsigned char *ring = smem + kCtlBytes;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t k = ptx::cluster_nctarank();
    const uint32_t crank = ptx::cluster_ctarank();
    const uint32_t cid = ptx::cluster_id_x();
    const uint32_t ncl = ptx::ncluster_x();
    const uint32_t full0 = ptx::smem_addr(&ctl.full[0]);
    const uint32_t empty0 = ptx::smem_addr(&ctl.empty[0]);

    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            ptx::mbar_init(full0 + 8u * s, 1);
            ptx::mbar_init(empty0 + 8u * s, kConsumerWarps);
        }
        ptx::mbar_init(ptx::smem_addr(&ctl.stat[0]), k);
        ptx::mbar_init(ptx::smem_addr(&ctl.stat[1]), k);
        ctl.abort = 0;
        ptx::fence_mbar_init_cluster();
    }
    __syncthreads();
    ptx::cluster_sync();  // every CTA's barriers exist before anyone signals them

    const int64_t n_iter = (static_cast<int64_t>(cid) < p.N) ? (p.N - 1 - cid) / ncl + 1 : 0;
    volatile int *abort = &ctl.abort;

    if (warp == kConsumerWarps) {
        if (lane == 0) produce<BF16>(p, ctl, ptx::smem_addr(ring), cid, ncl, crank, n_iter);
        __syncwarp();
    } else {
        // The label census of this call must be complete before it is read.
        ptx::griddep_wait();
        const int64_t n_valid = p.counts[0];
        float scale0 = p.grad_scale;
        if (p.reduction == VLMCE_MEAN)
            scale0 = n_valid > 0 ? p.grad_scale / static_cast<float>(n_valid) : 0.f;
        const float T = p.softcap;
        const float k2 = SOFTCAP ? -2.f * kLog2e / T : 0.f;

        int64_t q = 0;  // ring position of the row's first chunk, in step with the producer
        for (int64_t it = 0; it < n_iter; ++it) {
            const int pp = static_cast<int>(it & 1);
            const int64_t r = static_cast<int64_t>(cid) + it * ncl;
            const int64_t y = p.labels[r];
            const bool ignored = (y == p.ignore_index);
            const bool valid = !ignored && y >= 0 && y < p.V;
            const RowGeo g = row_geo<BF16>(p, r, crank);
            const int nch = (g.n_my + kChunkGranules - 1) / kChunkGranules;
            const int gy = valid ? static_cast<int>((y + g.lead) / EPG) - g.g_beg : -1;
            const int ly = valid ? static_cast<int>((y + g.lead) % EPG) : 0;

            // ---- pass A over the slice as its slots land
            Acc a;
            a.mv = -INFINITY;
            a.midx = INT_MAX;
            a.mz = -INFINITY;
            a.nmL = pk(INFINITY, INFINITY);
            a.s = pk(0.f, 0.f);
            a.sz = pk(0.f, 0.f);
            float zy = 0.f;
            for (int c = 0; c < nch; ++c) {
                const int64_t qc = q + c;
                const int slot = static_cast<int>(qc % kSlots);
                bounded_wait<false, true>(full0 + 8u * slot,
                                          static_cast<uint32_t>((qc / kSlots) & 1), abort, p.err);
                const int gl = c * kChunkGranules + tid;
                if (gl < g.n_my) {
                    const uint4 w =
                        *reinterpret_cast<const uint4 *>(ring + slot * kChunkBytes + 16 * tid);
                    pass_a_granule<BF16, SOFTCAP>(a, w, (g.g_beg + gl) * EPG - g.lead, p.V, T, k2);
                    if (gl == gy) {  // the label's logit
                        float xv[EPG];
                        unpack<BF16>(w, xv);
                        float xy = xv[0];
#pragma unroll
                        for (int l = 1; l < EPG; ++l)
                            if (l == ly) xy = xv[l];
                        zy = softcap_z<SOFTCAP>(xy, T, k2).z;
                    }
                }
            }
            RowPart part = part_identity();
            part.mx = a.mv;
            part.idx = a.midx;
            part.mz = a.mz;
            {
                float s0, s1, z0, z1;
                upk(a.s, s0, s1);
                upk(a.sz, z0, z1);
                part.s = s0 + s1;
                part.sz = z0 + z1;
            }
            part.zy = zy;
            warp_allreduce(part);

            // ---- the CTA's partial (the consumer warps meet on named barrier
            // 1), published by the first consumer warp to every CTA of the
            // cluster (lane c to CTA c, in parallel); then every warp merges
            // the k CTA partials of the row (same order everywhere)
            if (lane == 0) ctl.wslot[pp][warp] = part;
            consumers_sync();
            if (warp == 0) {
                RowPart cp = part_identity();
                if (lane < kConsumerWarps) cp = ctl.wslot[pp][lane];
                warp_allreduce(cp);
                if (static_cast<uint32_t>(lane) < k) {
                    const uint32_t dst = ptx::smem_addr(&ctl.xslot[pp][crank]);
                    const uint32_t bar = ptx::smem_addr(&ctl.stat[pp]);
                    const uint4 v0 = make_uint4(__float_as_uint(cp.mx), static_cast<uint32_t>(cp.idx),
                                                __float_as_uint(cp.mz), __float_as_uint(cp.s));
                    const uint4 v1 = make_uint4(__float_as_uint(cp.sz), __float_as_uint(cp.zy), 0u, 0u);
                    const uint32_t ra = ptx::mapa(dst, static_cast<uint32_t>(lane));
                    ptx::st_dsmem_v4(ra, v0);
                    ptx::st_dsmem_v4(ra + 16, v1);
                    ptx::mbar_remote_arrive_release(ptx::mapa(bar, static_cast<uint32_t>(lane)));
                }
            }
            bounded_wait<true, false>(ptx::smem_addr(&ctl.stat[pp]),
                                      static_cast<uint32_t>((it >> 1) & 1), abort, p.err);
            RowPart rp = part_identity();
            if (static_cast<uint32_t>(lane) < k) rp = ctl.xslot[pp][lane];
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

            // ---- pass B: gradient from shared memory, stored over the logits
            unsigned char *grow = reinterpret_cast<unsigned char *>(g.gbase) + 16 * g.g_beg;
            const float scale = p.token_scale ? scale0 * p.token_scale[r] : scale0;
            const float c_smooth = scale * (p.eps / static_cast<float>(p.V));  // scale eps / V
            const float c_label = c_smooth + scale * (1.f - p.eps);            // + scale (1 - eps)
            const ExpCoef ec = grad_exp_coef(lse, scale);
            const uint64_t nlseL2 = pk(ec.nlseL, ec.nlseL);
            const uint64_t scale2 = pk(ec.scale, ec.scale);
            const uint64_t negc2 = pk(-c_smooth, -c_smooth);
            for (int c = 0; c < nch && p.want_grad; ++c) {
                const int slot = static_cast<int>((q + c) % kSlots);
                const int gl = c * kChunkGranules + tid;
                if (gl < g.n_my) {
                    const int jg = (g.g_beg + gl) * EPG - g.lead;
                    if (valid) {
                        const uint4 w =
                            *reinterpret_cast<const uint4 *>(ring + slot * kChunkBytes + 16 * tid);
                        pass_b_granule<BF16, SOFTCAP>(w, jg, p.V, grow + 16 * gl, T, k2, nlseL2,
                                                      scale2, negc2, gl == gy ? ly : -1, ec.scale,
                                                      c_label);
                    } else {
                        store_zero_granule<BF16>(jg, p.V, grow + 16 * gl);
                    }
                }
            }
            // ---- the row's slots are free again
            __syncwarp();
            if (lane == 0) {
                for (int c = 0; c < nch; ++c)
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                                     empty0 + 8u * static_cast<uint32_t>((q + c) % kSlots))
                                 : "memory");
            }
            q += nch;
        }
    }
    ptx::griddep_launch_dependents();
    __syncthreads();
    ptx::cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

// The V-split kernel for the given softcap, per element type (ce_split_bf16.cu,
// ce_split_f32.cu).
SplitKernel split_kernel_bf16(bool softcap);
SplitKernel split_kernel_f32(bool softcap);

}  // namespace split
}  // namespace ce
}  // namespace vlmce
