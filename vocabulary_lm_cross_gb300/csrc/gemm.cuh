// gemm.cuh -- persistent tcgen05 GEMM for sm_103a, run by CTA pairs, with the
// fused linear-cross-entropy epilogues.
//
// C[M, N] = A[M, K] * B[N, K]^T with bf16 operands and fp32 accumulation in
// tensor memory.  Either operand may be stored K-major (K contiguous) or
// MN-major (M or N contiguous), so the three products of the fused linear
// cross-entropy need no transposed copies:
//   logits  S   = h' W_c^T     A = h' [N, H] K-major,   B = W_c [Vc, H] K-major
//   grad_h     += G_c W_c      A = G_c [N, Vc] K-major,  B = W_c: N(=H)-major
//   grad_W_c    = G_c^T h'     A = G_c: M(=Vc)-major,    B = h': N(=H)-major
//
// One launch runs up to kMaxProblems independent products ("problems") over
// one persistent grid: their 256 x 256 tiles are numbered one after the
// other and strided over the clusters, so a launch has a single tail.
//
// Cluster = 2 CTAs on two SMs ("pair"); the pair computes one 256 x 256 tile
// with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16 per instruction).
// Each CTA stages its own 128 rows of A and its own 128 rows of B (K = 128
// per stage as two 64-wide halves, 128-byte swizzle) in a 3-stage ring of
// 64 KB stages: each operand row is requested as 256 contiguous bytes per
// stage and a stage costs one barrier round trip per 128 K (measured 5.8 %
// faster per fused linear CE call than six 32 KB stages of K = 64).  A CTA
// moves a third less operand data per flop than a single-SM 128 x 256 tile
// would, and each
// CTA's TMEM receives its 128 rows of the tile.  Every operand copy is a
// plain load into the issuing CTA's own shared memory.  CTA = 7 warps:
//   warp 0      one lane issues the TMA loads of this CTA's halves; the
//               copies of both CTAs count on the leader's "full" barrier;
//   warp 1      allocates 512 TMEM columns per SM (two 128 x 256 fp32
//               accumulators) with its peer; in the leader one lane issues
//               the pair MMAs and commits them to both CTAs' barriers;
//   warps 2-5   epilogue: each reads its 32-lane TMEM subpartition (one
//               accumulator row per thread) in 32-column chunks while the
//               MMA fills the other accumulator; both CTAs' epilogue warps
//               release an accumulator on the leader's "tmem empty" barrier;
//   warp 6      in the leader, with a tile counter, one lane takes the tile
//               numbers in order and publishes them to both CTAs (the tiles
//               in flight then stay a window of consecutive numbers, so the
//               row tiles that share a weight tile read it close in time).
// Without a counter the clusters stride over the tiles statically.
//
// Operand tile layouts in shared memory (per CTA and 64-wide K half, the
// second half 16 KB after the first; bf16, 128-byte swizzle atoms of 8 rows x
// 128 bytes):
//   K-major  (128 rows of M or N, 64 K-elements = 128 B per row): 8-row
//            groups 1024 B apart (SBO); a K-step of 16 elements advances the
//            start address by 32 B.
//   MN-major (64 rows of K, 128 B = 64 M/N-elements per row, one TMA box of
//            64 x 64 per 64 M/N): 8-row (K) groups 1024 B apart (SBO), the
//            two 64-wide M/N groups 8192 B apart (LBO); a K-step of 16 rows
//            advances by 2048 B.
//
// Every wait on an mbarrier is bounded (kWaitLimitNs); a wait that gives up
// sets VLMCE_DEVERR_TIMEOUT in the device error word and the CTA runs its
// remaining loops without waiting, so the launch always ends.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ce_common.cuh"
#include "gemm_types.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace vlmce {
namespace gemm {

// ------------------------------------------------------------ barriers
template <bool CLUSTER_ACQUIRE = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort,
                                         int *err) {
    auto try_once = [&] {
        return CLUSTER_ACQUIRE ? ptx::mbar_try_wait_cluster(bar, parity)
                               : ptx::mbar_try_wait(bar, parity);
    };
    if (try_once()) return true;
    if (*abort) return false;
    const unsigned long long t0 = ptx::globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (try_once()) return true;
        if (*abort) return false;
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            if (err) atomicOr(err, VLMCE_DEVERR_TIMEOUT);
            return false;
        }
    }
}
// Same, but never skipped: used where copies or MMAs may still be in flight.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, int *err) {
    volatile int no_abort = 0;
    wait_bar(bar, parity, &no_abort, err);
}

// ------------------------------------------------------------ tiles
struct Tile {
    int p, m0, n0;
};
// Pair tile t of the launch: problem, first row, first column.
__device__ __forceinline__ Tile tile_of(const Params &a, int t) {
    int p = 0;
#pragma unroll
    for (int i = 1; i < kMaxProblems; ++i)
        if (i < a.nprob && t >= a.p[i].tile0) p = i;
    const int lt = t - a.p[p].tile0;
    const int mt = a.p[p].mt;
    return Tile{p, (lt % mt) * BM, (lt / mt) * BN};
}

// ------------------------------------------------------------ epilogues
__device__ __forceinline__ void st_v4f(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}

// Two fp32 values -> a bf16x2 or fp16x2 word, round to nearest even.
__device__ __forceinline__ uint32_t pack16x2(float a, float b, bool f16) {
    if (!f16) return ce::pack_bf16x2(a, b);
    const __half2 v = __floats2half2_rn(a, b);  // a in the low half, as for bf16
    uint32_t u;
    memcpy(&u, &v, 4);
    return u;
}
__device__ __forceinline__ uint16_t to16(float a, bool f16) {
    return f16 ? __half_as_ushort(__float2half_rn(a)) : __bfloat16_as_ushort(__float2bfloat16_rn(a));
}
__device__ __forceinline__ void store16x32(uint16_t *c16, const float (&o)[32], int nvalid, bool f16) {
    if (nvalid == 32) {
#pragma unroll
        for (int j = 0; j < 32; j += 8)
            *reinterpret_cast<uint4 *>(c16 + j) =
                make_uint4(pack16x2(o[j], o[j + 1], f16), pack16x2(o[j + 2], o[j + 3], f16),
                           pack16x2(o[j + 4], o[j + 5], f16), pack16x2(o[j + 6], o[j + 7], f16));
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < nvalid) c16[j] = to16(o[j], f16);
    }
}

// Per-row state of the statistics epilogue (pass 1 of the fused linear CE).
struct StatAcc {
    float mx;
    int idx;
    float mz, s, sz, zy;
};

// fp32 / 16-bit output modes on one 32-column chunk of one row; the
// accumulator is multiplied by `sc` first.
template <int MODE>
__device__ __forceinline__ void store_chunk(const Problem &P, const float (&v)[32], int row,
                                            int cbase, int nvalid, float sc, bool f16) {
    float o[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] = v[j] * sc;
    if constexpr (MODE == kStoreF32 || MODE == kAccF32 || MODE == kAccToBF16) {
        float *c = P.C + static_cast<int64_t>(row) * P.ldc + cbase;
        if constexpr (MODE != kStoreF32) {
            if (nvalid == 32) {
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 old = *reinterpret_cast<const float4 *>(c + j);
                    o[j] += old.x;
                    o[j + 1] += old.y;
                    o[j + 2] += old.z;
                    o[j + 3] += old.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < nvalid) o[j] += c[j];
            }
        }
        if constexpr (MODE == kAccToBF16) {
            store16x32(P.C16 + static_cast<int64_t>(row) * P.ldc16 + cbase, o, nvalid, f16);
        } else {
            if (nvalid == 32) {
#pragma unroll
                for (int j = 0; j < 32; j += 4) st_v4f(c + j, o[j], o[j + 1], o[j + 2], o[j + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < nvalid) c[j] = o[j];
            }
        }
    } else {  // kStoreBF16
        uint16_t *c16 = P.C16 + static_cast<int64_t>(row) * P.ldc16 + cbase;
        if (nvalid == 32 && (P.ldc16 % 8) == 0) {
            store16x32(c16, o, 32, f16);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < nvalid) c16[j] = to16(o[j], f16);
        }
    }
}

// Statistics of one 32-column chunk of a logits row (max / first argmax of
// S, online sum of exp(z - m_z), sum of z, z at the label).
__device__ __forceinline__ void stats_chunk(const Params &a, const Problem &P,
                                            const float (&v)[32], int cbase, int nvalid,
                                            StatAcc &st, int64_t y) {
    float cm = -INFINITY;
    int ci = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j < nvalid && v[j] > cm) {
            cm = v[j];
            ci = j;
        }
    const bool cap = a.T > 0.f;
    if (cm > st.mx) {
        const float nz = cap ? ce::softcap_z<true>(cm, a.T, a.k2).z : cm;
        const float f = ptx::ex2((st.mz - nz) * ce::kLog2e);
        st.s = (st.s == 0.f) ? 0.f : st.s * f;
        st.mx = cm;
        st.idx = P.col0 + cbase + ci;
        st.mz = nz;
    }
    const float nm = -st.mz * ce::kLog2e;
    float s0 = 0.f, s1 = 0.f, z0 = 0.f, z1 = 0.f;
    if (cap) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float za = ce::softcap_z<true>(v[j], a.T, a.k2).z;
            const float zb = ce::softcap_z<true>(v[j + 1], a.T, a.k2).z;
            if (j < nvalid) {
                s0 += ptx::ex2(fmaf(za, ce::kLog2e, nm));
                z0 += za;
            }
            if (j + 1 < nvalid) {
                s1 += ptx::ex2(fmaf(zb, ce::kLog2e, nm));
                z1 += zb;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            if (j < nvalid) {
                s0 += ptx::ex2(fmaf(v[j], ce::kLog2e, nm));
                z0 += v[j];
            }
            if (j + 1 < nvalid) {
                s1 += ptx::ex2(fmaf(v[j + 1], ce::kLog2e, nm));
                z1 += v[j + 1];
            }
        }
    }
    st.s += s0 + s1;
    st.sz += z0 + z1;
    const int64_t yl = y - P.col0 - cbase;  // label column within this chunk
    if (yl >= 0 && yl < nvalid) {
        float xy = v[0];
#pragma unroll
        for (int j = 1; j < 32; ++j)
            if (j == yl) xy = v[j];
        st.zy = cap ? ce::softcap_z<true>(xy, a.T, a.k2).z : xy;
    }
}

// Gradient tile of one 32-column chunk: (softmax - q) (1 - t^2) times m (the
// launch's power-of-two grad_mul for a valid row, 0 otherwise) -> 16-bit.
// The rows' common scale is applied by the products that consume the tile.
__device__ __forceinline__ void grad_chunk(const Params &a, const Problem &P, const float (&v)[32],
                                           int row, int cbase, int nvalid, int64_t y, float m,
                                           float nlseL) {
    const bool cap = a.T > 0.f;
    const float c_smooth = m * (a.eps / static_cast<float>(a.V));
    const float c_label = c_smooth + m * (1.f - a.eps);
    const int64_t yl = y - P.col0 - cbase;
    float g[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        float z = v[j], dz = 1.f;
        if (cap) {
            const ce::Capped cz = ce::softcap_z<true>(v[j], a.T, a.k2);
            z = cz.z;
            dz = cz.dz;
        }
        const float pr = ptx::ex2(fmaf(z, ce::kLog2e, nlseL));
        g[j] = fmaf(pr, m, (j == yl) ? -c_label : -c_smooth) * dz;
    }
    store16x32(P.C16 + static_cast<int64_t>(row) * P.ldc16 + cbase, g, nvalid, a.f16 != 0);
}

// ------------------------------------------------------------ the kernel
// Launched with clusters of 2 CTAs (one pair; CTA 0 is its leader) and a
// grid of co-resident clusters; needs kSmemBytes of dynamic shared memory.
__global__ void __launch_bounds__(kThreads, 1)
    vlmce_gemm_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Params a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBarriers);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *tq = reinterpret_cast<volatile int *>(tmem_slot + 4);  // [kTileQ] tile numbers
    const uint32_t ring = ptx::smem_addr(smem);
    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
    const uint32_t drain = bar0 + 8u * (2 * kStages + 4);
    auto qfull = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + i); };
    auto qempty = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + kTileQ + i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t prank = ptx::cluster_ctarank();  // 0: the pair's leader
    const uint16_t pair_ctas = 3u;
    const int cluster = static_cast<int>(ptx::cluster_id_x());
    const int nclusters = static_cast<int>(ptx::ncluster_x());

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // leader: its producer's arrival + the bytes of both CTAs of the pair
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);  // one commit from the leader's MMA issuer
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull(b), 1);
            ptx::mbar_init(tempty(b), 8);  // leader: 4 epilogue warps x 2 CTAs
        }
        ptx::mbar_init(drain, 1);
        for (int i = 0; i < kTileQ; ++i) {
            ptx::mbar_init(qfull(i), 1);                 // the leader producer's release-arrive
            ptx::mbar_init(qempty(i), kTileQConsumers);  // used at the leader only
        }
        *abort = 0;
        ptx::fence_mbar_init_cluster();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < a.nprob; ++i) {
            tc::prefetch_tensormap(&maps.a[i]);
            tc::prefetch_tensormap(&maps.b[i]);
        }
    }
    if (warp == 1) {
        tc::tmem_alloc_pair(ptx::smem_addr(tmem_slot), kTmemCols);
        tc::tmem_relinquish_pair();
    }
    tc::fence_before_sync();
    ptx::cluster_sync_any();  // barrier inits and the TMEM address visible to the cluster
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // The j-th tile this cluster runs (-1: none left).  Static order: tile
    // cluster + j * #clusters.  Dynamic order (a.tile_ctr): the leader's
    // scheduler warp takes tile numbers from the counter, up to kTileQ ahead
    // of the slowest role, and publishes each to queue slot j % kTileQ of both
    // CTAs; every role reads the slot and releases it on the leader.  A wait
    // that gives up ends the sequence (the error bit is set).
    const bool dyn = a.tile_ctr != nullptr;
    auto static_tile = [&](int j) {
        const int64_t t = cluster + static_cast<int64_t>(j) * nclusters;
        return t < a.tiles ? static_cast<int>(t) : -1;
    };
    auto publish = [&](int j) {  // the leader's scheduler lane
        const int slot = j % kTileQ;
        int t = -1;
        if (j < kTileQ || wait_bar<true>(qempty(slot), ((j / kTileQ) - 1) & 1, abort, a.err)) {
            const unsigned int u = atomicAdd(a.tile_ctr, 1u);
            t = u < static_cast<unsigned int>(a.tiles) ? static_cast<int>(u) : -1;
        }
        tq[slot] = t;
        ptx::st_dsmem_u32(ptx::mapa(ptx::smem_addr(const_cast<int *>(tq) + slot), 1),
                          static_cast<uint32_t>(t));
        ptx::mbar_arrive(qfull(slot));
        ptx::mbar_remote_arrive_release(ptx::mapa(qfull(slot), 1));
        return t;
    };
    auto consume = [&](int j) {  // every other role; all lanes of a warp call it
        const int slot = j % kTileQ;
        int t = -1;
        if (wait_bar<true>(qfull(slot), (j / kTileQ) & 1, abort, a.err)) t = tq[slot];
        __syncwarp(__activemask());  // every lane has read the slot
        if (lane == 0) {
            if (prank == 0)
                ptx::mbar_arrive(qempty(slot));
            else
                ptx::mbar_remote_arrive_release(ptx::mapa(qempty(slot), 0));
        }
        return t;
    };

    if (warp == 0) {
        // ---- TMA producer (every CTA): this CTA's 128 rows of A and its
        // 128-row half of the pair's B tile.  Every copy counts on the full
        // barrier of the pair leader.
        if (lane == 0) {
            const uint32_t full_leader = ptx::mapa(full(0), 0);
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            for (int j = 0;; ++j) {
                const int t = dyn ? consume(j) : static_tile(j);
                if (t < 0) break;
                const Tile tl = tile_of(a, t);
                const Problem &P = a.p[tl.p];
                const CUtensorMap *ma = &maps.a[tl.p];
                const CUtensorMap *mb = &maps.b[tl.p];
                const int ar = tl.m0 + kHalf * static_cast<int>(prank);
                const int br = tl.n0 + kHalf * static_cast<int>(prank);
                const int kblocks = (P.K + BK - 1) / BK;
                for (int kb = 0; kb < kblocks; ++kb) {
                    wait_bar(empty(s), ph ^ 1, abort, a.err);
                    if (prank == 0) ptx::mbar_arrive_expect_tx(full(s), 2 * kStageBytes);
                    const uint32_t sa = ring + s * kStageBytes, sb = sa + kOpBytes;
                    const uint32_t fb = full_leader + 8u * s;
                    // per 64 K: K-major one 64 x 128 box; MN-major two 64 x 64 boxes
#pragma unroll
                    for (int hk = 0; hk < BK / 64; ++hk) {
                        const int kc = kb * BK + 64 * hk;
                        const uint32_t oa = sa + 16384u * hk, ob = sb + 16384u * hk;
                        if (!P.a_mn) {
                            tc::tma_load_2d_pair(oa, ma, kc, ar, fb);
                        } else {
                            tc::tma_load_2d_pair(oa, ma, ar, kc, fb);
                            tc::tma_load_2d_pair(oa + 8192, ma, ar + 64, kc, fb);
                        }
                        if (!P.b_mn) {
                            tc::tma_load_2d_pair(ob, mb, kc, br, fb);
                        } else {
                            tc::tma_load_2d_pair(ob, mb, br, kc, fb);
                            tc::tma_load_2d_pair(ob + 8192, mb, br + 64, kc, fb);
                        }
                    }
                    ++issued;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            // at a leader, every copy into its pair has landed once the full
            // phases of the last kStages loads completed
            if (prank == 0) {
                for (int i = 0; i < kStages && i < issued; ++i) {
                    const int64_t q = issued - 1 - i;
                    drain_bar(full(static_cast<int>(q % kStages)),
                              static_cast<uint32_t>((q / kStages) & 1), a.err);
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer (pair leader)
        if (prank == 0 && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int it = 0;; ++it) {
                const int t = dyn ? consume(it) : static_tile(it);
                if (t < 0) break;
                const Tile tl = tile_of(a, t);
                const Problem &P = a.p[tl.p];
                const uint32_t idesc = tc::idesc_bf16_f32(BM, BN, P.a_mn != 0, P.b_mn != 0, a.f16 != 0);
                const int kblocks = (P.K + BK - 1) / BK;
                const int b = it & 1;
                wait_bar<true>(tempty(b), ((it >> 1) & 1) ^ 1, abort, a.err);
                tc::fence_after_sync();
                const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
                for (int kb = 0; kb < kblocks; ++kb) {
                    wait_bar(full(s), ph, abort, a.err);
                    tc::fence_after_sync();
                    const uint32_t sa = ring + s * kStageBytes, sb = sa + kOpBytes;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint32_t kh = 16384u * (kk >> 2), kq = kk & 3;
                        const uint64_t ad = P.a_mn ? tc::smem_desc_sw128(sa + kh + 2048 * kq, 8192, 1024)
                                                   : tc::smem_desc_sw128(sa + kh + 32 * kq, 16, 1024);
                        const uint64_t bd = P.b_mn ? tc::smem_desc_sw128(sb + kh + 2048 * kq, 8192, 1024)
                                                   : tc::smem_desc_sw128(sb + kh + 32 * kq, 16, 1024);
                        tc::mma_bf16_pair(d, ad, bd, idesc, (kb | kk) != 0);
                    }
                    tc::mma_commit_pair(empty(s), pair_ctas);  // the stage is free in both CTAs
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                tc::mma_commit_pair(tfull(b), pair_ctas);
            }
            tc::mma_commit_pair(drain, static_cast<uint16_t>(1u << prank));
            drain_bar(drain, 0, a.err);
        }
    } else if (warp == 6) {
        // ---- tile scheduler (pair leader, dynamic order only)
        if (dyn && prank == 0 && lane == 0) {
            for (int j = 0;; ++j)
                if (publish(j) < 0) break;
        }
    } else {
        // ---- epilogue: warps 2-5 of every CTA, TMEM subpartition warp % 4
        const int q = warp & 3;
        const int rl = static_cast<int>(prank) * kHalf + q * 32 + lane;
        const uint32_t tempty_leader = ptx::mapa(tempty(0), 0);
        for (int it = 0;; ++it) {
            const int t = dyn ? consume(it) : static_tile(it);
            if (t < 0) break;
            const Tile tl = tile_of(a, t);
            const Problem &P = a.p[tl.p];
            const int b = it & 1;
            wait_bar(tfull(b), (it >> 1) & 1, abort, a.err);
            tc::fence_after_sync();
            const int row = tl.m0 + rl;
            const bool row_ok = row < P.M;
            int64_t y = -1;
            float m = 0.f, nlseL = 0.f;
            if ((P.mode == kStats || P.mode == kGrad) && row_ok) {
                y = a.labels[row];
                if (P.mode == kGrad) {
                    m = a.row_scale[row] != 0.f ? a.grad_mul : 0.f;
                    nlseL = -a.lse[row] * ce::kLog2e;
                }
            }
            const float sc = a.out_scale ? *a.out_scale : 1.f;
            const bool f16 = a.f16 != 0;
            StatAcc st;
            st.mx = -INFINITY;
            st.idx = INT_MAX;
            st.mz = -INFINITY;
            st.s = 0.f;
            st.sz = 0.f;
            st.zy = 0.f;
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tc::tmem_ld32(tbase + 32 * c, r);
                tc::tmem_ld_wait();
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                const int cbase = tl.n0 + 32 * c;
                const int nvalid = min(32, P.N - cbase);
                if (nvalid <= 0 || !row_ok) continue;
                switch (P.mode) {
                    case kStats: stats_chunk(a, P, v, cbase, nvalid, st, y); break;
                    case kGrad: grad_chunk(a, P, v, row, cbase, nvalid, y, m, nlseL); break;
                    case kStoreF32: store_chunk<kStoreF32>(P, v, row, cbase, nvalid, sc, f16); break;
                    case kAccF32: store_chunk<kAccF32>(P, v, row, cbase, nvalid, sc, f16); break;
                    case kStoreBF16: store_chunk<kStoreBF16>(P, v, row, cbase, nvalid, sc, f16); break;
                    default: store_chunk<kAccToBF16>(P, v, row, cbase, nvalid, sc, f16); break;
                }
            }
            if (P.mode == kStats && row_ok) {
                ce::RowPart p;
                p.mx = st.mx;
                p.idx = st.idx;
                p.mz = st.mz;
                p.s = st.s;
                p.sz = st.sz;
                p.zy = st.zy;
                p.pad0 = p.pad1 = 0.f;
                P.part[static_cast<int64_t>(tl.n0 / BN) * P.part_ld + row] = p;
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_remote_arrive_release(tempty_leader + 8u * b);
        }
    }
    // teardown: every MMA of the cluster has completed (drain) and every copy
    // into it has landed; the cluster meets before TMEM is released and any
    // CTA exits
    tc::fence_before_sync();
    __syncthreads();
    ptx::cluster_sync_any();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace gemm
}  // namespace vlmce
