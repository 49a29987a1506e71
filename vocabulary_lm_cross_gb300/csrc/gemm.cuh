// gemm.cuh -- persistent tcgen05 GEMM for sm_103a with the fused
// linear-cross-entropy epilogues.
//
// C[M, N] = A[M, K] * B[N, K]^T with bf16 operands and fp32 accumulation in
// tensor memory.  Either operand may be stored K-major (K contiguous) or
// MN-major (M or N contiguous), so the three products of the fused linear
// cross-entropy need no transposed copies:
//   logits  S   = h' W_c^T     A = h' [N, H] K-major,   B = W_c [Vc, H] K-major
//   grad_h     += G_c W_c      A = G_c [N, Vc] K-major,  B = W_c: N(=H)-major
//   grad_W_c    = G_c^T h'     A = G_c: M(=Vc)-major,    B = h': N(=H)-major
//
// CTA = 6 warps, one per SM (persistent, tiles strided over the grid):
//   warp 0      one lane issues the TMA loads of A and B tiles (128x64 and
//               256x64 bf16, 128-byte swizzle) into a 4-stage ring;
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators)
//               and one lane issues tcgen05.mma (M=128, N=256, K=16 per
//               instruction), committing to the ring's empty barriers and,
//               per tile, to the accumulator's full barrier;
//   warps 2-5   epilogue: each reads its 32-lane TMEM subpartition (one
//               accumulator row per thread) in 32-column chunks while the
//               MMA fills the other accumulator.
//
// Operand tile layouts in shared memory (bf16, 128-byte swizzle atoms of
// 8 rows x 128 bytes):
//   K-major  (rows = M or N, 64 K-elements = 128 B per row): consecutive
//            8-row groups 1024 B apart (SBO); one K-step of 16 elements
//            advances the start address by 32 B.
//   MN-major (rows = K, 64 M/N-elements = 128 B per row, one TMA box of
//            64 x 64 per 64 M/N): 8-row (K) groups 1024 B apart (SBO), 64-wide
//            M/N groups 8192 B apart (LBO); a K-step of 16 rows advances by
//            2048 B.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "ce_common.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace vlmce {
namespace gemm {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;  // 16 KB
constexpr int kBBytes = BN * BK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kTmemCols = 2 * BN;
constexpr int kBarriers = 2 * kStages + 5;  // full, empty, tmem full x2, tmem empty x2, drain
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 8 * kBarriers + 16;
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

enum Mode : int {
    kStoreF32 = 0,   // C = acc (fp32)
    kAccF32 = 1,     // C += acc (fp32)
    kStats = 2,      // row statistics of the logits tile (fused linear CE, pass 1)
    kGrad = 3,       // gradient tile G = scale (p - q) (1 - t^2) -> bf16 (pass 2)
    kStoreBF16 = 4,  // C16 = bf16(acc)
    kAccToBF16 = 5,  // C16 = bf16(C + acc)
};

struct Args {
    int M, N, K;
    float *C;                  // fp32 [M, ldc]
    int64_t ldc;
    __nv_bfloat16 *C16;        // bf16 [M, ldc16]
    int64_t ldc16;
    // cross-entropy epilogues
    const int64_t *labels;     // [M]
    int64_t ignore_index;
    int col0;                  // vocabulary column of n = 0
    int V;                     // vocabulary size
    float eps, T, k2;          // smoothing, softcap (0 = off), -2 log2e / T
    ce::RowPart *part;         // kStats: part[n_tile * part_ld + row]
    int64_t part_ld;
    const float *lse;          // kGrad: [M]
    const float *row_scale;    // kGrad: [M] scale of a valid row, 0 otherwise
    int *err;                  // device error word
};

// ------------------------------------------------------------ barriers
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort,
                                         int *err) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    const unsigned long long t0 = ptx::globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
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

__device__ __forceinline__ void bar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// ------------------------------------------------------------ epilogues
__device__ __forceinline__ void st_v4f(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}

// Per-row state of the statistics epilogue (pass 1 of the fused linear CE).
struct StatAcc {
    float mx;
    int idx;
    float mz, s, sz, zy;
};

template <int MODE>
__device__ __forceinline__ void epilogue_chunk(const Args &a, const float (&v)[32], int row,
                                               int cbase, StatAcc &st, int64_t y, float rscale,
                                               float nlseL) {
    const int nvalid = min(32, a.N - cbase);
    if (nvalid <= 0 || row >= a.M) return;
    if constexpr (MODE == kStoreF32 || MODE == kAccF32 || MODE == kAccToBF16) {
        float *c = a.C + static_cast<int64_t>(row) * a.ldc + cbase;
        float o[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = v[j];
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
            __nv_bfloat16 *c16 = a.C16 + static_cast<int64_t>(row) * a.ldc16 + cbase;
            if (nvalid == 32) {
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    *reinterpret_cast<uint4 *>(c16 + j) =
                        make_uint4(ce::pack_bf16x2(o[j], o[j + 1]), ce::pack_bf16x2(o[j + 2], o[j + 3]),
                                   ce::pack_bf16x2(o[j + 4], o[j + 5]), ce::pack_bf16x2(o[j + 6], o[j + 7]));
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < nvalid) c16[j] = __float2bfloat16_rn(o[j]);
            }
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
    } else if constexpr (MODE == kStoreBF16) {
        __nv_bfloat16 *c16 = a.C16 + static_cast<int64_t>(row) * a.ldc16 + cbase;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < nvalid) c16[j] = __float2bfloat16_rn(v[j]);
    } else if constexpr (MODE == kStats) {
        // chunk max and its first column among the valid ones
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
            st.idx = a.col0 + cbase + ci;
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
        const int64_t yl = y - a.col0 - cbase;  // label column within this chunk
        if (yl >= 0 && yl < nvalid) {
            float xy = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j)
                if (j == yl) xy = v[j];
            st.zy = cap ? ce::softcap_z<true>(xy, a.T, a.k2).z : xy;
        }
    } else if constexpr (MODE == kGrad) {
        const bool cap = a.T > 0.f;
        const float c_smooth = rscale * (a.eps / static_cast<float>(a.V));
        const float c_label = c_smooth + rscale * (1.f - a.eps);
        const int64_t yl = y - a.col0 - cbase;
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
            g[j] = fmaf(pr, rscale, (j == yl) ? -c_label : -c_smooth) * dz;
        }
        __nv_bfloat16 *c16 = a.C16 + static_cast<int64_t>(row) * a.ldc16 + cbase;
        if (nvalid == 32) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                *reinterpret_cast<uint4 *>(c16 + j) =
                    make_uint4(ce::pack_bf16x2(g[j], g[j + 1]), ce::pack_bf16x2(g[j + 2], g[j + 3]),
                               ce::pack_bf16x2(g[j + 4], g[j + 5]), ce::pack_bf16x2(g[j + 6], g[j + 7]));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < nvalid) c16[j] = __float2bfloat16_rn(g[j]);
        }
    }
}

// ------------------------------------------------------------ the kernel
template <int MODE, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
    vlmce_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const Args a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBarriers);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t ring = ptx::smem_addr(smem);
    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
    const uint32_t drain = bar0 + 8u * (2 * kStages + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Mt = (a.M + BM - 1) / BM, Nt = (a.N + BN - 1) / BN;
    const int tiles = Mt * Nt;
    const int kblocks = (a.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull(b), 1);
            ptx::mbar_init(tempty(b), 4);
        }
        ptx::mbar_init(drain, 1);
        *abort = 0;
        ptx::fence_mbar_init_cluster();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tensormap(&tmA);
        tc::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tc::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---- TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
                const int m0 = (t % Mt) * BM, n0 = (t / Mt) * BN;
                for (int kb = 0; kb < kblocks; ++kb) {
                    wait_bar(empty(s), ph ^ 1, abort, a.err);
                    ptx::mbar_arrive_expect_tx(full(s), kStageBytes);
                    const uint32_t sa = ring + s * kStageBytes, sb = sa + kABytes;
                    if constexpr (!A_MN) {
                        tc::tma_load_2d(sa, &tmA, kb * BK, m0, full(s));
                    } else {
                        tc::tma_load_2d(sa, &tmA, m0, kb * BK, full(s));
                        tc::tma_load_2d(sa + 8192, &tmA, m0 + 64, kb * BK, full(s));
                    }
                    if constexpr (!B_MN) {
                        tc::tma_load_2d(sb, &tmB, kb * BK, n0, full(s));
                    } else {
#pragma unroll
                        for (int i = 0; i < BN / 64; ++i)
                            tc::tma_load_2d(sb + 8192 * i, &tmB, n0 + 64 * i, kb * BK, full(s));
                    }
                    ++issued;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            // every issued copy has landed before teardown
            for (int i = 0; i < kStages && i < issued; ++i) {
                const int64_t q = issued - 1 - i;
                drain_bar(full(static_cast<int>(q % kStages)),
                          static_cast<uint32_t>((q / kStages) & 1), a.err);
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN, A_MN, B_MN);
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
                const int b = it & 1;
                wait_bar(tempty(b), ((it >> 1) & 1) ^ 1, abort, a.err);
                tc::fence_after_sync();
                const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
                for (int kb = 0; kb < kblocks; ++kb) {
                    wait_bar(full(s), ph, abort, a.err);
                    tc::fence_after_sync();
                    const uint32_t sa = ring + s * kStageBytes, sb = sa + kABytes;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = A_MN ? tc::smem_desc_sw128(sa + 2048 * kk, 8192, 1024)
                                                 : tc::smem_desc_sw128(sa + 32 * kk, 16, 1024);
                        const uint64_t bd = B_MN ? tc::smem_desc_sw128(sb + 2048 * kk, 8192, 1024)
                                                 : tc::smem_desc_sw128(sb + 32 * kk, 16, 1024);
                        tc::mma_bf16(d, ad, bd, idesc, (kb | kk) != 0);
                    }
                    tc::mma_commit(empty(s));
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                tc::mma_commit(tfull(b));
            }
            tc::mma_commit(drain);
            drain_bar(drain, 0, a.err);
        }
    } else {
        // ---- epilogue: warps 2-5, TMEM subpartition warp % 4
        const int q = warp & 3;
        const int rl = q * 32 + lane;
        int it = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            const int b = it & 1;
            const int m0 = (t % Mt) * BM, n0 = (t / Mt) * BN;
            wait_bar(tfull(b), (it >> 1) & 1, abort, a.err);
            tc::fence_after_sync();
            const int row = m0 + rl;
            int64_t y = -1;
            float rscale = 0.f, nlseL = 0.f;
            if constexpr (MODE == kStats || MODE == kGrad) {
                if (row < a.M) {
                    y = a.labels[row];
                    if constexpr (MODE == kGrad) {
                        rscale = a.row_scale[row];
                        nlseL = -a.lse[row] * ce::kLog2e;
                    }
                }
            }
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
                epilogue_chunk<MODE>(a, v, row, n0 + 32 * c, st, y, rscale, nlseL);
            }
            if constexpr (MODE == kStats) {
                if (row < a.M) {
                    ce::RowPart p;
                    p.mx = st.mx;
                    p.idx = st.idx;
                    p.mz = st.mz;
                    p.s = st.s;
                    p.sz = st.sz;
                    p.zy = st.zy;
                    p.pad0 = p.pad1 = 0.f;
                    a.part[static_cast<int64_t>(t / Mt) * a.part_ld + row] = p;
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) bar_arrive(tempty(b));
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace gemm
}  // namespace vlmce
