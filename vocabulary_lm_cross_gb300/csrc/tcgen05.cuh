// tcgen05.cuh -- inline-PTX wrappers for the sm_100-family tensor cores,
// in their CTA-pair form (.cta_group::2: one MMA spans the tensor cores of
// two SMs of a cluster): tensor-memory (TMEM) allocation, tcgen05.mma with
// bf16 operands and fp32 accumulators, commits that arrive on the mbarriers
// of both CTAs of the pair, TMEM loads, tiled TMA loads, and the
// shared-memory / instruction descriptors the MMA consumes.  Every tcgen05
// instruction of a kernel must use the same .cta_group.
#pragma once

#include <cuda.h>

#include <cstdint>

namespace vlmce {
namespace tc {

// ------------------------------------------------------------------- TMEM
// Allocate `ncols` TMEM columns (power of two >= 32) in both SMs of the CTA
// pair; one warp of each CTA executes it, and each gets the (common) address
// in its own shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------- MMA
// Pair MMA, issued by one thread of the leader CTA: D (+)= A B^T with A's M
// rows split between the two CTAs (each CTA's half at the same shared-memory
// offset, described by a_desc) and B's N rows likewise (b_desc); each CTA's
// TMEM receives its own M half x all N columns.  bf16 x bf16 -> fp32.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Once every pair MMA this thread issued so far has completed, arrive once on
// the mbarrier at shared-memory offset `mbar` of each CTA in `cta_mask`.
__device__ __forceinline__ void mma_commit_pair(uint32_t mbar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(mbar),
        "h"(cta_mask)
        : "memory");
}

// 32 lanes x 32 consecutive fp32 columns of TMEM into 32 registers per thread
// (thread i of the warp gets lane base + i).  Complete with tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------- TMA
// 2-D tiled bulk tensor loads into this CTA's shared memory at `dst`.  c0 is
// the innermost coordinate (elements; its byte offset must be a multiple of
// 16).
// Pair form: the completed bytes are counted on the mbarrier at
// shared::cluster address `mbar_leader`, the barrier of the pair's leader
// (even) CTA.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *tm, int c0,
                                                 int c1, uint32_t mbar_leader) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tm), "r"(c0), "r"(c1), "r"(mbar_leader)
        : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}

// ------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
// lbo / sbo: leading / stride byte offsets (see the operand layouts in gemm.cuh).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: bf16 (or, with f16, fp16)
// A and B, fp32 D, M x N tile; a_mn / b_mn: operand stored M- (N-) major
// instead of K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn,
                                                      bool f16 = false) {
    return (1u << 4)                                    // D format: f32
           | (static_cast<uint32_t>(!f16) << 7)         // A format: bf16 (1) or f16 (0)
           | (static_cast<uint32_t>(!f16) << 10)        // B format: bf16 (1) or f16 (0)
           | (static_cast<uint32_t>(a_mn) << 15)        // A major
           | (static_cast<uint32_t>(b_mn) << 16)        // B major
           | (static_cast<uint32_t>(N >> 3) << 17)      // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);     // M / 16
}

}  // namespace tc
}  // namespace vlmce
