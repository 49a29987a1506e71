// flce.cu -- entry point flce_fwd_bwd: fused linear cross-entropy forward +
// backward, and vlmce_gemm_bf16 (the tcgen05 GEMM engine on its own).
//
// Method ("Add Liger Kernel support for Muse Glimmer", Summary and Details):
// the lm_head product h' W^T is never materialised as an [N, V] tensor; the
// softcap multiplier is folded into the hidden states by the caller; grad
// weight is accumulated in fp32.
//
// Schedule (V-chunked, logits recomputed; all products on tcgen05):
//   1. label census                                            (1 CTA)
//   2. S = h' W^T over the whole vocabulary, epilogue = per (row, 256-column
//      tile) statistics: max / first argmax of S, online sum exp(z - m),
//      sum z, z at the label                                   (GEMM, kStats)
//   3. per row: merge the tile statistics in column order -> lse, loss,
//      argmax, gradient scale                                  (1 warp / row)
//   4. for chunk c = 0 .. C of Vc = 8192 vocabulary columns, one grouped
//      GEMM launch each (tiles run in this order):
//        grad_h  (+)= G_{c-1} W_{c-1}   (fp32 [N, H]; the last chunk writes bf16)
//        G_c = scale (softmax - q) (1 - t^2), recomputed from S_c = h' W_c^T
//              and stored in bf16 [N, Vc] (two buffers, alternating)
//        grad_W_{c-1} (+)= G_{c-1}^T h' (fp32, rows of the chunk)
//      so the two products of a chunk share a launch with the next chunk's
//      gradient tile and every launch has one tail.
//   5. reduced loss and accuracy                               (1 CTA)
// Executed tensor work 8 N V H (the logits twice); algorithmic 6 N V H.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "ce_common.cuh"
#include "gemm_launch.h"
#include "host_util.h"
#include "ptx.cuh"
#include "vlmce.h"

namespace vlmce {
namespace flce {
namespace {

using ce::RowPart;

constexpr int kChunk = 8192;  // vocabulary columns per gradient chunk
// Factor of the fp16 gradient tile ((p - q)(1 - t^2) has |.| <= 1; x 2^14 stays
// below the fp16 maximum and keeps small probabilities out of the subnormals).
constexpr float kF16GradMul = 16384.f;
constexpr int64_t kWsHeader = 256;

// ----------------------------------------------------------------- kernels

__global__ void __launch_bounds__(1024) flce_count_kernel(const int64_t *__restrict__ labels,
                                                          int64_t N, int64_t V, int64_t ignore_index,
                                                          int64_t *counts, int *err,
                                                          unsigned int *tile_ctr, int n_ctr) {
    // the GEMM launches' tile counters start from zero in every call
    for (int i = threadIdx.x; i < n_ctr; i += blockDim.x) tile_ctr[i] = 0u;
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
        nv = lane < static_cast<int>(blockDim.x >> 5) ? sv[lane] : 0;
        nb = lane < static_cast<int>(blockDim.x >> 5) ? sb[lane] : 0;
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

// One warp per row: merge the row's tile statistics (fixed order) into lse,
// loss, argmax and the gradient scale of the row.
__global__ void __launch_bounds__(256) flce_merge_kernel(
    const RowPart *__restrict__ part, int64_t part_ld, int ntiles, const int64_t *__restrict__ labels,
    int64_t N, int64_t V, int64_t ignore_index, float eps, float grad_scale, int reduction,
    const int64_t *counts, float *lse, float *row_scale, float *loss, int64_t *argmax,
    float inv_grad_mul, float *out_scale) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row == 0 && lane == 0) {
        // the scale every valid row shares, divided by the gradient tile's factor:
        // the two gradient products multiply their accumulators by it
        float s = grad_scale;
        if (reduction == VLMCE_MEAN) {
            const long long nv = counts[0];
            s = nv > 0 ? grad_scale / static_cast<float>(nv) : 0.f;
        }
        *out_scale = s * inv_grad_mul;
    }
    if (row >= N) return;
    RowPart a = ce::part_identity();
    for (int t = lane; t < ntiles; t += 32) {
        const RowPart p = part[static_cast<int64_t>(t) * part_ld + row];
        ce::part_merge(a, p.mx, p.idx, p.mz, p.s, p.sz, p.zy);
    }
    ce::warp_allreduce(a);
    if (lane == 0) {
        const float l = a.mz + logf(a.s);
        const int64_t y = labels[row];
        const bool ignored = y == ignore_index;
        const bool valid = !ignored && y >= 0 && y < V;
        float sc = 0.f;
        if (valid) {
            sc = grad_scale;
            if (reduction == VLMCE_MEAN) {
                const long long nv = counts[0];
                sc = nv > 0 ? grad_scale / static_cast<float>(nv) : 0.f;
            }
        }
        lse[row] = l;
        row_scale[row] = sc;
        float lo = 0.f;
        if (valid)
            lo = l - fmaf(1.f - eps, a.zy, (eps / static_cast<float>(V)) * a.sz);
        else if (!ignored)
            lo = __int_as_float(0x7fc00000);
        loss[row] = lo;
        argmax[row] = a.idx;
    }
}

__global__ void __launch_bounds__(1024) flce_finalize_kernel(
    const float *__restrict__ loss, const int64_t *__restrict__ argmax,
    const int64_t *__restrict__ labels, int64_t N, int64_t V, int64_t ignore_index, int reduction,
    const int64_t *counts, const int *err, float *out_reduced, int64_t *out_counts) {
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
        acc = lane < static_cast<int>(blockDim.x >> 5) ? sa[lane] : 0.0;
        nc = lane < static_cast<int>(blockDim.x >> 5) ? sc[lane] : 0;
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

// Row-chunked schedule: the scale every valid row's gradient shares, divided
// by the factor of the 16-bit gradient (the products multiply their
// accumulators by it); the same value flce_merge_kernel writes.
__global__ void flce_rows_scale_kernel(const int64_t *counts, float grad_scale, int reduction,
                                       float inv_grad_mul, float *out_scale) {
    float s = grad_scale;
    if (reduction == VLMCE_MEAN) {
        const long long nv = counts[0];
        s = nv > 0 ? grad_scale / static_cast<float>(nv) : 0.f;
    }
    *out_scale = s * inv_grad_mul;
}

// Row-chunked schedule: G[r, j] = 16-bit(S[r, j]) for j < V (bf16, or fp16
// with F16; round to nearest even), four columns per thread, rows strided
// over grid.y.  S rows are 16-byte aligned (lds % 4 == 0) and G rows 8-byte
// aligned (ldg % 4 == 0).
template <bool F16>
__global__ void __launch_bounds__(256) flce_cast16_kernel(const float *__restrict__ S, int64_t lds,
                                                          uint16_t *__restrict__ G, int64_t ldg,
                                                          int64_t rows, int64_t V) {
    const int64_t j = 4 * (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x);
    if (j >= V) return;
    auto pack = [](float a, float b) -> uint32_t {
        uint32_t u;
        if constexpr (F16) {
            const __half2 h = __floats2half2_rn(a, b);
            memcpy(&u, &h, 4);
        } else {
            const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
            memcpy(&u, &h, 4);
        }
        return u;
    };
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const float *src = S + r * lds + j;
        uint16_t *dst = G + r * ldg + j;
        if (j + 4 <= V) {
            const float4 v = *reinterpret_cast<const float4 *>(src);
            *reinterpret_cast<uint2 *>(dst) = make_uint2(pack(v.x, v.y), pack(v.z, v.w));
        } else {
            for (int64_t k = 0; j + k < V; ++k) dst[k] = static_cast<uint16_t>(pack(src[k], 0.f));
        }
    }
}

// ----------------------------------------------------------------- workspace
struct Ws {
    int64_t *counts;
    int *err;
    RowPart *part;  // [ntiles][N]
    float *lse, *row_scale, *loss;
    int64_t *argmax;
    uint16_t *g[2];       // two [N, kChunk] gradient tiles (bf16 or fp16 bits)
    float *out_scale;     // scale of the gradient products' accumulators
    float *gh;            // [N, H] grad_h accumulator
    unsigned int *tile_ctr;  // [nchunks + 2]: one tile counter per GEMM launch
};

int64_t ntiles_of(int64_t V) { return (V + gemm::BN - 1) / gemm::BN; }
// GEMM launches of a vocabulary-chunked call: statistics + one per chunk + one.
int64_t n_gemm_launches(int64_t V) { return (V + kChunk - 1) / kChunk + 2; }

size_t ws_bytes(int64_t N, int64_t H, int64_t V) {
    int64_t b = kWsHeader;
    b += round_up(ntiles_of(V) * N * static_cast<int64_t>(sizeof(RowPart)), 256);
    b += 3 * round_up(4 * N, 256) + round_up(8 * N, 256);
    b += 2 * round_up(2 * N * static_cast<int64_t>(kChunk), 256);
    b += round_up(4 * N * H, 256);
    b += round_up(4 * n_gemm_launches(V), 256);
    return static_cast<size_t>(b);
}

Ws carve(void *ws, int64_t N, int64_t H, int64_t V) {
    unsigned char *p = static_cast<unsigned char *>(ws);
    Ws w;
    w.counts = reinterpret_cast<int64_t *>(p);
    w.err = reinterpret_cast<int *>(p + 64);
    w.out_scale = reinterpret_cast<float *>(p + 128);
    p += kWsHeader;
    w.part = reinterpret_cast<RowPart *>(p);
    p += round_up(ntiles_of(V) * N * static_cast<int64_t>(sizeof(RowPart)), 256);
    w.lse = reinterpret_cast<float *>(p);
    p += round_up(4 * N, 256);
    w.row_scale = reinterpret_cast<float *>(p);
    p += round_up(4 * N, 256);
    w.loss = reinterpret_cast<float *>(p);
    p += round_up(4 * N, 256);
    w.argmax = reinterpret_cast<int64_t *>(p);
    p += round_up(8 * N, 256);
    for (int i = 0; i < 2; ++i) {
        w.g[i] = reinterpret_cast<uint16_t *>(p);
        p += round_up(2 * N * static_cast<int64_t>(kChunk), 256);
    }
    w.gh = reinterpret_cast<float *>(p);
    p += round_up(4 * N * H, 256);
    w.tile_ctr = reinterpret_cast<unsigned int *>(p);
    return w;
}

// With no rows, d loss / dW is zero: an overwritten grad_weight is cleared
// (stream-ordered memset), an accumulated one is left as it is.
vlmce_status clear_grad_weight_if_empty(int64_t N, int64_t H, int64_t V, float *grad_weight,
                                        int32_t accumulate_grad_weight, cudaStream_t cs) {
    if (N != 0 || !grad_weight || accumulate_grad_weight) return VLMCE_OK;
    if (V > (INT64_MAX / 4) / H) return VLMCE_ERR_TOO_LARGE;
    return launch_status(cudaMemsetAsync(grad_weight, 0, static_cast<size_t>(4 * V * H), cs),
                         "cudaMemsetAsync(grad_weight)");
}

// Sizes for which the workspace arithmetic stays in range.
bool sizes_ok(int64_t N, int64_t H, int64_t V) {
    return N >= 0 && H >= 1 && V >= 1 && N <= INT_MAX && H <= INT_MAX && V <= INT_MAX;
}

// Argument checks of both schedules; ws_needed: the schedule's workspace bytes.
vlmce_status check_args(const void *hidden, int32_t dtype, int64_t hidden_stride, const void *weight,
                        int64_t weight_stride, const int64_t *labels, int64_t N, int64_t H,
                        int64_t V, float label_smoothing, float softcap, int32_t reduction,
                        float grad_scale, const float *out_loss, const int64_t *out_argmax,
                        const float *out_reduced, const int64_t *out_counts,
                        const void *grad_hidden, const float *grad_weight, const void *workspace,
                        size_t workspace_bytes_given, size_t ws_needed) {
    if (dtype != VLMCE_BF16 && dtype != VLMCE_F16) return VLMCE_ERR_UNSUPPORTED_DTYPE;
    if (N < 0 || H < 1 || V < 1) return VLMCE_ERR_INVALID_ARG;
    if (N > INT_MAX || H > INT_MAX || V > INT_MAX) return VLMCE_ERR_TOO_LARGE;
    if (hidden_stride < H || weight_stride < H) return VLMCE_ERR_INVALID_ARG;
    if (N > 0 && (!hidden || !weight || !labels || !grad_hidden || !grad_weight))
        return VLMCE_ERR_INVALID_ARG;
    if (!(label_smoothing >= 0.f && label_smoothing <= 1.f)) return VLMCE_ERR_INVALID_ARG;
    if (!(softcap >= 0.f) || !std::isfinite(softcap)) return VLMCE_ERR_INVALID_ARG;
    if (!std::isfinite(grad_scale)) return VLMCE_ERR_INVALID_ARG;
    if (reduction != VLMCE_MEAN && reduction != VLMCE_SUM) return VLMCE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes_given < ws_needed) return VLMCE_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 256)) return VLMCE_ERR_MISALIGNED;
    if (N > 0 && (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(grad_hidden, 16) ||
                  !aligned(grad_weight, 16) || !aligned(labels, 8)))
        return VLMCE_ERR_MISALIGNED;
    if (H % 8 || hidden_stride % 8 || weight_stride % 8) return VLMCE_ERR_MISALIGNED;
    if ((out_loss && !aligned(out_loss, 4)) || (out_argmax && !aligned(out_argmax, 8)) ||
        (out_reduced && !aligned(out_reduced, 4)) || (out_counts && !aligned(out_counts, 8)))
        return VLMCE_ERR_MISALIGNED;
    return VLMCE_OK;
}

// Row-chunked schedule workspace: counts / error word / product scale, the
// per-token losses and argmax of all N rows, the fp32 logits of one chunk of
// rows (row stride lds = V rounded up to 4), its 16-bit gradient (row stride
// ldg = V rounded up to 8) and the workspace of the CE call on the chunk.
struct RowsWs {
    int64_t *counts;
    int *err;
    float *out_scale;
    float *loss;
    int64_t *argmax;
    float *S;
    uint16_t *G;
    void *ce;
    size_t ce_bytes;
    int64_t nc, lds, ldg;
};

int64_t rows_chunk(int64_t N, int64_t chunk_rows) { return chunk_rows < N ? chunk_rows : N; }

size_t rows_ws_bytes(int64_t N, int64_t V, int64_t chunk_rows) {
    const int64_t nc = rows_chunk(N, chunk_rows);
    const int64_t lds = round_up(V, 4), ldg = round_up(V, 8);
    int64_t b = kWsHeader + round_up(4 * N, 256) + round_up(8 * N, 256);
    b += round_up(4 * nc * lds, 256) + round_up(2 * nc * ldg, 256);
    b += static_cast<int64_t>(vlmce_ce_workspace_bytes(nc, V, VLMCE_F32));
    return static_cast<size_t>(b);
}

RowsWs rows_carve(void *ws, int64_t N, int64_t V, int64_t chunk_rows) {
    unsigned char *p = static_cast<unsigned char *>(ws);
    RowsWs w;
    w.nc = rows_chunk(N, chunk_rows);
    w.lds = round_up(V, 4);
    w.ldg = round_up(V, 8);
    w.counts = reinterpret_cast<int64_t *>(p);
    w.err = reinterpret_cast<int *>(p + 64);
    w.out_scale = reinterpret_cast<float *>(p + 128);
    p += kWsHeader;
    w.loss = reinterpret_cast<float *>(p);
    p += round_up(4 * N, 256);
    w.argmax = reinterpret_cast<int64_t *>(p);
    p += round_up(8 * N, 256);
    w.S = reinterpret_cast<float *>(p);
    p += round_up(4 * w.nc * w.lds, 256);
    w.G = reinterpret_cast<uint16_t *>(p);
    p += round_up(2 * w.nc * w.ldg, 256);
    w.ce = p;
    w.ce_bytes = vlmce_ce_workspace_bytes(w.nc, V, VLMCE_F32);
    return w;
}

thread_local cudaEvent_t t_prof_begin = nullptr;
thread_local cudaEvent_t t_prof_end = nullptr;

}  // namespace
}  // namespace flce
}  // namespace vlmce

using namespace vlmce;
using namespace vlmce::flce;

extern "C" void vlmce_flce_profile_events(void *ev_begin, void *ev_end) {
    t_prof_begin = static_cast<cudaEvent_t>(ev_begin);
    t_prof_end = static_cast<cudaEvent_t>(ev_end);
}

extern "C" size_t vlmce_flce_workspace_bytes(int64_t N, int64_t H, int64_t V) {
    if (N < 0 || H < 1 || V < 1) return 0;
    return ws_bytes(N, H, V);
}

extern "C" vlmce_status vlmce_gemm(const void *A, int32_t a_mn, const void *B, int32_t b_mn,
                                   float *C, int64_t M, int64_t N, int64_t K, int64_t lda,
                                   int64_t ldb, int64_t ldc, int32_t accumulate, int32_t dtype,
                                   vlmce_stream_t stream) {
    if (dtype != VLMCE_BF16 && dtype != VLMCE_F16) return VLMCE_ERR_UNSUPPORTED_DTYPE;
    const bool f16 = dtype == VLMCE_F16;
    if (!A || !B || !C || M < 1 || N < 1 || K < 1) return VLMCE_ERR_INVALID_ARG;
    if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return VLMCE_ERR_TOO_LARGE;
    if (lda < (a_mn ? M : K) || ldb < (b_mn ? N : K) || ldc < N) return VLMCE_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || lda % 8 || ldb % 8 || ldc % 4)
        return VLMCE_ERR_MISALIGNED;
    DeviceInfo dev;
    vlmce_status st = current_device(&dev);
    if (st != VLMCE_OK) return st;
    gemm::Maps maps;
    if (!gemm::make_operand_map(&maps.a[0], A, a_mn != 0, M, K, lda, f16) ||
        !gemm::make_operand_map(&maps.b[0], B, b_mn != 0, N, K, ldb, f16)) {
        record_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
        return VLMCE_ERR_CUDA;
    }
    gemm::Params g = {};
    g.nprob = 1;
    g.f16 = f16 ? 1 : 0;
    gemm::Problem &p = g.p[0];
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.mode = accumulate ? gemm::kAccF32 : gemm::kStoreF32;
    p.a_mn = a_mn != 0;
    p.b_mn = b_mn != 0;
    p.C = C;
    p.ldc = ldc;
    g.err = nullptr;  // no device error word: a wait that gives up only ends the kernel
    return launch_status(gemm::launch_group(maps, g, reinterpret_cast<cudaStream_t>(stream)),
                         "vlmce_gemm_kernel");
}

extern "C" vlmce_status vlmce_gemm_bf16(const void *A, int32_t a_mn, const void *B, int32_t b_mn,
                                        float *C, int64_t M, int64_t N, int64_t K, int64_t lda,
                                        int64_t ldb, int64_t ldc, int32_t accumulate,
                                        vlmce_stream_t stream) {
    return vlmce_gemm(A, a_mn, B, b_mn, C, M, N, K, lda, ldb, ldc, accumulate, VLMCE_BF16, stream);
}

extern "C" vlmce_status flce_fwd_bwd_ex(const void *hidden, int32_t dtype, int64_t hidden_stride,
                                     const void *weight,
                                     int64_t weight_stride, const int64_t *labels, int64_t N,
                                     int64_t H, int64_t V, int64_t ignore_index,
                                     float label_smoothing, float softcap, int32_t reduction,
                                     float grad_scale, float *out_loss, int64_t *out_argmax,
                                     float *out_reduced, int64_t *out_counts, void *grad_hidden,
                                     float *grad_weight, int32_t accumulate_grad_weight,
                                     void *workspace, size_t workspace_bytes_given,
                                     vlmce_stream_t stream) {
    // ---- host-side argument checks; nothing is enqueued on failure
    vlmce_status st = check_args(hidden, dtype, hidden_stride, weight, weight_stride, labels, N, H, V,
                                 label_smoothing, softcap, reduction, grad_scale, out_loss,
                                 out_argmax, out_reduced, out_counts, grad_hidden, grad_weight,
                                 workspace, workspace_bytes_given,
                                 sizes_ok(N, H, V) ? ws_bytes(N, H, V) : 0);
    if (st != VLMCE_OK) return st;
    const bool f16 = dtype == VLMCE_F16;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != VLMCE_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    Ws w = carve(workspace, N, H, V);
    float *loss = out_loss ? out_loss : w.loss;
    int64_t *amax = out_argmax ? out_argmax : w.argmax;

    flce_count_kernel<<<1, 1024, 0, cs>>>(labels, N, V, ignore_index, w.counts, w.err, w.tile_ctr,
                                          static_cast<int>(n_gemm_launches(V)));
    st = launch_status(cudaSuccess, "flce_count_kernel");
    if (st != VLMCE_OK) return st;
    st = clear_grad_weight_if_empty(N, H, V, grad_weight, accumulate_grad_weight, cs);
    if (st != VLMCE_OK) return st;

    if (N > 0) {
        const float T = softcap;
        gemm::Params base = {};
        base.labels = labels;
        base.ignore_index = ignore_index;
        base.V = static_cast<int>(V);
        base.eps = label_smoothing;
        base.T = T;
        base.k2 = T > 0.f ? -2.f * ce::kLog2e / T : 0.f;
        base.lse = w.lse;
        base.row_scale = w.row_scale;
        base.err = w.err;
        base.f16 = f16 ? 1 : 0;
        // fp16 keeps the scale-free gradient tile (|.| <= 1) away from underflow
        base.grad_mul = f16 ? kF16GradMul : 1.f;
        base.out_scale = w.out_scale;

        cudaEvent_t eb = t_prof_begin, ee = t_prof_end;
        t_prof_begin = t_prof_end = nullptr;
        if (eb && (st = launch_status(cudaEventRecord(eb, cs), "cudaEventRecord")) != VLMCE_OK)
            return st;
        auto map_fail = [] {
            record_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
            return VLMCE_ERR_CUDA;
        };

        // ---- pass 1: statistics of S = h' W^T over the whole vocabulary
        {
            gemm::Maps maps;
            if (!gemm::make_operand_map(&maps.a[0], hidden, false, N, H, hidden_stride, f16) ||
                !gemm::make_operand_map(&maps.b[0], weight, false, V, H, weight_stride, f16))
                return map_fail();
            gemm::Params g = base;
            g.nprob = 1;
            gemm::Problem &p = g.p[0];
            p.M = static_cast<int>(N);
            p.N = static_cast<int>(V);
            p.K = static_cast<int>(H);
            p.mode = gemm::kStats;
            p.col0 = 0;
            p.part = w.part;
            p.part_ld = N;
            g.tile_ctr = w.tile_ctr;
            st = launch_status(gemm::launch_group(maps, g, cs), "vlmce_gemm_kernel(stats)");
            if (st != VLMCE_OK) return st;
        }

        flce_merge_kernel<<<static_cast<unsigned>((N + 7) / 8), 256, 0, cs>>>(
            w.part, N, static_cast<int>(ntiles_of(V)), labels, N, V, ignore_index, label_smoothing,
            grad_scale, reduction, w.counts, w.lse, w.row_scale, loss, amax,
            1.f / (f16 ? kF16GradMul : 1.f), w.out_scale);
        st = launch_status(cudaSuccess, "flce_merge_kernel");
        if (st != VLMCE_OK) return st;

        // ---- pass 2: launch c = the products of chunk c - 1 and the gradient tile of chunk c,
        // in the order grad_h, gradient tile, grad_W: the persistent grid runs the
        // tiles in problem order, and grad_W's (the shortest, K = N) end the launch
        const int64_t nchunks = (V + kChunk - 1) / kChunk;
        for (int64_t c = 0; c <= nchunks; ++c) {
            gemm::Maps maps;
            gemm::Params g = base;
            int n = 0;
            const int64_t cp = c - 1;  // the chunk whose products this launch computes
            const int64_t pv0 = cp * kChunk;
            const int64_t pvc = c >= 1 ? ((V - pv0) < kChunk ? (V - pv0) : kChunk) : 0;
            const uint16_t *gc = c >= 1 ? w.g[cp & 1] : nullptr;
            if (c >= 1) {
                const uint16_t *wc = static_cast<const uint16_t *>(weight) + pv0 * weight_stride;
                // grad_h (+)= G_c W_c: A = G_c K-major [N, Vc], B = W_c N(=H)-major
                if (!gemm::make_operand_map(&maps.a[n], gc, false, N, pvc, kChunk, f16) ||
                    !gemm::make_operand_map(&maps.b[n], wc, true, H, pvc, weight_stride, f16))
                    return map_fail();
                gemm::Problem &ph = g.p[n++];
                ph.M = static_cast<int>(N);
                ph.N = static_cast<int>(H);
                ph.K = static_cast<int>(pvc);
                ph.mode = nchunks == 1       ? gemm::kStoreBF16
                          : cp == 0           ? gemm::kStoreF32
                          : cp == nchunks - 1 ? gemm::kAccToBF16
                                              : gemm::kAccF32;
                ph.a_mn = 0;
                ph.b_mn = 1;
                ph.C = w.gh;
                ph.ldc = H;
                ph.C16 = static_cast<uint16_t *>(grad_hidden);
                ph.ldc16 = hidden_stride;
            }
            if (c < nchunks) {
                const int64_t v0 = c * kChunk;
                const int64_t vc = (V - v0) < kChunk ? (V - v0) : kChunk;
                const uint16_t *wc = static_cast<const uint16_t *>(weight) + v0 * weight_stride;
                // G_c = scale (softmax - q) (1 - t^2) from the recomputed S_c = h' W_c^T
                if (!gemm::make_operand_map(&maps.a[n], hidden, false, N, H, hidden_stride, f16) ||
                    !gemm::make_operand_map(&maps.b[n], wc, false, vc, H, weight_stride, f16))
                    return map_fail();
                gemm::Problem &pg = g.p[n++];
                pg.M = static_cast<int>(N);
                pg.N = static_cast<int>(vc);
                pg.K = static_cast<int>(H);
                pg.mode = gemm::kGrad;
                pg.col0 = static_cast<int>(v0);
                pg.C16 = w.g[c & 1];
                pg.ldc16 = kChunk;
            }
            if (c >= 1) {
                // grad_W_c (+)= G_c^T h': A = G_c^T M(=Vc)-major, B = h' N(=H)-major
                if (!gemm::make_operand_map(&maps.a[n], gc, true, pvc, N, kChunk, f16) ||
                    !gemm::make_operand_map(&maps.b[n], hidden, true, H, N, hidden_stride, f16))
                    return map_fail();
                gemm::Problem &pw = g.p[n++];
                pw.M = static_cast<int>(pvc);
                pw.N = static_cast<int>(H);
                pw.K = static_cast<int>(N);
                pw.mode = accumulate_grad_weight ? gemm::kAccF32 : gemm::kStoreF32;
                pw.a_mn = 1;
                pw.b_mn = 1;
                pw.C = grad_weight + pv0 * H;
                pw.ldc = H;
            }
            g.nprob = n;
            g.tile_ctr = w.tile_ctr + 1 + c;
            st = launch_status(gemm::launch_group(maps, g, cs), "vlmce_gemm_kernel(chunk)");
            if (st != VLMCE_OK) return st;
        }
        if (ee && (st = launch_status(cudaEventRecord(ee, cs), "cudaEventRecord")) != VLMCE_OK)
            return st;
    }

    flce_finalize_kernel<<<1, 1024, 0, cs>>>(loss, amax, labels, N, V, ignore_index, reduction,
                                             w.counts, w.err, out_reduced, out_counts);
    return launch_status(cudaSuccess, "flce_finalize_kernel");
}

extern "C" vlmce_status flce_fwd_bwd(const void *hidden, int64_t hidden_stride, const void *weight,
                                     int64_t weight_stride, const int64_t *labels, int64_t N,
                                     int64_t H, int64_t V, int64_t ignore_index,
                                     float label_smoothing, float softcap, int32_t reduction,
                                     float grad_scale, float *out_loss, int64_t *out_argmax,
                                     float *out_reduced, int64_t *out_counts, void *grad_hidden,
                                     float *grad_weight, int32_t accumulate_grad_weight,
                                     void *workspace, size_t workspace_bytes_given,
                                     vlmce_stream_t stream) {
    return flce_fwd_bwd_ex(hidden, VLMCE_BF16, hidden_stride, weight, weight_stride, labels, N, H,
                           V, ignore_index, label_smoothing, softcap, reduction, grad_scale,
                           out_loss, out_argmax, out_reduced, out_counts, grad_hidden,
                           grad_weight, accumulate_grad_weight, workspace, workspace_bytes_given,
                           stream);
}

extern "C" size_t vlmce_flce_rows_workspace_bytes(int64_t N, int64_t H, int64_t V,
                                                  int64_t chunk_rows) {
    if (!sizes_ok(N, H, V) || chunk_rows < 1) return 0;
    return rows_ws_bytes(N, V, chunk_rows);
}

// The row-chunked schedule (the comparison point of the vocabulary-chunked
// one above): for each block of chunk_rows rows,
//   S_k = h'_k W^T                  fp32 [nc, V] in the workspace   (GEMM)
//   ce_fwd_bwd_ex on S_k: losses, argmax, and in place grad_mul (p - q)(1 - t^2)
//                                   for the valid rows, 0 for the others
//   G_k = 16-bit(S_k)                                              (cast)
//   grad_h_k = G_k W, grad_W (+)= G_k^T h'_k, both times the shared scale
//                                   (one grouped GEMM launch)
// Executed tensor work 6 N V H (no recompute), at the price of the logits of a
// chunk in HBM and of one read-modify-write of the fp32 grad_W per chunk after
// the first.
extern "C" vlmce_status flce_fwd_bwd_rows(const void *hidden, int32_t dtype, int64_t hidden_stride,
                                          const void *weight, int64_t weight_stride,
                                          const int64_t *labels, int64_t N, int64_t H, int64_t V,
                                          int64_t ignore_index, float label_smoothing,
                                          float softcap, int32_t reduction, float grad_scale,
                                          float *out_loss, int64_t *out_argmax,
                                          float *out_reduced, int64_t *out_counts,
                                          void *grad_hidden, float *grad_weight,
                                          int32_t accumulate_grad_weight, int64_t chunk_rows,
                                          void *workspace, size_t workspace_bytes_given,
                                          vlmce_stream_t stream) {
    // ---- host-side argument checks; nothing is enqueued on failure
    if (chunk_rows < 1) return VLMCE_ERR_INVALID_ARG;
    vlmce_status st = check_args(hidden, dtype, hidden_stride, weight, weight_stride, labels, N, H, V,
                                 label_smoothing, softcap, reduction, grad_scale, out_loss,
                                 out_argmax, out_reduced, out_counts, grad_hidden, grad_weight,
                                 workspace, workspace_bytes_given,
                                 sizes_ok(N, H, V) ? rows_ws_bytes(N, V, chunk_rows) : 0);
    if (st != VLMCE_OK) return st;
    if (V > vlmce_ce_max_vocab(VLMCE_F32)) return VLMCE_ERR_TOO_LARGE;
    const bool f16 = dtype == VLMCE_F16;

    DeviceInfo dev;
    st = current_device(&dev);
    if (st != VLMCE_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    RowsWs w = rows_carve(workspace, N, V, chunk_rows);
    float *loss = out_loss ? out_loss : w.loss;
    int64_t *amax = out_argmax ? out_argmax : w.argmax;
    const float gmul = f16 ? kF16GradMul : 1.f;

    flce_count_kernel<<<1, 1024, 0, cs>>>(labels, N, V, ignore_index, w.counts, w.err, nullptr, 0);
    st = launch_status(cudaSuccess, "flce_count_kernel");
    if (st != VLMCE_OK) return st;
    st = clear_grad_weight_if_empty(N, H, V, grad_weight, accumulate_grad_weight, cs);
    if (st != VLMCE_OK) return st;

    if (N > 0) {
        flce_rows_scale_kernel<<<1, 1, 0, cs>>>(w.counts, grad_scale, reduction, 1.f / gmul,
                                                w.out_scale);
        if ((st = launch_status(cudaSuccess, "flce_rows_scale_kernel")) != VLMCE_OK) return st;
        cudaEvent_t eb = t_prof_begin, ee = t_prof_end;
        t_prof_begin = t_prof_end = nullptr;
        if (eb && (st = launch_status(cudaEventRecord(eb, cs), "cudaEventRecord")) != VLMCE_OK)
            return st;
        auto map_fail = [] {
            record_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
            return VLMCE_ERR_CUDA;
        };
        const int64_t gx = (round_up(V, 4) / 4 + 255) / 256;
        if (gx > INT_MAX) return VLMCE_ERR_TOO_LARGE;
        for (int64_t n0 = 0; n0 < N; n0 += w.nc) {
            const int64_t rows = (N - n0) < w.nc ? (N - n0) : w.nc;
            const uint16_t *hk = static_cast<const uint16_t *>(hidden) + n0 * hidden_stride;

            // S_k = h'_k W^T, fp32
            {
                gemm::Maps maps;
                if (!gemm::make_operand_map(&maps.a[0], hk, false, rows, H, hidden_stride, f16) ||
                    !gemm::make_operand_map(&maps.b[0], weight, false, V, H, weight_stride, f16))
                    return map_fail();
                gemm::Params g = {};
                g.nprob = 1;
                g.f16 = f16 ? 1 : 0;
                g.err = w.err;
                gemm::Problem &p = g.p[0];
                p.M = static_cast<int>(rows);
                p.N = static_cast<int>(V);
                p.K = static_cast<int>(H);
                p.mode = gemm::kStoreF32;
                p.C = w.S;
                p.ldc = w.lds;
                st = launch_status(gemm::launch_group(maps, g, cs), "vlmce_gemm_kernel(logits)");
                if (st != VLMCE_OK) return st;
            }

            // losses, argmax and grad_mul (p - q)(1 - t^2), in place
            st = ce_fwd_bwd_ex(w.S, VLMCE_F32, labels + n0, rows, V, w.lds, ignore_index,
                               label_smoothing, softcap, VLMCE_SUM, gmul, nullptr, 1, loss + n0,
                               amax + n0, nullptr, nullptr, w.ce, w.ce_bytes, stream);
            if (st != VLMCE_OK) return st;

            // G_k = 16-bit(S_k)
            {
                const int64_t gy = rows < 65535 ? rows : 65535;
                const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
                if (f16)
                    flce_cast16_kernel<true><<<grid, 256, 0, cs>>>(w.S, w.lds, w.G, w.ldg, rows, V);
                else
                    flce_cast16_kernel<false><<<grid, 256, 0, cs>>>(w.S, w.lds, w.G, w.ldg, rows, V);
                if ((st = launch_status(cudaSuccess, "flce_cast16_kernel")) != VLMCE_OK) return st;
            }

            // grad_h_k = G_k W and grad_W (+)= G_k^T h'_k, scaled by *out_scale
            {
                gemm::Maps maps;
                gemm::Params g = {};
                g.f16 = f16 ? 1 : 0;
                g.err = w.err;
                g.out_scale = w.out_scale;
                // grad_h_k: A = G_k K-major [rows, V], B = W N(=H)-major
                if (!gemm::make_operand_map(&maps.a[0], w.G, false, rows, V, w.ldg, f16) ||
                    !gemm::make_operand_map(&maps.b[0], weight, true, H, V, weight_stride, f16))
                    return map_fail();
                gemm::Problem &ph = g.p[0];
                ph.M = static_cast<int>(rows);
                ph.N = static_cast<int>(H);
                ph.K = static_cast<int>(V);
                ph.mode = gemm::kStoreBF16;
                ph.a_mn = 0;
                ph.b_mn = 1;
                ph.C16 = static_cast<uint16_t *>(grad_hidden) + n0 * hidden_stride;
                ph.ldc16 = hidden_stride;
                // grad_W: A = G_k^T M(=V)-major, B = h'_k N(=H)-major
                if (!gemm::make_operand_map(&maps.a[1], w.G, true, V, rows, w.ldg, f16) ||
                    !gemm::make_operand_map(&maps.b[1], hk, true, H, rows, hidden_stride, f16))
                    return map_fail();
                gemm::Problem &pw = g.p[1];
                pw.M = static_cast<int>(V);
                pw.N = static_cast<int>(H);
                pw.K = static_cast<int>(rows);
                pw.mode = (n0 == 0 && !accumulate_grad_weight) ? gemm::kStoreF32 : gemm::kAccF32;
                pw.a_mn = 1;
                pw.b_mn = 1;
                pw.C = grad_weight;
                pw.ldc = H;
                g.nprob = 2;
                st = launch_status(gemm::launch_group(maps, g, cs), "vlmce_gemm_kernel(products)");
                if (st != VLMCE_OK) return st;
            }
        }
        if (ee && (st = launch_status(cudaEventRecord(ee, cs), "cudaEventRecord")) != VLMCE_OK)
            return st;
    }

    flce_finalize_kernel<<<1, 1024, 0, cs>>>(loss, amax, labels, N, V, ignore_index, reduction,
                                             w.counts, w.err, out_reduced, out_counts);
    return launch_status(cudaSuccess, "flce_finalize_kernel");
}
