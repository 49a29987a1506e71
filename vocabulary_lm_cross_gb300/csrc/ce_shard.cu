// ce_shard.cu -- the vocabulary-sharded cross-entropy: the kernels each rank
// of a tensor-parallel group runs on its shard of the logits (columns
// [vocab_start, vocab_start + V_local) of every row), with the exchange of the
// per-row statistics left to the caller.
//
// Method ("Add Megatron-LM cross-entropy integration", Summary; "Add opt-in
// Liger vocab-parallel cross entropy through ops/loss", What does this PR do):
//   1. ce_shard_stats   -- per row of the shard: largest raw logit and its
//                          smallest global column, online sum of exp(z - m),
//                          sum of z, z at the label when the shard holds it;
//                          the row kernel's first pass, one CTA per row (the
//                          argmax column resolved once, after the merge).
//   2. (caller)         -- gather every shard's statistics.
//   3. ce_merge_stats   -- merge k shards' statistics in shard order (the same
//                          operator the kernels use between warps), so every
//                          rank obtains bit-identical global statistics.
//   4. ce_shard_fwd_bwd -- label census; per row the loss from the global
//                          statistics and the gradient of the shard's columns
//                          written in place (the row kernel's second pass with
//                          the global lse and the global V); reduced loss.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "ce_census.cuh"
#include "ce_rows.cuh"
#include "host_util.h"
#include "ptx.cuh"
#include "vlmce.h"

namespace vlmce {
namespace ce {
namespace shard {
namespace {

static_assert(sizeof(RowPart) == sizeof(vlmce_row_stats), "row statistics layout");

struct ShardParams {
    unsigned char *logits;
    const int64_t *labels;
    int V_local;
    int64_t vocab_start;
    int V;                  // global vocabulary
    int64_t stride_bytes;
    int64_t ignore_index;
    float eps, softcap, grad_scale;
    int reduction;
    RowPart *stats;         // stats kernel: out [N]; grad kernel: k gathered records [k][N]
    int k;                  // grad kernel: records per row, merged in order (1: already merged)
    int64_t N;
    float *loss;
    int64_t *argmax;
    const int64_t *counts;
};

// Row geometry in 16-byte granules (as the row kernel): whole granules are
// [gs, ge); granule 0 is partial when the row starts inside a granule, G - 1
// when it ends inside one.
struct Geo {
    unsigned char *gbase;  // the row's first 16-byte granule
    int lead, G, gs, ge, tail_tid;
    bool head;
    __device__ __forceinline__ const uint4 *row() const {
        return reinterpret_cast<const uint4 *>(gbase);
    }
};
__device__ __forceinline__ uintptr_t row_addr(const ShardParams &p) {
    return reinterpret_cast<uintptr_t>(p.logits) + static_cast<int64_t>(blockIdx.x) * p.stride_bytes;
}
template <bool BF16, int THREADS>
__device__ __forceinline__ Geo geometry(const ShardParams &p) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    constexpr int ELT = Elem<BF16>::kBytes;
    Geo g;
    const uintptr_t a0 = row_addr(p);
    g.gbase = reinterpret_cast<unsigned char *>(a0 & ~static_cast<uintptr_t>(15));
    g.lead = static_cast<int>((a0 & 15) / ELT);
    g.G = (g.lead + p.V_local + EPG - 1) / EPG;
    g.gs = g.lead > 0 ? 1 : 0;
    g.ge = ((g.lead + p.V_local) % EPG != 0) ? g.G - 1 : g.G;
    g.head = g.gs == 1;
    const bool tail = g.ge == g.G - 1 && g.G - 1 >= g.gs;
    g.tail_tid = tail ? (g.G - 1 - g.gs) % THREADS : -1;
    return g;
}

template <bool BF16>
__device__ __forceinline__ float load_x(uintptr_t a0, int64_t col) {
    const unsigned char *py = reinterpret_cast<const unsigned char *>(a0) + Elem<BF16>::kBytes * col;
    if constexpr (BF16)
        return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(py)) << 16);
    else
        return *reinterpret_cast<const float *>(py);
}

// CTAs per SM of the shard kernels: as the row kernel's, but four 256-thread
// softcap CTAs (the shard bookkeeping needs more than 48 registers there).
constexpr int min_blocks(int threads, bool softcap) {
    return (softcap && threads == rows::kShortThreads) ? 4 : rows::min_blocks(threads, softcap);
}

template <bool BF16, bool SOFTCAP, int THREADS>
__global__ void __launch_bounds__(THREADS, min_blocks(THREADS, SOFTCAP))
    ce_shard_stats_kernel(const ShardParams p) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    constexpr int kWarps = THREADS / 32;
    // a dependent launch that follows (the merge or a census, each waiting
    // for this grid before it reads anything) may be scheduled once every CTA
    // has started
    ptx::griddep_launch_dependents();
    __shared__ RowPart wpart[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const Geo g = geometry<BF16, THREADS>(p);
    const float T = p.softcap;
    const rows::CapK k = rows::cap_k<SOFTCAP>(T);
    bool poly_ok = true;
    rows::Acc a;
    rows::acc_init(a);
    if (g.head && tid == 0)
        rows::fold_partial<BF16, SOFTCAP, true>(a, rows::ld_v4(g.row()), -g.lead, p.V_local, k);
    int gl = g.gs + tid;
    for (; gl + THREADS < g.ge; gl += 2 * THREADS) {  // two loads in flight, column order kept
        const uint4 w0 = rows::ld_v4(g.row() + gl), w1 = rows::ld_v4(g.row() + gl + THREADS);
        if (gl + 3 * THREADS < g.ge) {  // the next iteration's pair, into L2 (as the row kernel)
            ptx::prefetch_l2(g.row() + gl + 2 * THREADS);
            ptx::prefetch_l2(g.row() + gl + 3 * THREADS);
        }
        rows::fold_full<BF16, SOFTCAP, true, true>(a, w0, gl * EPG - g.lead, p.V_local, k, poly_ok);
        rows::fold_full<BF16, SOFTCAP, true, true>(a, w1, (gl + THREADS) * EPG - g.lead, p.V_local,
                                                   k, poly_ok);
    }
    for (; gl < g.ge; gl += THREADS)
        rows::fold_full<BF16, SOFTCAP, true, true>(a, rows::ld_v4(g.row() + gl), gl * EPG - g.lead,
                                                   p.V_local, k, poly_ok);
    if (tid == g.tail_tid)
        rows::fold_partial<BF16, SOFTCAP, true>(a, rows::ld_v4(g.row() + (g.G - 1)),
                                                (g.G - 1) * EPG - g.lead, p.V_local, k);
    RowPart pt = rows::acc_part<SOFTCAP>(a, T);
    warp_allreduce(pt);
    if (lane == 0) wpart[warp] = pt;
    __syncthreads();
    if (warp == 0) {
        RowPart q = lane < kWarps ? wpart[lane] : part_identity();
        warp_allreduce(q);
        if (lane == 0) {
            // the granule of the shard's first maximum (pass 1 records only
            // the granule), whose column is resolved here; its load overlaps
            // the label's
            const uint4 wm = q.idx != INT_MAX
                                 ? rows::ld_v4(g.row() + (q.idx + g.lead) / EPG)
                                 : make_uint4(0u, 0u, 0u, 0u);
            const int64_t yl = p.labels[blockIdx.x] - p.vocab_start;
            q.zy = 0.f;
            if (yl >= 0 && yl < p.V_local)
                q.zy = rows::z_of<SOFTCAP>(load_x<BF16>(row_addr(p), yl), k);
            if (q.idx != INT_MAX) q.idx = rows::first_max_col<BF16>(wm, q.mx, q.idx, p.V_local);
            q.idx = q.idx == INT_MAX ? INT_MAX : static_cast<int>(q.idx + p.vocab_start);
            q.pad0 = q.pad1 = 0.f;
            p.stats[blockIdx.x] = q;
        }
    }
}

// One thread per row: out[r] = merge of shards[0][r], ..., shards[k-1][r]
// in that order (out may be shards[0]).
__global__ void __launch_bounds__(256) ce_merge_stats_kernel(const RowPart *shards, int k,
                                                            int64_t N, RowPart *out) {
    ptx::griddep_wait();  // the gathered records (launched dependent on their producer)
    const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r >= N) return;
    RowPart a = shards[r];
    for (int i = 1; i < k; ++i) {
        const RowPart b = shards[static_cast<int64_t>(i) * N + r];
        part_merge(a, b.mx, b.idx, b.mz, b.s, b.sz, b.zy);
    }
    out[r] = a;
}

// The gradient kernel keeps two granules in flight per thread; without a
// softcap its 256-thread CTAs run five per SM (48 registers) to hold them;
// its 128-thread CTAs keep sixteen per SM (all 2432 rows of a wave at once).
constexpr int grad_min_blocks(int threads, bool softcap) {
    if (!softcap && threads == rows::kShortThreads) return 5;
    if (!softcap && threads == rows::kTinyThreads) return 16;
    return min_blocks(threads, softcap);
}

template <bool BF16, bool SOFTCAP, int THREADS>
__global__ void __launch_bounds__(THREADS, grad_min_blocks(THREADS, SOFTCAP))
    ce_shard_grad_kernel(const ShardParams p) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    // the finalize kernel (dependent on this grid, waiting for it before it
    // reads anything) may be scheduled once every CTA has started
    ptx::griddep_launch_dependents();
    const int tid = threadIdx.x;
    const int64_t r = blockIdx.x;
    const Geo g = geometry<BF16, THREADS>(p);
    const float T = p.softcap;
    const rows::CapK k = rows::cap_k<SOFTCAP>(T);
    // the row's statistics over the whole vocabulary: its k gathered records
    // merged in shard order (the operator and order of ce_merge_stats) by the
    // first warp -- lane i loads record i, so the k loads are in flight
    // together -- and shared with the CTA
    __shared__ RowPart srow;
    if (tid < 32) {
        RowPart st = part_identity();
        for (int base = 0; base < p.k; base += 32) {
            RowPart mine = part_identity();
            if (base + tid < p.k) mine = p.stats[static_cast<int64_t>(base + tid) * p.N + r];
            const int n = p.k - base < 32 ? p.k - base : 32;
            for (int i = 0; i < n; ++i) {
                const float mx = __shfl_sync(0xffffffffu, mine.mx, i);
                const int idx = __shfl_sync(0xffffffffu, mine.idx, i);
                const float mz = __shfl_sync(0xffffffffu, mine.mz, i);
                const float s = __shfl_sync(0xffffffffu, mine.s, i);
                const float sz = __shfl_sync(0xffffffffu, mine.sz, i);
                const float zy = __shfl_sync(0xffffffffu, mine.zy, i);
                if (base + i == 0) {
                    st.mx = mx;
                    st.idx = idx;
                    st.mz = mz;
                    st.s = s;
                    st.sz = sz;
                    st.zy = zy;
                } else {
                    part_merge(st, mx, idx, mz, s, sz, zy);
                }
            }
        }
        if (tid == 0) srow = st;
    }
    __syncthreads();
    const float lse = srow.mz + logf(srow.s);
    const int64_t y = p.labels[r];
    const bool ignored = y == p.ignore_index;
    const bool valid = !ignored && y >= 0 && y < p.V;
    // The label census of this call (launched just before, this kernel
    // dependent on it; the merged statistics were complete before the census
    // started).  Every CTA waits, so that the grid completes after the census
    // and the finalize kernel, dependent on this grid, may read its counts.
    ptx::griddep_wait();
    if (valid) {
        const int64_t n_valid = p.counts[0];
        rows::GradCoef c;
        float scale = p.grad_scale;
        if (p.reduction == VLMCE_MEAN)
            scale = n_valid > 0 ? p.grad_scale / static_cast<float>(n_valid) : 0.f;
        rows::set_coef(c, lse, scale, p.eps, p.V);
        c.k = k;
        // the label's granule and lane when this shard holds it
        const int64_t yl = y - p.vocab_start;
        const bool mine = yl >= 0 && yl < p.V_local;
        const int gy = mine ? static_cast<int>((yl + g.lead) / EPG) : -1;
        const int ly = mine ? static_cast<int>((yl + g.lead) % EPG) : -1;
        float gr[EPG];
        if (g.head && tid == 0) {
            rows::grad_values<BF16, SOFTCAP, rows::kCapColumn>(rows::ld_v4(g.row()), c,
                                                               gy == 0 ? ly : -1, gr);
            rows::store_partial<BF16>(g.gbase, -g.lead, p.V_local, gr);
        }
        // two granules loaded before either is stored (the stores would
        // otherwise keep each load waiting for the previous iteration)
        int gl = g.gs + tid;
        for (; gl + THREADS < g.ge; gl += 2 * THREADS) {
            const uint4 w0 = rows::ld_v4(g.row() + gl), w1 = rows::ld_v4(g.row() + gl + THREADS);
            rows::grad_values<BF16, SOFTCAP>(w0, c, gl == gy ? ly : -1, gr);
            ptx::st_global_cs_v4(g.gbase + 16 * gl, rows::pack_granule<BF16>(gr));
            rows::grad_values<BF16, SOFTCAP>(w1, c, gl + THREADS == gy ? ly : -1, gr);
            ptx::st_global_cs_v4(g.gbase + 16 * (gl + THREADS), rows::pack_granule<BF16>(gr));
        }
        for (; gl < g.ge; gl += THREADS) {
            rows::grad_values<BF16, SOFTCAP>(rows::ld_v4(g.row() + gl), c, gl == gy ? ly : -1, gr);
            ptx::st_global_cs_v4(g.gbase + 16 * gl, rows::pack_granule<BF16>(gr));
        }
        if (tid == g.tail_tid) {
            rows::grad_values<BF16, SOFTCAP, rows::kCapColumn>(rows::ld_v4(g.row() + (g.G - 1)), c,
                                             gy == g.G - 1 ? ly : -1, gr);
            rows::store_partial<BF16>(g.gbase + 16 * (g.G - 1), (g.G - 1) * EPG - g.lead,
                                      p.V_local, gr);
        }
    } else {
        float z[EPG];
#pragma unroll
        for (int l = 0; l < EPG; ++l) z[l] = 0.f;
        if (g.head && tid == 0) rows::store_partial<BF16>(g.gbase, -g.lead, p.V_local, z);
        for (int gl = g.gs + tid; gl < g.ge; gl += THREADS)
            ptx::st_global_cs_v4(g.gbase + 16 * gl, make_uint4(0u, 0u, 0u, 0u));
        if (tid == g.tail_tid)
            rows::store_partial<BF16>(g.gbase + 16 * (g.G - 1), (g.G - 1) * EPG - g.lead,
                                      p.V_local, z);
    }
    if (tid == 0) {  // the row's loss and argmax (the same on every shard)
        float l = 0.f;
        if (valid)
            l = lse - fmaf(1.f - p.eps, srow.zy, (p.eps / static_cast<float>(p.V)) * srow.sz);
        else if (!ignored)
            l = __int_as_float(0x7fc00000);  // bad label: NaN
        if (p.loss) p.loss[r] = l;
        if (p.argmax) p.argmax[r] = srow.idx;
    }
}

using ShardKernel = void (*)(ShardParams);
template <int TH>
ShardKernel stats_kernel_t(bool bf16, bool softcap) {
    if (bf16) return softcap ? ce_shard_stats_kernel<true, true, TH> : ce_shard_stats_kernel<true, false, TH>;
    return softcap ? ce_shard_stats_kernel<false, true, TH> : ce_shard_stats_kernel<false, false, TH>;
}
template <int TH>
ShardKernel grad_kernel_t(bool bf16, bool softcap) {
    if (bf16) return softcap ? ce_shard_grad_kernel<true, true, TH> : ce_shard_grad_kernel<true, false, TH>;
    return softcap ? ce_shard_grad_kernel<false, true, TH> : ce_shard_grad_kernel<false, false, TH>;
}
ShardKernel stats_kernel(bool bf16, bool softcap, int threads) {
    if (threads == rows::kTinyThreads)  // no softcap
        return bf16 ? ce_shard_stats_kernel<true, false, rows::kTinyThreads>
                    : ce_shard_stats_kernel<false, false, rows::kTinyThreads>;
    return threads == rows::kShortThreads ? stats_kernel_t<rows::kShortThreads>(bf16, softcap)
                                          : stats_kernel_t<rows::kThreads>(bf16, softcap);
}
ShardKernel grad_kernel(bool bf16, bool softcap, int threads) {
    if (threads == rows::kTinyThreads)  // no softcap
        return bf16 ? ce_shard_grad_kernel<true, false, rows::kTinyThreads>
                    : ce_shard_grad_kernel<false, false, rows::kTinyThreads>;
    return threads == rows::kShortThreads ? grad_kernel_t<rows::kShortThreads>(bf16, softcap)
                                          : grad_kernel_t<rows::kThreads>(bf16, softcap);
}
// The row kernel's CTA size for the shard's rows (the same arithmetic order).
int shard_threads(const void *logits, int32_t dtype, int64_t V_local, int64_t row_stride,
                  bool softcap) {
    const bool bf16 = dtype == VLMCE_BF16;
    return rows::threads_for(
        rows::row_granules(bf16, V_local, rows::rows_aligned(logits, row_stride, bf16 ? 2 : 4)),
        softcap);
}

// Launch a kernel dependent on the previous work on the stream (programmatic
// dependent launch): it may start while its predecessor finishes and waits for
// it with griddepcontrol.wait before using its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                             Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int64_t kMaxVocab = int64_t(1) << 28;

// Checks shared by the shard entry points (nothing is enqueued on failure).
vlmce_status check_shard(const void *logits, int32_t dtype, const int64_t *labels, int64_t N,
                         int64_t V_local, int64_t row_stride, int64_t vocab_start, int64_t V,
                         float softcap) {
    if (dtype != VLMCE_F32 && dtype != VLMCE_BF16) return VLMCE_ERR_UNSUPPORTED_DTYPE;
    if (N < 0 || V_local < 1 || row_stride < V_local || vocab_start < 0 || V < 1 ||
        vocab_start + V_local > V)
        return VLMCE_ERR_INVALID_ARG;
    if (N > 0 && (!logits || !labels)) return VLMCE_ERR_INVALID_ARG;
    if (!(softcap >= 0.f) || !std::isfinite(softcap)) return VLMCE_ERR_INVALID_ARG;
    if (V > kMaxVocab || N > INT_MAX) return VLMCE_ERR_TOO_LARGE;
    const int64_t elt = dtype == VLMCE_BF16 ? 2 : 4;
    if (N > 0 && row_stride > (INT64_MAX / elt) / N) return VLMCE_ERR_TOO_LARGE;
    if (logits && !aligned(logits, static_cast<uintptr_t>(elt))) return VLMCE_ERR_MISALIGNED;
    if (labels && !aligned(labels, 8)) return VLMCE_ERR_MISALIGNED;
    return VLMCE_OK;
}

}  // namespace
}  // namespace shard
}  // namespace ce
}  // namespace vlmce

using namespace vlmce;
using namespace vlmce::ce;
using namespace vlmce::ce::shard;

extern "C" vlmce_status ce_shard_stats(const void *logits, int32_t dtype, const int64_t *labels,
                                       int64_t N, int64_t V_local, int64_t row_stride,
                                       int64_t vocab_start, int64_t V, float softcap,
                                       vlmce_row_stats *out_stats, vlmce_stream_t stream) {
    vlmce_status st = check_shard(logits, dtype, labels, N, V_local, row_stride, vocab_start, V,
                                  softcap);
    if (st != VLMCE_OK) return st;
    if (N > 0 && !out_stats) return VLMCE_ERR_INVALID_ARG;
    if (out_stats && !aligned(out_stats, 16)) return VLMCE_ERR_MISALIGNED;
    if (N == 0) return VLMCE_OK;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != VLMCE_OK) return st;
    ShardParams p = {};
    p.logits = static_cast<unsigned char *>(const_cast<void *>(logits));
    p.labels = labels;
    p.V_local = static_cast<int>(V_local);
    p.vocab_start = vocab_start;
    p.V = static_cast<int>(V);
    p.stride_bytes = row_stride * (dtype == VLMCE_BF16 ? 2 : 4);
    p.softcap = softcap;
    p.stats = reinterpret_cast<RowPart *>(out_stats);
    const int th = shard_threads(logits, dtype, V_local, row_stride, softcap > 0.f);
    stats_kernel(dtype == VLMCE_BF16, softcap > 0.f, th)
        <<<static_cast<unsigned>(N), th, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    return launch_status(cudaSuccess, "ce_shard_stats_kernel");
}

extern "C" vlmce_status ce_merge_stats(const vlmce_row_stats *shards, int32_t k, int64_t N,
                                       vlmce_row_stats *out, vlmce_stream_t stream) {
    if (k < 1 || N < 0) return VLMCE_ERR_INVALID_ARG;
    if (N > 0 && (!shards || !out)) return VLMCE_ERR_INVALID_ARG;
    if (N > INT_MAX) return VLMCE_ERR_TOO_LARGE;
    if ((shards && !aligned(shards, 16)) || (out && !aligned(out, 16))) return VLMCE_ERR_MISALIGNED;
    if (N == 0) return VLMCE_OK;
    DeviceInfo dev;
    vlmce_status st = current_device(&dev);
    if (st != VLMCE_OK) return st;
    return launch_status(
        launch_dependent(ce_merge_stats_kernel, dim3(static_cast<unsigned>((N + 255) / 256)),
                         dim3(256), reinterpret_cast<cudaStream_t>(stream),
                         reinterpret_cast<const RowPart *>(shards), k, N,
                         reinterpret_cast<RowPart *>(out)),
        "ce_merge_stats_kernel");
}

namespace vlmce {
namespace ce {
namespace shard {
namespace {

// ce_shard_fwd_bwd on k gathered records per row ([k][N]; k = 1: merged).
vlmce_status shard_fwd_bwd(void *logits, int32_t dtype, const int64_t *labels, int64_t N,
                           int64_t V_local, int64_t row_stride, int64_t vocab_start, int64_t V,
                           int64_t ignore_index, float label_smoothing, float softcap,
                           int32_t reduction, float grad_scale, const vlmce_row_stats *stats,
                           int32_t k, float *out_loss, int64_t *out_argmax, float *out_reduced,
                           int64_t *out_counts, void *workspace, size_t workspace_bytes_given,
                           vlmce_stream_t stream) {
    vlmce_status st = check_shard(logits, dtype, labels, N, V_local, row_stride, vocab_start, V,
                                  softcap);
    if (st != VLMCE_OK) return st;
    if (!(label_smoothing >= 0.f && label_smoothing <= 1.f)) return VLMCE_ERR_INVALID_ARG;
    if (!std::isfinite(grad_scale)) return VLMCE_ERR_INVALID_ARG;
    if (reduction != VLMCE_MEAN && reduction != VLMCE_SUM && reduction != VLMCE_NONE)
        return VLMCE_ERR_INVALID_ARG;
    if (k < 1) return VLMCE_ERR_INVALID_ARG;
    if (N > 0 && !stats) return VLMCE_ERR_INVALID_ARG;
    if (stats && !aligned(stats, 16)) return VLMCE_ERR_MISALIGNED;
    const size_t need = vlmce_ce_workspace_bytes(N, V, dtype);
    if (!workspace || workspace_bytes_given < need) return VLMCE_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return VLMCE_ERR_MISALIGNED;
    if ((out_loss && !aligned(out_loss, 4)) || (out_argmax && !aligned(out_argmax, 8)) ||
        (out_reduced && !aligned(out_reduced, 4)) || (out_counts && !aligned(out_counts, 8)))
        return VLMCE_ERR_MISALIGNED;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != VLMCE_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // workspace: counts [4] and the error word at the front, then loss / argmax
    unsigned char *wb = static_cast<unsigned char *>(workspace);
    int64_t *counts = reinterpret_cast<int64_t *>(wb);
    int *err = reinterpret_cast<int *>(wb + 64);
    float *loss = out_loss ? out_loss : reinterpret_cast<float *>(wb + 256);
    int64_t *amax = out_argmax ? out_argmax
                               : reinterpret_cast<int64_t *>(wb + 256 + round_up(4 * N, 256));

    if ((st = launch_status(launch_dependent(ce_count_kernel, dim3(1), dim3(1024), cs, labels, N,
                                             V, ignore_index, counts, err),
                            "ce_count_kernel")) != VLMCE_OK)
        return st;
    if (N > 0) {
        ShardParams p = {};
        p.logits = static_cast<unsigned char *>(logits);
        p.labels = labels;
        p.V_local = static_cast<int>(V_local);
        p.vocab_start = vocab_start;
        p.V = static_cast<int>(V);
        p.stride_bytes = row_stride * (dtype == VLMCE_BF16 ? 2 : 4);
        p.ignore_index = ignore_index;
        p.eps = label_smoothing;
        p.softcap = softcap;
        p.grad_scale = grad_scale;
        p.reduction = reduction;
        p.stats = reinterpret_cast<RowPart *>(const_cast<vlmce_row_stats *>(stats));
        p.k = k;
        p.N = N;
        p.loss = loss;
        p.argmax = amax;
        p.counts = counts;
        const int th = shard_threads(logits, dtype, V_local, row_stride, softcap > 0.f);
        st = launch_status(launch_dependent(grad_kernel(dtype == VLMCE_BF16, softcap > 0.f, th),
                                            dim3(static_cast<unsigned>(N)), dim3(th), cs, p),
                           "ce_shard_grad_kernel");
        if (st != VLMCE_OK) return st;
    }
    return launch_status(
        launch_dependent(ce_finalize_kernel, dim3(1), dim3(1024), cs,
                         static_cast<const float *>(loss), static_cast<const int64_t *>(amax),
                         labels, N, V, ignore_index, static_cast<int>(reduction),
                         static_cast<const int64_t *>(counts), static_cast<const int *>(err),
                         out_reduced, out_counts),
        "ce_finalize_kernel");
}

}  // namespace
}  // namespace shard
}  // namespace ce
}  // namespace vlmce

extern "C" vlmce_status ce_shard_fwd_bwd(void *logits, int32_t dtype, const int64_t *labels,
                                         int64_t N, int64_t V_local, int64_t row_stride,
                                         int64_t vocab_start, int64_t V, int64_t ignore_index,
                                         float label_smoothing, float softcap, int32_t reduction,
                                         float grad_scale, const vlmce_row_stats *global_stats,
                                         float *out_loss, int64_t *out_argmax, float *out_reduced,
                                         int64_t *out_counts, void *workspace,
                                         size_t workspace_bytes_given, vlmce_stream_t stream) {
    return shard_fwd_bwd(logits, dtype, labels, N, V_local, row_stride, vocab_start, V,
                         ignore_index, label_smoothing, softcap, reduction, grad_scale,
                         global_stats, 1, out_loss, out_argmax, out_reduced, out_counts, workspace,
                         workspace_bytes_given, stream);
}

extern "C" vlmce_status ce_shard_fwd_bwd_gathered(
    void *logits, int32_t dtype, const int64_t *labels, int64_t N, int64_t V_local,
    int64_t row_stride, int64_t vocab_start, int64_t V, int64_t ignore_index,
    float label_smoothing, float softcap, int32_t reduction, float grad_scale,
    const vlmce_row_stats *gathered, int32_t k, float *out_loss, int64_t *out_argmax,
    float *out_reduced, int64_t *out_counts, void *workspace, size_t workspace_bytes_given,
    vlmce_stream_t stream) {
    return shard_fwd_bwd(logits, dtype, labels, N, V_local, row_stride, vocab_start, V,
                         ignore_index, label_smoothing, softcap, reduction, grad_scale, gathered, k,
                         out_loss, out_argmax, out_reduced, out_counts, workspace,
                         workspace_bytes_given, stream);
}
