// ce.cu -- entry point ce_fwd_bwd: fused cross-entropy forward + backward over
// [N, V] logits, with the gradient written in place of the logits.
//
// Method (web pages on Liger-Kernel / Megatron-LM cross-entropy): per row, an
// online softmax (running max and sum-exp) over the vocabulary, the loss with
// ignore_index, label smoothing and an optional final-logit softcap
// T tanh(x/T), the argmax with smallest-index ties, and the gradient
// scale (softmax - smoothed one-hot) (1 - t^2) stored over the logits, so the
// softmax is never materialised.
//
// Three launches on the caller's stream:
//   1. ce_count_kernel    -- label census (n_valid for the mean, bad labels).
//   2. the row work, by one of two kernels:
//      ce_rows_kernel  (ce_rows.cuh)  -- one CTA per row, two passes, the second
//                    served mostly by L2; the default: every SM busy once N >= 304;
//      ce_split_kernel (ce_split.cuh) -- a thread-block cluster per row,
//                    the row split over its CTAs in shared memory and merged
//                    through distributed shared memory; for few, wide rows,
//                    where one CTA per row would leave most SMs idle.
//   3. ce_finalize_kernel -- fixed-order float-float reduction of the
//      per-row losses and correct-prediction count.
// All three use programmatic dependent launch, so that each is resident
// when its predecessor on the stream completes: the census waits for that
// predecessor before it reads anything, the row work overlaps the census,
// and the finalize waits for the row work.  No floating-point atomics:
// results are bit-reproducible.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <tuple>

#include "ce_census.cuh"
#include "ce_rows.cuh"
#include "ce_split.cuh"
#include "host_util.h"
#include "ptx.cuh"
#include "vlmce.h"

namespace vlmce {
namespace ce {
namespace {

// ------------------------------------------------------------------ host side

struct Workspace {
    int64_t *counts;  // [4]
    int *err;
    float *loss;      // [N]
    int64_t *argmax;  // [N]
};

constexpr int64_t kWsHeader = 256;
constexpr int64_t kMaxVocab = int64_t(1) << 28;

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

using rows::row_granules;
using rows::rows_aligned;

// ---- V-split plans (cluster per row)

struct SplitPlan {
    int k = 0;             // CTAs per cluster (row split)
    int gran_per_cta = 0;  // granules of a row per CTA
    int max_clusters = 0;  // co-resident clusters (persistent grid)
    split::SplitKernel kernel = nullptr;
};

// Smallest cluster whose per-CTA slice fits kPreferredChunks ring slots (two
// rows in flight per CTA); past 8 CTAs, slices of up to the whole ring.
// Tuning override: environment VLMCE_CE_SPLIT = "k".
bool shape_split(int64_t G, SplitPlan *pl) {
    int fk = 0;
    const char *e = getenv("VLMCE_CE_SPLIT");
    if (e && *e) {
        int a = 0;
        if (sscanf(e, "%d", &a) == 1 && a >= 1 && a <= split::kMaxCluster) fk = a;
    }
    const int64_t pref = static_cast<int64_t>(split::kPreferredChunks) * split::kChunkGranules;
    const int64_t cap = static_cast<int64_t>(split::kSlots) * split::kChunkGranules;
    int k = fk ? fk : static_cast<int>((G + pref - 1) / pref);
    if (k < 1) k = 1;
    if (k > split::kMaxCluster) k = split::kMaxCluster;
    const int64_t gc = (G + k - 1) / k;
    if (gc > cap) return false;
    pl->k = k;
    pl->gran_per_cta = static_cast<int>(gc);
    return true;
}

std::mutex g_mu;
std::map<std::tuple<int, bool, bool, int64_t, std::string>, SplitPlan> g_plans;
std::set<std::pair<int, split::SplitKernel>> g_attr_set;

vlmce_status get_split_plan(const DeviceInfo &d, bool bf16, bool softcap, int64_t G,
                            SplitPlan *out) {
    const char *e = getenv("VLMCE_CE_SPLIT");
    const auto key = std::make_tuple(d.device, bf16, softcap, G, std::string(e ? e : ""));
    std::lock_guard<std::mutex> lk(g_mu);
    auto itp = g_plans.find(key);
    if (itp != g_plans.end()) {
        *out = itp->second;
        return VLMCE_OK;
    }
    SplitPlan pl;
    if (!shape_split(G, &pl)) return VLMCE_ERR_TOO_LARGE;
    if (d.smem_optin < split::kSmemBytes) return VLMCE_ERR_UNSUPPORTED_DEVICE;
    pl.kernel = bf16 ? split::split_kernel_bf16(softcap) : split::split_kernel_f32(softcap);
    if (!g_attr_set.count({d.device, pl.kernel})) {
        if (record_cuda(cudaFuncSetAttribute(pl.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             split::kSmemBytes),
                        "cudaFuncSetAttribute(ce_split_kernel)") != cudaSuccess)
            return VLMCE_ERR_CUDA;
        g_attr_set.insert({d.device, pl.kernel});
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.k * d.sm_count, 1, 1);
    cfg.blockDim = dim3(split::kThreads, 1, 1);
    cfg.dynamicSmemBytes = split::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pl.k;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int ncl = 0;
    if (record_cuda(cudaOccupancyMaxActiveClusters(&ncl, pl.kernel, &cfg),
                    "cudaOccupancyMaxActiveClusters(ce_split_kernel)") != cudaSuccess)
        return VLMCE_ERR_CUDA;
    if (ncl < 1) return VLMCE_ERR_TOO_LARGE;
    pl.max_clusters = ncl;
    g_plans[key] = pl;
    *out = pl;
    return VLMCE_OK;
}

// Which kernel does the row work.  The V-split kernel spreads each row over a
// cluster of k CTAs; it pays when the rows are wide (k >= 3) and so few that
// all N k CTAs run at once with room to spare (N k <= 5/3 SMs): measured on
// GB300 over 1..128 rows of 32000..262144 columns, the row kernel (one CTA
// per row, the second pass served by L2) is as fast or faster beyond that.
// Override: environment VLMCE_CE_PATH = "rows" or "split".
bool use_split(int64_t N, int64_t G, const DeviceInfo &d) {
    const char *e = getenv("VLMCE_CE_PATH");
    const int64_t cap = static_cast<int64_t>(split::kMaxCluster) * split::kSlots *
                        split::kChunkGranules;
    if (e && strcmp(e, "split") == 0) return G <= cap;
    if (e && strcmp(e, "rows") == 0) return false;
    if (G > cap) return false;
    const int64_t pref = static_cast<int64_t>(split::kPreferredChunks) * split::kChunkGranules;
    int64_t k = (G + pref - 1) / pref;
    if (k > split::kMaxCluster) k = split::kMaxCluster;
    return k >= 3 && 3 * N * k <= 5 * static_cast<int64_t>(d.sm_count);
}

// Launch the row kernel over N <= INT_MAX rows, one CTA per row, after the
// previous launch on the stream when pdl is set (programmatic dependent
// launch: the kernel waits for it before pass 2).
vlmce_status launch_rows(rows::Kernel kern, const rows::Params &p, int64_t N, int threads, bool pdl,
                         cudaStream_t cs) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(N), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = cs;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return launch_status(cudaLaunchKernelEx(&cfg, kern, p), "ce_rows_kernel");
}

thread_local cudaEvent_t t_prof_begin = nullptr;
thread_local cudaEvent_t t_prof_end = nullptr;

}  // namespace
}  // namespace ce
}  // namespace vlmce

using namespace vlmce;
using namespace vlmce::ce;

extern "C" void vlmce_profile_events(void *ev_begin, void *ev_end) {
    t_prof_begin = static_cast<cudaEvent_t>(ev_begin);
    t_prof_end = static_cast<cudaEvent_t>(ev_end);
}

extern "C" int64_t vlmce_ce_max_vocab(int32_t dtype) {
    if (dtype != VLMCE_F32 && dtype != VLMCE_BF16) return 0;
    return kMaxVocab;
}

extern "C" int32_t vlmce_ce_describe_plan(int64_t N, int64_t V, int32_t dtype, float softcap,
                                          int32_t aligned_rows, int32_t *out) {
    if (!out || N < 0 || V < 1 || V > kMaxVocab || (dtype != VLMCE_F32 && dtype != VLMCE_BF16))
        return VLMCE_ERR_INVALID_ARG;
    DeviceInfo dev;
    vlmce_status st = current_device(&dev);
    if (st != VLMCE_OK) return st;
    const bool bf16 = dtype == VLMCE_BF16;
    const int64_t G = row_granules(bf16, V, aligned_rows != 0);
    if (use_split(N, G, dev)) {
        SplitPlan pl;
        st = get_split_plan(dev, bf16, softcap > 0.f, G, &pl);
        if (st != VLMCE_OK) return st;
        out[0] = 1;
        out[1] = pl.k;
        out[2] = pl.gran_per_cta;
        out[3] = pl.max_clusters;
        out[4] = split::kThreads;
        out[5] = split::kSmemBytes;
    } else {
        out[0] = 0;
        const int th = rows::threads_for(G, softcap > 0.f);
        out[1] = 1;
        out[2] = static_cast<int32_t>(G);
        out[3] = rows::min_blocks(th, softcap > 0.f) * dev.sm_count;
        out[4] = th;
        out[5] = 0;
    }
    return VLMCE_OK;
}

extern "C" size_t vlmce_ce_workspace_bytes(int64_t N, int64_t V, int32_t dtype) {
    (void)V;
    (void)dtype;
    if (N < 0) return 0;
    return workspace_bytes(N);
}

namespace vlmce {
namespace ce {
namespace {

// ce_fwd_bwd itself; allow_split = false keeps the row work on the row kernel
// (plain loads and stores only), for logits in host memory.
vlmce_status run_ce(void *logits, int32_t dtype, const int64_t *labels, int64_t N, int64_t V,
                    int64_t row_stride, int64_t ignore_index, float label_smoothing, float softcap,
                    int32_t reduction, float grad_scale, const float *token_scale, bool want_grad,
                    float *out_loss, int64_t *out_argmax, float *out_reduced,
                    int64_t *out_counts, void *workspace, size_t workspace_bytes_given,
                    vlmce_stream_t stream, bool allow_split) {
    // ---- host-side argument checks; nothing is enqueued on failure
    if (dtype != VLMCE_F32 && dtype != VLMCE_BF16) return VLMCE_ERR_UNSUPPORTED_DTYPE;
    if (N < 0 || V < 1 || row_stride < V) return VLMCE_ERR_INVALID_ARG;
    if (N > 0 && (!logits || !labels)) return VLMCE_ERR_INVALID_ARG;
    if (!(label_smoothing >= 0.f && label_smoothing <= 1.f)) return VLMCE_ERR_INVALID_ARG;
    if (!(softcap >= 0.f) || !std::isfinite(softcap)) return VLMCE_ERR_INVALID_ARG;
    if (!std::isfinite(grad_scale)) return VLMCE_ERR_INVALID_ARG;
    if (reduction != VLMCE_MEAN && reduction != VLMCE_SUM && reduction != VLMCE_NONE)
        return VLMCE_ERR_INVALID_ARG;
    if (V > kMaxVocab || N > INT_MAX) return VLMCE_ERR_TOO_LARGE;
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
    if (token_scale && !aligned(token_scale, 4)) return VLMCE_ERR_MISALIGNED;

    DeviceInfo dev;
    vlmce_status st = current_device(&dev);
    if (st != VLMCE_OK) return st;

    const bool bf16 = dtype == VLMCE_BF16;
    const bool capped = softcap > 0.f;
    const int64_t G = row_granules(bf16, V, rows_aligned(logits, row_stride, elt));
    const bool split_path = allow_split && N > 0 && use_split(N, G, dev);
    SplitPlan pl;
    if (split_path) {
        st = get_split_plan(dev, bf16, capped, G, &pl);
        if (st != VLMCE_OK) return st;
    }

    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    Workspace w = carve(workspace, N);
    float *loss = out_loss ? out_loss : w.loss;
    int64_t *amax = out_argmax ? out_argmax : w.argmax;

    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    {
        cudaLaunchConfig_t cc = {};
        cc.gridDim = dim3(1, 1, 1);
        cc.blockDim = dim3(1024, 1, 1);
        cc.stream = cs;
        cc.attrs = attr;
        cc.numAttrs = 1;
        st = launch_status(cudaLaunchKernelEx(&cc, ce_count_kernel, labels, N, V, ignore_index,
                                              w.counts, w.err),
                           "ce_count_kernel");
        if (st != VLMCE_OK) return st;
    }

    if (N > 0) {
        cudaEvent_t eb = t_prof_begin, ee = t_prof_end;
        t_prof_begin = t_prof_end = nullptr;
        if (eb && (st = launch_status(cudaEventRecord(eb, cs), "cudaEventRecord")) != VLMCE_OK)
            return st;
        if (split_path) {
            split::SplitParams p;
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
            p.token_scale = token_scale;
            p.want_grad = want_grad ? 1 : 0;
            const int64_t ncl = N < pl.max_clusters ? N : pl.max_clusters;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(ncl * pl.k), 1, 1);
            cfg.blockDim = dim3(split::kThreads, 1, 1);
            cfg.dynamicSmemBytes = split::kSmemBytes;
            cfg.stream = cs;
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = pl.k;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 2;
            st = launch_status(cudaLaunchKernelEx(&cfg, pl.kernel, p), "ce_split_kernel");
        } else {
            rows::Params p;
            p.logits = static_cast<unsigned char *>(logits);
            p.labels = labels;
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
            p.token_scale = token_scale;
            p.want_grad = want_grad ? 1 : 0;
            const int th = rows::threads_for(G, capped);
            st = launch_rows(bf16 ? rows::kernel_bf16(capped, th, !want_grad)
                                  : rows::kernel_f32(capped, th, !want_grad),
                             p, N, th, true, cs);
        }
        if (st != VLMCE_OK) return st;
        if (ee && (st = launch_status(cudaEventRecord(ee, cs), "cudaEventRecord")) != VLMCE_OK)
            return st;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(1024, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = cs;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_status(
        cudaLaunchKernelEx(&cfg, ce_finalize_kernel, static_cast<const float *>(loss),
                           static_cast<const int64_t *>(amax), labels, N, V, ignore_index,
                           static_cast<int>(reduction), static_cast<const int64_t *>(w.counts),
                           static_cast<const int *>(w.err), out_reduced, out_counts),
        "ce_finalize_kernel");
}

}  // namespace
}  // namespace ce
}  // namespace vlmce

extern "C" vlmce_status ce_fwd_bwd(void *logits, int32_t dtype, const int64_t *labels, int64_t N,
                                   int64_t V, int64_t row_stride, int64_t ignore_index,
                                   float label_smoothing, float softcap, int32_t reduction,
                                   float grad_scale, float *out_loss, int64_t *out_argmax,
                                   float *out_reduced, int64_t *out_counts, void *workspace,
                                   size_t workspace_bytes_given, vlmce_stream_t stream) {
    return run_ce(logits, dtype, labels, N, V, row_stride, ignore_index, label_smoothing, softcap,
                  reduction, grad_scale, nullptr, true, out_loss, out_argmax, out_reduced,
                  out_counts, workspace, workspace_bytes_given, stream, true);
}

extern "C" vlmce_status ce_fwd_bwd_ex(void *logits, int32_t dtype, const int64_t *labels,
                                      int64_t N, int64_t V, int64_t row_stride,
                                      int64_t ignore_index, float label_smoothing, float softcap,
                                      int32_t reduction, float grad_scale,
                                      const float *grad_per_token, int32_t compute_grad,
                                      float *out_loss, int64_t *out_argmax, float *out_reduced,
                                      int64_t *out_counts, void *workspace,
                                      size_t workspace_bytes_given, vlmce_stream_t stream) {
    return run_ce(logits, dtype, labels, N, V, row_stride, ignore_index, label_smoothing, softcap,
                  reduction, grad_scale, grad_per_token, compute_grad != 0, out_loss, out_argmax,
                  out_reduced, out_counts, workspace, workspace_bytes_given, stream, true);
}

namespace vlmce {
namespace ce {
namespace {

// The device address of a pointer the kernels may dereference: device or
// managed memory as is, page-locked host memory through its device mapping.
// False for memory the device cannot address (pageable host memory).
bool device_alias(const void *p, void **out, bool *is_host) {
    *is_host = false;
    if (!p) {
        *out = nullptr;
        return true;
    }
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *out = const_cast<void *>(p);
        return true;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer) {
        // the mapping of this address within its page-locked allocation
        *out = static_cast<char *>(a.devicePointer) +
               (static_cast<const char *>(p) - static_cast<const char *>(a.hostPointer));
        *is_host = true;
        return true;
    }
    return false;
}

// ---- staged pipeline for logits in host memory
constexpr int kRing = 3;                       // staging slots
constexpr int64_t kChunkTarget = 32ll << 20;   // bytes of logits per chunk
constexpr int kMaxPipeDevices = 64;

int64_t chunk_rows(int64_t N, int64_t row_stride, int64_t elt) {
    int64_t r = kChunkTarget / (row_stride * elt);
    if (r < 1) r = 1;
    return r < N ? r : (N > 0 ? N : 1);
}
int64_t slot_bytes(int64_t rows, int64_t row_stride, int64_t elt) {
    return round_up(16 + rows * row_stride * elt, 256);
}
size_t host_workspace_bytes(int64_t N, int64_t row_stride, int64_t elt) {
    return workspace_bytes(N) +
           static_cast<size_t>(kRing * slot_bytes(chunk_rows(N, row_stride, elt), row_stride, elt));
}

// Per device: the copy-in and copy-out streams and the ring's events.
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t loaded[kRing] = {}, computed[kRing] = {}, stored[kRing] = {};
};
std::mutex g_pipe_mu;
HostPipe g_pipes[kMaxPipeDevices];

vlmce_status get_pipe(int device, HostPipe **out) {
    if (device < 0 || device >= kMaxPipeDevices) return VLMCE_ERR_UNSUPPORTED_DEVICE;
    HostPipe &hp = g_pipes[device];
    if (!hp.ready) {
        const unsigned f = cudaEventDisableTiming;
        cudaError_t e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, f);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.done, f);
        for (int b = 0; b < kRing && e == cudaSuccess; ++b) {
            e = cudaEventCreateWithFlags(&hp.loaded[b], f);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.computed[b], f);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.stored[b], f);
        }
        if (record_cuda(e, "host pipeline streams and events") != cudaSuccess) return VLMCE_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return VLMCE_OK;
}

// Same checks and results as run_ce (row kernel); the logits live in host
// memory and pass through the device in chunks of rows: copy in (stream
// `in`), compute (the caller's stream), copy the gradient columns back
// (stream `out`), three chunks in flight.  Staged rows keep the caller's row
// stride and 16-byte phase, so the kernel sees the same layout.
vlmce_status run_ce_staged(void *host_logits, int32_t dtype, const int64_t *labels, int64_t N,
                           int64_t V, int64_t row_stride, int64_t ignore_index,
                           float label_smoothing, float softcap, int32_t reduction,
                           float grad_scale, float *loss_out, int64_t *amax_out,
                           float *out_reduced, int64_t *out_counts, void *workspace,
                           size_t workspace_bytes_given, cudaStream_t cs) {
    if (dtype != VLMCE_F32 && dtype != VLMCE_BF16) return VLMCE_ERR_UNSUPPORTED_DTYPE;
    if (N < 0 || V < 1 || row_stride < V) return VLMCE_ERR_INVALID_ARG;
    if (N > 0 && (!host_logits || !labels)) return VLMCE_ERR_INVALID_ARG;
    if (!(label_smoothing >= 0.f && label_smoothing <= 1.f)) return VLMCE_ERR_INVALID_ARG;
    if (!(softcap >= 0.f) || !std::isfinite(softcap)) return VLMCE_ERR_INVALID_ARG;
    if (!std::isfinite(grad_scale)) return VLMCE_ERR_INVALID_ARG;
    if (reduction != VLMCE_MEAN && reduction != VLMCE_SUM && reduction != VLMCE_NONE)
        return VLMCE_ERR_INVALID_ARG;
    if (V > kMaxVocab || N > INT_MAX) return VLMCE_ERR_TOO_LARGE;
    const int64_t elt = dtype == VLMCE_BF16 ? 2 : 4;
    if (N > 0 && row_stride > (INT64_MAX / elt) / N) return VLMCE_ERR_TOO_LARGE;
    if (!workspace || workspace_bytes_given < host_workspace_bytes(N, row_stride, elt))
        return VLMCE_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 256)) return VLMCE_ERR_MISALIGNED;
    if (!aligned(host_logits, static_cast<uintptr_t>(elt))) return VLMCE_ERR_MISALIGNED;
    if (labels && !aligned(labels, 8)) return VLMCE_ERR_MISALIGNED;
    if (loss_out && !aligned(loss_out, 4)) return VLMCE_ERR_MISALIGNED;
    if (amax_out && !aligned(amax_out, 8)) return VLMCE_ERR_MISALIGNED;
    if (out_reduced && !aligned(out_reduced, 4)) return VLMCE_ERR_MISALIGNED;
    if (out_counts && !aligned(out_counts, 8)) return VLMCE_ERR_MISALIGNED;

    DeviceInfo dev;
    vlmce_status st = current_device(&dev);
    if (st != VLMCE_OK) return st;
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe *hp = nullptr;
    if ((st = get_pipe(dev.device, &hp)) != VLMCE_OK) return st;

    const bool bf16 = dtype == VLMCE_BF16;
    const int64_t stride_bytes = row_stride * elt;
    const int64_t R = chunk_rows(N, row_stride, elt);
    const int64_t sb = slot_bytes(R, row_stride, elt);
    Workspace w = carve(workspace, N);
    unsigned char *ring = static_cast<unsigned char *>(workspace) + workspace_bytes(N);
    float *loss = loss_out ? loss_out : w.loss;
    int64_t *amax = amax_out ? amax_out : w.argmax;
    unsigned char *hbase = static_cast<unsigned char *>(host_logits);

    auto fail = [](cudaError_t e, const char *where) { return launch_status(e, where); };
    if ((st = fail(cudaEventRecord(hp->start, cs), "cudaEventRecord")) != VLMCE_OK) return st;
    if ((st = fail(cudaStreamWaitEvent(hp->in, hp->start, 0), "cudaStreamWaitEvent")) != VLMCE_OK)
        return st;
    if ((st = fail(cudaStreamWaitEvent(hp->out, hp->start, 0), "cudaStreamWaitEvent")) != VLMCE_OK)
        return st;

    ce_count_kernel<<<1, 1024, 0, cs>>>(labels, N, V, ignore_index, w.counts, w.err);
    if ((st = launch_status(cudaSuccess, "ce_count_kernel")) != VLMCE_OK) return st;

    // the CTA size ce_fwd_bwd would pick for these rows (the same arithmetic order)
    const int th = rows::threads_for(
        rows::row_granules(bf16, V, rows::rows_aligned(host_logits, row_stride, elt)), softcap > 0.f);
    const rows::Kernel kern =
        bf16 ? rows::kernel_bf16(softcap > 0.f, th, false) : rows::kernel_f32(softcap > 0.f, th, false);
    const int64_t nchunks = N > 0 ? (N + R - 1) / R : 0;
    for (int64_t i = 0; i < nchunks; ++i) {
        const int b = static_cast<int>(i % kRing);
        const int64_t r0 = i * R;
        const int64_t rows_i = (N - r0) < R ? (N - r0) : R;
        unsigned char *hrow = hbase + r0 * stride_bytes;
        // the chunk's first row keeps its 16-byte phase in the slot
        unsigned char *slot = ring + b * sb + (reinterpret_cast<uintptr_t>(hrow) & 15u);
        // copy in: whole rows, but not past the last row's V columns
        if (i >= kRing &&
            (st = fail(cudaStreamWaitEvent(hp->in, hp->stored[b], 0), "cudaStreamWaitEvent")) != VLMCE_OK)
            return st;
        if ((st = fail(cudaMemcpyAsync(slot, hrow, (rows_i - 1) * stride_bytes + V * elt,
                                       cudaMemcpyDefault, hp->in),
                       "cudaMemcpyAsync(host to device)")) != VLMCE_OK)
            return st;
        if ((st = fail(cudaEventRecord(hp->loaded[b], hp->in), "cudaEventRecord")) != VLMCE_OK) return st;
        // compute on the caller's stream
        if ((st = fail(cudaStreamWaitEvent(cs, hp->loaded[b], 0), "cudaStreamWaitEvent")) != VLMCE_OK)
            return st;
        rows::Params p;
        p.logits = slot;
        p.labels = labels + r0;
        p.V = static_cast<int>(V);
        p.stride_bytes = stride_bytes;
        p.ignore_index = ignore_index;
        p.eps = label_smoothing;
        p.softcap = softcap;
        p.grad_scale = grad_scale;
        p.reduction = reduction;
        p.loss = loss + r0;
        p.argmax = amax + r0;
        p.counts = w.counts;
        p.token_scale = nullptr;
        p.want_grad = 1;
        if ((st = launch_rows(kern, p, rows_i, th, false, cs)) != VLMCE_OK) return st;
        if ((st = fail(cudaEventRecord(hp->computed[b], cs), "cudaEventRecord")) != VLMCE_OK) return st;
        // copy the gradient columns [0, V) of each row back
        if ((st = fail(cudaStreamWaitEvent(hp->out, hp->computed[b], 0), "cudaStreamWaitEvent")) !=
            VLMCE_OK)
            return st;
        if ((st = fail(cudaMemcpy2DAsync(hrow, stride_bytes, slot, stride_bytes, V * elt, rows_i,
                                         cudaMemcpyDefault, hp->out),
                       "cudaMemcpy2DAsync(device to host)")) != VLMCE_OK)
            return st;
        if ((st = fail(cudaEventRecord(hp->stored[b], hp->out), "cudaEventRecord")) != VLMCE_OK) return st;
    }
    if ((st = fail(cudaEventRecord(hp->done, hp->out), "cudaEventRecord")) != VLMCE_OK) return st;
    if ((st = fail(cudaStreamWaitEvent(cs, hp->done, 0), "cudaStreamWaitEvent")) != VLMCE_OK) return st;

    ce_finalize_kernel<<<1, 1024, 0, cs>>>(loss, amax, labels, N, V, ignore_index,
                                           static_cast<int>(reduction), w.counts, w.err,
                                           out_reduced, out_counts);
    return launch_status(cudaSuccess, "ce_finalize_kernel");
}

}  // namespace
}  // namespace ce
}  // namespace vlmce

extern "C" size_t vlmce_ce_host_workspace_bytes(int64_t N, int64_t V, int64_t row_stride,
                                                int32_t dtype) {
    if (N < 0 || V < 1 || row_stride < V || (dtype != VLMCE_F32 && dtype != VLMCE_BF16)) return 0;
    return host_workspace_bytes(N, row_stride, dtype == VLMCE_BF16 ? 2 : 4);
}

extern "C" vlmce_status ce_fwd_bwd_host(void *logits, int32_t dtype, const int64_t *labels,
                                        int64_t N, int64_t V, int64_t row_stride,
                                        int64_t ignore_index, float label_smoothing, float softcap,
                                        int32_t reduction, float grad_scale, float *out_loss,
                                        int64_t *out_argmax, float *out_reduced,
                                        int64_t *out_counts, void *workspace,
                                        size_t workspace_bytes_given, vlmce_stream_t stream) {
    void *d[6];
    bool host[6];
    const void *h[6] = {logits, labels, out_loss, out_argmax, out_reduced, out_counts};
    for (int i = 0; i < 6; ++i)
        if (!device_alias(h[i], &d[i], &host[i])) return VLMCE_ERR_INVALID_ARG;
    if (!host[0])  // device logits: ce_fwd_bwd, with host labels / outputs read and written in place
        return run_ce(d[0], dtype, static_cast<const int64_t *>(d[1]), N, V, row_stride,
                      ignore_index, label_smoothing, softcap, reduction, grad_scale, nullptr, true,
                      static_cast<float *>(d[2]), static_cast<int64_t *>(d[3]),
                      static_cast<float *>(d[4]), static_cast<int64_t *>(d[5]), workspace,
                      workspace_bytes_given, stream, true);
    return run_ce_staged(logits, dtype, static_cast<const int64_t *>(d[1]), N, V, row_stride,
                         ignore_index, label_smoothing, softcap, reduction, grad_scale,
                         static_cast<float *>(d[2]), static_cast<int64_t *>(d[3]),
                         static_cast<float *>(d[4]), static_cast<int64_t *>(d[5]), workspace,
                         workspace_bytes_given, reinterpret_cast<cudaStream_t>(stream));
}
