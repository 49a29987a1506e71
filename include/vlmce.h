/*
 * vlmce.h -- C ABI of the GB300 (sm_103a) fused large-vocabulary language-model
 * cross-entropy library (libvlmce.so).
 *
 * Plain pointers and sizes only.  Every buffer argument is DEVICE memory that
 * the caller allocates and owns; the library never allocates, frees or
 * synchronises.  All work is enqueued on the caller's stream, in stream order,
 * and a call returns as soon as it is enqueued.  Arguments are checked on the
 * host before anything is enqueued; a non-zero status means nothing was
 * enqueued (except VLMCE_ERR_CUDA, which reports a failed launch).
 *
 * Notation (per row r of an [N, V] logits tensor; x_j the input logit):
 *   t_j = tanh(x_j / T), z_j = T t_j  when the softcap T > 0, else z_j = x_j
 *   q_j = (1 - eps) [j = y] + eps / V          (label smoothing eps, label y)
 *   lse = log sum_j exp(z_j),  p_j = exp(z_j - lse)
 *   loss_r = lse - (1 - eps) z_y - (eps / V) sum_j z_j
 *   grad_j = scale (p_j - q_j) (T > 0 ? 1 - t_j^2 : 1)
 * with scale = grad_scale / n_valid for the mean reduction and grad_scale for
 * the sum, n_valid = the number of rows whose label is in [0, V).
 *
 * Sources (web pages on Liger-Kernel / Megatron-LM cross-entropy):
 *  - "Add Megatron-LM cross-entropy integration", Summary: ignore_index and
 *    label_smoothing arguments; online softmax; gradient written in place of
 *    the logits; no full-softmax materialisation.
 *  - "Add opt-in Liger vocab-parallel cross entropy through ops/loss", What
 *    does this PR do: fp32 per-token losses, gradient kept in the incoming
 *    dtype, optional global argmax with smallest-index ties; Contribution
 *    process: strided inputs and arbitrary upstream gradients.
 *  - "Add Liger Kernel support for Muse Glimmer", Summary and Details: token
 *    accuracy, the final-logit softcap T tanh(x/T) with the multiplier folded
 *    into the hidden states, and a fused linear cross-entropy that never
 *    builds the [B, S, V] logits and keeps grad_weight in fp32; the native
 *    Blackwell fused path accepts only 16-bit inputs and mean/sum.
 */
#ifndef VLMCE_H_
#define VLMCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *vlmce_stream_t;

typedef enum {
    VLMCE_OK = 0,
    VLMCE_ERR_INVALID_ARG = 1,        /* NULL pointer, bad size, bad option value   */
    VLMCE_ERR_UNSUPPORTED_DTYPE = 2,  /* dtype not accepted by this entry point      */
    VLMCE_ERR_MISALIGNED = 3,         /* a pointer is not aligned as documented      */
    VLMCE_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
    VLMCE_ERR_WORKSPACE_TOO_SMALL = 5,/* workspace NULL or smaller than the query    */
    VLMCE_ERR_CUDA = 6,               /* a CUDA runtime call or launch failed        */
    VLMCE_ERR_TOO_LARGE = 7           /* a size beyond what the kernels support      */
} vlmce_status;

/* VLMCE_F16: fp16, accepted by flce_fwd_bwd_ex and vlmce_gemm only. */
typedef enum { VLMCE_F32 = 0, VLMCE_BF16 = 1, VLMCE_F16 = 2 } vlmce_dtype;
/* VLMCE_NONE: per-token losses only; the gradient is not averaged (each row
 * is scaled by grad_scale, and by grad_per_token[r] where given) and
 * out_reduced[0] is the sum of the losses.  Not accepted by flce_fwd_bwd. */
typedef enum { VLMCE_NONE = 0, VLMCE_MEAN = 1, VLMCE_SUM = 2 } vlmce_reduction;

/* Bits of out_counts[3]: errors the kernels detected on the device. */
#define VLMCE_DEVERR_TIMEOUT 1 /* an on-chip wait gave up; results are invalid */

/* Largest vocabulary ce_fwd_bwd accepts, in elements, for the given dtype. */
int64_t vlmce_ce_max_vocab(int32_t dtype);

/* The launch plan ce_fwd_bwd uses for N rows of V elements on the current
 * device: out[6] = {kernel (0: one CTA per row, 1: a cluster per row),
 * CTAs per row, 16-byte granules per CTA, co-resident CTAs (kernel 0) or
 * clusters (kernel 1), threads per CTA, dynamic shared-memory bytes per CTA}.
 * aligned_rows: every row starts on a 16-byte boundary.  Returns a
 * vlmce_status. */
int32_t vlmce_ce_describe_plan(int64_t N, int64_t V, int32_t dtype, float softcap,
                               int32_t aligned_rows, int32_t *out);

/* Bytes of device workspace ce_fwd_bwd needs for N rows (16-byte aligned). */
size_t vlmce_ce_workspace_bytes(int64_t N, int64_t V, int32_t dtype);

/*
 * ce_fwd_bwd -- fused cross-entropy forward + backward over N rows, in place.
 *
 * logits       in:  [N, row_stride] elements of `dtype` (VLMCE_F32 or
 *                   VLMCE_BF16), rows of V valid elements; the element pointer
 *                   must be aligned to the element size.
 *              out: columns [0, V) of every row hold grad_j in the same dtype
 *                   (fp32 -> bf16 rounding is round-to-nearest-even).  Columns
 *                   [V, row_stride) are neither read nor written.  The input
 *                   logits are destroyed.
 * labels       [N] int64, device, 8-byte aligned.  A row whose label equals
 *              ignore_index gets loss 0 and a zero gradient.  A label outside
 *              [0, V) that is not ignore_index is a caller error: that row's
 *              loss is NaN, its gradient zero, and it is counted in
 *              out_counts[2] (the reduced loss is then NaN).
 * N >= 0, 1 <= V <= vlmce_ce_max_vocab(dtype), row_stride >= V (elements).
 * label_smoothing in [0, 1]; softcap T >= 0 and finite (0 = off).  The
 * stated tolerances hold for 1e-4 <= T <= 1e4: the row kernels evaluate
 * tanh(x/T) for |x| <= 0.55 T by a polynomial in x whose coefficients carry
 * powers of 1/T up to the ninth, which leave the fp32 normal range outside it;
 * reduction VLMCE_MEAN (over rows with labels in [0, V); 0 when there are none),
 * VLMCE_SUM or VLMCE_NONE; grad_scale finite: the upstream gradient of the
 * reduced loss.
 * out_loss     [N] fp32 per-token loss (0 for ignored rows), or NULL.
 * out_argmax   [N] int64, or NULL: per row the smallest j with x_j = max_k x_k
 *              (raw input values), written for ignored rows too.
 * out_reduced  [2] fp32, or NULL: reduced loss, token accuracy
 *              (n_correct / n_valid, 0 when n_valid = 0).
 * out_counts   [4] int64, or NULL: n_valid, n_correct (argmax = label among
 *              valid rows), n_bad_labels, device error bits (VLMCE_DEVERR_*).
 * workspace    device, >= vlmce_ce_workspace_bytes(N, V, dtype) bytes,
 *              16-byte aligned; contents need no initialisation and are
 *              scratch between calls.  Calls that share a workspace or
 *              output buffers must be ordered on one stream.
 * stream       the stream every kernel is launched on.
 *
 * Deterministic: the same inputs give bit-identical outputs (fixed-order
 * reductions, no floating-point atomics).
 */
vlmce_status ce_fwd_bwd(void *logits, int32_t dtype, const int64_t *labels, int64_t N, int64_t V,
                        int64_t row_stride, int64_t ignore_index, float label_smoothing,
                        float softcap, int32_t reduction, float grad_scale, float *out_loss,
                        int64_t *out_argmax, float *out_reduced, int64_t *out_counts,
                        void *workspace, size_t workspace_bytes, vlmce_stream_t stream);

/*
 * ce_fwd_bwd_ex -- ce_fwd_bwd with a per-token upstream gradient and a
 * forward-only mode ("Add opt-in Liger vocab-parallel cross entropy through
 * ops/loss", Contribution process: arbitrary upstream gradients).
 *   grad_per_token  device fp32 [N], 4-byte aligned, or NULL: row r's gradient
 *                   is further multiplied by grad_per_token[r] (the upstream
 *                   gradient of a VLMCE_NONE reduction; also allowed with MEAN
 *                   and SUM).
 *   compute_grad    0: forward only -- the logits are read once and left
 *                   unchanged; losses, argmax, reduced values and counts are
 *                   written as usual.  Otherwise as ce_fwd_bwd.
 * All other arguments, results and errors are those of ce_fwd_bwd, which is
 * ce_fwd_bwd_ex(..., grad_per_token = NULL, compute_grad = 1, ...).
 */
vlmce_status ce_fwd_bwd_ex(void *logits, int32_t dtype, const int64_t *labels, int64_t N,
                           int64_t V, int64_t row_stride, int64_t ignore_index,
                           float label_smoothing, float softcap, int32_t reduction,
                           float grad_scale, const float *grad_per_token, int32_t compute_grad,
                           float *out_loss, int64_t *out_argmax, float *out_reduced,
                           int64_t *out_counts, void *workspace, size_t workspace_bytes,
                           vlmce_stream_t stream);

/*
 * ce_fwd_bwd_host -- ce_fwd_bwd for data that lives in host memory.  logits
 * (read, then overwritten by the gradient), labels and the outputs may be
 * page-locked host memory (cudaHostAlloc / cudaMallocHost / cudaHostRegister)
 * as well as device memory.  The pages have no counterpart: it serves callers
 * whose logits are produced or consumed on the host.
 *
 * Host logits pass through the device in chunks of about 32 MB of rows: a
 * copy in on a library-owned stream, the row kernel on `stream`, a copy of
 * the gradient columns [0, V) back on a second library-owned stream, three
 * chunks in flight, so both directions of the host-device link (NVLink-C2C on
 * GB300) stay busy.  Labels and the outputs are read and written in place by
 * the kernels.  Results are those of ce_fwd_bwd with its row kernel (bit-
 * identical on the same inputs).  Device logits are handled by ce_fwd_bwd
 * itself (host labels / outputs still allowed).
 *
 * Arguments, layout, results and errors are those of ce_fwd_bwd, except:
 *   - every non-NULL pointer but the workspace is checked with
 *     cudaPointerGetAttributes before anything is enqueued; one the device
 *     cannot address (pageable host memory) gives VLMCE_ERR_INVALID_ARG;
 *   - with host logits the workspace (device, 256-byte aligned) must hold
 *     vlmce_ce_host_workspace_bytes(N, V, row_stride, dtype) bytes (it
 *     includes the staging ring);
 *   - the library creates, once per device, two non-blocking streams and a
 *     few events for the pipeline, and enqueue is serialised by a mutex.
 * The host buffers hold the results once `stream` has reached the end of the
 * call (synchronise it before reading them).
 */
vlmce_status ce_fwd_bwd_host(void *logits, int32_t dtype, const int64_t *labels, int64_t N,
                             int64_t V, int64_t row_stride, int64_t ignore_index,
                             float label_smoothing, float softcap, int32_t reduction,
                             float grad_scale, float *out_loss, int64_t *out_argmax,
                             float *out_reduced, int64_t *out_counts, void *workspace,
                             size_t workspace_bytes, vlmce_stream_t stream);

/* Bytes of device workspace ce_fwd_bwd_host needs when the logits are in
 * host memory: ce_fwd_bwd's workspace and a ring of three chunk buffers of
 * whole rows (row_stride elements each, about 32 MB per chunk). */
size_t vlmce_ce_host_workspace_bytes(int64_t N, int64_t V, int64_t row_stride, int32_t dtype);

/*
 * Vocabulary-sharded cross-entropy ("Add Megatron-LM cross-entropy
 * integration", Summary; "Add opt-in Liger vocab-parallel cross entropy
 * through ops/loss", What does this PR do): each rank of a tensor-parallel
 * group holds the columns [vocab_start, vocab_start + V_local) of every row
 * (V = the whole vocabulary).  Per call sequence on each rank:
 *   ce_shard_stats  -> this shard's row statistics [N];
 *   (the caller gathers all k shards' statistics, e.g. an all-gather, as a
 *    [k][N] array in shard order);
 *   ce_merge_stats  -> the whole vocabulary's statistics [N] (identical bits
 *                      on every rank that merges the same array);
 *   ce_shard_fwd_bwd -> per-token loss / argmax / reduced loss and accuracy
 *                      (the same on every rank) and the gradient of this
 *                      shard's columns, written in place;
 *   or, in place of the last two, ce_shard_fwd_bwd_gathered on the gathered
 *   array itself.
 * With one shard (vocab_start 0, V_local = V) this is ce_fwd_bwd.
 */
typedef struct vlmce_row_stats {
    float x_max;     /* largest raw logit of the columns merged so far */
    int32_t argmax;  /* its smallest global column (INT32_MAX before any column) */
    float m;         /* reference of s, >= every z_j merged (z = T tanh(x/T), or
                        x): z at x_max, or up to 8 above it */
    float s;         /* sum over the columns of exp(z_j - m) */
    float sum_z;     /* sum over the columns of z_j */
    float z_y;       /* z at the row's label column if merged so far, else 0 */
    float reserved[2];
} vlmce_row_stats;   /* 32 bytes; lse = m + log(s) */

/* Statistics of one shard.  logits: device, N rows of row_stride elements
 * (>= V_local) holding the shard's V_local columns (not modified); labels:
 * [N] int64 global labels; 0 <= vocab_start, vocab_start + V_local <= V <=
 * vlmce_ce_max_vocab(dtype); softcap as in ce_fwd_bwd.  out_stats: device
 * [N], 16-byte aligned.  Argument errors as ce_fwd_bwd. */
vlmce_status ce_shard_stats(const void *logits, int32_t dtype, const int64_t *labels, int64_t N,
                            int64_t V_local, int64_t row_stride, int64_t vocab_start, int64_t V,
                            float softcap, vlmce_row_stats *out_stats, vlmce_stream_t stream);

/* out[r] = merge of shards[0][r] .. shards[k-1][r] in that order: the
 * largest x_max (smallest argmax on ties), the sums of exp rescaled to the
 * larger reference, the sums of sum_z and z_y.  shards: device [k][N]
 * (contiguous), k >= 1; out: device [N], may be shards itself (block 0). */
vlmce_status ce_merge_stats(const vlmce_row_stats *shards, int32_t k, int64_t N,
                            vlmce_row_stats *out, vlmce_stream_t stream);

/* Loss and this shard's gradient from the whole vocabulary's statistics.
 * Arguments as ce_fwd_bwd (logits: the shard, overwritten by the gradient of
 * its V_local columns; label validity, the mean's n_valid and eps / V use
 * the global V), plus vocab_start, V and global_stats (device [N], the merge
 * of every shard's statistics).  workspace: vlmce_ce_workspace_bytes(N, V,
 * dtype) bytes of device memory.  out_* as ce_fwd_bwd; their values are the
 * same on every rank. */
vlmce_status ce_shard_fwd_bwd(void *logits, int32_t dtype, const int64_t *labels, int64_t N,
                              int64_t V_local, int64_t row_stride, int64_t vocab_start, int64_t V,
                              int64_t ignore_index, float label_smoothing, float softcap,
                              int32_t reduction, float grad_scale,
                              const vlmce_row_stats *global_stats, float *out_loss,
                              int64_t *out_argmax, float *out_reduced, int64_t *out_counts,
                              void *workspace, size_t workspace_bytes, vlmce_stream_t stream);

/* ce_merge_stats followed by ce_shard_fwd_bwd in one call, with no merged
 * statistics buffer: gathered is the device [k][N] array of every shard's
 * statistics in shard order (as an all-gather of the k ranks' ce_shard_stats
 * outputs leaves it), k >= 1, 16-byte aligned.  Each row's k records are
 * merged inside the gradient kernel with ce_merge_stats' operator and order,
 * so every result is bit-identical to the two calls; one launch fewer on the
 * rank's step.  Other arguments, results and errors as ce_shard_fwd_bwd. */
vlmce_status ce_shard_fwd_bwd_gathered(void *logits, int32_t dtype, const int64_t *labels,
                                       int64_t N, int64_t V_local, int64_t row_stride,
                                       int64_t vocab_start, int64_t V, int64_t ignore_index,
                                       float label_smoothing, float softcap, int32_t reduction,
                                       float grad_scale, const vlmce_row_stats *gathered,
                                       int32_t k, float *out_loss, int64_t *out_argmax,
                                       float *out_reduced, int64_t *out_counts, void *workspace,
                                       size_t workspace_bytes, vlmce_stream_t stream);

/*
 * Fused gate-up SwiGLU ("[Megatron] Add SwiGLU integration", Summary and
 * Background).  x: device [T, x_stride] elements of `dtype` (VLMCE_BF16 or
 * VLMCE_F32), the gate in columns [0, n) and the up projection in [n, 2n) of
 * every row (x_stride >= 2n).  Arithmetic in fp32, results rounded to
 * nearest even.  Argument errors are returned before anything is enqueued.
 *
 * swiglu_fwd: y [T, y_stride >= n] = silu(gate) * up, silu(a) = a / (1 + e^-a).
 *             y must not overlap x.
 * swiglu_bwd: dx [T, dx_stride >= 2n] = (d_gate | d_up) for dy [T, dy_stride
 *             >= n]: d_up = dy silu(gate), d_gate = dy up silu'(gate).  dx may
 *             be x itself with the same stride (in place); otherwise the
 *             buffers must not overlap.
 * 16-byte vector accesses when n, the strides and the bases allow it, else
 * one element per thread.
 */
vlmce_status swiglu_fwd(const void *x, int32_t dtype, int64_t T, int64_t n, int64_t x_stride,
                        void *y, int64_t y_stride, vlmce_stream_t stream);
vlmce_status swiglu_bwd(const void *x, int64_t x_stride, const void *dy, int64_t dy_stride,
                        void *dx, int64_t dx_stride, int32_t dtype, int64_t T, int64_t n,
                        vlmce_stream_t stream);

/* Bytes of device workspace flce_fwd_bwd needs (256-byte aligned): per-row
 * statistics of every 256-column logits tile, two bf16 [N, 8192] gradient
 * tiles, an fp32 [N, H] grad_hidden accumulator and one 4-byte tile counter
 * per GEMM launch of the call (the workspace of a call in flight belongs to
 * that call: two calls at once need two workspaces). */
size_t vlmce_flce_workspace_bytes(int64_t N, int64_t H, int64_t V);

/*
 * flce_fwd_bwd -- fused linear cross-entropy forward + backward: the logits
 * S = h' W^T are formed tile by tile on the tensor cores and never stored as an
 * [N, V] tensor ("Add Liger Kernel support for Muse Glimmer", Summary and
 * Details: Softcap; its Memory section: grad_weight in fp32).
 *
 * hidden       bf16 [N, hidden_stride], rows of H valid elements: h' = m h, the
 *              hidden states already multiplied by the logit multiplier m.
 * weight       bf16 [V, weight_stride], rows of H valid elements (lm_head).
 * labels, ignore_index, label_smoothing, softcap, reduction, grad_scale,
 * out_loss, out_argmax, out_reduced, out_counts: as ce_fwd_bwd, applied to
 *              the logits S (argmax over the fp32 S).
 * grad_hidden  out: bf16 [N, hidden_stride], d(grad_scale * loss) / d h'
 *              (the caller multiplies by m for d / d h).
 * grad_weight  fp32 [V, H] contiguous: overwritten with d(...)/dW, or added
 *              to when accumulate_grad_weight != 0 (with N = 0 an overwritten
 *              grad_weight is set to zero; it may then be NULL).
 * workspace    >= vlmce_flce_workspace_bytes(N, H, V) bytes, 256-byte aligned.
 * H, hidden_stride, weight_stride must be multiples of 8; every pointer
 * 16-byte aligned.  bf16 only (like the native Blackwell path on the pages).
 * Deterministic: no floating-point atomics.
 */
vlmce_status flce_fwd_bwd(const void *hidden, int64_t hidden_stride, const void *weight,
                          int64_t weight_stride, const int64_t *labels, int64_t N, int64_t H,
                          int64_t V, int64_t ignore_index, float label_smoothing, float softcap,
                          int32_t reduction, float grad_scale, float *out_loss,
                          int64_t *out_argmax, float *out_reduced, int64_t *out_counts,
                          void *grad_hidden, float *grad_weight, int32_t accumulate_grad_weight,
                          void *workspace, size_t workspace_bytes, vlmce_stream_t stream);

/*
 * flce_fwd_bwd_ex -- flce_fwd_bwd for bf16 or fp16 hidden states and weight
 * (dtype VLMCE_BF16 or VLMCE_F16; grad_hidden in the same dtype, grad_weight
 * fp32), like the SM100 fused linear cross-entropy of "Add Liger Kernel
 * support for Muse Glimmer" (FP16/BF16 input and weight, mean/sum).  The
 * gradient tile between the products is kept without the row scale (times
 * 2^14 in fp16, so that small probabilities do not underflow); the two
 * gradient products apply the scale in their epilogues.  Other arguments,
 * results and errors as flce_fwd_bwd, which is flce_fwd_bwd_ex(VLMCE_BF16).
 */
vlmce_status flce_fwd_bwd_ex(const void *hidden, int32_t dtype, int64_t hidden_stride,
                             const void *weight, int64_t weight_stride, const int64_t *labels,
                             int64_t N, int64_t H, int64_t V, int64_t ignore_index,
                             float label_smoothing, float softcap, int32_t reduction,
                             float grad_scale, float *out_loss, int64_t *out_argmax,
                             float *out_reduced, int64_t *out_counts, void *grad_hidden,
                             float *grad_weight, int32_t accumulate_grad_weight, void *workspace,
                             size_t workspace_bytes, vlmce_stream_t stream);

/* Bytes of device workspace flce_fwd_bwd_rows needs (256-byte aligned): the
 * per-token losses and argmax, the fp32 logits and the 16-bit gradient of one
 * chunk of min(chunk_rows, N) rows, and the ce_fwd_bwd workspace of a chunk.
 * 0 for arguments flce_fwd_bwd_rows rejects by size. */
size_t vlmce_flce_rows_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t chunk_rows);

/*
 * flce_fwd_bwd_rows -- flce_fwd_bwd_ex on a row-chunked schedule instead of
 * the vocabulary-chunked one: for each block of chunk_rows rows the logits
 * S_k = h'_k W^T are written in fp32 to the workspace, ce_fwd_bwd_ex turns
 * them into the block's losses, argmax and gradient in place, and two GEMMs
 * give the block's grad_hidden and add its share to grad_weight.  The logits
 * are formed once (tensor work 6 N V H instead of 8 N V H) at the cost of an
 * [chunk_rows, V] fp32 logits block in device memory and a read-modify-write
 * of the fp32 grad_weight for every block after the first.  Its precision is
 * that of flce_fwd_bwd_ex (fp32 logits, 16-bit gradient between the products).
 *
 * chunk_rows   rows per block, >= 1 (VLMCE_ERR_INVALID_ARG otherwise); a value
 *              >= N makes one block.
 * workspace    >= vlmce_flce_rows_workspace_bytes(N, H, V, chunk_rows) bytes,
 *              256-byte aligned.
 * V must not exceed vlmce_ce_max_vocab(VLMCE_F32) (VLMCE_ERR_TOO_LARGE).
 * Every other argument, result and error as flce_fwd_bwd_ex.  Deterministic.
 */
vlmce_status flce_fwd_bwd_rows(const void *hidden, int32_t dtype, int64_t hidden_stride,
                               const void *weight, int64_t weight_stride, const int64_t *labels,
                               int64_t N, int64_t H, int64_t V, int64_t ignore_index,
                               float label_smoothing, float softcap, int32_t reduction,
                               float grad_scale, float *out_loss, int64_t *out_argmax,
                               float *out_reduced, int64_t *out_counts, void *grad_hidden,
                               float *grad_weight, int32_t accumulate_grad_weight,
                               int64_t chunk_rows, void *workspace, size_t workspace_bytes,
                               vlmce_stream_t stream);

/* vlmce_gemm -- vlmce_gemm_bf16 with the operand type as an argument
 * (VLMCE_BF16 or VLMCE_F16; A and B share it). */
vlmce_status vlmce_gemm(const void *A, int32_t a_mn, const void *B, int32_t b_mn, float *C,
                        int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        int32_t accumulate, int32_t dtype, vlmce_stream_t stream);

/*
 * vlmce_gemm_bf16 -- the library's tcgen05 GEMM on its own:
 * C[M, N] (+)= A[M, K] B[N, K]^T, bf16 inputs, fp32 accumulation and output.
 * A is stored K-major ([M, lda], a_mn = 0) or M-major ([K, lda], a_mn = 1);
 * B is stored K-major ([N, ldb], b_mn = 0) or N-major ([K, ldb], b_mn = 1);
 * C is [M, ldc] fp32.  lda, ldb multiples of 8, ldc of 4, pointers 16-byte
 * aligned.  accumulate != 0 adds to C.
 */
vlmce_status vlmce_gemm_bf16(const void *A, int32_t a_mn, const void *B, int32_t b_mn, float *C,
                             int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                             int64_t ldc, int32_t accumulate, vlmce_stream_t stream);

/* Profiling hook of flce_fwd_bwd: like vlmce_profile_events, the next call on
 * this host thread records the two events around its tensor-core work (the
 * statistics GEMM, the row merge and every chunk's three GEMMs; for
 * flce_fwd_bwd_rows every block's GEMMs, cross-entropy call and cast). */
void vlmce_flce_profile_events(void *ev_begin, void *ev_end);

/*
 * ce_fwd_bwd_noalloc -- ce_fwd_bwd without a workspace argument, for callers
 * that cannot allocate device memory (for instance code inside a framework
 * whose allocator owns all device memory, or latency-critical code that
 * cannot afford cudaMalloc's implicit device synchronisation).  The pages have
 * no counterpart of this entry point; it exists for such callers only.
 *
 * Arguments, outputs, errors and results are those of ce_fwd_bwd.  Its
 * scratch is a fixed array of 786,688 bytes in the library's device image
 * (256 B + 12 B per row), which every GPU that loads the library holds until
 * the process exits.  N may not exceed vlmce_ce_noalloc_max_rows() (65536):
 * larger N returns VLMCE_ERR_TOO_LARGE before anything is enqueued.  No
 * device memory is allocated or freed.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress, a host-side query).
 * Every call on a device shares the one array:
 * calls that overlap on the GPU (different streams without ordering between
 * them) race on it and must not be issued; calls ordered on one stream are
 * safe.  The array keeps the last call's contents, none of which a call needs
 * to start at zero.  The looked-up address is kept for the life of the
 * process: the entry point serves the primary context of each device (the
 * one the CUDA runtime uses), and not calls made after cudaDeviceReset.
 */
vlmce_status ce_fwd_bwd_noalloc(void *logits, int32_t dtype, const int64_t *labels, int64_t N,
                                int64_t V, int64_t row_stride, int64_t ignore_index,
                                float label_smoothing, float softcap, int32_t reduction,
                                float grad_scale, float *out_loss, int64_t *out_argmax,
                                float *out_reduced, int64_t *out_counts, vlmce_stream_t stream);

/* Rows ce_fwd_bwd_noalloc accepts (the size of its fixed scratch). */
int64_t vlmce_ce_noalloc_max_rows(void);

/*
 * Profiling hook: the next ce_fwd_bwd call made by this host thread records
 * `ev_begin` immediately before and `ev_end` immediately after its row kernel
 * (the dominant kernel) on the call's stream, then forgets both.  The two
 * arguments are cudaEvent_t handles created by the caller (NULL clears the
 * hook).  Recording the events costs the overlap of that one launch with its
 * neighbours, so time whole calls without the hook.
 */
void vlmce_profile_events(void *ev_begin, void *ev_end);

/* The last failed CUDA call made by this library on this host thread, as
 * "where: cudaErrorName (description)"; "" if none.  Valid until the next
 * failing call on the same thread. */
const char *vlmce_last_error(void);

/* Static, human-readable name of a status code. */
const char *vlmce_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* VLMCE_H_ */
