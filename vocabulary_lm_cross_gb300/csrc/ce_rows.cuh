// ce_rows.cuh -- the cross-entropy row kernel (default path): one CTA per
// row; 1024 threads (two CTAs, 64 warps per SM) for long rows, 256 threads
// (eight CTAs per SM) for rows of at most kShortGranules granules and (five
// per SM, for their registers) for softcap rows, 128 threads (sixteen per SM)
// for rows of at most kTinyGranules granules.
//
//   pass 1: stream the row from HBM in 16-byte granules: max and first argmax
//           of the raw logits, online sum of exp(z - m) and sum of z;
//   merge:  warp shuffles, then the warp partials (fixed order);
//   pass 2: read the row again, last granule first (the lines pass 1 read
//           last are the likeliest still in L2) -- without a softcap it is
//           mostly still in the 129 MB L2, since at most 2 x 152 rows (78 MB
//           for 256 KB rows) are in flight; softcap rows exceed L2 and are
//           prefetched into it ahead, two granules in flight per thread --
//           and store the gradient scale (p - q) (1 - t^2), rounded to the
//           storage dtype, with 16-byte evict-first stores over the logits.
// Without a softcap HBM sees about one read and one write of every byte.
// The label census of the call is only needed by pass 2, so the kernel waits
// for it (programmatic dependent launch) after pass 1, in one warp while
// another merges the warp partials.
//
// Pass 1 keeps two 16-byte loads in flight per thread and prefetches the
// next iteration's pair into L2, so that enough bytes are outstanding per SM
// to cover the DRAM latency.  Its arithmetic is the rest of its cost.  With
// 16 to 80 granules per thread some lane of a warp meets a new maximum in
// most granules, so the branch a new maximum takes (new_max) is kept short:
// the reference of the exponentials moves lazily, and softcap rows, whose
// pass 1 is bound by instruction issue, record only the granule of the
// first maximum -- the column within it is found once per row, after the
// merge (first_max_col); so do forward-only calls, which have no pass 2.
// With a gradient, rows without a softcap locate the column in new_max:
// measured on GB300, deferring it there saved 29 % of the instructions but
// cost 4-6 % of the time (more of pass 2 missed L2).
// Instruction issue bounds the kernel (softcap rows at full size: DRAM, with
// the pass-2 re-reads), so the inner loops run over whole
// granules only, with no per-element tests: the at most two partial granules
// at the ends of a row are handled apart (the first one before a thread's
// main loop, the last one after it, so every thread still meets its granules
// in column order), the label column's gradient is stored over the smoothed
// value after pass 2's loop by the thread that owns it, and the sum of z is
// only formed when label smoothing needs it.
#pragma once

#include <type_traits>

#include "ce_common.cuh"

namespace vlmce {
namespace ce {
namespace rows {

// CTA sizes: 1024 threads for long rows, 256 (eight CTAs per SM) for rows of
// at most kShortGranules 16-byte granules, so that every thread still folds
// several granules per row.
constexpr int kThreads = 1024;
constexpr int kShortThreads = 256;
constexpr int kShortGranules = 8192;
// Rows of at most kTinyGranules granules (16384 bf16 columns, e.g. one
// tensor-parallel shard of a 128K vocabulary): 128-thread CTAs, sixteen per
// SM, so that 2432 rows run in a single wave.
constexpr int kTinyThreads = 128;
constexpr int kTinyGranules = 2048;
// CTAs per SM the launch bounds ask for (the softcap variants need more
// registers per thread: 48 at five 256-thread CTAs per SM, which also keeps
// fewer softcap rows in flight for L2 to hold until pass 2).
constexpr int min_blocks(int threads, bool softcap) {
    return threads == kThreads ? (softcap ? 1 : 2)
                               : threads == kTinyThreads ? 16 : (softcap ? 5 : 8);
}

// What the merge hands every thread of the row: lse, the row's maximum with
// its first column (deferred: the first column of its granule), and the
// row's gradient scale.
struct RowBcast {
    float lse, mx;
    int idx;
    float scale;
};

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
    const int64_t *counts;      // [0] n_valid (written by the count kernel)
    const float *token_scale;   // [N] per-row factor of the gradient, or null
    int want_grad;              // 0: forward only, the logits are not written
};

using Kernel = void (*)(Params);

__device__ __forceinline__ uint4 ld_v4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Pass-1 state of one thread.  The sums run over even and odd columns in
// the two halves of packed fp32x2 registers.
struct Acc {
    float mv;    // max raw logit seen
    int midx;    // first column of mv; softcap rows: first column of its granule
    float mz;    // reference of s, at least the largest z seen
    float nmL;   // -mz log2e
    float xthr;  // largest x whose z mz is known to cover
    uint64_t s;  // sums of exp(z - mz) (even, odd columns)
    uint64_t z;  // sums of z, or of tanh(x/T) when a softcap is set (even, odd columns)
};

__device__ __forceinline__ void acc_init(Acc &a) {
    a.mv = -INFINITY;
    a.midx = INT_MAX;
    a.mz = -INFINITY;
    a.nmL = INFINITY;
    a.xthr = -INFINITY;
    a.s = a.z = pk(0.f, 0.f);
}

// The thread's statistics as a RowPart (sum of z scaled back by T under a softcap).
template <bool SOFTCAP>
__device__ __forceinline__ RowPart acc_part(const Acc &a, float T) {
    RowPart pt = part_identity();
    float s0, s1, z0, z1;
    upk(a.s, s0, s1);
    upk(a.z, z0, z1);
    pt.mx = a.mv;
    pt.idx = a.midx;  // softcap rows: a granule's first column, resolved by first_max_col
    pt.mz = a.mz;
    pt.s = s0 + s1;
    pt.sz = SOFTCAP ? T * (z0 + z1) : z0 + z1;
    return pt;
}

// The softcap's constants of a thread: T, -2 log2e / T and the polynomial's.
struct CapK {
    float T, k2;
    PolyCap pc;
    float q[5];  // tanh(x/T) = x Q(x^2) within the polynomial's range: Q's coefficients
};
template <bool SOFTCAP>
__device__ __forceinline__ CapK cap_k(float T) {
    CapK k;
    k.T = T;
    k.k2 = SOFTCAP ? -2.f * kLog2e / T : 0.f;
    k.pc = SOFTCAP ? poly_cap(T) : PolyCap{};
    // tanh(u)/u = P(u^2), u = x / T: Q's i-th coefficient is P's divided by T^(2i+1)
    const float c[5] = {kTanhP0, kTanhP1, kTanhP2, kTanhP3, kTanhP4};
    const float r = SOFTCAP ? k.pc.rT : 0.f, r2 = r * r;
    float f = r;
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        k.q[i] = c[i] * f;
        f *= r2;
    }
    return k;
}
// tanh(x/T) of two columns (each |x| <= 0.55 T) by the polynomial.
__device__ __forceinline__ uint64_t tanh_q2(uint64_t x, const CapK &k) {
    const uint64_t s = mul2(x, x);
    uint64_t a = fma2(pk(k.q[4], k.q[4]), s, pk(k.q[3], k.q[3]));
    a = fma2(a, s, pk(k.q[2], k.q[2]));
    a = fma2(a, s, pk(k.q[1], k.q[1]));
    a = fma2(a, s, pk(k.q[0], k.q[0]));
    return mul2(x, a);
}
// tanh(x/T) of one column: the polynomial within its range, else softcap2's arithmetic.
__device__ __forceinline__ float cap_t_any(float x, const CapK &k) {
    if (fabsf(x) <= k.pc.lim) {
        float t0, t1;
        upk(tanh_q2(pk(x, x), k), t0, t1);
        return t0;
    }
    return softcap_t1(x, k.k2);
}

// z of one column: the logit, or T tanh(x/T) under a softcap.
template <bool SOFTCAP>
__device__ __forceinline__ float z_of(float x, const CapK &k) {
    if constexpr (SOFTCAP)
        return k.T * cap_t_any(x, k);
    else
        return x;
}

// Margin (natural-log units) by which the sums' reference is set above a new
// maximum, so that later maxima seldom move it: every term exp(z - mz) stays
// <= 1, and one below e^-8 loses nothing (fp32 precision is relative).
constexpr float kRefMargin = 8.f;

// New maximum gm in the granule starting at column jg: record its first
// column (DEFER: the granule's first column); only when gm passes
// xthr, move the reference of the running sums to z(gm) + kRefMargin and
// rescale them.  (z grows no faster than x, so mz covers every x <= gm +
// kRefMargin.)
template <bool BF16, bool SOFTCAP, bool DEFER>
__device__ __forceinline__ void new_max(Acc &a, const float (&x)[Elem<BF16>::kPerGranule],
                                        float gm, int jg, int V, const CapK &k) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    a.mv = gm;
    if constexpr (DEFER) {
        a.midx = jg;
    } else {
        int li = EPG - 1;
#pragma unroll
        for (int l = EPG - 1; l >= 0; --l)
            if (x[l] == gm && jg + l >= 0 && jg + l < V) li = l;
        a.midx = jg + li;
    }
    if (gm > a.xthr) {
        const float nz = z_of<SOFTCAP>(gm, k) + kRefMargin;
        const float f = ptx::ex2((a.mz - nz) * kLog2e);
        float s0, s1;
        upk(a.s, s0, s1);
        s0 = (s0 == 0.f) ? 0.f : s0 * f;
        s1 = (s1 == 0.f) ? 0.f : s1 * f;
        a.s = pk(s0, s1);
        a.mz = nz;
        a.nmL = -nz * kLog2e;
        a.xthr = gm + kRefMargin;
    }
}

// A softcap row's argmax from its merged statistics: the first column in
// [0, V) of granule w (first column jg) that holds the maximum mv.  Threads visit
// their granules in column order and keep the first granule that reaches
// their maximum, and the merges keep the smallest granule among equal
// maxima, so this is the smallest column holding the row's maximum.
template <bool BF16>
__device__ __forceinline__ int first_max_col(const uint4 w, float mv, int jg, int V) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    float x[EPG];
    unpack<BF16>(w, x);
    int li = EPG - 1;
#pragma unroll
    for (int l = EPG - 1; l >= 0; --l)
        if (x[l] == mv && jg + l >= 0 && jg + l < V) li = l;
    return jg + li;
}

// Fold a whole granule (every column valid), two columns per packed op.
// Under a softcap the exponent is t (T log2e) - mz log2e with t = tanh(x/T),
// by the polynomial when the whole granule is within its range (else ok is
// cleared and softcap2 is used).
template <bool BF16, bool SOFTCAP, bool SUMZ, bool DEFER = SOFTCAP>
__device__ __forceinline__ void fold_full(Acc &a, const uint4 w, int jg, int V, const CapK &k,
                                          bool &ok) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    float x[EPG];
    unpack<BF16>(w, x);
    const float gm = granule_max<BF16>(w);
    if (gm > a.mv) new_max<BF16, SOFTCAP, DEFER>(a, x, gm, jg, V, k);
    const float L = SOFTCAP ? k.T * kLog2e : kLog2e;
    const uint64_t L2 = pk(L, L), nmL2 = pk(a.nmL, a.nmL);
    if constexpr (SOFTCAP) {
        if (granule_in_poly_range<BF16>(w, k.pc)) {
#pragma unroll
            for (int l = 0; l < EPG; l += 2) {
                const uint64_t v = tanh_q2(pk(x[l], x[l + 1]), k);
                a.s = add2(a.s, ex2x2(fma2(v, L2, nmL2)));
                if constexpr (SUMZ) a.z = add2(a.z, v);
            }
            return;
        }
        ok = false;
    }
#pragma unroll
    for (int l = 0; l < EPG; l += 2) {
        uint64_t v;
        if constexpr (SOFTCAP)
            v = softcap2(x[l], x[l + 1], k.k2).t;
        else
            v = pk(x[l], x[l + 1]);
        a.s = add2(a.s, ex2x2(fma2(v, L2, nmL2)));
        if constexpr (SUMZ) a.z = add2(a.z, v);
    }
}

// Fold a granule of which only the columns in [0, V) count (into the even sums).
template <bool BF16, bool SOFTCAP, bool DEFER = SOFTCAP>
__device__ __forceinline__ void fold_partial(Acc &a, const uint4 w, int jg, int V, const CapK &k) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    float x[EPG];
    unpack<BF16>(w, x);
    float gm = -INFINITY;
#pragma unroll
    for (int l = 0; l < EPG; ++l)
        if (jg + l >= 0 && jg + l < V) gm = fmaxf(gm, x[l]);
    if (gm > a.mv) new_max<BF16, SOFTCAP, DEFER>(a, x, gm, jg, V, k);
    const float L = SOFTCAP ? k.T * kLog2e : kLog2e;
    float s0, s1, z0, z1;
    upk(a.s, s0, s1);
    upk(a.z, z0, z1);
#pragma unroll
    for (int l = 0; l < EPG; ++l) {
        if (jg + l >= 0 && jg + l < V) {
            const float v = SOFTCAP ? cap_t_any(x[l], k) : x[l];
            s0 += ptx::ex2(fmaf(v, L, a.nmL));
            z0 += v;
        }
    }
    a.s = pk(s0, s1);
    a.z = pk(z0, z1);
}

struct GradCoef {
    float nlseL;     // -lse log2e (+ the exponent bias)
    float scale;     // coefficient of 2^e: the row scale (times 2^-bias)
    float c_smooth;  // scale eps / V (unbiased row scale)
    float c_label;   // scale (1 - eps + eps / V)
    CapK k;          // the softcap's constants
};

// GradCoef of a row with this lse and (unbiased) scale; the softcap's
// constants set apart.
__device__ __forceinline__ void set_coef(GradCoef &c, float lse, float scale, float eps, int V) {
    c.c_smooth = scale * (eps / static_cast<float>(V));
    c.c_label = c.c_smooth + scale * (1.f - eps);
    const ExpCoef ec = grad_exp_coef(lse, scale);
    c.nlseL = ec.nlseL;
    c.scale = ec.scale;
}

// Gradient of one column with target term q_coef = scale q_j (c_smooth, or
// c_label at the label): under a softcap by the polynomial within its range
// (g = scale (p - q) (1 - t^2)), else by softcap2 (g = 4 scale (p - q) a r^2,
// the factor 4 of dz/dx = 4 a r^2 folded into the coefficients, exactly).
template <bool SOFTCAP>
__device__ __forceinline__ float column_grad(float x, float q_coef, const GradCoef &c) {
    if constexpr (SOFTCAP) {
        const float L = c.k.T * kLog2e;
        if (fabsf(x) <= c.k.pc.lim) {
            float t, t_;
            upk(tanh_q2(pk(x, x), c.k), t, t_);
            const float pr = ptx::ex2(fmaf(t, L, c.nlseL));
            return fmaf(pr, c.scale, -q_coef) * fmaf(-t, t, 1.f);
        }
        const Cap2 cz = softcap2(x, x, c.k.k2);
        float t, t_, ar2, ar2_;
        upk(cz.t, t, t_);
        upk(cz.ar2, ar2, ar2_);
        const float pr = ptx::ex2(fmaf(t, L, c.nlseL));
        return fmaf(pr, 4.f * c.scale, -4.f * q_coef) * ar2;
    } else {
        const float pr = ptx::ex2(fmaf(x, kLog2e, c.nlseL));
        return fmaf(pr, c.scale, -q_coef);
    }
}
// Gradient of the label column: q_y = 1 - eps + eps/V.
template <bool SOFTCAP>
__device__ __forceinline__ float label_grad(float x, const GradCoef &c) {
    return column_grad<SOFTCAP>(x, c.c_label, c);
}

// How pass 2 forms the softcap's tanh of a granule: the polynomial if the
// whole granule is within its range, else softcap2 (kCapCheck: the decision
// pass 1 took for the same granule); the polynomial without the test
// (kCapPoly: pass 1 found every whole granule of the row in range); column by
// column (kCapColumn: the partial granules at the ends of a row, which pass 1
// also folds column by column).
enum CapMode : int { kCapCheck = 0, kCapPoly = 1, kCapColumn = 2 };

// Gradients of the EPG elements of a granule, in fp32, two per packed op;
// label_lane >= 0: the label column's lane.
template <bool BF16, bool SOFTCAP, int MODE = kCapCheck>
__device__ __forceinline__ void grad_values(const uint4 w, const GradCoef &c, int label_lane,
                                            float (&g)[Elem<BF16>::kPerGranule]) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    float x[EPG];
    unpack<BF16>(w, x);
    const float L = SOFTCAP ? c.k.T * kLog2e : kLog2e;
    const uint64_t L2 = pk(L, L), nlseL2 = pk(c.nlseL, c.nlseL);
    if constexpr (SOFTCAP && MODE == kCapColumn) {
#pragma unroll
        for (int l = 0; l < EPG; ++l) g[l] = column_grad<SOFTCAP>(x[l], c.c_smooth, c);
    } else if (SOFTCAP && (MODE == kCapPoly || granule_in_poly_range<BF16>(w, c.k.pc))) {
        // g = (c_smooth - scale p) (t^2 - 1) = scale (p - q) (1 - t^2)
        const uint64_t nscale2 = pk(-c.scale, -c.scale), c2 = pk(c.c_smooth, c.c_smooth);
        const uint64_t m_one = pk(-1.f, -1.f);
#pragma unroll
        for (int l = 0; l < EPG; l += 2) {
            const uint64_t t = tanh_q2(pk(x[l], x[l + 1]), c.k);
            const uint64_t g2 =
                mul2(fma2(ex2x2(fma2(t, L2, nlseL2)), nscale2, c2), fma2(t, t, m_one));
            upk(g2, g[l], g[l + 1]);
        }
    } else {
        const float f = SOFTCAP ? 4.f : 1.f;
        const uint64_t scale2 = pk(f * c.scale, f * c.scale);
        const uint64_t nc2 = pk(-f * c.c_smooth, -f * c.c_smooth);
#pragma unroll
        for (int l = 0; l < EPG; l += 2) {
            uint64_t g2;
            if constexpr (SOFTCAP) {
                const Cap2 cz = softcap2(x[l], x[l + 1], c.k.k2);
                g2 = mul2(fma2(ex2x2(fma2(cz.t, L2, nlseL2)), scale2, nc2), cz.ar2);
            } else {
                g2 = fma2(ex2x2(fma2(pk(x[l], x[l + 1]), L2, nlseL2)), scale2, nc2);
            }
            upk(g2, g[l], g[l + 1]);
        }
    }
    if (label_lane >= 0) {  // the label column (rare)
#pragma unroll
        for (int l = 0; l < EPG; ++l)
            if (l == label_lane) g[l] = label_grad<SOFTCAP>(x[l], c);
    }
}

template <bool BF16>
__device__ __forceinline__ uint4 pack_granule(const float (&g)[Elem<BF16>::kPerGranule]) {
    if constexpr (BF16) {
        return make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]),
                          pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7]));
    } else {
        return make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                          __float_as_uint(g[3]));
    }
}

// Store only the elements of a partial granule that lie in [0, V).
template <bool BF16>
__device__ __forceinline__ void store_partial(unsigned char *dst, int jg, int V,
                                              const float (&g)[Elem<BF16>::kPerGranule]) {
    constexpr int EPG = Elem<BF16>::kPerGranule;
    constexpr int ELT = Elem<BF16>::kBytes;
#pragma unroll
    for (int l = 0; l < EPG; ++l)
        if (jg + l >= 0 && jg + l < V) store_elem<BF16>(dst + ELT * l, g[l]);
}

template <bool BF16, bool SOFTCAP, bool SUMZ, int THREADS, bool DEFER>
__device__ __forceinline__ void row_work(const Params &p, RowPart *wpart, RowBcast *bc) {
    constexpr int kWarps = THREADS / 32;
    constexpr int EPG = Elem<BF16>::kPerGranule;
    constexpr int ELT = Elem<BF16>::kBytes;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p.logits) + r * p.stride_bytes;
    unsigned char *gbase = reinterpret_cast<unsigned char *>(a0 & ~static_cast<uintptr_t>(15));
    const uint4 *row = reinterpret_cast<const uint4 *>(gbase);
    const int lead = static_cast<int>((a0 & 15) / ELT);
    const int G = (lead + p.V + EPG - 1) / EPG;
    // Whole granules are [gs, ge); granule 0 is partial when lead > 0 and
    // granule G - 1 when the row does not end on a granule boundary.
    const int gs = lead > 0 ? 1 : 0;
    const int ge = ((lead + p.V) % EPG != 0) ? G - 1 : G;
    const bool head = gs == 1;                     // granule 0 partial (thread 0)
    const bool tail = ge == G - 1 && G - 1 >= gs;  // granule G-1 partial, distinct from 0
    const int tail_tid = tail ? (G - 1 - gs) % THREADS : -1;
    const float T = p.softcap;
    const CapK k = cap_k<SOFTCAP>(T);
    // Pass 2 walks the row backwards, so that it starts on the lines pass 1
    // read last, the ones most likely still in L2.  Where the rows in flight
    // exceed L2 -- softcap rows (five 256-thread CTAs per SM, up to 760 rows
    // in flight) -- it keeps two granules in flight and prefetches ahead.
    constexpr bool kAhead2 = SOFTCAP;

    // ---- pass 1
    Acc a;
    acc_init(a);
    bool poly_ok = true;  // every whole granule of this thread took the polynomial softcap
    if (head && tid == 0) fold_partial<BF16, SOFTCAP, DEFER>(a, ld_v4(row), -lead, p.V, k);
    // two granules in flight per thread (the loads of a warp would otherwise
    // leave too few bytes outstanding to cover the DRAM latency); the folds
    // keep the thread's column order
    int gl = gs + tid;
    for (; gl + THREADS < ge; gl += 2 * THREADS) {
        const uint4 w0 = ld_v4(row + gl), w1 = ld_v4(row + gl + THREADS);
        if (gl + 3 * THREADS < ge) {  // the next iteration's pair, into L2
            ptx::prefetch_l2(row + gl + 2 * THREADS);
            ptx::prefetch_l2(row + gl + 3 * THREADS);
        }
        fold_full<BF16, SOFTCAP, SUMZ, DEFER>(a, w0, gl * EPG - lead, p.V, k, poly_ok);
        fold_full<BF16, SOFTCAP, SUMZ, DEFER>(a, w1, (gl + THREADS) * EPG - lead, p.V, k, poly_ok);
    }
    for (; gl < ge; gl += THREADS)
        fold_full<BF16, SOFTCAP, SUMZ, DEFER>(a, ld_v4(row + gl), gl * EPG - lead, p.V, k, poly_ok);
    if (tid == tail_tid)
        fold_partial<BF16, SOFTCAP, DEFER>(a, ld_v4(row + (G - 1)), (G - 1) * EPG - lead, p.V, k);

    RowPart pt = acc_part<SOFTCAP>(a, T);
    warp_allreduce(pt);
    if (lane == 0) wpart[warp] = pt;

    const int64_t y = p.labels[r];
    const bool ignored = (y == p.ignore_index);
    const bool valid = !ignored && y >= 0 && y < p.V;
    // every whole granule of the row took the polynomial softcap in pass 1
    const bool row_poly = __syncthreads_and(poly_ok) != 0;
    if (warp == 0) {
        // the label's logit, loaded while the warp merges
        float xy = 0.f;
        if (lane == 0 && valid) {
            const unsigned char *py = reinterpret_cast<const unsigned char *>(a0) + ELT * y;
            if constexpr (BF16)
                xy = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(py)) << 16);
            else
                xy = *reinterpret_cast<const float *>(py);
        }
        RowPart q = lane < kWarps ? wpart[lane] : part_identity();
        warp_allreduce(q);
        if (lane == 0) {
            const float lse = q.mz + logf(q.s);
            float l = 0.f;
            if (valid) {
                const float zy = z_of<SOFTCAP>(xy, k);
                l = lse - fmaf(1.f - p.eps, zy, (p.eps / static_cast<float>(p.V)) * q.sz);
            } else if (!ignored) {
                l = __int_as_float(0x7fc00000);  // bad label: NaN
            }
            p.loss[r] = l;
            if (!DEFER || q.idx == INT_MAX) p.argmax[r] = q.idx;  // INT_MAX: every logit -inf or NaN
            bc->lse = lse;
            bc->mx = q.mx;
            bc->idx = q.idx;
        }
    } else if (warp == 1 && lane == 0 && valid && p.want_grad) {
        // meanwhile the row's gradient scale, from the label census of this
        // call (waited for here; every thread waits again below)
        ptx::griddep_wait();
        float scale = p.grad_scale;
        if (p.reduction == VLMCE_MEAN) {
            const int64_t n_valid = p.counts[0];
            scale = n_valid > 0 ? p.grad_scale / static_cast<float>(n_valid) : 0.f;
        }
        if (p.token_scale) scale *= p.token_scale[r];
        bc->scale = scale;
    }
    __syncthreads();
    // DEFER: the argmax column; the granule of the row's first maximum is
    // resolved by the thread that stores it in pass 2 (under every branch
    // below), before it does so; so no other thread writes it, and no barrier
    // waits for the load.
    if (DEFER && bc->idx != INT_MAX) {
        const int gb = (bc->idx + lead) / EPG;
        const bool rev = valid && p.want_grad;  // pass 2 proper walks backwards, the zeroing forwards
        const int owner = (head && gb == 0)       ? 0
                          : (tail && gb == G - 1) ? tail_tid
                                                  : (rev ? ge - 1 - gb : gb - gs) % THREADS;
        if (tid == owner) p.argmax[r] = first_max_col<BF16>(ld_v4(row + gb), bc->mx, bc->idx, p.V);
    }
    // The label census of this call, which pass 2 reads.  Every CTA waits (not
    // only those that read it), so the grid completes after the census: the
    // finalize kernel, launched dependent on this grid, reads its counts.
    ptx::griddep_wait();
    if (!p.want_grad) return;  // forward only

    // ---- pass 2
    if (valid) {
        GradCoef c;
        set_coef(c, bc->lse, bc->scale, p.eps, p.V);
        c.k = k;
        const int gy = static_cast<int>((y + lead) / EPG);
        const int ly = static_cast<int>((y + lead) % EPG);
        // The label column in a whole granule: the thread that owns the
        // granule reads x_y now (the loop overwrites it), stores the granule
        // like any other in the loop, then overwrites the one element with the
        // label gradient, so the loop itself has no label test.
        const int y_owner =
            (gy >= gs && gy < ge) ? (ge - 1 - gy) % THREADS : -1;
        unsigned char *py = gbase + ELT * (static_cast<int64_t>(y) + lead);
        float xy = 0.f;
        if (tid == y_owner) {
            if constexpr (BF16)
                xy = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(py)) << 16);
            else
                xy = *reinterpret_cast<const float *>(py);
        }
        float g[EPG];
        if (head && tid == 0) {
            grad_values<BF16, SOFTCAP, kCapColumn>(ld_v4(row), c, gy == 0 ? ly : -1, g);
            store_partial<BF16>(gbase, -lead, p.V, g);
        }
        // the whole granules: without the range test when pass 1 found the
        // whole row within the polynomial's range
        auto whole = [&](auto mode) {
            constexpr int M = decltype(mode)::value;
            int gl = ge - 1 - tid;
            if constexpr (kAhead2) {
                for (; gl - THREADS >= gs; gl -= 2 * THREADS) {
                    // the pair two iterations ahead, into L2 (the row has partly
                    // left L2 since pass 1)
                    if (gl - 3 * THREADS >= gs) {
                        ptx::prefetch_l2(row + gl - 2 * THREADS);
                        ptx::prefetch_l2(row + gl - 3 * THREADS);
                    }
                    const uint4 w0 = ld_v4(row + gl), w1 = ld_v4(row + gl - THREADS);
                    grad_values<BF16, SOFTCAP, M>(w0, c, -1, g);
                    ptx::st_global_cs_v4(gbase + 16 * gl, pack_granule<BF16>(g));
                    grad_values<BF16, SOFTCAP, M>(w1, c, -1, g);
                    ptx::st_global_cs_v4(gbase + 16 * (gl - THREADS), pack_granule<BF16>(g));
                }
            }
            for (; gl >= gs; gl -= THREADS) {
                grad_values<BF16, SOFTCAP, M>(ld_v4(row + gl), c, -1, g);
                ptx::st_global_cs_v4(gbase + 16 * gl, pack_granule<BF16>(g));
            }
        };
        if (!SOFTCAP || row_poly)
            whole(std::integral_constant<int, kCapPoly>{});
        else
            whole(std::integral_constant<int, kCapCheck>{});
        if (tid == y_owner) store_elem<BF16>(py, label_grad<SOFTCAP>(xy, c));
        if (tid == tail_tid) {
            grad_values<BF16, SOFTCAP, kCapColumn>(ld_v4(row + (G - 1)), c, gy == G - 1 ? ly : -1,
                                                   g);
            store_partial<BF16>(gbase + 16 * (G - 1), (G - 1) * EPG - lead, p.V, g);
        }
    } else {
        float z[EPG];
#pragma unroll
        for (int l = 0; l < EPG; ++l) z[l] = 0.f;
        if (head && tid == 0) store_partial<BF16>(gbase, -lead, p.V, z);
        for (int gl = gs + tid; gl < ge; gl += THREADS)
            ptx::st_global_cs_v4(gbase + 16 * gl, make_uint4(0u, 0u, 0u, 0u));
        if (tid == tail_tid) store_partial<BF16>(gbase + 16 * (G - 1), (G - 1) * EPG - lead, p.V, z);
    }
}

// Long rows: two CTAs of 1024 threads per SM (32 registers per thread); short
// rows: eight CTAs of 256.  Softcap rows: 256-thread CTAs, five per SM (48
// registers).
template <bool BF16, bool SOFTCAP, int THREADS, bool DEFER = SOFTCAP>
__global__ void __launch_bounds__(THREADS, min_blocks(THREADS, SOFTCAP)) ce_rows_kernel(const Params p) {
    __shared__ RowPart wpart[THREADS / 32];
    __shared__ RowBcast bcast;
    // the finalize kernel (launched dependent on this grid, and waiting for it
    // before it reads anything) may be scheduled once every CTA has started
    ptx::griddep_launch_dependents();
    // sum z only matters with label smoothing; skip the adds without it
    if (p.eps > 0.f)
        row_work<BF16, SOFTCAP, true, THREADS, DEFER>(p, wpart, &bcast);
    else
        row_work<BF16, SOFTCAP, false, THREADS, DEFER>(p, wpart, &bcast);
}

// Granules (16 B) of a row: exact when every row starts on a 16-byte boundary,
// else the worst case over the possible offsets of its first element.
inline int64_t row_granules(bool bf16, int64_t V, bool aligned_rows) {
    const int64_t epg = bf16 ? 8 : 4;
    return aligned_rows ? (V + epg - 1) / epg : (epg - 1 + V + epg - 1) / epg;
}
inline bool rows_aligned(const void *logits, int64_t row_stride, int64_t elt) {
    return (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && ((row_stride * elt) % 16) == 0;
}

// CTA size of the row kernel for rows of G granules (with or without a softcap).
// Softcap rows always take 256-thread CTAs: five of them per SM keep more
// warps resident than one CTA of 1024 at 64 registers, and their barriers
// stall fewer warps at a time.
inline int threads_for(int64_t G, bool softcap) {
    if (!softcap && G <= kTinyGranules) return kTinyThreads;
    return (softcap || G <= kShortGranules) ? kShortThreads : kThreads;
}
// The row kernel for the given softcap, CTA size and mode (forward only: the
// argmax column deferred also without a softcap), per element type
// (ce_rows_bf16.cu, ce_rows_f32.cu).
Kernel kernel_bf16(bool softcap, int threads, bool fwd_only);
Kernel kernel_f32(bool softcap, int threads, bool fwd_only);

}  // namespace rows
}  // namespace ce
}  // namespace vlmce
