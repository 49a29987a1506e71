/*
 * ce_oracle.c -- plain fp64 CPU oracle for the fused large-vocabulary LM
 * cross-entropy forward + backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or helper with the CUDA library, and it never imports
 * or calls it.
 *
 * What it computes (sources: "Add Megatron-LM cross-entropy integration",
 * Summary: ignore_index / label_smoothing arguments, online softmax with the
 * gradient written over the logits; "Add opt-in Liger vocab-parallel cross
 * entropy through ops/loss", What does this PR do: fp32 per-token losses,
 * gradient in the incoming dtype, global argmax with smallest-index ties;
 * "Add Liger Kernel support for Muse Glimmer", Summary and Details: token
 * accuracy and the final-logit softcap T*tanh(x/T)).  The pages name the
 * operation as the same one torch.nn.functional.cross_entropy computes, so
 * the label-smoothing target is PyTorch's: q_j = (1-eps)[j=y] + eps/V.
 *
 * Per row r, with x_j the input logit widened exactly to fp64:
 *   t_j = tanh(x_j/T), z_j = T t_j           if softcap T > 0, else z_j = x_j
 *   argmax_r = smallest j with x_j = max_k x_k   (raw input values)
 *   lse = m + ln sum_j exp(z_j - m),  m = max_j z_j
 *   loss_r = lse - (1-eps) z_y - (eps/V) sum_j z_j
 *   g_j = scale (exp(z_j - lse) - q_j) (T > 0 ? 1 - t_j^2 : 1)
 * Rows whose label equals ignore_index: loss 0, gradient 0.
 * Rows whose label is neither ignore_index nor in [0, V) (a caller error):
 * loss NaN, gradient 0 (the library's documented convention).
 *
 * Everything is computed in fp64 in the order written above; there is no
 * blocking, fusion or reordering.  Rows are independent and are spread over
 * POSIX threads; each row is computed by one thread start to finish, so the
 * result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

/* Exact widening of one stored element to fp64. */
static double load_elem(const unsigned char *row, int dtype, int64_t j) {
    if (dtype == ORACLE_F32) {
        float f;
        memcpy(&f, row + 4 * j, 4);
        return (double)f;
    }
    if (dtype == ORACLE_BF16) {
        uint16_t h;
        uint32_t u;
        float f;
        memcpy(&h, row + 2 * j, 2);
        u = (uint32_t)h << 16; /* bf16 is the top half of an fp32 */
        memcpy(&f, &u, 4);
        return (double)f;
    }
    {
        double d;
        memcpy(&d, row + 8 * j, 8);
        return d;
    }
}

static size_t elem_size(int dtype) {
    return dtype == ORACLE_F32 ? 4 : dtype == ORACLE_BF16 ? 2 : 8;
}

typedef struct {
    const unsigned char *x;
    int dtype;
    int64_t n_rows, V, row_stride;
    const int64_t *labels;
    int64_t ignore_index;
    double eps, softcap, scale;
    double *loss;    /* [n_rows] */
    int64_t *argmax; /* [n_rows] */
    double *grad;    /* [n_rows * V] or NULL */
    int64_t row_begin, row_end;
} job_t;

/* One row, start to finish, in the order of the header comment. */
static void one_row(const job_t *jb, int64_t r, double *z, double *t) {
    const unsigned char *row = jb->x + (size_t)r * (size_t)jb->row_stride * elem_size(jb->dtype);
    const int64_t V = jb->V;
    const int64_t y = jb->labels[r];
    double *g = jb->grad ? jb->grad + (size_t)r * (size_t)V : NULL;
    int64_t j, best = 0;
    double xbest = load_elem(row, jb->dtype, 0);

    /* argmax over the raw inputs, first occurrence wins */
    for (j = 1; j < V; ++j) {
        double xj = load_elem(row, jb->dtype, j);
        if (xj > xbest) {
            xbest = xj;
            best = j;
        }
    }
    jb->argmax[r] = best;

    if (y == jb->ignore_index || y < 0 || y >= V) {
        jb->loss[r] = (y == jb->ignore_index) ? 0.0 : NAN;
        if (g)
            for (j = 0; j < V; ++j) g[j] = 0.0;
        return;
    }

    /* softcap */
    for (j = 0; j < V; ++j) {
        double xj = load_elem(row, jb->dtype, j);
        if (jb->softcap > 0.0) {
            t[j] = tanh(xj / jb->softcap);
            z[j] = jb->softcap * t[j];
        } else {
            t[j] = 0.0;
            z[j] = xj;
        }
    }

    /* log-sum-exp */
    double m = z[0];
    for (j = 1; j < V; ++j)
        if (z[j] > m) m = z[j];
    double s = 0.0, sumz = 0.0;
    for (j = 0; j < V; ++j) {
        s += exp(z[j] - m);
        sumz += z[j];
    }
    const double lse = m + log(s);

    /* smoothed-target loss */
    jb->loss[r] = lse - (1.0 - jb->eps) * z[y] - (jb->eps / (double)V) * sumz;

    /* gradient of scale * loss with respect to x */
    if (g) {
        for (j = 0; j < V; ++j) {
            double q = jb->eps / (double)V + (j == y ? 1.0 - jb->eps : 0.0);
            double d = exp(z[j] - lse) - q;
            if (jb->softcap > 0.0) d *= 1.0 - t[j] * t[j];
            g[j] = jb->scale * d;
        }
    }
}

static void *worker(void *arg) {
    job_t *jb = (job_t *)arg;
    double *z = (double *)malloc(sizeof(double) * (size_t)jb->V);
    double *t = (double *)malloc(sizeof(double) * (size_t)jb->V);
    if (!z || !t) {
        free(z);
        free(t);
        return (void *)1;
    }
    for (int64_t r = jb->row_begin; r < jb->row_end; ++r) one_row(jb, r, z, t);
    free(z);
    free(t);
    return NULL;
}

/* Number of threads the oracle uses when asked for 0. */
int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n < 1 ? 1 : (int)n;
}

/*
 * Per-row loss, argmax and (optionally) gradient for n_rows rows.
 * x: n_rows rows of `row_stride` elements of `dtype`; only the first V of each
 * row are read.  scale: the gradient factor of a valid row (grad_scale / n_valid
 * for the mean, grad_scale for the sum; the caller decides, see
 * oracle_ce_scale).  grad (fp64, dense [n_rows, V]) may be NULL.
 * Returns 0 on success, 1 on an argument or allocation error.
 */
int oracle_ce_rows(const void *x, int dtype, int64_t n_rows, int64_t V, int64_t row_stride,
                   const int64_t *labels, int64_t ignore_index, double eps, double softcap,
                   double scale, double *loss, int64_t *argmax, double *grad, int n_threads) {
    if (!x || !labels || !loss || !argmax || V < 1 || n_rows < 0 || row_stride < V) return 1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return 1;
    if (n_rows == 0) return 0;
    if (n_threads <= 0) n_threads = oracle_default_threads();
    if (n_threads > n_rows) n_threads = (int)n_rows;

    job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return 1;
    }
    int rc = 0;
    for (int i = 0; i < n_threads; ++i) {
        job_t *jb = &jobs[i];
        jb->x = (const unsigned char *)x;
        jb->dtype = dtype;
        jb->n_rows = n_rows;
        jb->V = V;
        jb->row_stride = row_stride;
        jb->labels = labels;
        jb->ignore_index = ignore_index;
        jb->eps = eps;
        jb->softcap = softcap;
        jb->scale = scale;
        jb->loss = loss;
        jb->argmax = argmax;
        jb->grad = grad;
        jb->row_begin = n_rows * i / n_threads;
        jb->row_end = n_rows * (i + 1) / n_threads;
        if (pthread_create(&th[i], NULL, worker, jb) != 0) {
            /* run it here instead */
            if (worker(jb) != NULL) rc = 1;
            th[i] = 0;
        }
    }
    for (int i = 0; i < n_threads; ++i) {
        if (th[i]) {
            void *ret = NULL;
            pthread_join(th[i], &ret);
            if (ret != NULL) rc = 1;
        }
    }
    free(jobs);
    free(th);
    return rc;
}

/*
 * Gradient of some columns of some rows when the row's log-sum-exp is known
 * (the full-vocabulary sum is formed elsewhere): the gradient line of
 * one_row(), g_j = scale_r (exp(z_j - lse_r) - q_j) (T > 0 ? 1 - t_j^2 : 1),
 * for x: n_rows x n_cols fp64 logits of columns col[0..n_cols) of a V-wide
 * vocabulary; q_j = eps/V + (col[j] == y_r ? 1 - eps : 0).  Rows whose
 * label is ignore_index or outside [0, V) get zeros.
 */
void oracle_ce_grad_columns(const double *x, int64_t n_rows, int64_t n_cols, const int64_t *col,
                            int64_t V, const int64_t *labels, int64_t ignore_index,
                            const double *lse, const double *scale, double eps, double softcap,
                            double *grad) {
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t y = labels[r];
        const int valid = y != ignore_index && y >= 0 && y < V;
        for (int64_t j = 0; j < n_cols; ++j) {
            double g = 0.0;
            if (valid) {
                const double xj = x[r * n_cols + j];
                double t = 0.0, z = xj;
                if (softcap > 0.0) {
                    t = tanh(xj / softcap);
                    z = softcap * t;
                }
                const double q = eps / (double)V + (col[j] == y ? 1.0 - eps : 0.0);
                g = exp(z - lse[r]) - q;
                if (softcap > 0.0) g *= 1.0 - t * t;
                g *= scale[r];
            }
            grad[r * n_cols + j] = g;
        }
    }
}

/*
 * Label census: n_valid = #labels in [0, V); n_bad = #labels that are neither
 * ignore_index nor in [0, V).  The mean reduction divides by n_valid.
 */
void oracle_ce_count(const int64_t *labels, int64_t n, int64_t V, int64_t ignore_index,
                     int64_t *n_valid, int64_t *n_bad) {
    int64_t v = 0, b = 0;
    for (int64_t r = 0; r < n; ++r) {
        int64_t y = labels[r];
        if (y == ignore_index) continue;
        if (y >= 0 && y < V)
            ++v;
        else
            ++b;
    }
    *n_valid = v;
    *n_bad = b;
}

/*
 * Gradient factor of one valid row: reduction 1 = mean (grad_scale / n_valid,
 * 0 when no row is valid), 2 = sum (grad_scale).
 */
double oracle_ce_scale(int reduction, double grad_scale, int64_t n_valid) {
    if (reduction == 1) return n_valid > 0 ? grad_scale / (double)n_valid : 0.0;
    return grad_scale;
}

/*
 * Reduced loss and token accuracy, summed in row order in fp64.
 * Reduced loss: sum of loss_r over rows whose label is not ignore_index
 * (a bad label's NaN propagates), divided by n_valid for the mean
 * (0 when n_valid = 0).  n_correct = #rows with a label in [0, V) whose
 * argmax equals the label; accuracy = n_correct / n_valid (0 when n_valid = 0).
 */
void oracle_ce_reduce(const double *loss, const int64_t *argmax, const int64_t *labels, int64_t n,
                      int64_t V, int64_t ignore_index, int reduction, double *reduced_loss,
                      double *accuracy, int64_t *n_correct_out) {
    double acc = 0.0;
    int64_t nv = 0, nc = 0;
    for (int64_t r = 0; r < n; ++r) {
        int64_t y = labels[r];
        if (y == ignore_index) continue;
        acc += loss[r];
        if (y >= 0 && y < V) {
            ++nv;
            if (argmax[r] == y) ++nc;
        }
    }
    if (reduction == 1) acc = nv > 0 ? acc / (double)nv : 0.0;
    *reduced_loss = acc;
    *accuracy = nv > 0 ? (double)nc / (double)nv : 0.0;
    *n_correct_out = nc;
}

/*
 * Round fp64 values to bfloat16 bits, round-to-nearest-even, directly from
 * fp64 (no intermediate fp32 rounding).  bf16 keeps 8 significant bits and
 * fp32's exponent range: the quantum of a value in [2^(e-1), 2^e) is
 * 2^(e-8), never finer than the subnormal quantum 2^-133.
 */
void oracle_round_bf16(const double *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        double v = in[i];
        uint16_t sign = signbit(v) ? 0x8000u : 0u;
        if (isnan(v)) {
            out[i] = 0x7fc0u;
            continue;
        }
        double a = fabs(v);
        if (isinf(a) || a == 0.0) {
            out[i] = sign | (isinf(a) ? 0x7f80u : 0u);
            continue;
        }
        int e;
        (void)frexp(a, &e);
        int qexp = e - 8;
        if (qexp < -133) qexp = -133;
        double k = nearbyint(ldexp(a, -qexp)); /* default mode: ties to even */
        float f = (float)ldexp(k, qexp);       /* exact, or +inf past the top */
        uint32_t u;
        memcpy(&u, &f, 4);
        out[i] = sign | (uint16_t)(u >> 16);
    }
}
