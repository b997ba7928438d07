/*
 * ce_oracle.c -- plain fp64 CPU oracle for softmax cross-entropy, forward and
 * backward, over a [n_rows, vocab] logits matrix.
 *
 * TEST INFRASTRUCTURE ONLY. This file is used by the tests, by the smoke
 * check and by the CPU-baseline leg of the benchmark. The CUDA library never
 * links, loads or calls it, and it shares no code with the CUDA library.
 *
 * What it computes (the plain definition, written out row by row in double
 * precision; the GPU method reaches the same values, it does not approximate):
 *
 *   valid row i: target t_i != ignore_index and 0 <= t_i < V
 *   m_i   = max_c x_ic
 *   S_i   = sum_c exp(x_ic - m_i),  LSE_i = m_i + log S_i
 *   lp_ic = x_ic - LSE_i                      (log-softmax)
 *   loss_i = -(1-eps) * w_{t_i} * lp_{i,t_i} - (eps/V) * sum_c w_c * lp_ic
 *   loss_i = 0 for rows that are not valid
 *   p_ic  = exp(lp_ic)
 *   dL/dx_ic = s_i * [ (1-eps) * w_{t_i} * (p_ic - [c == t_i])
 *                      + (eps/V) * (p_ic * W_all - w_c) ],   0 on invalid rows
 *   W_all = sum_c w_c,   W_y = sum_{valid i} w_{t_i}
 *   s_i = g / W_y (mean), g (sum), g_i (none)
 *
 * Sources (pages, sections):
 *  - Liger-Kernel PR #1268, review diff: the smoothing term "X_block += -eps"
 *    subtracted from every gradient element and the weighted gradient
 *    "(1 - label_smoothing) * softmax_X" with (1 - label_smoothing) taken
 *    off at the true class.
 *  - Liger-Kernel PR #1622, Summary: eps = label_smoothing / V multiplies the
 *    class-weight sum; mean divides by the non-ignored count or the
 *    target-weight sum; sum and none do not divide.
 *  - Liger-Kernel commit #1329 (quoted on PR #1268): dx_y = (softmax(x_y) - 1)/N
 *    at eps = 0, w = 1.
 *  - TransformerEngine PR #2325, description and sequence diagram: the
 *    gradient is formed in fp32 (here: fp64) from the saved row statistics
 *    m, d, X_y and the smoothing sum.
 *  Mean with every row ignored is read as loss 0, gradient 0 (the pages are
 *  silent there; this oracle and the CUDA path agree on that reading).
 *
 * Options (next to the method on the Liger-Kernel #1268 page, whose CE suite
 * covers "class weights, softcap, label smoothing, z-loss, and ignore_index"
 * and whose dx_y correction keeps "softcap factors"; the pages name them but
 * do not define them, so the plain definitions are taken):
 *   softcap c > 0: every logit is replaced by z = c * tanh(x / c) before the
 *     loss; the gradient with respect to x is the gradient with respect to z
 *     times dz/dx = 1 - tanh^2(x / c).
 *   z-loss lambda > 0: loss_i += lambda * LSE_i^2 on valid rows (LSE over the
 *     capped logits), reduced like the other terms; its gradient adds
 *     s_i * 2 * lambda * LSE_i * p_ic.
 *   argmax: the first column holding the row maximum (token accuracy is the
 *     share of valid rows whose argmax is the target).
 *
 * Per-row statistics returned for the forward/backward split:
 *   stats[i] = { m_i, s_i, x_{i,t_i}, r_i } with
 *   s_i = sum_{c != t_i} exp(x_ic - m_i)   (all c on invalid rows)
 *   r_i = sum_c w_c * (x_ic - m_i)         (the smoothing sum, relative to m)
 *   x_{i,t_i} = 0 on invalid rows.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2, OR_F64 = 3 };
enum { OR_NONE = 0, OR_MEAN = 1, OR_SUM = 2 };

/* Exact decode of one stored element to double. */
static double or_load(const void *base, int dtype, int64_t idx)
{
    switch (dtype) {
    case OR_F32:
        return (double)((const float *)base)[idx];
    case OR_BF16: {
        /* bfloat16 is the upper half of an IEEE binary32 */
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    case OR_F16: {
        /* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits */
        uint16_t h = ((const uint16_t *)base)[idx];
        int sign = (h >> 15) & 1;
        int e = (h >> 10) & 0x1f;
        int f = h & 0x3ff;
        double v;
        if (e == 0)
            v = ldexp((double)f, -24);
        else if (e == 31)
            v = f ? NAN : INFINITY;
        else
            v = ldexp((double)(f + 1024), e - 25);
        return sign ? -v : v;
    }
    default:
        return ((const double *)base)[idx];
    }
}

static int64_t or_target(const void *target, int is_int32, int64_t i)
{
    return is_int32 ? (int64_t)((const int32_t *)target)[i] : ((const int64_t *)target)[i];
}

static int or_valid(int64_t t, int64_t ignore_index, int64_t vocab)
{
    return t != ignore_index && t >= 0 && t < vocab;
}

/*
 * Normalisers over all rows: out[0] = number of valid rows, out[1] = W_y,
 * out[2] = W_all (V when unweighted). Returns the number of rows whose target
 * is neither ignore_index nor inside [0, V).
 */
int64_t ce_oracle_normalizers(const void *target, int target_is_int32, int64_t n_rows,
                              int64_t vocab, int64_t ignore_index,
                              const double *class_weight, double *out)
{
    double n = 0.0, wy = 0.0, wall = 0.0;
    int64_t bad = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        int64_t t = or_target(target, target_is_int32, i);
        if (or_valid(t, ignore_index, vocab)) {
            n += 1.0;
            wy += class_weight ? class_weight[t] : 1.0;
        } else if (t != ignore_index) {
            ++bad;
        }
    }
    if (class_weight) {
        for (int64_t c = 0; c < vocab; ++c)
            wall += class_weight[c];
    } else {
        wall = (double)vocab;
    }
    out[0] = n;
    out[1] = wy;
    out[2] = wall;
    return bad;
}

typedef struct {
    double softcap;      /* 0: off */
    double z_loss;       /* lambda, 0: off */
    int64_t *argmax;     /* [n_rows] or NULL */
} or_opts;

typedef struct {
    const void *logits;
    int dtype;
    int64_t vocab, ld;
    const void *target;
    int target_is_int32;
    int64_t ignore_index;
    const double *w;
    double eps;
    int reduction;
    const double *grad_output;
    int grad_output_per_row;
    double norm_wy, w_all;
    double *row_loss, *stats, *grad;
    int64_t row_begin, row_end;
    or_opts opt;
} or_job;

static void or_one_row(const or_job *J, int64_t i, double *xbuf)
{
    const int64_t V = J->vocab;
    const double eps = J->eps;
    const double cap = J->opt.softcap;
    for (int64_t c = 0; c < V; ++c) {
        double x = or_load(J->logits, J->dtype, i * J->ld + c);
        xbuf[c] = cap > 0.0 ? cap * tanh(x / cap) : x;
    }

    int64_t t = or_target(J->target, J->target_is_int32, i);
    int valid = or_valid(t, J->ignore_index, V);

    /* pass 1: max (and its first column) */
    double m = -INFINITY;
    int64_t am = 0;
    for (int64_t c = 0; c < V; ++c)
        if (xbuf[c] > m) {
            m = xbuf[c];
            am = c;
        }
    if (J->opt.argmax)
        J->opt.argmax[i] = am;
    /* pass 2: exp-sum, off-target exp-sum, smoothing sum */
    double S = 0.0, s_off = 0.0, r = 0.0;
    for (int64_t c = 0; c < V; ++c) {
        double e = exp(xbuf[c] - m);
        S += e;
        if (!valid || c != t)
            s_off += e;
        r += (J->w ? J->w[c] : 1.0) * (xbuf[c] - m);
    }
    double lse = m + log(S);

    if (J->stats) {
        double *st = J->stats + 4 * i;
        st[0] = m;
        st[1] = s_off;
        st[2] = valid ? xbuf[t] : 0.0;
        st[3] = r;
    }

    double loss = 0.0;
    if (valid) {
        double wy = J->w ? J->w[t] : 1.0;
        double smooth = 0.0; /* sum_c w_c * lp_c */
        for (int64_t c = 0; c < V; ++c)
            smooth += (J->w ? J->w[c] : 1.0) * (xbuf[c] - lse);
        loss = -(1.0 - eps) * wy * (xbuf[t] - lse) - (eps / (double)V) * smooth;
        loss += J->opt.z_loss * lse * lse;
    }
    if (J->row_loss)
        J->row_loss[i] = loss;

    if (J->grad) {
        double *gr = J->grad + i * V;
        if (!valid) {
            for (int64_t c = 0; c < V; ++c)
                gr[c] = 0.0;
            return;
        }
        double g = J->grad_output ? J->grad_output[J->grad_output_per_row ? i : 0] : 1.0;
        double scale;
        if (J->reduction == OR_MEAN)
            scale = J->norm_wy != 0.0 ? g / J->norm_wy : 0.0;
        else
            scale = g;
        double wy = J->w ? J->w[t] : 1.0;
        for (int64_t c = 0; c < V; ++c) {
            double p = exp(xbuf[c] - lse);
            double onehot = (c == t) ? 1.0 : 0.0;
            double wc = J->w ? J->w[c] : 1.0;
            double G = (1.0 - eps) * wy * (p - onehot) + (eps / (double)V) * (p * J->w_all - wc);
            G += 2.0 * J->opt.z_loss * lse * p;
            if (cap > 0.0) {
                /* chain rule through z = cap * tanh(x / cap): dz/dx = 1 - (z / cap)^2 */
                double th = xbuf[c] / cap;
                G *= 1.0 - th * th;
            }
            gr[c] = scale * G;
        }
    }
}

static void *or_worker(void *arg)
{
    or_job *J = (or_job *)arg;
    double *xbuf = (double *)malloc(sizeof(double) * (size_t)(J->vocab > 0 ? J->vocab : 1));
    if (!xbuf)
        return (void *)1;
    for (int64_t i = J->row_begin; i < J->row_end; ++i)
        or_one_row(J, i, xbuf);
    free(xbuf);
    return NULL;
}

/*
 * Row losses, statistics and gradient for rows [0, n_rows) of the given
 * block. The normalisers norm_wy and w_all come from ce_oracle_normalizers
 * over the whole batch (a row block may be a sample of a larger batch).
 * row_loss [n_rows], stats [n_rows][4] and grad [n_rows][vocab] may each be
 * NULL. grad_output is [1] (or [n_rows] with grad_output_per_row) or NULL
 * for 1.0. Returns 0 on success.
 */
int ce_oracle_rows_ex(const void *logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                      const void *target, int target_is_int32, int64_t ignore_index,
                      const double *class_weight, double label_smoothing, int reduction,
                      const double *grad_output, int grad_output_per_row, double norm_wy,
                      double w_all, double *row_loss, double *stats, double *grad, int n_threads,
                      double softcap, double z_loss, int64_t *argmax)
{
    if (n_rows < 0 || vocab < 1 || ld < vocab)
        return 1;
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > n_rows)
        n_threads = n_rows > 0 ? (int)n_rows : 1;
    or_job *jobs = (or_job *)calloc((size_t)n_threads, sizeof(or_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return 2;
    }
    int rc = 0;
    for (int k = 0; k < n_threads; ++k) {
        or_job *J = &jobs[k];
        J->logits = logits;
        J->dtype = dtype;
        J->vocab = vocab;
        J->ld = ld;
        J->target = target;
        J->target_is_int32 = target_is_int32;
        J->ignore_index = ignore_index;
        J->w = class_weight;
        J->eps = label_smoothing;
        J->reduction = reduction;
        J->grad_output = grad_output;
        J->grad_output_per_row = grad_output_per_row;
        J->norm_wy = norm_wy;
        J->w_all = w_all;
        J->row_loss = row_loss;
        J->stats = stats;
        J->grad = grad;
        J->row_begin = n_rows * k / n_threads;
        J->row_end = n_rows * (k + 1) / n_threads;
        J->opt.softcap = softcap;
        J->opt.z_loss = z_loss;
        J->opt.argmax = argmax;
    }
    int started = 0;
    for (int k = 1; k < n_threads; ++k) {
        if (pthread_create(&tid[k], NULL, or_worker, &jobs[k]) != 0) {
            rc = 3;
            break;
        }
        started = k;
    }
    if (or_worker(&jobs[0]) != NULL)
        rc = 2;
    for (int k = 1; k <= started; ++k) {
        void *ret = NULL;
        pthread_join(tid[k], &ret);
        if (ret != NULL)
            rc = 2;
    }
    if (rc == 3) /* run what did not start on this thread */
        for (int k = started + 1; k < n_threads; ++k)
            or_worker(&jobs[k]);
    free(jobs);
    free(tid);
    return rc == 3 ? 0 : rc;
}

/* mean: sum / norm_wy (0 when norm_wy is 0), sum: sum, none: not reduced. */
double ce_oracle_reduce(const double *row_loss, int64_t n_rows, int reduction, double norm_wy)
{
    double s = 0.0;
    for (int64_t i = 0; i < n_rows; ++i)
        s += row_loss[i];
    if (reduction == OR_MEAN)
        return norm_wy != 0.0 ? s / norm_wy : 0.0;
    return s;
}

int ce_oracle_rows(const void *logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                   const void *target, int target_is_int32, int64_t ignore_index,
                   const double *class_weight, double label_smoothing, int reduction,
                   const double *grad_output, int grad_output_per_row, double norm_wy,
                   double w_all, double *row_loss, double *stats, double *grad, int n_threads)
{
    return ce_oracle_rows_ex(logits, dtype, n_rows, vocab, ld, target, target_is_int32, ignore_index,
                             class_weight, label_smoothing, reduction, grad_output, grad_output_per_row,
                             norm_wy, w_all, row_loss, stats, grad, n_threads, 0.0, 0.0, NULL);
}
