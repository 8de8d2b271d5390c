/*
 * Plain fp64 CPU oracle for jagged Generalized Dot-Product Attention (GDPA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path includes, links or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no header, helper, table or constant with the
 * CUDA library: the activation codes below are re-declared here on purpose.
 *
 * What it computes (the plain definition, evaluated pair by pair):
 *
 *   For every segment b and head h, with Lq = q_off[b+1]-q_off[b] and
 *   Lkv = kv_off[b+1]-kv_off[b], segment-local indices i < Lq, j < Lkv, and
 *   valid(i,j) = (j < Lkv) and (not causal or j <= i)
 *                and (window == 0 or |i - j| < window):
 *
 *     x_ij = s * <q_i, k_j> + bias[h][clamp(i-j, -R, R) + R]   (bias optional,
 *                                                               R = (T-1)/2)
 *     GELU / SiLU : O_i = sum_{valid j} act(x_ij) v_j           (no normalisation)
 *     SOFTMAX     : O_i = sum_{valid j} exp(x_ij - LSE_i) v_j,
 *                   LSE_i = log sum_{valid j} exp(x_ij)
 *
 * Sources.  "GEM Training: How Meta Doubled the Efficiency of Its ..." (page
 * globalainews.in), section "What to watch": the attention modules are two
 * matrix multiplications with an element-wise activation in between, softmax
 * replaced by GELU or SiLU; section "What happened": JFA runs flash attention
 * directly on jagged tensors with custom attention biases, asymmetric
 * query/key-value lengths and a backward pass.  "Meta redesigns AI training
 * infrastructure ..." (aiuniverse.news), section "Custom Kernels and 5D
 * Parallelism ...": GDPA with GELU/SiLU activations.  The pages print no
 * formula; the readings taken where they are silent are:
 *   - no 1/L or row-sum normalisation in GELU/SiLU mode;
 *   - GELU is the exact erf form x*Phi(x);
 *   - the bias is a per-head table of T = 2R+1 entries indexed by
 *     clamp(i-j, -R, R)+R with segment-local i, j, added after scaling;
 *   - the scale multiplies q.k only;
 *   - causal masking is top-left aligned (j <= i);
 *   - sliding-window attention ("Meta redesigns AI training infrastructure
 *     ...", section "Custom Kernels and 5D Parallelism ...", names it without
 *     defining it; the GEM page's opening list speaks of long sequences with
 *     short attention windows) keeps the pairs with |i - j| < window, again
 *     with segment-local indices; window = 0 means no window, and with causal
 *     masking the two conditions combine (i - window < j <= i);
 *   - a row with no valid key gives O_i = 0 (and LSE_i = -inf in softmax mode);
 *   - PMA-style pooling ("GEM Training ...", section "What to watch": learned
 *     seed queries shared across the batch): with q_shared = S > 0, q holds S
 *     rows that every segment reads as its query rows 0..S-1 (each segment
 *     then has Lq = S, and q_off still places its O, dO and LSE rows); the
 *     gradient of the shared rows is the sum over segments of each segment's
 *     dQ, added in segment order.
 *
 * The backward pass is the analytic gradient of L = sum O * dO:
 *   dP_ij = <dO_i, v_j>
 *   GELU / SiLU : dS_ij = dP_ij act'(x_ij),        dV_j += act(x_ij) dO_i
 *   SOFTMAX     : P_ij = exp(x_ij - LSE_i), D_i = <dO_i, O_i>,
 *                 dS_ij = P_ij (dP_ij - D_i),       dV_j += P_ij dO_i
 *   dQ_i += s dS_ij k_j,  dK_j += s dS_ij q_i,  dbias[h][clamp(i-j)+R] += dS_ij
 *
 * Layouts: q, out, dout, dq are [total_q][H][d]; k, v, dk, dv are
 * [total_kv][H][d]; lse is [H][total_q]; bias and dbias are [H][T].
 * All floating point is double.  OpenMP parallelises over (segment, head)
 * units only; every unit runs the same sequential loops.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_GELU = 0, ORACLE_SILU = 1, ORACLE_SOFTMAX = 2, ORACLE_IDENTITY = 3 };

/* Standard normal density and distribution function. */
static double phi_pdf(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }
static double phi_cdf(double x) { return 0.5 * (1.0 + erf(x / sqrt(2.0))); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* act(x) and act'(x) for the element-wise modes (not softmax). */
static void act_eval(int act, double x, double* y, double* dy) {
    switch (act) {
    case ORACLE_GELU: {            /* GELU(x) = x Phi(x), GELU'(x) = Phi(x) + x phi(x) */
        double c = phi_cdf(x);
        *y = x * c;
        *dy = c + x * phi_pdf(x);
        break;
    }
    case ORACLE_SILU: {            /* SiLU(x) = x sigma(x), SiLU' = sigma (1 + x (1 - sigma)) */
        double sg = sigmoid(x);
        *y = x * sg;
        *dy = sg * (1.0 + x * (1.0 - sg));
        break;
    }
    default:                       /* identity: test mode for the associativity check */
        *y = x;
        *dy = 1.0;
        break;
    }
}

int oracle_act_eval(int32_t act, const double* x, int64_t n, double* y, double* dy) {
    if (act != ORACLE_GELU && act != ORACLE_SILU && act != ORACLE_IDENTITY) return 1;
    for (int64_t t = 0; t < n; ++t) act_eval(act, x[t], &y[t], &dy[t]);
    return 0;
}

typedef struct {
    const double *q, *k, *v, *dout, *bias;
    const int32_t *q_off, *kv_off;
    int32_t batch, heads, d, act, bias_len, causal, window, q_shared;
    double scale;
} problem;

/* Query row i of segment b, head h (the shared rows when q_shared > 0). */
static const double* q_row(const problem* p, int32_t b, int64_t i, int32_t h) {
    const int64_t hd = (int64_t)p->heads * p->d;
    const int64_t row = p->q_shared > 0 ? i : (int64_t)p->q_off[b] + i;
    return p->q + row * hd + (int64_t)h * p->d;
}

static int valid_pair(const problem* p, int64_t i, int64_t j, int64_t lkv) {
    if (j >= lkv) return 0;
    if (p->causal && j > i) return 0;
    if (p->window > 0 && (i - j >= p->window || j - i >= p->window)) return 0;
    return 1;
}

/* Index into the bias table of head h for local (i, j). */
static int64_t bias_index(const problem* p, int64_t i, int64_t j) {
    int64_t r = (p->bias_len - 1) / 2;
    int64_t rel = i - j;
    if (rel < -r) rel = -r;
    if (rel > r) rel = r;
    return rel + r;
}

/* x_ij = s <q_i, k_j> + bias. */
static double logit(const problem* p, int32_t b, int32_t h, int64_t i, int64_t j) {
    const int64_t hd = (int64_t)p->heads * p->d;
    const double* qi = q_row(p, b, i, h);
    const double* kj = p->k + ((int64_t)p->kv_off[b] + j) * hd + (int64_t)h * p->d;
    double dot = 0.0;
    for (int32_t c = 0; c < p->d; ++c) dot += qi[c] * kj[c];
    double x = p->scale * dot;
    if (p->bias_len > 0) x += p->bias[(int64_t)h * p->bias_len + bias_index(p, i, j)];
    return x;
}

/* Forward of query row i of segment b, head h: writes O_i (d values at oi)
 * and returns LSE_i.  x is scratch for the row's Lkv logits. */
static double fwd_row(const problem* p, int32_t b, int32_t h, int64_t i, double* x, double* oi) {
    const int64_t lkv = p->kv_off[b + 1] - p->kv_off[b];
    const int64_t hd = (int64_t)p->heads * p->d;
    for (int32_t c = 0; c < p->d; ++c) oi[c] = 0.0;
    double m = -INFINITY;
    for (int64_t j = 0; j < lkv; ++j) {
        if (!valid_pair(p, i, j, lkv)) continue;
        x[j] = logit(p, b, h, i, j);
        if (x[j] > m) m = x[j];
    }
    double l = 0.0;
    if (p->act == ORACLE_SOFTMAX) {
        for (int64_t j = 0; j < lkv; ++j)
            if (valid_pair(p, i, j, lkv)) l += exp(x[j] - m);
    }
    for (int64_t j = 0; j < lkv; ++j) {
        if (!valid_pair(p, i, j, lkv)) continue;
        double w, dw;
        if (p->act == ORACLE_SOFTMAX) w = exp(x[j] - m) / l;
        else act_eval(p->act, x[j], &w, &dw);
        const double* vj = p->v + ((int64_t)p->kv_off[b] + j) * hd + (int64_t)h * p->d;
        for (int32_t c = 0; c < p->d; ++c) oi[c] += w * vj[c];
    }
    return (l > 0.0) ? m + log(l) : -INFINITY;
}

/* Forward of one (segment, head) unit: O rows and LSE of that unit.
 * Returns nonzero if its scratch cannot be allocated. */
static int fwd_unit(const problem* p, int32_t b, int32_t h, double* out, double* lse,
                     int64_t total_q) {
    const int64_t lq = p->q_off[b + 1] - p->q_off[b];
    const int64_t lkv = p->kv_off[b + 1] - p->kv_off[b];
    const int64_t hd = (int64_t)p->heads * p->d;
    double* x = (double*)malloc(sizeof(double) * (size_t)(lkv > 0 ? lkv : 1));
    if (!x) return 1;
    for (int64_t i = 0; i < lq; ++i) {
        double* oi = out + ((int64_t)p->q_off[b] + i) * hd + (int64_t)h * p->d;
        const double l = fwd_row(p, b, h, i, x, oi);
        if (lse) lse[(int64_t)h * total_q + p->q_off[b] + i] = l;
    }
    free(x);
    return 0;
}

/* Backward quantities of one valid pair (i, j): P_ij (the act value, or the
 * softmax probability exp(x_ij - LSE_i)) and dS_ij = dP_ij act'(x_ij), or
 * P_ij (dP_ij - D_i) in softmax mode, with dP_ij = <dO_i, v_j>. */
static void pair_grad(const problem* p, int32_t b, int32_t h, int64_t i, int64_t j,
                      const double* doi, double lse_i, double di, double* pij, double* ds) {
    const int64_t hd = (int64_t)p->heads * p->d;
    const double* vj = p->v + ((int64_t)p->kv_off[b] + j) * hd + (int64_t)h * p->d;
    double x = logit(p, b, h, i, j);
    double dp = 0.0;
    for (int32_t c = 0; c < p->d; ++c) dp += doi[c] * vj[c];
    if (p->act == ORACLE_SOFTMAX) {
        *pij = exp(x - lse_i);
        *ds = *pij * (dp - di);
    } else {
        double da;
        act_eval(p->act, x, pij, &da);
        *ds = dp * da;
    }
}

/* Backward of one unit.  dq/dk/dv rows of the unit are overwritten; the
 * unit's dbias contribution is written to dbias_unit[T] (zeroed here).  With
 * shared queries dq is the unit's own [S][d] buffer instead. */
static int bwd_unit(const problem* p, int32_t b, int32_t h, double* dq, double* dk,
                    double* dv, double* dbias_unit) {
    const int64_t lq = p->q_off[b + 1] - p->q_off[b];
    const int64_t lkv = p->kv_off[b + 1] - p->kv_off[b];
    const int32_t d = p->d;
    const int64_t hd = (int64_t)p->heads * d;
    const int64_t q0 = p->q_off[b], k0 = p->kv_off[b];
    if (dbias_unit) memset(dbias_unit, 0, sizeof(double) * (size_t)p->bias_len);
    const int shared = p->q_shared > 0;
    for (int64_t i = 0; i < lq; ++i) {
        double* dqi = shared ? dq + i * d : dq + (q0 + i) * hd + (int64_t)h * d;
        for (int32_t c = 0; c < d; ++c) dqi[c] = 0.0;
    }
    for (int64_t j = 0; j < lkv; ++j) {
        double* dkj = dk + (k0 + j) * hd + (int64_t)h * d;
        double* dvj = dv + (k0 + j) * hd + (int64_t)h * d;
        for (int32_t c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
    }
    /* Softmax mode needs O_i and LSE_i of this unit: recompute them here. */
    double* o = NULL;
    double* lse = NULL;
    if (p->act == ORACLE_SOFTMAX && lq > 0) {
        /* A private single-unit problem whose output rows start at 0. */
        int32_t qoff2[2] = {0, (int32_t)lq};
        int32_t koff2[2] = {0, (int32_t)lkv};
        problem sub = *p;
        sub.q = shared ? p->q : p->q + q0 * hd;
        sub.q_shared = 0;
        sub.k = p->k + k0 * hd;
        sub.v = p->v + k0 * hd;
        sub.q_off = qoff2;
        sub.kv_off = koff2;
        sub.batch = 1;
        o = (double*)calloc((size_t)(lq * hd), sizeof(double));
        lse = (double*)calloc((size_t)(lq * p->heads), sizeof(double));
        if (!o || !lse || fwd_unit(&sub, 0, h, o, lse, lq)) {
            free(o);
            free(lse);
            return 1;
        }
    }
    for (int64_t i = 0; i < lq; ++i) {
        const double* qi = q_row(p, b, i, h);
        const double* doi = p->dout + (q0 + i) * hd + (int64_t)h * d;
        double* dqi = shared ? dq + i * d : dq + (q0 + i) * hd + (int64_t)h * d;
        double di = 0.0, lse_i = 0.0;
        if (o) {
            const double* oi = o + i * hd + (int64_t)h * d;
            for (int32_t c = 0; c < d; ++c) di += doi[c] * oi[c];
            lse_i = lse[(int64_t)h * lq + i];
        }
        for (int64_t j = 0; j < lkv; ++j) {
            if (!valid_pair(p, i, j, lkv)) continue;
            const double* kj = p->k + (k0 + j) * hd + (int64_t)h * d;
            double* dkj = dk + (k0 + j) * hd + (int64_t)h * d;
            double* dvj = dv + (k0 + j) * hd + (int64_t)h * d;
            double pij, ds;
            pair_grad(p, b, h, i, j, doi, lse_i, di, &pij, &ds);
            for (int32_t c = 0; c < d; ++c) {
                dvj[c] += pij * doi[c];
                dqi[c] += p->scale * ds * kj[c];
                dkj[c] += p->scale * ds * qi[c];
            }
            if (dbias_unit) dbias_unit[bias_index(p, i, j)] += ds;
        }
    }
    free(o);
    free(lse);
    return 0;
}

static int check_problem(const problem* p) {
    if (p->batch < 0 || p->heads < 1 || p->d < 1) return 1;
    if (p->act < ORACLE_GELU || p->act > ORACLE_IDENTITY) return 1;
    if (p->bias_len < 0 || (p->bias_len > 0 && (p->bias_len % 2) == 0)) return 1;
    if (p->bias_len > 0 && !p->bias) return 1;
    if (p->window < 0) return 1;
    if (p->batch > 0 && (p->q_off[0] != 0 || p->kv_off[0] != 0)) return 1;
    for (int32_t b = 0; b < p->batch; ++b)
        if (p->q_off[b + 1] < p->q_off[b] || p->kv_off[b + 1] < p->kv_off[b]) return 1;
    if (p->q_shared < 0) return 1;
    if (p->q_shared > 0)  /* every segment reads the S shared rows */
        for (int32_t b = 0; b < p->batch; ++b)
            if (p->q_off[b + 1] - p->q_off[b] != p->q_shared) return 1;
    return 0;
}

static void set_threads(int32_t threads) {
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

/*
 * Forward.  units/n_units select (segment, head) units as b*H + h; units ==
 * NULL means all of them.  Only the selected units' rows of out and lse are
 * written.  lse may be NULL.  Returns 0, 1 on invalid arguments, or 2 if
 * scratch memory cannot be allocated.
 */
int oracle_fwd(const double* q, const double* k, const double* v,
               const int32_t* q_off, const int32_t* kv_off, int32_t batch,
               int32_t heads, int32_t d, int32_t act, double scale,
               const double* bias, int32_t bias_len, int32_t causal, int32_t window,
               int32_t q_shared, const int32_t* units, int32_t n_units, int32_t threads,
               double* out, double* lse) {
    problem p = {q, k, v, NULL, bias, q_off, kv_off, batch, heads, d, act, bias_len, causal, window,
                 q_shared, scale};
    if (check_problem(&p)) return 1;
    const int64_t total_q = batch > 0 ? q_off[batch] : 0;
    const int32_t n = units ? n_units : batch * heads;
    int failed = 0;
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t u = 0; u < n; ++u) {
        int32_t id = units ? units[u] : u;
        if (fwd_unit(&p, id / heads, id % heads, out, lse, total_q)) {
#pragma omp atomic write
            failed = 1;
        }
    }
    return failed ? 2 : 0;
}

/*
 * Backward.  Overwrites the selected units' rows of dq, dk, dv; dbias (may be
 * NULL) receives the sum over the selected units, reduced in unit order.
 * Returns 0, 1 on invalid arguments, or 2 if scratch memory cannot be
 * allocated (the outputs are then incomplete).
 */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
               const int32_t* q_off, const int32_t* kv_off, int32_t batch,
               int32_t heads, int32_t d, int32_t act, double scale,
               const double* bias, int32_t bias_len, int32_t causal, int32_t window,
               int32_t q_shared, const int32_t* units, int32_t n_units, int32_t threads,
               double* dq, double* dk, double* dv, double* dbias) {
    problem p = {q, k, v, dout, bias, q_off, kv_off, batch, heads, d, act, bias_len, causal, window,
                 q_shared, scale};
    if (check_problem(&p)) return 1;
    const int32_t n = units ? n_units : batch * heads;
    const int32_t t = bias_len > 0 ? bias_len : 1;
    double* part = (dbias && bias_len > 0)
                       ? (double*)calloc((size_t)n * (size_t)t, sizeof(double)) : NULL;
    /* shared queries: each unit's dQ in its own [S][d] buffer, summed per
       head in unit (segment) order below */
    const int64_t sq = (int64_t)q_shared * d;
    double* dq_part = q_shared > 0 ? (double*)calloc((size_t)n * (size_t)(sq > 0 ? sq : 1), sizeof(double))
                                   : NULL;
    if ((dbias && bias_len > 0 && !part) || (q_shared > 0 && !dq_part)) {
        free(part);
        free(dq_part);
        return 2;
    }
    int failed = 0;
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t u = 0; u < n; ++u) {
        int32_t id = units ? units[u] : u;
        if (bwd_unit(&p, id / heads, id % heads, dq_part ? dq_part + (int64_t)u * sq : dq, dk, dv,
                     part ? part + (int64_t)u * t : NULL)) {
#pragma omp atomic write
            failed = 1;
        }
    }
    if (failed) {
        free(part);
        free(dq_part);
        return 2;
    }
    if (dq_part) {
        memset(dq, 0, sizeof(double) * (size_t)q_shared * (size_t)heads * (size_t)d);
        for (int32_t u = 0; u < n; ++u) {
            int32_t h = (units ? units[u] : u) % heads;
            for (int64_t i = 0; i < q_shared; ++i)
                for (int32_t c = 0; c < d; ++c)
                    dq[(i * heads + h) * d + c] += dq_part[(int64_t)u * sq + i * d + c];
        }
        free(dq_part);
    }
    if (part) {
        memset(dbias, 0, sizeof(double) * (size_t)heads * (size_t)bias_len);
        for (int32_t u = 0; u < n; ++u) {
            int32_t id = units ? units[u] : u;
            int32_t h = id % heads;
            for (int32_t e = 0; e < bias_len; ++e)
                dbias[(int64_t)h * bias_len + e] += part[(int64_t)u * t + e];
        }
        free(part);
    }
    return 0;
}

/*
 * Backward of one (segment b, head h) unit restricted to some of its rows:
 * dQ_i for the segment-local query rows q_rows[0..n_q) and dK_j, dV_j for
 * the key rows kv_rows[0..n_kv), each an explicit sum over its valid
 * partners with the per-pair quantities of the full backward, taken in the
 * same order (ascending j for dQ_i, ascending i for dK_j and dV_j), so the
 * rows equal those of oracle_bwd.  In softmax mode LSE_i and D_i = <dO_i, O_i>
 * come from the forward of each query row involved.  dq_rows is [n_q][d],
 * dk_rows and dv_rows are [n_kv][d].  OpenMP runs over the selected rows.
 * Returns 0, 1 on invalid arguments (including a row outside the segment,
 * or shared queries, which this entry point does not take), or 2 if scratch
 * memory cannot be allocated.
 */
int oracle_bwd_rows(const double* q, const double* k, const double* v, const double* dout,
                    const int32_t* q_off, const int32_t* kv_off, int32_t batch,
                    int32_t heads, int32_t d, int32_t act, double scale,
                    const double* bias, int32_t bias_len, int32_t causal, int32_t window,
                    int32_t b, int32_t h, const int32_t* q_rows, int32_t n_q,
                    const int32_t* kv_rows, int32_t n_kv, int32_t threads,
                    double* dq_rows, double* dk_rows, double* dv_rows) {
    problem p = {q, k, v, dout, bias, q_off, kv_off, batch, heads, d, act, bias_len, causal, window,
                 0, scale};
    if (check_problem(&p)) return 1;
    if (b < 0 || b >= batch || h < 0 || h >= heads || n_q < 0 || n_kv < 0) return 1;
    const int64_t lq = q_off[b + 1] - q_off[b];
    const int64_t lkv = kv_off[b + 1] - kv_off[b];
    for (int32_t r = 0; r < n_q; ++r)
        if (q_rows[r] < 0 || q_rows[r] >= lq) return 1;
    for (int32_t r = 0; r < n_kv; ++r)
        if (kv_rows[r] < 0 || kv_rows[r] >= lkv) return 1;
    const int64_t hd = (int64_t)heads * d;
    const int64_t q0 = q_off[b], k0 = kv_off[b];
    const int softmax = act == ORACLE_SOFTMAX;
    /* softmax: LSE_i and D_i of every query row (the key rows meet them all) */
    double* lse = NULL;
    double* dd = NULL;
    int failed = 0;
    set_threads(threads);
    if (softmax && lq > 0) {
        lse = (double*)malloc(sizeof(double) * (size_t)lq);
        dd = (double*)malloc(sizeof(double) * (size_t)lq);
        if (!lse || !dd) {
            free(lse);
            free(dd);
            return 2;
        }
#pragma omp parallel
        {
            double* x = (double*)malloc(sizeof(double) * (size_t)(lkv > 0 ? lkv : 1));
            double* oi = (double*)malloc(sizeof(double) * (size_t)d);
            if (!x || !oi) {
#pragma omp atomic write
                failed = 1;
            }
#pragma omp for schedule(dynamic, 16)
            for (int64_t i = 0; i < lq; ++i) {
                if (!x || !oi) continue;
                lse[i] = fwd_row(&p, b, h, i, x, oi);
                const double* doi = dout + (q0 + i) * hd + (int64_t)h * d;
                double di = 0.0;
                for (int32_t c = 0; c < d; ++c) di += doi[c] * oi[c];
                dd[i] = di;
            }
            free(x);
            free(oi);
        }
        if (failed) {
            free(lse);
            free(dd);
            return 2;
        }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < n_q; ++r) {
        const int64_t i = q_rows[r];
        const double* doi = dout + (q0 + i) * hd + (int64_t)h * d;
        double* dqi = dq_rows + (int64_t)r * d;
        for (int32_t c = 0; c < d; ++c) dqi[c] = 0.0;
        for (int64_t j = 0; j < lkv; ++j) {
            if (!valid_pair(&p, i, j, lkv)) continue;
            const double* kj = k + (k0 + j) * hd + (int64_t)h * d;
            double pij, ds;
            pair_grad(&p, b, h, i, j, doi, softmax ? lse[i] : 0.0, softmax ? dd[i] : 0.0, &pij, &ds);
            for (int32_t c = 0; c < d; ++c) dqi[c] += scale * ds * kj[c];
        }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < n_kv; ++r) {
        const int64_t j = kv_rows[r];
        double* dkj = dk_rows + (int64_t)r * d;
        double* dvj = dv_rows + (int64_t)r * d;
        for (int32_t c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
        for (int64_t i = 0; i < lq; ++i) {
            if (!valid_pair(&p, i, j, lkv)) continue;
            const double* qi = q + (q0 + i) * hd + (int64_t)h * d;
            const double* doi = dout + (q0 + i) * hd + (int64_t)h * d;
            double pij, ds;
            pair_grad(&p, b, h, i, j, doi, softmax ? lse[i] : 0.0, softmax ? dd[i] : 0.0, &pij, &ds);
            for (int32_t c = 0; c < d; ++c) {
                dvj[c] += pij * doi[c];
                dkj[c] += scale * ds * qi[c];
            }
        }
    }
    free(lse);
    free(dd);
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
