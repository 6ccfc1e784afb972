/*
 * oracle.c -- plain, slow, fp64 CPU reference for the online-softmax attention
 * forward.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * helper with the GPU path and includes nothing from it.
 *
 * Every routine below is the plain definition (or the pages' algorithm, step
 * by step) written in fp64 with no blocking, fusion or reordering:
 *
 *   oracle_attention      three-pass safe softmax attention, S materialised
 *                         per query row.  "Online Softmax 算法详解" section 2.1
 *                         (the three passes), section 8.1 (LSE definition);
 *                         masked-row convention from section 7.2/7.3.
 *   oracle_online_blocks  the blockwise (m, l, O) recurrence with a caller
 *                         chosen block partition and block order.
 *                         "在线Softmax算法解析" section 3.2; "01 -- La
 *                         recurrencia del online softmax", section "La
 *                         recurrencia"; -inf reference point from
 *                         "Online Softmax 算法详解" section 7.1.
 *   oracle_merge          the two-block merge rule folded over P parts
 *                         (airsota.com online-softmax card, section 三,
 *                         "Running Combined Updates"; associativity per
 *                         "La recurrencia del online softmax", practice 4).
 *   oracle_softmax_two_pass
 *                         Milakov & Gimelshein two-pass normaliser
 *                         ("Online Softmax 算法详解" section 2.2).
 *   oracle_softmax_rows   the same over the rows of a matrix.
 *   oracle_attention_bwd  gradients dQ, dK, dV of the attention forward
 *                         ("Online Softmax 算法详解" section 8.3).
 *   oracle_attention_fp8  the FP8 (E4M3) forward with Max_offset = 8
 *                         ("Online Softmax 算法详解" section 6); oracle_e4m3.
 *
 *   oracle_attention_window
 *                         the same with a local (sliding-window) mask.
 *
 * Causal convention (not fixed by the pages; the reading used throughout):
 * key j is visible to query i iff j <= i + (nk - nq)  (bottom-right aligned).
 * Local window (named but not defined by the pages, "Online Softmax 算法详解"
 * section 3.2; the reading used throughout): key j is visible to query i iff
 * i + off - wl <= j <= i + off + wr with off = nk - nq; a negative wl or wr
 * leaves that side unbounded.  Causal is the window (-1, 0).
 *
 * All routines are re-entrant.  oracle_attention splits its rows over
 * `nthreads` POSIX threads (nthreads <= 0 means one thread).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Three-pass safe-softmax attention                                          */
/* ------------------------------------------------------------------------ */

/* One query row.  s is caller scratch of nk doubles. */
static void attention_row(const double *qi, const double *k, const double *v,
                          int64_t nk, int64_t d, double scale,
                          int64_t first_visible, int64_t last_visible,
                          double *s, double *oi, double *lse_i)
{
    /* Materialise the score row S_j = scale * <q_i, k_j>; -inf where masked. */
    for (int64_t j = 0; j < nk; ++j) {
        if (j > last_visible || j < first_visible) {
            s[j] = -INFINITY;
            continue;
        }
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += qi[c] * k[j * d + c];
        s[j] = scale * acc;
    }

    /* Pass 1: m = max_j S_j. */
    double m = -INFINITY;
    for (int64_t j = 0; j < nk; ++j)
        if (s[j] > m)
            m = s[j];

    /* A row with no visible key: O = 0 and LSE = -inf. */
    if (m == -INFINITY) {
        for (int64_t c = 0; c < d; ++c)
            oi[c] = 0.0;
        *lse_i = -INFINITY;
        return;
    }

    /* Pass 2: l = sum_j exp(S_j - m). */
    double l = 0.0;
    for (int64_t j = 0; j < nk; ++j)
        l += exp(s[j] - m);

    /* Pass 3: P_j = exp(S_j - m) / l and O = sum_j P_j v_j. */
    for (int64_t c = 0; c < d; ++c)
        oi[c] = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
        double p = exp(s[j] - m) / l;
        for (int64_t c = 0; c < d; ++c)
            oi[c] += p * v[j * d + c];
    }

    /* LSE = ln sum_j exp(S_j) = m + ln l. */
    *lse_i = m + log(l);
}

typedef struct {
    const double *q, *k, *v;
    int64_t nq, nk, d;
    double scale;
    int causal;
    int64_t wl, wr; /* window (used when causal == 2) */
    const int64_t *rows;
    int64_t row_begin, row_end;
    double *o, *lse;
    int status;
} attention_job;

static void *attention_worker(void *arg)
{
    attention_job *job = (attention_job *)arg;
    double *s = (double *)malloc((size_t)(job->nk > 0 ? job->nk : 1) * sizeof(double));
    if (!s) {
        job->status = -1;
        return NULL;
    }
    for (int64_t r = job->row_begin; r < job->row_end; ++r) {
        int64_t i = job->rows ? job->rows[r] : r;
        int64_t first_visible = 0;
        int64_t last_visible = job->causal ? i + (job->nk - job->nq) : job->nk - 1;
        if (job->causal == 2) { /* local window */
            int64_t off = job->nk - job->nq;
            first_visible = job->wl < 0 ? 0 : i + off - job->wl;
            last_visible = job->wr < 0 ? job->nk - 1 : i + off + job->wr;
        }
        attention_row(job->q + i * job->d, job->k, job->v, job->nk, job->d,
                      job->scale, first_visible, last_visible, s,
                      job->o + r * job->d, job->lse + r);
    }
    free(s);
    job->status = 0;
    return NULL;
}

/*
 * q [nq][d], k [nk][d], v [nk][d] : one head, row-major fp64.
 * rows[nrows] : query rows to compute (NULL: all nq rows, nrows must be nq).
 * o [nrows][d], lse [nrows] : outputs, in the order of `rows`.
 * Returns 0, or -1 on a bad argument / allocation failure.
 */
static int run_attention(const double *q, int64_t nq, const double *k,
                         const double *v, int64_t nk, int64_t d, double scale,
                         int causal, int64_t wl, int64_t wr,
                         const int64_t *rows, int64_t nrows, double *o,
                         double *lse, int nthreads)
{
    if (!q || !k || !v || !o || !lse || nq < 0 || nk < 0 || d <= 0 || nrows < 0)
        return -1;
    if (!rows && nrows != nq)
        return -1;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= nq)
            return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nrows)
        nthreads = nrows > 0 ? (int)nrows : 1;

    attention_job *jobs = (attention_job *)calloc((size_t)nthreads, sizeof(attention_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -1;
    }
    int64_t per = (nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        attention_job *job = &jobs[t];
        job->q = q; job->k = k; job->v = v;
        job->nq = nq; job->nk = nk; job->d = d;
        job->scale = scale; job->causal = causal;
        job->wl = wl; job->wr = wr;
        job->rows = rows;
        job->row_begin = (int64_t)t * per < nrows ? (int64_t)t * per : nrows;
        job->row_end = job->row_begin + per < nrows ? job->row_begin + per : nrows;
        job->o = o; job->lse = lse;
        job->status = -1;
    }
    int rc = 0;
    int *created = (int *)calloc((size_t)nthreads, sizeof(int));
    if (!created) {
        free(jobs);
        free(tids);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        if (nthreads > 1 && pthread_create(&tids[t], NULL, attention_worker, &jobs[t]) == 0)
            created[t] = 1;
        else
            attention_worker(&jobs[t]); /* single thread, or no thread available */
    }
    for (int t = 0; t < nthreads; ++t)
        if (created[t])
            pthread_join(tids[t], NULL);
    free(created);
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != 0)
            rc = -1;
    free(jobs);
    free(tids);
    return rc;
}

int oracle_attention(const double *q, int64_t nq, const double *k,
                     const double *v, int64_t nk, int64_t d, double scale,
                     int causal, const int64_t *rows, int64_t nrows,
                     double *o, double *lse, int nthreads)
{
    return run_attention(q, nq, k, v, nk, d, scale, causal ? 1 : 0, -1, -1,
                         rows, nrows, o, lse, nthreads);
}

/* As oracle_attention, with the local window [i + off - wl, i + off + wr]. */
int oracle_attention_window(const double *q, int64_t nq, const double *k,
                            const double *v, int64_t nk, int64_t d,
                            double scale, int64_t wl, int64_t wr,
                            const int64_t *rows, int64_t nrows, double *o,
                            double *lse, int nthreads)
{
    return run_attention(q, nq, k, v, nk, d, scale, 2, wl, wr, rows, nrows, o,
                         lse, nthreads);
}

/* ------------------------------------------------------------------------ */
/* The blockwise online recurrence, one row                                   */
/* ------------------------------------------------------------------------ */

/*
 * s[n] : the row's (already scaled) scores, -inf allowed.
 * v[n][dv] : value rows.
 * block_start[nb], block_len[nb] : the blocks, in processing order (any
 *   order; together they should cover each index once).
 * Outputs: *m_out, *l_out (running max and sum at the end), o_out[dv] = O/l
 * (0 when l = 0), *lse_out = m + ln l (-inf when l = 0).
 *
 * State starts at m = -inf, l = 0, O = 0.  Per block:
 *   m_blk = max of the block; m_new = max(m, m_blk)
 *   ref   = m_new, or 0 when m_new is -inf (no NaN from -inf - -inf)
 *   alpha = exp(m - ref); l <- alpha * l; O <- alpha * O
 *   p_j   = exp(s_j - ref); l <- l + sum p_j; O <- O + sum p_j v_j
 *   m     <- m_new
 * Finally O <- O / l.
 */
int oracle_online_blocks(const double *s, const double *v, int64_t n,
                         int64_t dv, const int64_t *block_start,
                         const int64_t *block_len, int64_t nb,
                         double *m_out, double *l_out, double *o_out,
                         double *lse_out)
{
    if (!s || !v || !block_start || !block_len || !m_out || !l_out || !o_out ||
        !lse_out || n < 0 || dv <= 0 || nb < 0)
        return -1;
    double m = -INFINITY, l = 0.0;
    double *o = (double *)calloc((size_t)dv, sizeof(double));
    if (!o)
        return -1;

    for (int64_t b = 0; b < nb; ++b) {
        int64_t j0 = block_start[b], len = block_len[b];
        if (j0 < 0 || len < 0 || j0 + len > n) {
            free(o);
            return -1;
        }
        double m_blk = -INFINITY;
        for (int64_t j = j0; j < j0 + len; ++j)
            if (s[j] > m_blk)
                m_blk = s[j];
        double m_new = m > m_blk ? m : m_blk;
        double ref = (m_new == -INFINITY) ? 0.0 : m_new;
        double alpha = exp(m - ref);
        l = l * alpha;
        for (int64_t c = 0; c < dv; ++c)
            o[c] = o[c] * alpha;
        for (int64_t j = j0; j < j0 + len; ++j) {
            double p = exp(s[j] - ref);
            l = l + p;
            for (int64_t c = 0; c < dv; ++c)
                o[c] = o[c] + p * v[j * dv + c];
        }
        m = m_new;
    }

    *m_out = m;
    *l_out = l;
    for (int64_t c = 0; c < dv; ++c)
        o_out[c] = (l == 0.0) ? 0.0 : o[c] / l;
    *lse_out = (l == 0.0) ? -INFINITY : m + log(l);
    free(o);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The two-block merge rule, folded left over P parts                         */
/* ------------------------------------------------------------------------ */

/*
 * Part p carries (m[p], l[p], o[p][dv]) with o normalised (O_p / l_p, or 0
 * when l_p = 0).  Two parts combine as
 *   m   = max(m1, m2)
 *   l   = l1 exp(m1 - m) + l2 exp(m2 - m)
 *   O   = O1 (l1 exp(m1 - m) / l) + O2 (l2 exp(m2 - m) / l)
 * with an empty part (m = -inf, l = 0) contributing nothing.  The fold runs
 * left to right; outputs are the merged (m, l, O) and LSE = m + ln l
 * (-inf and O = 0 when every part is empty).
 */
int oracle_merge(const double *m, const double *l, const double *o,
                 int64_t nparts, int64_t dv, double *m_out, double *l_out,
                 double *o_out, double *lse_out)
{
    if (!m || !l || !o || !m_out || !l_out || !o_out || !lse_out || nparts < 1 || dv <= 0)
        return -1;
    double m1 = m[0], l1 = l[0];
    for (int64_t c = 0; c < dv; ++c)
        o_out[c] = o[c];
    for (int64_t p = 1; p < nparts; ++p) {
        double m2 = m[p], l2 = l[p];
        const double *o2 = o + p * dv;
        double mm = m1 > m2 ? m1 : m2;
        if (mm == -INFINITY) { /* both sides empty so far */
            m1 = -INFINITY;
            l1 = 0.0;
            for (int64_t c = 0; c < dv; ++c)
                o_out[c] = 0.0;
            continue;
        }
        double w1 = (m1 == -INFINITY) ? 0.0 : l1 * exp(m1 - mm);
        double w2 = (m2 == -INFINITY) ? 0.0 : l2 * exp(m2 - mm);
        double ll = w1 + w2;
        for (int64_t c = 0; c < dv; ++c)
            o_out[c] = (ll == 0.0) ? 0.0 : o_out[c] * (w1 / ll) + o2[c] * (w2 / ll);
        m1 = mm;
        l1 = ll;
    }
    if (l1 == 0.0) {
        for (int64_t c = 0; c < dv; ++c)
            o_out[c] = 0.0;
    }
    *m_out = m1;
    *l_out = l1;
    *lse_out = (l1 == 0.0) ? -INFINITY : m1 + log(l1);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Two-pass online normaliser                                                 */
/* ------------------------------------------------------------------------ */

/*
 * Pass 1 fuses the max and the sum element by element:
 *   m_new = max(m, x_i); l = exp(m - m_new) l + exp(x_i - m_new); m = m_new
 * Pass 2: p_i = exp(x_i - m) / l.
 * A row of all -inf yields p = 0 (the -inf reference point is replaced by 0,
 * as in the blockwise recurrence).  Returns LSE = m + ln l in *lse_out.
 */
int oracle_softmax_two_pass(const double *x, int64_t n, double *p, double *lse_out)
{
    if (!x || !p || !lse_out || n < 0)
        return -1;
    double m = -INFINITY, l = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double m_new = m > x[i] ? m : x[i];
        double ref = (m_new == -INFINITY) ? 0.0 : m_new;
        l = exp(m - ref) * l + exp(x[i] - ref);
        m = m_new;
    }
    double ref = (m == -INFINITY) ? 0.0 : m;
    for (int64_t i = 0; i < n; ++i)
        p[i] = (l == 0.0) ? 0.0 : exp(x[i] - ref) / l;
    *lse_out = (l == 0.0) ? -INFINITY : m + log(l);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 (E4M3) forward with Max_offset = 8                                      */
/* ------------------------------------------------------------------------ */

/*
 * Round a non-negative value to the nearest FP8 E4M3 value (ties to even),
 * saturating at the largest finite value 448: 1 sign bit, 4 exponent bits
 * (bias 7), 3 mantissa bits; normals (1 + f/8) 2^e for e in [-6, 8],
 * subnormals f 2^-9 for f in 1..7.  Negative inputs round their magnitude.
 */
double oracle_e4m3(double x)
{
    if (x != x)
        return x;
    double a = fabs(x);
    if (a >= 448.0)
        return x < 0 ? -448.0 : 448.0;
    double spacing;
    if (a < ldexp(1.0, -6)) {
        spacing = ldexp(1.0, -9); /* subnormal grid */
    } else {
        int e;
        frexp(a, &e); /* a = f 2^e, f in [0.5, 1): exponent of the leading bit is e - 1 */
        spacing = ldexp(1.0, (e - 1) - 3);
    }
    double r = nearbyint(a / spacing) * spacing; /* default rounding mode: ties to even */
    if (r > 448.0)
        r = 448.0;
    return x < 0 ? -r : r;
}

/*
 * One head, FP8 inputs: q, k, v hold E4M3 values (exact in fp64) whose real
 * values are q * q_descale, k * k_descale, v * v_descale.  The online steps of
 * "Online Softmax 算法详解" section 6 over key blocks of `block` keys, in order:
 *   s_j   = scale * q_descale * k_descale * <q_i, k_j>        (-inf where masked)
 *   m'    = max(m, max_j s_j);   alpha = exp(m - m')  (0 while m = -inf)
 *   P'_j  = 2^((s_j - m') log2(e) + 8)                          (Max_offset = 8: P' in [0, 256])
 *   l    <- alpha l + sum_j P'_j          (the sum of the unquantised P')
 *   acc  <- alpha acc + sum_j E4M3(P'_j) v_j                    (P cast to FP8 for the P.V product)
 * then sum_scale: l <- l / 2^8, LSE = m + ln l, O = acc * (v_descale / 2^8) / l
 * (the final_scale that undoes the 2^8 in P); a row with l = 0 gets O = 0,
 * LSE = -inf.  s is in natural-log units of the scaled logits, as in
 * oracle_attention.  Causal: bottom-right aligned, as elsewhere.
 */
static void attention_fp8_row(const double *qi, const double *k, const double *v, int64_t nk,
                              int64_t d, double scale_qk, double v_descale, int64_t last_visible,
                              int64_t block, double *s, double *acc, double *oi, double *lse_i)
{
    const double log2e = 1.4426950408889634;
    for (int64_t j = 0; j < nk; ++j) {
        if (j > last_visible) {
            s[j] = -INFINITY;
            continue;
        }
        double t = 0.0;
        for (int64_t c = 0; c < d; ++c)
            t += k[j * d + c] * qi[c];
        s[j] = scale_qk * t;
    }
    double m = -INFINITY, l = 0.0;
    for (int64_t c = 0; c < d; ++c)
        acc[c] = 0.0;
    for (int64_t j0 = 0; j0 < nk; j0 += block) {
        int64_t j1 = j0 + block < nk ? j0 + block : nk;
        double m_new = m;
        for (int64_t j = j0; j < j1; ++j)
            if (s[j] > m_new)
                m_new = s[j];
        if (m_new == -INFINITY)
            continue; /* nothing visible yet */
        double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        l *= alpha;
        for (int64_t c = 0; c < d; ++c)
            acc[c] *= alpha;
        for (int64_t j = j0; j < j1; ++j) {
            if (s[j] == -INFINITY)
                continue;
            double pp = exp2((s[j] - m_new) * log2e + 8.0);
            l += pp;
            double p8 = oracle_e4m3(pp);
            for (int64_t c = 0; c < d; ++c)
                acc[c] += p8 * v[j * d + c];
        }
        m = m_new;
    }
    l *= 1.0 / 256.0; /* sum_scale */
    if (l == 0.0) {
        for (int64_t c = 0; c < d; ++c)
            oi[c] = 0.0;
        *lse_i = -INFINITY;
        return;
    }
    const double final_scale = v_descale / 256.0;
    for (int64_t c = 0; c < d; ++c)
        oi[c] = acc[c] * final_scale / l;
    *lse_i = log(l) + m;
}

int oracle_attention_fp8(const double *q, int64_t nq, const double *k, const double *v,
                         int64_t nk, int64_t d, double scale, double q_descale, double k_descale,
                         double v_descale, int causal, int64_t block, const int64_t *rows,
                         int64_t nrows, double *o, double *lse)
{
    if (!q || !k || !v || !o || !lse || nq < 0 || nk < 0 || d <= 0 || nrows < 0 || block < 1)
        return -1;
    if (!rows && nrows != nq)
        return -1;
    double *s = (double *)malloc((size_t)(nk > 0 ? nk : 1) * sizeof(double));
    double *acc = (double *)malloc((size_t)d * sizeof(double));
    if (!s || !acc) {
        free(s);
        free(acc);
        return -1;
    }
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= nq) {
            free(s);
            free(acc);
            return -1;
        }
        int64_t last = causal ? i + (nk - nq) : nk - 1;
        attention_fp8_row(q + i * d, k, v, nk, d, scale * q_descale * k_descale, v_descale, last,
                          block, s, acc, o + r * d, lse + r);
    }
    free(s);
    free(acc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Attention backward                                                         */
/* ------------------------------------------------------------------------ */
/*
 * Gradients of O = softmax(scale * Q K^T + mask) V for one head, given dO
 * ("Online Softmax 算法详解" section 8.3: recompute S, restore P from LSE,
 * then dQ, dK, dV; the pages leave the gradient formulas to a page not in the
 * set, so these are the derivative of the forward written out):
 *   P_ij  = exp(scale * S_ij - LSE_i)          (0 where masked)
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = <dO_i, v_j>
 *   D_i   = sum_j P_ij dP_ij                   (= <dO_i, O_i>)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j  = scale sum_i dS_ij q_i
 * A row with no visible key (LSE = -inf) has P = 0 and contributes nothing
 * (section 7.3).  Three sweeps: per row LSE and D; per key dK and dV; per row
 * dQ -- each a plain loop, threads split the rows or the keys.
 */
typedef struct {
    const double *q, *k, *v, *dout;
    int64_t nq, nk, d;
    double scale;
    int64_t wl, wr;
    double *lse, *dd; /* per row */
    double *dq, *dk, *dv;
    int64_t begin, end;
    int sweep;
} bwd_job;

static int visible(int64_t i, int64_t j, int64_t nq, int64_t nk, int64_t wl, int64_t wr)
{
    int64_t off = nk - nq;
    if (wl >= 0 && j < i + off - wl)
        return 0;
    if (wr >= 0 && j > i + off + wr)
        return 0;
    return 1;
}

static double dot(const double *a, const double *b, int64_t d)
{
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c)
        acc += a[c] * b[c];
    return acc;
}

/* P_ij from the row's LSE; 0 if masked or the row is empty. */
static double prob(const bwd_job *J, int64_t i, int64_t j)
{
    if (!visible(i, j, J->nq, J->nk, J->wl, J->wr) || J->lse[i] == -INFINITY)
        return 0.0;
    return exp(J->scale * dot(J->q + i * J->d, J->k + j * J->d, J->d) - J->lse[i]);
}

static void *bwd_worker(void *arg)
{
    bwd_job *J = (bwd_job *)arg;
    const int64_t d = J->d;
    if (J->sweep == 0) { /* rows: LSE_i, then D_i = sum_j P_ij dP_ij */
        for (int64_t i = J->begin; i < J->end; ++i) {
            double m = -INFINITY;
            for (int64_t j = 0; j < J->nk; ++j)
                if (visible(i, j, J->nq, J->nk, J->wl, J->wr)) {
                    double sij = J->scale * dot(J->q + i * d, J->k + j * d, d);
                    if (sij > m)
                        m = sij;
                }
            if (m == -INFINITY) {
                J->lse[i] = -INFINITY;
                J->dd[i] = 0.0;
                continue;
            }
            double l = 0.0;
            for (int64_t j = 0; j < J->nk; ++j)
                if (visible(i, j, J->nq, J->nk, J->wl, J->wr))
                    l += exp(J->scale * dot(J->q + i * d, J->k + j * d, d) - m);
            J->lse[i] = m + log(l);
            double di = 0.0;
            for (int64_t j = 0; j < J->nk; ++j) {
                double p = prob(J, i, j);
                if (p != 0.0)
                    di += p * dot(J->dout + i * d, J->v + j * d, d);
            }
            J->dd[i] = di;
        }
    } else if (J->sweep == 1) { /* keys: dV_j and dK_j */
        for (int64_t j = J->begin; j < J->end; ++j) {
            double *dvj = J->dv + j * d, *dkj = J->dk + j * d;
            for (int64_t c = 0; c < d; ++c)
                dvj[c] = dkj[c] = 0.0;
            for (int64_t i = 0; i < J->nq; ++i) {
                double p = prob(J, i, j);
                if (p == 0.0)
                    continue;
                double ds = p * (dot(J->dout + i * d, J->v + j * d, d) - J->dd[i]);
                for (int64_t c = 0; c < d; ++c) {
                    dvj[c] += p * J->dout[i * d + c];
                    dkj[c] += J->scale * ds * J->q[i * d + c];
                }
            }
        }
    } else { /* rows: dQ_i */
        for (int64_t i = J->begin; i < J->end; ++i) {
            double *dqi = J->dq + i * d;
            for (int64_t c = 0; c < d; ++c)
                dqi[c] = 0.0;
            for (int64_t j = 0; j < J->nk; ++j) {
                double p = prob(J, i, j);
                if (p == 0.0)
                    continue;
                double ds = p * (dot(J->dout + i * d, J->v + j * d, d) - J->dd[i]);
                for (int64_t c = 0; c < d; ++c)
                    dqi[c] += J->scale * ds * J->k[j * d + c];
            }
        }
    }
    return NULL;
}

static void run_sweep(bwd_job *base, int sweep, int64_t n, int nthreads)
{
    bwd_job jobs[256];
    pthread_t tids[256];
    int created[256];
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if (nthreads > n)
        nthreads = n > 0 ? (int)n : 1;
    int64_t per = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *base;
        jobs[t].sweep = sweep;
        jobs[t].begin = (int64_t)t * per < n ? (int64_t)t * per : n;
        jobs[t].end = jobs[t].begin + per < n ? jobs[t].begin + per : n;
        created[t] = 0;
    }
    for (int t = 0; t < nthreads; ++t) {
        if (nthreads > 1 && pthread_create(&tids[t], NULL, bwd_worker, &jobs[t]) == 0)
            created[t] = 1;
        else
            bwd_worker(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (created[t])
            pthread_join(tids[t], NULL);
}

/*
 * q [nq][d], k, v [nk][d], dout [nq][d]: one head, fp64.  Mask: the window
 * (wl, wr) of oracle_attention_window (causal = (-1, 0), none = (-1, -1)).
 * Outputs dq [nq][d], dk, dv [nk][d], and lse [nq], dd [nq] (D_i).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_attention_bwd(const double *q, int64_t nq, const double *k, const double *v,
                         int64_t nk, int64_t d, double scale, int64_t wl, int64_t wr,
                         const double *dout, double *dq, double *dk, double *dv, double *lse,
                         double *dd, int nthreads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || !lse || !dd || nq < 0 || nk < 0 || d <= 0)
        return -1;
    bwd_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.dout = dout;
    J.nq = nq; J.nk = nk; J.d = d;
    J.scale = scale; J.wl = wl; J.wr = wr;
    J.lse = lse; J.dd = dd; J.dq = dq; J.dk = dk; J.dv = dv;
    run_sweep(&J, 0, nq, nthreads);
    run_sweep(&J, 1, nk, nthreads);
    run_sweep(&J, 2, nq, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The two-pass normaliser over the rows of a matrix                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    const double *x;
    int64_t cols;
    const int64_t *sel;
    int64_t r_begin, r_end;
    double *p, *lse;
} softmax_rows_job;

static void *softmax_rows_worker(void *arg)
{
    softmax_rows_job *job = (softmax_rows_job *)arg;
    for (int64_t r = job->r_begin; r < job->r_end; ++r) {
        int64_t i = job->sel ? job->sel[r] : r;
        oracle_softmax_two_pass(job->x + i * job->cols, job->cols, job->p + r * job->cols,
                                job->lse + r);
    }
    return NULL;
}

/*
 * x [rows][cols] row-major fp64; sel[nsel] : rows to compute (NULL: all rows,
 * nsel must equal rows).  p [nsel][cols], lse [nsel] : oracle_softmax_two_pass
 * of each selected row, in the order of `sel`.  Rows are spread over
 * `nthreads` POSIX threads.  Returns 0, or -1 on a bad argument.
 */
int oracle_softmax_rows(const double *x, int64_t rows, int64_t cols, const int64_t *sel,
                        int64_t nsel, double *p, double *lse, int nthreads)
{
    if (!x || !p || !lse || rows < 0 || cols < 0 || nsel < 0)
        return -1;
    if (!sel && nsel != rows)
        return -1;
    for (int64_t r = 0; sel && r < nsel; ++r)
        if (sel[r] < 0 || sel[r] >= rows)
            return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nsel)
        nthreads = nsel > 0 ? (int)nsel : 1;
    softmax_rows_job jobs[256];
    pthread_t tids[256];
    int created[256];
    if (nthreads > 256)
        nthreads = 256;
    int64_t per = (nsel + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].x = x;
        jobs[t].cols = cols;
        jobs[t].sel = sel;
        jobs[t].r_begin = (int64_t)t * per < nsel ? (int64_t)t * per : nsel;
        jobs[t].r_end = jobs[t].r_begin + per < nsel ? jobs[t].r_begin + per : nsel;
        jobs[t].p = p;
        jobs[t].lse = lse;
        created[t] = 0;
    }
    for (int t = 0; t < nthreads; ++t) {
        if (nthreads > 1 && pthread_create(&tids[t], NULL, softmax_rows_worker, &jobs[t]) == 0)
            created[t] = 1;
        else
            softmax_rows_worker(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (created[t])
            pthread_join(tids[t], NULL);
    return 0;
}
