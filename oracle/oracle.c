/*
 * oracle.c -- plain fp64 CPU reference for the scaled-dot-product attention
 * forward pass.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it; the product path never does.
 *
 * What it computes (definition, not an algorithm):
 *   For batch b, query head h, query row i, with key/value head
 *   g = h / (Hq / Hkv)                     [grouped-query mapping: JAX Pallas
 *                                           attention_mgpu.py, `_attention_forward`,
 *                                           kv_head = q_head // q_heads_per_kv_head]
 *   s_j   = scale * sum_d q[b,i,h,d] * k[b,j,g,d]        for every visible key j
 *   m     = max_j s_j
 *   l     = sum_j exp(s_j - m)
 *   o[d]  = sum_j exp(s_j - m) * v[b,j,g,d] / l
 *   lse   = m + ln(l)                      (natural log-sum-exp of the scaled logits)
 * This is `attention_reference` of the Pallas page (fp32 einsum, max, exp,
 * divide by the row sum) written out in fp64, with the caller's scale applied
 * to the logits and a natural-log LSE.
 *
 * Visibility: without a mask (causal=0) every key 0..Skv-1 is visible.  With
 * causal=1 the mask is bottom-right aligned: key j is visible from query i iff
 * j <= i + (Skv - Sq).  With causal=2 it is top-left aligned: j <= i, the rule of
 * the Pallas page's reference (`mask = q_idx >= kv_idx`); the two coincide when
 * Sq == Skv.
 * A row with no visible key gets o = 0 and lse = -inf (the pages leave this
 * case open; this is the reading the tests and the GPU path share).
 *
 * Inputs are raw 16-bit patterns ([B,Sq,Hq,D] for q, [B,Skv,Hkv,D] for k and
 * v, D contiguous) of bf16 or, with f16 = 1, IEEE binary16 (the Pallas page
 * accepts both), widened exactly to fp64.  Nothing is blocked, fused or
 * reordered: each row is two passes over its keys (max, then sums).
 *
 * The partial-triple entry point returns the un-normalised (m, l, o) of a row
 * over a sub-range of keys; merging such triples is the rule of the kernbench
 * page (`_merge_running`), used by the tests to pin the one-shot definition.
 *
 * Backward (gradients; the Pallas page's `_attention_bwd`, written out as the
 * plain vector-Jacobian product of the definition above).  Given dO, the
 * gradient of L = sum dO[b,i,h,d] * o[b,i,h,d] with respect to q, k and v:
 *   p_ij    = exp(s_ij - lse_i)                 normalised weight, visible j only
 *   dp_ij   = sum_d dO[b,i,h,d] * v[b,j,g,d]
 *   delta_i = sum_j p_ij * dp_ij                (equals dO_i . o_i)
 *   ds_ij   = p_ij * (dp_ij - delta_i)          (Jacobian of the row softmax)
 *   dq[b,i,h,:] = scale * sum_j ds_ij * k[b,j,g,:]
 *   dk[b,j,g,:] = scale * sum_{h in group g} sum_i ds_ij * q[b,i,h,:]
 *   dv[b,j,g,:] =         sum_{h in group g} sum_i p_ij  * dO[b,i,h,:]
 * The page sums per-query-head dk/dv over each group of heads sharing a
 * key/value head; here the sums run over the group directly.  dO has q's
 * layout and element format.  Rows with no visible key contribute nothing.
 * The page's backward rejects the causal mask; these functions apply the same
 * visibility rule as the forward (a masked pair has p_ij = 0), the gradient of
 * the masked forward.
 * The page's backward kernel takes delta_i from the stored forward output
 * (its residual `out`, in the input's element type) rather than from the
 * exact o_i.  Each backward entry point therefore also accepts delta_i from
 * the caller (delta_in, [B,Hq,Sq]); dq, dk, dv are affine in it and the
 * other quantities are unchanged.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double widen_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: sign, 5-bit exponent (bias 15), 10-bit fraction; exact in fp64 */
static double widen_f16(uint16_t bits) {
    const int sign = bits >> 15, e = (bits >> 10) & 0x1F, frac = bits & 0x3FF;
    double mag;
    if (e == 0)
        mag = ldexp((double)frac, -24); /* zero and subnormals */
    else if (e == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), e - 25);
    return sign ? -mag : mag;
}

typedef struct {
    const uint16_t *q, *k, *v;
    long B, Sq, Skv, Hq, Hkv, D;
    int causal;
    double scale;
    int f16; /* element format of q, k, v: 0 bf16, 1 IEEE binary16 */
} problem_t;

static double widen(const problem_t *p, uint16_t bits) {
    return p->f16 ? widen_f16(bits) : widen_bf16(bits);
}

/* last visible key index + 1 for query row i (may be <= 0: no visible key) */
static long visible_end(const problem_t *p, long i) {
    if (p->causal == 0) return p->Skv;
    long end = (p->causal == 1) ? i + (p->Skv - p->Sq) + 1 : i + 1;
    return end < p->Skv ? end : p->Skv;
}

/* Un-normalised triple of one row over keys [j_lo, j_hi) intersected with the
 * visible set.  s_buf holds at least (j_hi - j_lo) doubles, qd at least D. */
static void row_triple(const problem_t *p, long b, long h, long i, long j_lo, long j_hi,
                       double *s_buf, double *qd, double *m_out, double *l_out,
                       double *o_out) {
    const long D = p->D;
    const long g = h / (p->Hq / p->Hkv);
    long end = visible_end(p, i);
    if (end > j_hi) end = j_hi;
    for (long d = 0; d < D; ++d) o_out[d] = 0.0;
    if (end <= j_lo) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    const uint16_t *qrow = p->q + ((b * p->Sq + i) * p->Hq + h) * D;
    for (long d = 0; d < D; ++d) qd[d] = widen(p, qrow[d]);

    /* pass 1: scaled logits and their maximum */
    double m = -INFINITY;
    for (long j = j_lo; j < end; ++j) {
        const uint16_t *krow = p->k + ((b * p->Skv + j) * p->Hkv + g) * D;
        double acc = 0.0;
        for (long d = 0; d < D; ++d) acc += qd[d] * widen(p, krow[d]);
        double s = p->scale * acc;
        s_buf[j - j_lo] = s;
        if (s > m) m = s;
    }
    /* pass 2: weights exp(s - m), their sum, and the weighted sum of v rows */
    double l = 0.0;
    for (long j = j_lo; j < end; ++j) {
        double w = exp(s_buf[j - j_lo] - m);
        l += w;
        const uint16_t *vrow = p->v + ((b * p->Skv + j) * p->Hkv + g) * D;
        for (long d = 0; d < D; ++d) o_out[d] += w * widen(p, vrow[d]);
    }
    *m_out = m;
    *l_out = l;
}

static int check_dims(long B, long Sq, long Skv, long Hq, long Hkv, long D) {
    if (B < 1 || Sq < 1 || Skv < 1 || Hq < 1 || Hkv < 1 || D < 1) return -1;
    if (Hq % Hkv != 0) return -1;
    return 0;
}

/*
 * Attention output for an explicit list of rows.
 * rows: nrows triples (b, h, i).  o_out: nrows*D doubles (normalised o).
 * lse_out: nrows doubles.  Returns 0, or -1 on bad arguments.
 */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, long B, long Sq,
                     long Skv, long Hq, long Hkv, long D, int causal, double scale, int f16,
                     long nrows, const long *rows, double *o_out, double *lse_out) {
    if (check_dims(B, Sq, Skv, Hq, Hkv, D) || causal < 0 || causal > 2) return -1;
    problem_t p = {q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, scale, f16 != 0};
    for (long r = 0; r < nrows; ++r) {
        const long *t = rows + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= Hq || t[2] < 0 || t[2] >= Sq)
            return -1;
    }
    int bad = 0;
#pragma omp parallel
    {
        double *s_buf = (double *)malloc(sizeof(double) * (size_t)Skv);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s_buf || !qd) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long r = 0; r < nrows; ++r) {
                const long *t = rows + 3 * r;
                double m, l;
                double *o = o_out + r * D;
                row_triple(&p, t[0], t[1], t[2], 0, Skv, s_buf, qd, &m, &l, o);
                if (l > 0.0) {
                    for (long d = 0; d < D; ++d) o[d] /= l;
                    lse_out[r] = m + log(l);
                } else {
                    lse_out[r] = -INFINITY;
                }
            }
        }
        free(s_buf);
        free(qd);
    }
    return bad ? -1 : 0;
}

/*
 * Attention output for every row.  o_out: [B,Sq,Hq,D] doubles; lse_out: [B,Hq,Sq].
 */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, long B, long Sq,
                    long Skv, long Hq, long Hkv, long D, int causal, double scale, int f16,
                    double *o_out, double *lse_out) {
    if (check_dims(B, Sq, Skv, Hq, Hkv, D) || causal < 0 || causal > 2) return -1;
    problem_t p = {q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, scale, f16 != 0};
    const long nrows = B * Hq * Sq;
    int bad = 0;
#pragma omp parallel
    {
        double *s_buf = (double *)malloc(sizeof(double) * (size_t)Skv);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s_buf || !qd) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long r = 0; r < nrows; ++r) {
                long b = r / (Hq * Sq), h = (r / Sq) % Hq, i = r % Sq;
                double m, l;
                double *o = o_out + ((b * Sq + i) * Hq + h) * D;
                row_triple(&p, b, h, i, 0, Skv, s_buf, qd, &m, &l, o);
                if (l > 0.0) {
                    for (long d = 0; d < D; ++d) o[d] /= l;
                    lse_out[(b * Hq + h) * Sq + i] = m + log(l);
                } else {
                    lse_out[(b * Hq + h) * Sq + i] = -INFINITY;
                }
            }
        }
        free(s_buf);
        free(qd);
    }
    return bad ? -1 : 0;
}

/*
 * Un-normalised partial triple (m, l, o) of one row over keys [j_lo, j_hi):
 * m = max of the visible scaled logits in the range (-inf if none),
 * l = sum exp(s_j - m), o = sum exp(s_j - m) v_j.
 */
int oracle_partial_triple(const uint16_t *q, const uint16_t *k, const uint16_t *v, long B,
                          long Sq, long Skv, long Hq, long Hkv, long D, int causal,
                          double scale, int f16, long b, long h, long i, long j_lo, long j_hi,
                          double *m_out, double *l_out, double *o_out) {
    if (check_dims(B, Sq, Skv, Hq, Hkv, D) || causal < 0 || causal > 2) return -1;
    if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Sq) return -1;
    if (j_lo < 0 || j_hi > Skv || j_lo > j_hi) return -1;
    problem_t p = {q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, scale, f16 != 0};
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)(j_hi - j_lo + 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    int rc = 0;
    if (!s_buf || !qd)
        rc = -1;
    else
        row_triple(&p, b, h, i, j_lo, j_hi, s_buf, qd, m_out, l_out, o_out);
    free(s_buf);
    free(qd);
    return rc;
}

/* ------------------------------------------------------------------ backward */

/* Weights and softmax-Jacobian terms of one row: on return p_buf[j] = p_ij and
 * ds_buf[j] = ds_ij for j < *end_out (the row's visible keys), and, if dq is not
 * NULL, dq[0..D) = scale * sum_j ds_ij k_j.  qd, dod: D doubles of scratch.
 * Three passes over the keys: logits and their max; weights, lse and dp_ij with
 * delta_i = sum_j p_ij dp_ij; ds_ij and dq.  delta_in (NULL: the exact delta_i
 * above) supplies delta_i instead, indexed [(b * Hq + h) * Sq + i]. */
static void row_grad(const problem_t *p, const uint16_t *dO, const double *delta_in, long b,
                     long h, long i, double *p_buf, double *ds_buf, double *qd, double *dod,
                     double *dq, long *end_out) {
    const long D = p->D;
    const long g = h / (p->Hq / p->Hkv);
    const long end = visible_end(p, i);
    *end_out = end > 0 ? end : 0;
    if (dq)
        for (long d = 0; d < D; ++d) dq[d] = 0.0;
    if (end <= 0) return;
    const long qoff = ((b * p->Sq + i) * p->Hq + h) * D;
    for (long d = 0; d < D; ++d) {
        qd[d] = widen(p, p->q[qoff + d]);
        dod[d] = widen(p, dO[qoff + d]);
    }
    /* pass 1: scaled logits (kept in p_buf) and their maximum */
    double m = -INFINITY;
    for (long j = 0; j < end; ++j) {
        const uint16_t *krow = p->k + ((b * p->Skv + j) * p->Hkv + g) * D;
        double acc = 0.0;
        for (long d = 0; d < D; ++d) acc += qd[d] * widen(p, krow[d]);
        p_buf[j] = p->scale * acc;
        if (p_buf[j] > m) m = p_buf[j];
    }
    double l = 0.0;
    for (long j = 0; j < end; ++j) l += exp(p_buf[j] - m);
    const double lse = m + log(l);
    /* pass 2: normalised weights, dp_ij (kept in ds_buf) and delta_i */
    double delta = 0.0;
    for (long j = 0; j < end; ++j) {
        p_buf[j] = exp(p_buf[j] - lse);
        const uint16_t *vrow = p->v + ((b * p->Skv + j) * p->Hkv + g) * D;
        double dp = 0.0;
        for (long d = 0; d < D; ++d) dp += dod[d] * widen(p, vrow[d]);
        ds_buf[j] = dp;
        delta += p_buf[j] * dp;
    }
    if (delta_in) delta = delta_in[(b * p->Hq + h) * p->Sq + i];
    /* pass 3: ds_ij and dq */
    for (long j = 0; j < end; ++j) {
        ds_buf[j] = p_buf[j] * (ds_buf[j] - delta);
        if (dq) {
            const uint16_t *krow = p->k + ((b * p->Skv + j) * p->Hkv + g) * D;
            for (long d = 0; d < D; ++d) dq[d] += ds_buf[j] * widen(p, krow[d]);
        }
    }
    if (dq)
        for (long d = 0; d < D; ++d) dq[d] *= p->scale;
}

/*
 * Every gradient.  dO: [B,Sq,Hq,D] 16-bit patterns in q's format; delta_in:
 * NULL (exact delta_i) or [B,Hq,Sq] doubles (see row_grad).
 * dq_out: [B,Sq,Hq,D] doubles; dk_out, dv_out: [B,Skv,Hkv,D] doubles.
 * Parallel over (b, g): each thread owns the dk/dv rows of its key/value head.
 */
int oracle_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dO,
                    const double *delta_in, long B, long Sq, long Skv, long Hq, long Hkv, long D,
                    int causal, double scale, int f16, double *dq_out, double *dk_out,
                    double *dv_out) {
    if (check_dims(B, Sq, Skv, Hq, Hkv, D) || causal < 0 || causal > 2) return -1;
    problem_t p = {q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, scale, f16 != 0};
    const long G = Hq / Hkv;
    int bad = 0;
#pragma omp parallel
    {
        double *p_buf = (double *)malloc(sizeof(double) * (size_t)Skv);
        double *ds_buf = (double *)malloc(sizeof(double) * (size_t)Skv);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *dod = (double *)malloc(sizeof(double) * (size_t)D);
        if (!p_buf || !ds_buf || !qd || !dod) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long bg = 0; bg < B * Hkv; ++bg) {
                const long b = bg / Hkv, g = bg % Hkv;
                for (long j = 0; j < Skv; ++j)
                    for (long d = 0; d < D; ++d) {
                        dk_out[((b * Skv + j) * Hkv + g) * D + d] = 0.0;
                        dv_out[((b * Skv + j) * Hkv + g) * D + d] = 0.0;
                    }
                for (long h = g * G; h < (g + 1) * G; ++h)
                    for (long i = 0; i < Sq; ++i) {
                        long end;
                        double *dq = dq_out + ((b * Sq + i) * Hq + h) * D;
                        row_grad(&p, dO, delta_in, b, h, i, p_buf, ds_buf, qd, dod, dq, &end);
                        for (long j = 0; j < end; ++j) {
                            double *dk = dk_out + ((b * Skv + j) * Hkv + g) * D;
                            double *dv = dv_out + ((b * Skv + j) * Hkv + g) * D;
                            for (long d = 0; d < D; ++d) {
                                dk[d] += scale * ds_buf[j] * qd[d];
                                dv[d] += p_buf[j] * dod[d];
                            }
                        }
                    }
            }
        }
        free(p_buf);
        free(ds_buf);
        free(qd);
        free(dod);
    }
    return bad ? -1 : 0;
}

/*
 * dq of an explicit list of rows: rows holds nrows triples (b, h, i);
 * dq_out: nrows*D doubles; delta_in as for oracle_attn_bwd.
 */
int oracle_attn_bwd_dq_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const uint16_t *dO, const double *delta_in, long B, long Sq, long Skv,
                            long Hq, long Hkv, long D, int causal, double scale, int f16, long nrows,
                            const long *rows, double *dq_out) {
    if (check_dims(B, Sq, Skv, Hq, Hkv, D) || causal < 0 || causal > 2) return -1;
    problem_t p = {q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, scale, f16 != 0};
    for (long r = 0; r < nrows; ++r) {
        const long *t = rows + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= Hq || t[2] < 0 || t[2] >= Sq)
            return -1;
    }
    int bad = 0;
#pragma omp parallel
    {
        double *p_buf = (double *)malloc(sizeof(double) * (size_t)Skv);
        double *ds_buf = (double *)malloc(sizeof(double) * (size_t)Skv);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *dod = (double *)malloc(sizeof(double) * (size_t)D);
        if (!p_buf || !ds_buf || !qd || !dod) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long r = 0; r < nrows; ++r) {
                const long *t = rows + 3 * r;
                long end;
                row_grad(&p, dO, delta_in, t[0], t[1], t[2], p_buf, ds_buf, qd, dod,
                         dq_out + r * D, &end);
            }
        }
        free(p_buf);
        free(ds_buf);
        free(qd);
        free(dod);
    }
    return bad ? -1 : 0;
}

/*
 * dk and dv of an explicit list of keys: keys holds nkeys triples (b, g, j)
 * with g a key/value head; dk_out, dv_out: nkeys*D doubles each.  For every
 * (b, g) that occurs, the per-row lse_i and delta_i of the group's query heads
 * are computed once (one row pass each), then each listed key sums over the
 * rows that see it.  delta_in as for oracle_attn_bwd.
 */
int oracle_attn_bwd_dkv_keys(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             const uint16_t *dO, const double *delta_in, long B, long Sq, long Skv,
                             long Hq, long Hkv, long D, int causal, double scale, int f16, long nkeys,
                             const long *keys, double *dk_out, double *dv_out) {
    if (check_dims(B, Sq, Skv, Hq, Hkv, D) || causal < 0 || causal > 2) return -1;
    problem_t p = {q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, scale, f16 != 0};
    for (long r = 0; r < nkeys; ++r) {
        const long *t = keys + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= Hkv || t[2] < 0 || t[2] >= Skv)
            return -1;
    }
    const long G = Hq / Hkv;
    double *lse = (double *)malloc(sizeof(double) * (size_t)(G * Sq));
    double *delta = (double *)malloc(sizeof(double) * (size_t)(G * Sq));
    char *done = (char *)calloc((size_t)(B * Hkv), 1);
    int bad = (!lse || !delta || !done);
    for (long r0 = 0; r0 < nkeys && !bad; ++r0) {
        const long b = keys[3 * r0], g = keys[3 * r0 + 1];
        if (done[b * Hkv + g]) continue;
        done[b * Hkv + g] = 1;
        /* lse_i and delta_i of every row of the group's heads */
#pragma omp parallel
        {
            double *p_buf = (double *)malloc(sizeof(double) * (size_t)Skv);
            double *ds_buf = (double *)malloc(sizeof(double) * (size_t)Skv);
            double *qd = (double *)malloc(sizeof(double) * (size_t)D);
            double *dod = (double *)malloc(sizeof(double) * (size_t)D);
            if (!p_buf || !ds_buf || !qd || !dod) {
#pragma omp atomic write
                bad = 1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (long hi = 0; hi < G * Sq; ++hi) {
                    const long h = g * G + hi / Sq, i = hi % Sq;
                    const long end = visible_end(&p, i);
                    if (end <= 0) {
                        lse[hi] = -INFINITY;
                        delta[hi] = 0.0;
                        continue;
                    }
                    const long qoff = ((b * Sq + i) * Hq + h) * D;
                    for (long d = 0; d < D; ++d) {
                        qd[d] = widen(&p, q[qoff + d]);
                        dod[d] = widen(&p, dO[qoff + d]);
                    }
                    double m = -INFINITY;
                    for (long j = 0; j < end; ++j) {
                        const uint16_t *krow = k + ((b * Skv + j) * Hkv + g) * D;
                        double acc = 0.0;
                        for (long d = 0; d < D; ++d) acc += qd[d] * widen(&p, krow[d]);
                        p_buf[j] = scale * acc;
                        if (p_buf[j] > m) m = p_buf[j];
                    }
                    double l = 0.0;
                    for (long j = 0; j < end; ++j) l += exp(p_buf[j] - m);
                    const double ls = m + log(l);
                    double dl = 0.0;
                    for (long j = 0; j < end; ++j) {
                        const uint16_t *vrow = v + ((b * Skv + j) * Hkv + g) * D;
                        double dp = 0.0;
                        for (long d = 0; d < D; ++d) dp += dod[d] * widen(&p, vrow[d]);
                        dl += exp(p_buf[j] - ls) * dp;
                    }
                    lse[hi] = ls;
                    delta[hi] = delta_in ? delta_in[(b * Hq + h) * Sq + i] : dl;
                }
            }
            free(p_buf);
            free(ds_buf);
            free(qd);
            free(dod);
        }
        if (bad) break;
        /* every listed key of this (b, g) */
#pragma omp parallel for schedule(dynamic, 1)
        for (long r = 0; r < nkeys; ++r) {
            if (keys[3 * r] != b || keys[3 * r + 1] != g) continue;
            const long j = keys[3 * r + 2];
            double *dk = dk_out + r * D;
            double *dv = dv_out + r * D;
            for (long d = 0; d < D; ++d) dk[d] = dv[d] = 0.0;
            const uint16_t *krow = k + ((b * Skv + j) * Hkv + g) * D;
            const uint16_t *vrow = v + ((b * Skv + j) * Hkv + g) * D;
            for (long hi = 0; hi < G * Sq; ++hi) {
                const long h = g * G + hi / Sq, i = hi % Sq;
                if (j >= visible_end(&p, i)) continue;
                const uint16_t *qrow = q + ((b * Sq + i) * Hq + h) * D;
                const uint16_t *dorow = dO + ((b * Sq + i) * Hq + h) * D;
                double s = 0.0, dp = 0.0;
                for (long d = 0; d < D; ++d) {
                    s += widen(&p, qrow[d]) * widen(&p, krow[d]);
                    dp += widen(&p, dorow[d]) * widen(&p, vrow[d]);
                }
                const double pij = exp(scale * s - lse[hi]);
                const double ds = pij * (dp - delta[hi]);
                for (long d = 0; d < D; ++d) {
                    dk[d] += scale * ds * widen(&p, qrow[d]);
                    dv[d] += pij * widen(&p, dorow[d]);
                }
            }
        }
    }
    free(lse);
    free(delta);
    free(done);
    return bad ? -1 : 0;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
