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

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
