/*
 * ref_attn.c -- fp64 reference for exact attention forward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.
 *
 * What it computes is the plain definition that the FlashAttention-4 method
 * reaches exactly (up to rounding order): "FlashAttention-4: Algorithm and
 * Kernel Pipelining Co-Design for Asymmetric Hardware Scaling", Method,
 * and §3.1.4 (the final 1/l normalisation recovers the exact
 * softmax-times-V output). For every (b, h, i):
 *
 *   g      = h / (Hq / Hkv)                       kv head of query head h
 *   x_j    = scale * sum_e q[b,i,h,e] * k[b,j,g,e]   (BF16 widened exactly)
 *   valid  = !causal || j <= i + (Sk - Sq)         bottom-right causal mask
 *   m      = max_{valid j} x_j
 *   w_j    = exp(x_j - m) for valid j, else 0
 *   l      = sum_j w_j
 *   O[b,i,h,:]  = sum_j w_j * v[b,j,g,:] / l
 *   LSE[b,h,i]  = m + ln(l)
 *
 * A row with no valid key gets O = 0 and LSE = -inf.
 *
 * Each row materialises its full score row (naive softmax). There is no
 * blocking, no online softmax and no reordering beyond the definition.
 * Layouts: q/o [B,Sq,Hq,d], k/v [B,Sk,Hkv,d] (BF16 bit patterns in, fp64
 * out), lse [B,Hq,Sq]. OpenMP parallelises over output rows only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_bits_to_f64(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int64_t B, Hq, Hkv, Sq, Sk, d;
    double scale;
    int causal;
} attn_args;

static int check_args(const attn_args *a)
{
    if (!a->q || !a->k || !a->v) return -1;
    if (a->B < 1 || a->Hq < 1 || a->Hkv < 1 || a->Sq < 0 || a->Sk < 0 || a->d < 1) return -1;
    if (a->Hq % a->Hkv != 0) return -1;
    if (!(a->scale > 0.0) || !isfinite(a->scale)) return -1;
    return 0;
}

/* Materialise x_j (scaled logits) for one query row; returns the number of
 * valid keys. xs must hold Sk doubles, qrow d doubles. */
static int64_t score_row(const attn_args *a, int64_t b, int64_t h, int64_t i,
                         double *qrow, double *xs, unsigned char *valid)
{
    const int64_t g = h / (a->Hq / a->Hkv);
    const uint16_t *qp = a->q + ((b * a->Sq + i) * a->Hq + h) * a->d;
    for (int64_t e = 0; e < a->d; ++e) qrow[e] = bf16_bits_to_f64(qp[e]);
    int64_t nvalid = 0;
    for (int64_t j = 0; j < a->Sk; ++j) {
        valid[j] = (unsigned char)(!a->causal || j <= i + (a->Sk - a->Sq));
        if (!valid[j]) { xs[j] = -INFINITY; continue; }
        const uint16_t *kp = a->k + ((b * a->Sk + j) * a->Hkv + g) * a->d;
        double dot = 0.0;
        for (int64_t e = 0; e < a->d; ++e) dot += qrow[e] * bf16_bits_to_f64(kp[e]);
        xs[j] = a->scale * dot;
        ++nvalid;
    }
    return nvalid;
}

/* O row (d doubles) and LSE for one (b, h, i). If probs is non-null it
 * receives the normalised softmax row P_ij (Sk doubles). */
static void attend_row(const attn_args *a, int64_t b, int64_t h, int64_t i,
                       double *qrow, double *xs, unsigned char *valid,
                       double *orow, double *lse, double *probs)
{
    const int64_t g = h / (a->Hq / a->Hkv);
    const int64_t nvalid = score_row(a, b, h, i, qrow, xs, valid);
    for (int64_t e = 0; e < a->d; ++e) orow[e] = 0.0;
    if (nvalid == 0) {
        *lse = -INFINITY;
        if (probs) for (int64_t j = 0; j < a->Sk; ++j) probs[j] = 0.0;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < a->Sk; ++j)
        if (valid[j] && xs[j] > m) m = xs[j];
    double l = 0.0;
    for (int64_t j = 0; j < a->Sk; ++j) {
        xs[j] = valid[j] ? exp(xs[j] - m) : 0.0; /* xs now holds w_j */
        l += xs[j];
    }
    for (int64_t j = 0; j < a->Sk; ++j) {
        if (xs[j] == 0.0) continue;
        const uint16_t *vp = a->v + ((b * a->Sk + j) * a->Hkv + g) * a->d;
        for (int64_t e = 0; e < a->d; ++e) orow[e] += xs[j] * bf16_bits_to_f64(vp[e]);
    }
    for (int64_t e = 0; e < a->d; ++e) orow[e] /= l;
    *lse = m + log(l);
    if (probs) for (int64_t j = 0; j < a->Sk; ++j) probs[j] = xs[j] / l;
}

/* Number of OpenMP threads a parallel region here will use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Evaluate the listed rows only. rows[r] = (b*Hq + h)*Sq + i; o_rows is
 * [n_rows, d], lse_rows [n_rows]. Returns 0, or -1 on bad arguments. */
int oracle_attn_fwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk,
                         int64_t d, double scale, int causal,
                         const int64_t *rows, int64_t n_rows,
                         double *o_rows, double *lse_rows)
{
    attn_args a = {q, k, v, B, Hq, Hkv, Sq, Sk, d, scale, causal};
    if (check_args(&a) || !rows || !o_rows || !lse_rows || n_rows < 0) return -1;
    const int64_t total = B * Hq * Sq;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= total) return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
        double *xs = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        unsigned char *valid = (unsigned char *)malloc((size_t)(Sk > 0 ? Sk : 1));
        if (!qrow || !xs || !valid) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t r = 0; r < n_rows; ++r) {
                const int64_t id = rows[r];
                const int64_t i = id % Sq;
                const int64_t h = (id / Sq) % Hq;
                const int64_t b = id / (Sq * Hq);
                attend_row(&a, b, h, i, qrow, xs, valid, o_rows + r * d, lse_rows + r, NULL);
            }
        }
        free(qrow); free(xs); free(valid);
    }
    return bad ? -2 : 0;
}

/* Every row: o [B,Sq,Hq,d], lse [B,Hq,Sq]. */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    double *o, double *lse,
                    int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d,
                    double scale, int causal)
{
    attn_args a = {q, k, v, B, Hq, Hkv, Sq, Sk, d, scale, causal};
    if (check_args(&a) || !o || !lse) return -1;
    const int64_t total = B * Hq * Sq;
    int bad = 0;
#pragma omp parallel
    {
        double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
        double *xs = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        unsigned char *valid = (unsigned char *)malloc((size_t)(Sk > 0 ? Sk : 1));
        if (!qrow || !xs || !valid) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t id = 0; id < total; ++id) {
                const int64_t i = id % Sq;
                const int64_t h = (id / Sq) % Hq;
                const int64_t b = id / (Sq * Hq);
                double *orow = o + ((b * Sq + i) * Hq + h) * d;
                attend_row(&a, b, h, i, qrow, xs, valid, orow, lse + id, NULL);
            }
        }
        free(qrow); free(xs); free(valid);
    }
    return bad ? -2 : 0;
}

/* Normalised softmax matrix P [Sq, Sk] for one (b, h): for invariant checks
 * on small inputs. */
int oracle_attn_probs(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d,
                      double scale, int causal, int64_t b, int64_t h, double *probs)
{
    attn_args a = {q, k, v, B, Hq, Hkv, Sq, Sk, d, scale, causal};
    if (check_args(&a) || !probs || b < 0 || b >= B || h < 0 || h >= Hq) return -1;
    double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
    double *xs = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
    unsigned char *valid = (unsigned char *)malloc((size_t)(Sk > 0 ? Sk : 1));
    double *orow = (double *)malloc(sizeof(double) * (size_t)d);
    int rc = 0;
    if (!qrow || !xs || !valid || !orow) {
        rc = -2;
    } else {
        for (int64_t i = 0; i < Sq; ++i) {
            double lse;
            attend_row(&a, b, h, i, qrow, xs, valid, orow, &lse, probs + i * Sk);
        }
    }
    free(qrow); free(xs); free(valid); free(orow);
    return rc;
}
