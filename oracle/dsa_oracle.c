/*
 * dsa_oracle.c -- host oracle for the DeepSeek-Sparse-Attention hot path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE: see dsa_oracle.h for who may call it,
 * the sources each function follows, and the argument conventions.
 *
 * Plain C11, double accumulation, no blocking or reordering beyond the plain
 * definition.  The optional OpenMP pragmas only split independent outputs (one
 * key, one head) between threads; every individual sum runs in index order, so
 * results are identical with any thread count.
 */
#include "dsa_oracle.h"

#include <math.h>
#include <omp.h>
#include <stdlib.h>
#include <string.h>

int oracle_set_threads(int32_t n) {
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
}

int oracle_index_scores(const float *q, const float *w, const float *keys,
                        int64_t n_keys, int32_t heads, int32_t dim, double *scores)
{
    if (n_keys < 0 || heads <= 0 || dim <= 0) return -1;
    if (n_keys > 0 && (!q || !w || !keys || !scores)) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n_keys; t++) {
        const float *kt = keys + t * (int64_t)dim;
        double s = 0.0;
        for (int32_t h = 0; h < heads; h++) {
            const float *qh = q + (int64_t)h * dim;
            double d = 0.0;
            for (int32_t i = 0; i < dim; i++) d += (double)qh[i] * (double)kt[i];
            double relu = d > 0.0 ? d : 0.0;          /* ReLU on the per-head dot */
            s += (double)w[h] * relu;                 /* weighted sum over heads  */
        }
        scores[t] = s;
    }
    return 0;
}

typedef struct {
    double s;
    int64_t i;
} scored_t;

/* Total order of the selection: higher score first, then lower index first. */
static int cmp_score_desc_index_asc(const void *pa, const void *pb)
{
    const scored_t *a = (const scored_t *)pa, *b = (const scored_t *)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i) ? 1 : 0;
}

static int cmp_i32_asc(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a < b) ? -1 : (a > b) ? 1 : 0;
}

int oracle_topk(const double *scores, int64_t n, int64_t k, int32_t *idx, int64_t *n_sel)
{
    if (n < 0 || k < 0 || !n_sel) return -1;
    if (n > 0 && (!scores || !idx)) return -1;
    if (n > INT32_MAX) return -1;
    if (n <= k) {                                     /* dense: every index */
        for (int64_t t = 0; t < n; t++) idx[t] = (int32_t)t;
        *n_sel = n;
        return 0;
    }
    scored_t *all = (scored_t *)malloc((size_t)n * sizeof(scored_t));
    if (!all) return -2;
    for (int64_t t = 0; t < n; t++) { all[t].s = scores[t]; all[t].i = t; }
    qsort(all, (size_t)n, sizeof(scored_t), cmp_score_desc_index_asc);
    for (int64_t j = 0; j < k; j++) idx[j] = (int32_t)all[j].i;
    free(all);
    qsort(idx, (size_t)k, sizeof(int32_t), cmp_i32_asc);   /* emit ascending */
    *n_sel = k;
    return 0;
}

int oracle_kpool_select(const double *pool_scores, int64_t L, int64_t k, int32_t kpool,
                        int32_t *idx, int64_t *n_sel)
{
    if (L < 0 || k <= 0 || kpool <= 0 || !n_sel || !idx) return -1;
    if (k % kpool != 0) return -1;
    if (L > INT32_MAX) return -1;
    int64_t n_pool = L / kpool;                       /* complete pools */
    int64_t keep = k / kpool;                         /* pools a query may keep */
    if (n_pool <= keep) {                             /* dense: every token */
        for (int64_t t = 0; t < L; t++) idx[t] = (int32_t)t;
        *n_sel = L;
        return 0;
    }
    if (!pool_scores) return -1;
    int32_t *pools = (int32_t *)malloc((size_t)keep * sizeof(int32_t));
    if (!pools) return -2;
    int64_t n_pools_sel = 0;
    int rc = oracle_topk(pool_scores, n_pool, keep, pools, &n_pools_sel);
    if (rc != 0) { free(pools); return rc; }
    int64_t m = 0;
    for (int64_t j = 0; j < n_pools_sel; j++)         /* expand pools to tokens */
        for (int32_t r = 0; r < kpool; r++) idx[m++] = (int32_t)((int64_t)pools[j] * kpool + r);
    for (int64_t t = n_pool * kpool; t < L; t++) idx[m++] = (int32_t)t;   /* unfilled tail */
    free(pools);
    *n_sel = m;
    return 0;
}

/* Softmax-weighted pooling of the latent for one head over a list of logits. */
static void attend_head(const double *z, const float *const *row_ptr, int64_t n, int32_t dv,
                        double *out_h, double *lse_h)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; j++) if (z[j] > m) m = z[j];
    double l = 0.0;
    for (int32_t c = 0; c < dv; c++) out_h[c] = 0.0;
    for (int64_t j = 0; j < n; j++) {
        if (z[j] == -INFINITY) continue;              /* masked row: weight exactly 0 */
        double p = exp(z[j] - m);
        l += p;
        const float *r = row_ptr[j];
        for (int32_t c = 0; c < dv; c++) out_h[c] += p * (double)r[c];
    }
    for (int32_t c = 0; c < dv; c++) out_h[c] /= l;
    if (lse_h) *lse_h = m + log(l);
}

static double dot_row(const float *q, const float *r, int32_t width)
{
    double a = 0.0;
    for (int32_t c = 0; c < width; c++) a += (double)q[c] * (double)r[c];
    return a;
}

/* (score, unit) pairs for the descending sort: larger score first, then the
 * smaller unit. */
typedef struct { double s; int64_t u; } unit_key;

static int cmp_desc(const void *pa, const void *pb)
{
    const unit_key *a = (const unit_key *)pa, *b = (const unit_key *)pb;
    if (a->s != b->s) return a->s > b->s ? -1 : 1;
    return (a->u > b->u) - (a->u < b->u);
}

int oracle_order_desc(const double *unit_scores, int64_t n_units, const int32_t *sel,
                      int64_t n_sel, int64_t L, int32_t kpool, int32_t *out)
{
    if (n_sel < 0 || kpool <= 0 || L < 0 || n_units < 0) return -1;
    if (n_sel > 0 && (!sel || !out || !unit_scores)) return -1;
    const int64_t tail = kpool > 1 ? L % kpool : 0;       /* rows of the unfilled pool */
    if (n_sel < tail || (n_sel - tail) % kpool != 0) return -1;
    const int64_t n = (n_sel - tail) / kpool;               /* selected units */
    unit_key *k = (unit_key *)malloc((size_t)(n > 0 ? n : 1) * sizeof(unit_key));
    if (!k) return -1;
    for (int64_t i = 0; i < n; i++) {
        const int64_t u = sel[i * kpool] / kpool;           /* the unit's first row / kpool */
        if (u < 0 || u >= n_units) { free(k); return -1; }
        k[i].s = unit_scores[u];
        k[i].u = u;
    }
    qsort(k, (size_t)n, sizeof(unit_key), cmp_desc);
    for (int64_t i = 0; i < n; i++)
        for (int32_t r = 0; r < kpool; r++) out[i * kpool + r] = (int32_t)(k[i].u * kpool + r);
    for (int64_t i = n * kpool; i < n_sel; i++) out[i] = sel[i];   /* the tail, as it was */
    free(k);
    return 0;
}

int oracle_sparse_mla(const float *q_abs, const float *rows, int64_t n_rows, int32_t heads,
                      int32_t width, int32_t dv, double scale, const int32_t *idx,
                      int64_t n_sel, double *out, double *lse)
{
    if (heads <= 0 || width <= 0 || dv <= 0 || dv > width || n_sel <= 0 || n_rows <= 0) return -1;
    if (!q_abs || !rows || !idx || !out) return -1;
    for (int64_t j = 0; j < n_sel; j++) if (idx[j] < 0 || idx[j] >= n_rows) return -1;
    const float **row_ptr = (const float **)malloc((size_t)n_sel * sizeof(float *));
    double *zall = (double *)malloc((size_t)n_sel * (size_t)heads * sizeof(double));
    if (!row_ptr || !zall) { free(row_ptr); free(zall); return -2; }
    for (int64_t j = 0; j < n_sel; j++) row_ptr[j] = rows + (int64_t)idx[j] * width;
#pragma omp parallel for schedule(static)
    for (int32_t h = 0; h < heads; h++) {
        const float *qh = q_abs + (int64_t)h * width;
        double *z = zall + (int64_t)h * n_sel;
        for (int64_t j = 0; j < n_sel; j++) z[j] = scale * dot_row(qh, row_ptr[j], width);
        attend_head(z, row_ptr, n_sel, dv, out + (int64_t)h * dv, lse ? lse + h : NULL);
    }
    free(zall);
    free(row_ptr);
    return 0;
}

int oracle_dense_masked_mla(const float *q_abs, const float *rows, int64_t n_rows,
                            int32_t heads, int32_t width, int32_t dv, double scale,
                            const uint8_t *mask, double *out, double *lse)
{
    if (heads <= 0 || width <= 0 || dv <= 0 || dv > width || n_rows <= 0) return -1;
    if (!q_abs || !rows || !mask || !out) return -1;
    int64_t n_on = 0;
    for (int64_t t = 0; t < n_rows; t++) n_on += mask[t] != 0;
    if (n_on == 0) return -1;
    const float **row_ptr = (const float **)malloc((size_t)n_rows * sizeof(float *));
    double *zall = (double *)malloc((size_t)n_rows * (size_t)heads * sizeof(double));
    if (!row_ptr || !zall) { free(row_ptr); free(zall); return -2; }
    for (int64_t t = 0; t < n_rows; t++) row_ptr[t] = rows + t * (int64_t)width;
#pragma omp parallel for schedule(static)
    for (int32_t h = 0; h < heads; h++) {
        const float *qh = q_abs + (int64_t)h * width;
        double *z = zall + (int64_t)h * n_rows;
        for (int64_t t = 0; t < n_rows; t++)
            z[t] = mask[t] ? scale * dot_row(qh, row_ptr[t], width) : -INFINITY;
        attend_head(z, row_ptr, n_rows, dv, out + (int64_t)h * dv, lse ? lse + h : NULL);
    }
    free(zall);
    free(row_ptr);
    return 0;
}

int oracle_decode_step(const float *q_idx, const float *w, const float *keys,
                       int32_t idx_heads, int32_t idx_dim, const float *q_abs,
                       const float *rows, int64_t L, int32_t heads, int32_t width,
                       int32_t dv, double scale, int64_t k, int32_t kpool,
                       double *scores_out, int32_t *idx, int64_t *n_sel,
                       double *out, double *lse)
{
    if (L <= 0 || kpool <= 0 || k <= 0) return -1;
    int64_t n_keys = L / kpool;
    double *sc = scores_out;
    if (!sc && n_keys > 0) {
        sc = (double *)malloc((size_t)n_keys * sizeof(double));
        if (!sc) return -2;
    }
    int rc = 0;
    /* The dense shortcut skips scoring entirely ([GLM-DOC] "The sparse-attention
     * path"); the scores are still produced here so callers can inspect them. */
    if (n_keys > 0) rc = oracle_index_scores(q_idx, w, keys, n_keys, idx_heads, idx_dim, sc);
    if (rc == 0) rc = oracle_kpool_select(sc, L, k, kpool, idx, n_sel);
    if (rc == 0) rc = oracle_sparse_mla(q_abs, rows, L, heads, width, dv, scale, idx, *n_sel, out, lse);
    if (sc != scores_out) free(sc);
    return rc;
}

int oracle_pool_compress(const float *cells, int64_t n_pools, const float *pos, int32_t kpool,
                         int32_t dim, double *out)
{
    if (n_pools < 0 || kpool <= 0 || dim <= 0) return -1;
    if (n_pools > 0 && (!cells || !pos || !out)) return -1;
    const int64_t cell_w = 2 * (int64_t)dim;               /* key then gate */
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < n_pools; p++) {
        const float *pool = cells + p * kpool * cell_w;
        for (int32_t c = 0; c < dim; c++) {
            /* logits of the slots: the cell's gate plus its slot's embedding */
            double zmax = -INFINITY;
            for (int32_t i = 0; i < kpool; i++) {
                const double z = (double)pool[i * cell_w + dim + c] + (double)pos[(int64_t)i * dim + c];
                if (z > zmax) zmax = z;
            }
            /* every slot masked (logit -inf): no weight anywhere, the key is 0 */
            if (zmax == -INFINITY) {
                out[p * dim + c] = 0.0;
                continue;
            }
            /* softmax over the slots (max-subtracted), weighted sum of the keys;
             * a masked slot has weight exp(-inf) = 0 */
            double den = 0.0, num = 0.0;
            for (int32_t i = 0; i < kpool; i++) {
                const double z = (double)pool[i * cell_w + dim + c] + (double)pos[(int64_t)i * dim + c];
                const double e = exp(z - zmax);
                den += e;
                num += e * (double)pool[i * cell_w + c];
            }
            out[p * dim + c] = num / den;
        }
    }
    return 0;
}

int oracle_new_pools(int64_t L, int64_t q_len, int32_t kpool, int64_t *j0, int64_t *j1)
{
    if (L < 0 || q_len < 0 || q_len > L || kpool <= 0 || !j0 || !j1) return -1;
    *j0 = (L - q_len) / kpool;
    *j1 = L / kpool;
    return 0;
}

int oracle_hadamard(const double *x, int32_t n, double *out)
{
    if (n <= 0 || (n & (n - 1)) != 0 || !x || !out || x == out) return -1;
    const double norm = 1.0 / sqrt((double)n);
    for (int32_t i = 0; i < n; i++) {
        double s = 0.0;
        for (int32_t j = 0; j < n; j++) {
            const int odd = __builtin_popcount((unsigned)(i & j)) & 1;   /* sign (-1)^popcount */
            s += odd ? -x[j] : x[j];
        }
        out[i] = s * norm;
    }
    return 0;
}

int oracle_rope(const float *x, int32_t dim, int32_t rope_dims, double base, int64_t pos,
                double *out)
{
    if (dim <= 0 || rope_dims < 0 || rope_dims > dim || (rope_dims & 1) || !(base > 0.0) ||
        !x || !out)
        return -1;
    for (int32_t i = 0; i < rope_dims / 2; i++) {
        const double theta = pow(base, -2.0 * i / (double)rope_dims);
        const double a = (double)pos * theta;
        const double c = cos(a), s = sin(a);
        const double x0 = x[2 * i], x1 = x[2 * i + 1];
        out[2 * i] = x0 * c - x1 * s;
        out[2 * i + 1] = x0 * s + x1 * c;
    }
    for (int32_t d = rope_dims; d < dim; d++) out[d] = x[d];
    return 0;
}

int oracle_index_prepare(const float *x, const int64_t *pos, int64_t n, int32_t dim,
                         int32_t rope_dims, double base, double *out)
{
    if (n < 0 || dim <= 0 || dim > 4096) return -1;
    if (n > 0 && (!x || !pos || !out)) return -1;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(|:bad)
    for (int64_t v = 0; v < n; v++) {
        double r[4096];
        bad |= oracle_rope(x + v * dim, dim, rope_dims, base, pos[v], r) != 0;   /* rope first */
        bad |= oracle_hadamard(r, dim, out + v * dim) != 0;                      /* then rotate */
    }
    return bad ? -1 : 0;
}

int oracle_absorb_q(const float *q, const float *w_uk, int32_t heads, int32_t nope, int32_t rope,
                    int32_t kv_lora, double *q_abs)
{
    if (heads <= 0 || nope < 0 || rope < 0 || kv_lora <= 0 || !q || !q_abs) return -1;
    if (nope > 0 && !w_uk) return -1;
    const int64_t qw = (int64_t)nope + rope, aw = (int64_t)kv_lora + rope;
#pragma omp parallel for schedule(static)
    for (int32_t h = 0; h < heads; h++) {
        const float *qh = q + h * qw;
        const float *wh = w_uk + (int64_t)h * nope * kv_lora;
        for (int32_t i = 0; i < kv_lora; i++) {
            double s = 0.0;
            for (int32_t d = 0; d < nope; d++) s += (double)qh[d] * (double)wh[(int64_t)d * kv_lora + i];
            q_abs[h * aw + i] = s;                       /* the query in the latent */
        }
        for (int32_t r = 0; r < rope; r++) q_abs[h * aw + kv_lora + r] = qh[nope + r];
    }
    return 0;
}

int oracle_up_project(const double *o, const float *w_uv, int32_t heads, int32_t kv_lora,
                      int32_t v_dim, double *out)
{
    if (heads <= 0 || kv_lora <= 0 || v_dim <= 0 || !o || !w_uv || !out) return -1;
#pragma omp parallel for schedule(static)
    for (int32_t h = 0; h < heads; h++) {
        const double *oh = o + (int64_t)h * kv_lora;
        const float *wh = w_uv + (int64_t)h * v_dim * kv_lora;
        for (int32_t v = 0; v < v_dim; v++) {
            double s = 0.0;
            for (int32_t i = 0; i < kv_lora; i++) s += (double)wh[(int64_t)v * kv_lora + i] * oh[i];
            out[(int64_t)h * v_dim + v] = s;
        }
    }
    return 0;
}
