/*
 * CPU oracle for the R-KV compression event -- TEST INFRASTRUCTURE ONLY.
 * Plain, slow, fp64 restatement of what the pages say R-KV computes; see
 * rkv_oracle.h for the sources and for every reading taken where the pages
 * are silent. Nothing here is shared with the CUDA library.
 */
#include "rkv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bf16 bit pattern (the upper half of an IEEE float). */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double dot_bf16(const uint16_t *a, const uint16_t *b, int d)
{
    double acc = 0.0;
    for (int c = 0; c < d; ++c)
        acc += bf16_value(a[c]) * bf16_value(b[c]);
    return acc;
}

/*
 * Importance ([RKV-blog] R-KV section, second step: multi-head attention
 * decides how much each cached token contributes; [RKV-review] "How R-KV
 * decides what to drop": the local window supplies the queries).
 * For each query row r: p_r = softmax_j(q_r . k_j / sqrt(d)) over all n keys
 * (readings R1-R3); I_j = mean_r p_r[j].
 */
void orc_importance(const uint16_t *q, int rows, const uint16_t *k, int n, int d, double *imp)
{
    double *logit = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    const double scale = 1.0 / sqrt((double)d);
    for (int j = 0; j < n; ++j)
        imp[j] = 0.0;
    for (int r = 0; r < rows; ++r) {
        const uint16_t *qr = q + (size_t)r * d;
        double mx = -INFINITY;
        for (int j = 0; j < n; ++j) {
            logit[j] = dot_bf16(qr, k + (size_t)j * d, d) * scale;
            if (logit[j] > mx)
                mx = logit[j];
        }
        double z = 0.0;
        for (int j = 0; j < n; ++j)
            z += exp(logit[j] - mx);
        for (int j = 0; j < n; ++j)
            imp[j] += exp(logit[j] - mx) / z / (double)rows;
    }
    free(logit);
}

/*
 * Redundancy ([RKV-blog] R-KV section, first step: cosine similarity of key
 * vectors flags repeated content). Pairwise definition, reading R4:
 * R_i = (1/(n-1)) * sum_{j != i} k_i.k_j / (|k_i| |k_j|).
 */
void orc_redundancy(const uint16_t *k, int n, int d, double *red)
{
    double *inv = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < n; ++i) {
        double nrm = sqrt(dot_bf16(k + (size_t)i * d, k + (size_t)i * d, d));
        inv[i] = nrm > 0.0 ? 1.0 / nrm : 0.0;
    }
    for (int i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int j = 0; j < n; ++j) {
            if (j == i)
                continue;
            acc += dot_bf16(k + (size_t)i * d, k + (size_t)j * d, d) * inv[i] * inv[j];
        }
        red[i] = n > 1 ? acc / (double)(n - 1) : 0.0;
    }
    free(inv);
}

/*
 * The same redundancy from the rank-one identity of the cosine sum: with
 * u_j = k_j / |k_j| (u_j = 0 for a zero key), sum_{j != i} cos(k_i, k_j) =
 * u_i . (sum_j u_j) - u_i . u_i, and u_i . u_i is 1 for a non-zero key, 0 for
 * a zero one. Exact algebra, so it equals orc_redundancy up to fp64 rounding;
 * it costs two passes over the keys instead of n^2 dot products.
 */
void orc_redundancy_closed(const uint16_t *k, int n, int d, double *red)
{
    double *inv = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *sum_u = (double *)calloc((size_t)(d > 0 ? d : 1), sizeof(double));
    for (int j = 0; j < n; ++j) {
        const uint16_t *kj = k + (size_t)j * d;
        double nrm = sqrt(dot_bf16(kj, kj, d));
        inv[j] = nrm > 0.0 ? 1.0 / nrm : 0.0;
        for (int c = 0; c < d; ++c)
            sum_u[c] += bf16_value(kj[c]) * inv[j];
    }
    for (int i = 0; i < n; ++i) {
        const uint16_t *ki = k + (size_t)i * d;
        double proj = 0.0;
        for (int c = 0; c < d; ++c)
            proj += bf16_value(ki[c]) * sum_u[c];
        const double self = inv[i] > 0.0 ? 1.0 : 0.0;
        red[i] = n > 1 ? (inv[i] * proj - self) / (double)(n - 1) : 0.0;
    }
    free(sum_u);
    free(inv);
}

/* Min-max normalisation over the head's n tokens (reading R5). */
void orc_minmax(const double *x, int n, double *out)
{
    double lo = INFINITY, hi = -INFINITY;
    for (int j = 0; j < n; ++j) {
        if (x[j] < lo) lo = x[j];
        if (x[j] > hi) hi = x[j];
    }
    for (int j = 0; j < n; ++j)
        out[j] = hi > lo ? (x[j] - lo) / (hi - lo) : 0.0;
}

/* Blend ([RKV-review]: mix_lambda blends the two signals; [RKV-blog]: keep
 * high importance and low redundancy, lambda about 0.1). Reading R6. */
void orc_mix(const double *imp_hat, const double *red_hat, int n, double lam, double *s)
{
    for (int j = 0; j < n; ++j)
        s[j] = lam * imp_hat[j] - (1.0 - lam) * red_hat[j];
}

static const double *g_sort_scores;

/* Larger score first; equal scores: lower index first. */
static int by_score_desc(const void *a, const void *b)
{
    int i = *(const int32_t *)a, j = *(const int32_t *)b;
    double si = g_sort_scores[i], sj = g_sort_scores[j];
    if (si > sj) return -1;
    if (si < sj) return 1;
    return (i > j) - (i < j);
}

static int by_index(const void *a, const void *b)
{
    int i = *(const int32_t *)a, j = *(const int32_t *)b;
    return (i > j) - (i < j);
}

/*
 * Selection ([RKV-review]: kv_budget tokens are kept and a local window of
 * window_size recent tokens is protected). Reading R7. keep[] receives the
 * kept indices ascending; entries past the kept count are set to -1
 * (keep must hold `budget` entries). Returns the kept count.
 * Not thread-safe (qsort comparator state); callers serialise it.
 */
int orc_select(const double *s, int n, int budget, int window, int32_t *keep)
{
    int kept;
    if (n <= budget) {
        for (int j = 0; j < n; ++j)
            keep[j] = j;
        kept = n;
    } else {
        int cand = n - window;
        int take = budget - window;
        int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)(cand > 0 ? cand : 1));
        for (int j = 0; j < cand; ++j)
            order[j] = j;
        g_sort_scores = s;
        qsort(order, (size_t)cand, sizeof(int32_t), by_score_desc);
        for (int t = 0; t < take; ++t)
            keep[t] = order[t];
        for (int t = 0; t < window; ++t)
            keep[take + t] = cand + t;
        qsort(keep, (size_t)budget, sizeof(int32_t), by_index);
        free(order);
        kept = budget;
    }
    for (int j = kept; j < budget; ++j)
        keep[j] = -1;
    return kept;
}

/* Address (in elements) of logical token t of head h, sequence b, layer l. */
static size_t row_offset(const orc_problem *p, const int32_t *block_table, int l, int b, int h, int t)
{
    const size_t d = (size_t)p->head_dim;
    if (!p->paged)
        return ((((size_t)l * p->batch + b) * p->kv_heads + h) * p->max_seq_len + t) * d;
    int blk = block_table[(size_t)b * p->max_blocks + t / p->block_size];
    return ((((size_t)l * p->num_blocks + blk) * p->block_size + t % p->block_size) * p->kv_heads + h) * d;
}

static int check_problem(const orc_problem *p, const int32_t *seq_lens, const int32_t *block_table)
{
    if (p->layers < 0 || p->batch < 0 || p->kv_heads <= 0 || p->q_heads <= 0 || p->head_dim <= 0)
        return -1;
    if (p->q_heads % p->kv_heads != 0 || p->window < 1 || p->window > p->budget)
        return -1;
    for (int b = 0; b < p->batch; ++b) {
        int n = seq_lens[b];
        if (n < 0 || n > p->max_seq_len)
            return -2;
        if (p->paged) {
            int nb = (n + p->block_size - 1) / p->block_size;
            if (nb > p->max_blocks)
                return -2;
            for (int i = 0; i < nb; ++i) {
                int blk = block_table[(size_t)b * p->max_blocks + i];
                if (blk < 0 || blk >= p->num_blocks)
                    return -3;
            }
        }
    }
    return 0;
}

/* Slot j <- token keep[j] for one head, in logical-slot space (reading R8).
 * The source rows are read from a snapshot, so the result equals an in-order
 * in-place gather. */
static int compact_head(const orc_problem *p, uint16_t *cache, const int32_t *block_table,
                        int l, int b, int h, int n, const int32_t *keep, int kept, uint16_t *snap)
{
    const int d = p->head_dim;
    for (int t = 0; t < n; ++t)
        memcpy(snap + (size_t)t * d, cache + row_offset(p, block_table, l, b, h, t), sizeof(uint16_t) * d);
    for (int j = 0; j < kept; ++j) {
        if (keep[j] < 0 || keep[j] >= n || (j > 0 && keep[j] <= keep[j - 1]))
            return -4;
        memcpy(cache + row_offset(p, block_table, l, b, h, j), snap + (size_t)keep[j] * d,
               sizeof(uint16_t) * d);
    }
    return 0;
}

int orc_freed_blocks(const orc_problem *p, const int32_t *seq_lens, const int32_t *block_table,
                     int32_t *freed_off, int32_t *freed_ids, int32_t *new_seq_lens)
{
    int rc = check_problem(p, seq_lens, block_table);
    if (rc)
        return rc;
    freed_off[0] = 0;
    for (int b = 0; b < p->batch; ++b) {
        int n = seq_lens[b];
        int kept = n < p->budget ? n : p->budget;
        new_seq_lens[b] = kept;
        int count = 0;
        if (p->paged) {
            int first = (kept + p->block_size - 1) / p->block_size;
            int last = (n + p->block_size - 1) / p->block_size;
            for (int i = first; i < last; ++i)
                freed_ids[freed_off[b] + count++] = block_table[(size_t)b * p->max_blocks + i];
        }
        freed_off[b + 1] = freed_off[b] + count;
    }
    return 0;
}

int orc_compact(const orc_problem *p, uint16_t *k_cache, uint16_t *v_cache,
                const int32_t *seq_lens, const int32_t *block_table, const int32_t *keep_idx)
{
    int rc = check_problem(p, seq_lens, block_table);
    if (rc)
        return rc;
    const int heads = p->layers * p->batch * p->kv_heads;
    int err = 0;
#pragma omp parallel
    {
        uint16_t *snap = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)p->max_seq_len * p->head_dim);
#pragma omp for schedule(dynamic)
        for (int e = 0; e < heads; ++e) {
            int h = e % p->kv_heads, b = (e / p->kv_heads) % p->batch, l = e / (p->kv_heads * p->batch);
            int n = seq_lens[b];
            int kept = n < p->budget ? n : p->budget;
            const int32_t *keep = keep_idx + (size_t)e * p->budget;
            if (compact_head(p, k_cache, block_table, l, b, h, n, keep, kept, snap) ||
                compact_head(p, v_cache, block_table, l, b, h, n, keep, kept, snap)) {
#pragma omp atomic write
                err = -4;
            }
        }
        free(snap);
    }
    return err;
}

static int compress_with(const orc_problem *p, int closed_form, uint16_t *k_cache, uint16_t *v_cache,
                         const uint16_t *q_window, const int32_t *seq_lens, const int32_t *block_table,
                         int32_t *keep_idx, int32_t *freed_off, int32_t *freed_ids,
                         int32_t *new_seq_lens, double *scores)
{
    int rc = check_problem(p, seq_lens, block_table);
    if (rc)
        return rc;
    const int L = p->layers, B = p->batch, H = p->kv_heads, d = p->head_dim, N = p->max_seq_len;
    const int G = p->q_heads / H, w = p->window, rows = G * w;
    const int heads = L * B * H;
    const size_t plane = (size_t)heads * N;
    if (scores)
        memset(scores, 0, sizeof(double) * 5 * plane);

    /* Scores and selection for every head, from the unmodified cache. */
#pragma omp parallel
    {
        uint16_t *kh = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)N * d);
        double *I = (double *)malloc(sizeof(double) * (size_t)N * 5);
        double *R = I + N, *Ih = R + N, *Rh = Ih + N, *S = Rh + N;
#pragma omp for schedule(dynamic)
        for (int e = 0; e < heads; ++e) {
            int h = e % H, b = (e / H) % B, l = e / (H * B);
            int n = seq_lens[b];
            int32_t *keep = keep_idx + (size_t)e * p->budget;
            for (int t = 0; t < n; ++t)
                memcpy(kh + (size_t)t * d, k_cache + row_offset(p, block_table, l, b, h, t),
                       sizeof(uint16_t) * d);
            /* q heads h*G .. h*G+G-1, each with w window rows: one [rows][d] block */
            const uint16_t *qh = q_window + ((((size_t)l * B + b) * p->q_heads + (size_t)h * G) * w) * d;
            orc_importance(qh, rows, kh, n, d, I);
            if (closed_form)
                orc_redundancy_closed(kh, n, d, R);
            else
                orc_redundancy(kh, n, d, R);
            orc_minmax(I, n, Ih);
            orc_minmax(R, n, Rh);
            orc_mix(Ih, Rh, n, p->mix_lambda, S);
#pragma omp critical(orc_select_sort)
            orc_select(S, n, p->budget, w, keep);
            if (scores) {
                for (int j = 0; j < n; ++j) {
                    scores[0 * plane + (size_t)e * N + j] = I[j];
                    scores[1 * plane + (size_t)e * N + j] = R[j];
                    scores[2 * plane + (size_t)e * N + j] = Ih[j];
                    scores[3 * plane + (size_t)e * N + j] = Rh[j];
                    scores[4 * plane + (size_t)e * N + j] = S[j];
                }
            }
        }
        free(kh);
        free(I);
    }
    rc = orc_compact(p, k_cache, v_cache, seq_lens, block_table, keep_idx);
    if (rc)
        return rc;
    return orc_freed_blocks(p, seq_lens, block_table, freed_off, freed_ids, new_seq_lens);
}

int orc_compress(const orc_problem *p, uint16_t *k_cache, uint16_t *v_cache,
                 const uint16_t *q_window, const int32_t *seq_lens, const int32_t *block_table,
                 int32_t *keep_idx, int32_t *freed_off, int32_t *freed_ids,
                 int32_t *new_seq_lens, double *scores)
{
    return compress_with(p, 0, k_cache, v_cache, q_window, seq_lens, block_table, keep_idx, freed_off,
                         freed_ids, new_seq_lens, scores);
}

int orc_compress_closed(const orc_problem *p, uint16_t *k_cache, uint16_t *v_cache,
                        const uint16_t *q_window, const int32_t *seq_lens, const int32_t *block_table,
                        int32_t *keep_idx, int32_t *freed_off, int32_t *freed_ids,
                        int32_t *new_seq_lens, double *scores)
{
    return compress_with(p, 1, k_cache, v_cache, q_window, seq_lens, block_table, keep_idx, freed_off,
                         freed_ids, new_seq_lens, scores);
}
