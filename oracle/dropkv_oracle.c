/*
 * DropKV scoring path: CPU oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 restatement of what the scoring path computes.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may call it;
 * the product library never links, loads or calls it, and this file shares no
 * code, header, table or constant with the CUDA library.
 *
 * Every step is the definition written out, in the pages' order:
 *
 *  [S1] window attention.  For KV head h of sequence b, every query head of its
 *       GQA group contributes its w window queries.  Query t sits at position
 *       n_b - w + t and sees keys j <= n_b - w + t ("DropKV: Exact single-entry
 *       output-perturbation scoring", Code mapping and limits: tail-aligned
 *       causality; "DropKV: Decoupling Residual-Output Perturbation for
 *       Near-Optimal KV-Cache Eviction", section 2.1: causal mask).
 *       x_j = q.k_j / sqrt(d), m = max_j x_j, e_j = exp(x_j - m), l = sum_j e_j,
 *       p_j = e_j / l, a = sum_j p_j v_j  ("... output-perturbation scoring",
 *       Core equation: p = softmax(Kq/sqrt d), a = sum_j p_j v_j).
 *  [S2] singular rule: a probability equal to 1 makes exact removal singular;
 *       it is rejected, never patched with an epsilon (same page, Algorithm 1
 *       summary).
 *  [S3] per-token perturbation, summed over the window: removing key j moves
 *       the output by Delta_j = p_j / (1 - p_j) (a - v_j); the score is
 *       s_j = sum_t ||Delta_j^(t)||^2 (same page, Core equation; "DropKV:
 *       Decoupling ...", sections 3.1 and 3.3).  1 - p_j is evaluated as
 *       (l - e_j) / l and ||a - v_j||^2 as the direct sum of squared
 *       differences; for the one key a row may give more than half its mass,
 *       Delta_j is taken in the equal deletion form p_j (a_{-j} - v_j), with
 *       the other keys' mass and output summed on their own (no cancellation
 *       as p_j -> 1).  Keys a query cannot see contribute nothing for it.
 *  [S4] local GQA averaging: the scores of the query heads that share a KV
 *       head are averaged (same page, Algorithm 1 summary).
 *  [S5] MaxPool1D along the sequence (kernel kappa, stride 1, window clipped to
 *       [0, n_b)), then the last `protect` slots are set to +inf (same page,
 *       Algorithm 1 summary: pooling, then recent-window protection).
 *  [S6] the k_b smallest final scores are evicted; among equal scores the lower
 *       position goes first; the kept positions are listed in ascending order
 *       (same page, Algorithm 1 summary: evict the smallest scores; "DropKV:
 *       Decoupling ...", section 2.2: eviction shrinks the resident cache).
 *  [S7] the kept K/V rows are gathered in that order (byte copies).
 *
 * Layer-wide selection (AdaDropKV: DropKV scores with an adaptive head
 * budget, "DropKV: Decoupling ...", section 5.3 and Appendix A.3; the pages
 * give no allocation rule, so the plainest one is taken): for each sequence,
 * the scores of all its KV heads form one pool; the evict_total[b] smallest
 * (score, head, position) triples are evicted, so each head keeps its own
 * number of slots.  Each head's kept positions are listed ascending.
 *
 * Prefill attention (the model's own causal attention over the prompt,
 * "DropKV: Decoupling ...", section 2.1, whose last-w rows give the window
 * statistics of S1 for free when the scorer is fused into it): every query
 * row i < n_b of every query head sees the keys j <= i of its KV head;
 * out_i = sum_j p_j v_j with p = softmax(x), x_j = q_i.k_j / sqrt(d).
 *
 * Score kind SnapKV (the attention-only baseline of "DropKV: Decoupling ...",
 * Appendix B, Table 14: MaxPool1d over the window sum of p_j): step S3 becomes
 * s_j = sum_t p_j^(t) and the singular rule S2 does not apply (nothing is
 * divided by 1 - p_j); S1, S4-S7 are unchanged.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "dropkv_oracle.h"

/* bf16 bit pattern -> exact double */
static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void* base, int dtype, size_t i) {
    if (dtype == ORACLE_BF16) return bf16_to_double(((const uint16_t*)base)[i]);
    return ((const double*)base)[i];
}

typedef struct {
    const oracle_shape* s;
    int dtype;
    const void *q, *k, *v;
    const int32_t* lengths;
    int pool_kernel, protect, kind;
    double *m_out, *l_out, *a_out, *raw_out, *final_out;
    double* s_heads;         /* [B * Hkv][g][n_max]: per query head sums of S3 */
    /* work distribution: items are (unit, query head) in phase 1, units in phase 2 */
    int next_item;
    int phase;
    pthread_mutex_t lock;
    int status;              /* ORACLE_OK or first error */
    int singular_unit;
} score_job;

static int take_item(score_job* job) {
    pthread_mutex_lock(&job->lock);
    int u = job->next_item++;
    pthread_mutex_unlock(&job->lock);
    return u;
}

static void set_status(score_job* job, int st, int unit) {
    pthread_mutex_lock(&job->lock);
    if (job->status == ORACLE_OK) {
        job->status = st;
        job->singular_unit = unit;
    }
    pthread_mutex_unlock(&job->lock);
}

/* One query head hl of one (b, KV head) unit: steps S1-S3 for its w window
 * rows, summed over the rows into s_head[0, n_b). */
static int score_head(score_job* job, int unit, int hl, double* x, double* e, double* qrow, double* a,
                      double* ar, double* s_head) {
    const oracle_shape* s = job->s;
    const int b = unit / s->Hkv, h = unit % s->Hkv;
    const int g = s->Hq / s->Hkv, d = s->d, w = s->w;
    const int nb = job->lengths[b];
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    const size_t kv_base = ((size_t)b * s->Hkv + h) * (size_t)s->n_max * d;
    const int hq = h * g + hl;

    for (int j = 0; j < nb; ++j) s_head[j] = 0.0;
    for (int t = 0; t < w; ++t) {
        const int pos = nb - w + t;            /* last visible key of this query */
        const size_t row = ((size_t)b * s->Hq + hq) * w + t;
        for (int c = 0; c < d; ++c) qrow[c] = load_elem(job->q, job->dtype, row * d + c);

        /* S1: logits, max, exponentials, normaliser */
        double m = -INFINITY;
        for (int j = 0; j <= pos; ++j) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += qrow[c] * load_elem(job->k, job->dtype, kv_base + (size_t)j * d + c);
            x[j] = acc * inv_sqrt_d;
            if (x[j] > m) m = x[j];
        }
        double l = 0.0;
        for (int j = 0; j <= pos; ++j) {
            e[j] = exp(x[j] - m);
            l += e[j];
        }
        /* a = sum_j p_j v_j */
        for (int c = 0; c < d; ++c) a[c] = 0.0;
        for (int j = 0; j <= pos; ++j) {
            const double p = e[j] / l;
            /* S2: a probability rounded to 1 is rejected */
            if (p == 1.0 && job->kind == ORACLE_KIND_DROPKV) return ORACLE_SINGULAR;
            for (int c = 0; c < d; ++c)
                a[c] += p * load_elem(job->v, job->dtype, kv_base + (size_t)j * d + c);
        }
        if (job->m_out) job->m_out[row] = m;
        if (job->l_out) job->l_out[row] = l;
        if (job->a_out)
            for (int c = 0; c < d; ++c) job->a_out[row * d + c] = a[c];

        if (job->kind == ORACLE_KIND_SNAPKV) {
            /* SnapKV: the attention probability of every visible key */
            for (int j = 0; j <= pos; ++j) s_head[j] += e[j] / l;
            continue;
        }
        /* S3: ||p_j / (1 - p_j) (a - v_j)||^2 for every visible key.  That
         * vector is the change of the output when key j is deleted,
         * a_{-j} - a, which also equals p_j (a_{-j} - v_j) (a = p_j v_j +
         * (1 - p_j) a_{-j}).  For the one key that may hold more than half of
         * the row's mass, a - v_j and l - e_j cancel as p_j nears 1 (at
         * 1 - p_j = 1e-14 the closed form keeps one digit), so its term is
         * taken in the second form, with the other keys' mass and output
         * summed on their own. */
        for (int j = 0; j <= pos; ++j) {
            if (e[j] > 0.5 * l) {
                double l_rest = 0.0;
                for (int c = 0; c < d; ++c) ar[c] = 0.0;
                for (int i = 0; i <= pos; ++i) {
                    if (i == j) continue;
                    l_rest += e[i];
                    for (int c = 0; c < d; ++c)
                        ar[c] += e[i] * load_elem(job->v, job->dtype, kv_base + (size_t)i * d + c);
                }
                /* l_rest > 0 here: otherwise p_j == 1.0 was rejected above */
                const double p_dom = e[j] / (e[j] + l_rest);
                double dist_rest = 0.0;
                for (int c = 0; c < d; ++c) {
                    const double diff = ar[c] / l_rest - load_elem(job->v, job->dtype, kv_base + (size_t)j * d + c);
                    dist_rest += diff * diff;
                }
                s_head[j] += p_dom * p_dom * dist_rest;
                continue;
            }
            const double p = e[j] / l;
            const double one_minus_p = (l - e[j]) / l;
            const double ratio = p / one_minus_p;
            double dist = 0.0;
            for (int c = 0; c < d; ++c) {
                const double diff = a[c] - load_elem(job->v, job->dtype, kv_base + (size_t)j * d + c);
                dist += diff * diff;
            }
            s_head[j] += ratio * ratio * dist;
        }
    }
    return ORACLE_OK;
}

/* Steps S4-S5 of one unit: the mean over its g query heads (summed in query
 * head order), MaxPool1D and protection. */
static void finish_unit(score_job* job, int unit) {
    const oracle_shape* s = job->s;
    const int b = unit / s->Hkv;
    const int g = s->Hq / s->Hkv;
    const int nb = job->lengths[b];
    const size_t n_max = (size_t)s->n_max;
    const double* heads = job->s_heads + (size_t)unit * g * n_max;

    /* S4: mean over the g query heads of the group */
    double* raw = job->raw_out + (size_t)unit * n_max;
    for (int j = 0; j < nb; ++j) {
        double sum = 0.0;
        for (int hl = 0; hl < g; ++hl) sum += heads[(size_t)hl * n_max + j];
        raw[j] = sum / (double)g;
    }
    for (size_t j = (size_t)nb; j < n_max; ++j) raw[j] = NAN;

    /* S5: MaxPool1D (window clipped to the sequence), then protection */
    double* fin = job->final_out + (size_t)unit * n_max;
    const int half = job->pool_kernel / 2;
    for (int j = 0; j < nb; ++j) {
        int lo = j - half, hi = j + half;
        if (lo < 0) lo = 0;
        if (hi > nb - 1) hi = nb - 1;
        double mx = raw[lo];
        for (int i = lo + 1; i <= hi; ++i)
            if (raw[i] > mx) mx = raw[i];
        fin[j] = mx;
    }
    for (int j = nb - job->protect; j < nb; ++j)
        if (j >= 0) fin[j] = INFINITY;
    for (size_t j = (size_t)nb; j < n_max; ++j) fin[j] = NAN;
}

static void* score_worker(void* arg) {
    score_job* job = (score_job*)arg;
    const oracle_shape* s = job->s;
    const int g = s->Hq / s->Hkv, units = s->B * s->Hkv;
    const size_t n = (size_t)s->n_max;
    if (job->phase == 2) {
        for (;;) {
            const int u = take_item(job);
            if (u >= units) break;
            finish_unit(job, u);
        }
        return NULL;
    }
    double* x = (double*)malloc(n * sizeof(double));
    double* e = (double*)malloc(n * sizeof(double));
    double* qrow = (double*)malloc((size_t)s->d * sizeof(double));
    double* a = (double*)malloc((size_t)s->d * sizeof(double));
    double* ar = (double*)malloc((size_t)s->d * sizeof(double));
    if (!x || !e || !qrow || !a || !ar) {
        set_status(job, ORACLE_NOMEM, -1);
    } else {
        for (;;) {
            const int it = take_item(job);
            if (it >= units * g) break;
            const int u = it / g, hl = it % g;
            const int st = score_head(job, u, hl, x, e, qrow, a, ar, job->s_heads + ((size_t)u * g + hl) * n);
            if (st != ORACLE_OK) set_status(job, st, u);
        }
    }
    free(x); free(e); free(qrow); free(a); free(ar);
    return NULL;
}

/* Run score_worker on nthreads threads (the calling thread included). */
static void run_phase(score_job* job, int phase, int nthreads) {
    job->phase = phase;
    job->next_item = 0;
    pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
    int started = 0;
    for (int i = 1; i < nthreads && th; ++i)
        if (pthread_create(&th[i], NULL, score_worker, job) == 0) started = i; else break;
    score_worker(job);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    free(th);
}

static int check_shape(const oracle_shape* s) {
    if (!s || s->B < 1 || s->Hq < 1 || s->Hkv < 1 || s->d < 1 || s->n_max < 1 || s->w < 1) return 0;
    if (s->Hq % s->Hkv != 0) return 0;
    return 1;
}

int oracle_score_kind(const oracle_shape* s, int kind, int dtype, const void* q, const void* k, const void* v,
                      const int32_t* lengths, int pool_kernel, int protect,
                      double* m_out, double* l_out, double* a_out, double* raw_out, double* final_out,
                      int nthreads, int32_t* singular_unit) {
    if (singular_unit) *singular_unit = -1;
    if (kind != ORACLE_KIND_DROPKV && kind != ORACLE_KIND_SNAPKV) return ORACLE_INVALID;
    if (!check_shape(s) || !q || !k || !v || !lengths || !raw_out || !final_out) return ORACLE_INVALID;
    if (dtype != ORACLE_F64 && dtype != ORACLE_BF16) return ORACLE_INVALID;
    if (pool_kernel < 1 || pool_kernel % 2 == 0 || protect < 0) return ORACLE_INVALID;
    for (int b = 0; b < s->B; ++b)
        if (lengths[b] < s->w || lengths[b] > s->n_max || protect > lengths[b]) return ORACLE_INVALID;

    score_job job;
    memset(&job, 0, sizeof job);
    job.s = s; job.dtype = dtype; job.q = q; job.k = k; job.v = v; job.lengths = lengths;
    job.pool_kernel = pool_kernel; job.protect = protect; job.kind = kind;
    job.m_out = m_out; job.l_out = l_out; job.a_out = a_out;
    job.raw_out = raw_out; job.final_out = final_out;
    job.status = ORACLE_OK; job.singular_unit = -1;
    const int units = s->B * s->Hkv, g = s->Hq / s->Hkv;
    job.s_heads = (double*)malloc((size_t)units * g * (size_t)s->n_max * sizeof(double));
    if (!job.s_heads) return ORACLE_NOMEM;
    pthread_mutex_init(&job.lock, NULL);

    if (nthreads < 1) nthreads = 1;
    /* phase 1: S1-S3 per (unit, query head); phase 2: S4-S5 per unit */
    run_phase(&job, 1, nthreads > units * g ? units * g : nthreads);
    if (job.status == ORACLE_OK) run_phase(&job, 2, nthreads > units ? units : nthreads);
    free(job.s_heads);
    pthread_mutex_destroy(&job.lock);
    if (singular_unit) *singular_unit = job.singular_unit;
    return job.status;
}

int oracle_score(const oracle_shape* s, int dtype, const void* q, const void* k, const void* v,
                 const int32_t* lengths, int pool_kernel, int protect,
                 double* m_out, double* l_out, double* a_out, double* raw_out, double* final_out,
                 int nthreads, int32_t* singular_unit) {
    return oracle_score_kind(s, ORACLE_KIND_DROPKV, dtype, q, k, v, lengths, pool_kernel, protect, m_out, l_out,
                             a_out, raw_out, final_out, nthreads, singular_unit);
}

/* S6: order by (final score, position), evict the first k_b. */
typedef struct { double key; int32_t idx; } keyed;

static int cmp_keyed(const void* pa, const void* pb) {
    const keyed* a = (const keyed*)pa;
    const keyed* b = (const keyed*)pb;
    if (a->key < b->key) return -1;
    if (a->key > b->key) return 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

static int cmp_i32(const void* pa, const void* pb) {
    const int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

int oracle_select(const oracle_shape* s, const double* final_scores, const int32_t* lengths,
                  const int32_t* evict_k, int protect, int32_t* kept_idx, int32_t* kept_len) {
    if (!check_shape(s) || !final_scores || !lengths || !evict_k || !kept_idx || !kept_len)
        return ORACLE_INVALID;
    for (int b = 0; b < s->B; ++b) {
        if (lengths[b] < 1 || lengths[b] > s->n_max) return ORACLE_INVALID;
        if (evict_k[b] < 0 || evict_k[b] > lengths[b] - protect) return ORACLE_INVALID;
    }
    const size_t n_max = (size_t)s->n_max;
    keyed* tmp = (keyed*)malloc(n_max * sizeof(keyed));
    if (!tmp) return ORACLE_NOMEM;
    for (int b = 0; b < s->B; ++b) {
        const int nb = lengths[b], kb = evict_k[b];
        kept_len[b] = nb - kb;
        for (int h = 0; h < s->Hkv; ++h) {
            const size_t unit = (size_t)b * s->Hkv + h;
            const double* fin = final_scores + unit * n_max;
            for (int j = 0; j < nb; ++j) { tmp[j].key = fin[j]; tmp[j].idx = j; }
            qsort(tmp, (size_t)nb, sizeof(keyed), cmp_keyed);
            int32_t* out = kept_idx + unit * n_max;
            for (int i = kb; i < nb; ++i) out[i - kb] = tmp[i].idx;
            qsort(out, (size_t)(nb - kb), sizeof(int32_t), cmp_i32);
        }
    }
    free(tmp);
    return ORACLE_OK;
}

/* Layer-wide S6: one pool per sequence over all its KV heads; ties go to the
 * lower head, then the lower position.  kept_len is [B][Hkv]. */
int oracle_select_layer(const oracle_shape* s, const double* final_scores, const int32_t* lengths,
                        const int32_t* evict_total, int protect, int32_t* kept_idx, int32_t* kept_len) {
    if (!check_shape(s) || !final_scores || !lengths || !evict_total || !kept_idx || !kept_len)
        return ORACLE_INVALID;
    for (int b = 0; b < s->B; ++b) {
        if (lengths[b] < 1 || lengths[b] > s->n_max) return ORACLE_INVALID;
        if (evict_total[b] < 0 || evict_total[b] > s->Hkv * (lengths[b] - protect)) return ORACLE_INVALID;
    }
    const size_t n_max = (size_t)s->n_max;
    keyed* tmp = (keyed*)malloc((size_t)s->Hkv * n_max * sizeof(keyed));
    char* keep = (char*)malloc((size_t)s->Hkv * n_max);
    if (!tmp || !keep) { free(tmp); free(keep); return ORACLE_NOMEM; }
    for (int b = 0; b < s->B; ++b) {
        const int nb = lengths[b];
        size_t m = 0;
        for (int h = 0; h < s->Hkv; ++h) {
            const double* fin = final_scores + ((size_t)b * s->Hkv + h) * n_max;
            for (int j = 0; j < nb; ++j) {
                tmp[m].key = fin[j];
                tmp[m].idx = (int32_t)((size_t)h * n_max + (size_t)j);
                ++m;
            }
        }
        qsort(tmp, m, sizeof(keyed), cmp_keyed);
        memset(keep, 0, (size_t)s->Hkv * n_max);
        for (size_t i = (size_t)evict_total[b]; i < m; ++i) keep[tmp[i].idx] = 1;
        for (int h = 0; h < s->Hkv; ++h) {
            int32_t* out = kept_idx + ((size_t)b * s->Hkv + h) * n_max;
            int c = 0;
            for (int j = 0; j < nb; ++j)
                if (keep[(size_t)h * n_max + (size_t)j]) out[c++] = j;
            kept_len[(size_t)b * s->Hkv + h] = c;
        }
    }
    free(tmp);
    free(keep);
    return ORACLE_OK;
}

/* S7 with a kept count per KV head (kept_len [B][Hkv]). */
int oracle_compact_heads(const oracle_shape* s, int elem_bytes, const void* k, const void* v,
                         const int32_t* kept_idx, const int32_t* kept_len, int out_rows,
                         void* k_out, void* v_out) {
    if (!check_shape(s) || elem_bytes < 1 || !k || !v || !kept_idx || !kept_len || !k_out || !v_out)
        return ORACLE_INVALID;
    const size_t row_bytes = (size_t)s->d * elem_bytes;
    const size_t n_max = (size_t)s->n_max;
    for (int u = 0; u < s->B * s->Hkv; ++u)
        if (kept_len[u] < 0 || kept_len[u] > out_rows) return ORACLE_INVALID;
    for (size_t unit = 0; unit < (size_t)s->B * s->Hkv; ++unit) {
        const int32_t* idx = kept_idx + unit * n_max;
        for (int i = 0; i < kept_len[unit]; ++i) {
            if (idx[i] < 0 || (size_t)idx[i] >= n_max) return ORACLE_INVALID;
            const size_t src = (unit * n_max + (size_t)idx[i]) * row_bytes;
            const size_t dst = (unit * (size_t)out_rows + (size_t)i) * row_bytes;
            memcpy((char*)k_out + dst, (const char*)k + src, row_bytes);
            memcpy((char*)v_out + dst, (const char*)v + src, row_bytes);
        }
    }
    return ORACLE_OK;
}

/* S7: gather the kept rows of K and V (elem_bytes per element). */
int oracle_compact(const oracle_shape* s, int elem_bytes, const void* k, const void* v,
                   const int32_t* kept_idx, const int32_t* kept_len, int out_rows,
                   void* k_out, void* v_out) {
    if (!check_shape(s) || elem_bytes < 1 || !k || !v || !kept_idx || !kept_len || !k_out || !v_out)
        return ORACLE_INVALID;
    const size_t row_bytes = (size_t)s->d * elem_bytes;
    const size_t n_max = (size_t)s->n_max;
    for (int b = 0; b < s->B; ++b)
        if (kept_len[b] < 0 || kept_len[b] > out_rows) return ORACLE_INVALID;
    for (int b = 0; b < s->B; ++b) {
        for (int h = 0; h < s->Hkv; ++h) {
            const size_t unit = (size_t)b * s->Hkv + h;
            const int32_t* idx = kept_idx + unit * n_max;
            for (int i = 0; i < kept_len[b]; ++i) {
                if (idx[i] < 0 || (size_t)idx[i] >= n_max) return ORACLE_INVALID;
                const size_t src = (unit * n_max + (size_t)idx[i]) * row_bytes;
                const size_t dst = (unit * (size_t)out_rows + (size_t)i) * row_bytes;
                memcpy((char*)k_out + dst, (const char*)k + src, row_bytes);
                memcpy((char*)v_out + dst, (const char*)v + src, row_bytes);
            }
        }
    }
    return ORACLE_OK;
}

/* Causal prefill attention over every query row (definition in the header
 * comment).  Items are (sequence, query head) pairs spread over the threads. */
typedef struct {
    const oracle_shape* s;
    int dtype;
    const void *q, *k, *v;
    const int32_t* lengths;
    double* out;
    int next_item;
    int status;
    pthread_mutex_t mu;
} prefill_job;

static void* prefill_worker(void* arg) {
    prefill_job* job = (prefill_job*)arg;
    const oracle_shape* s = job->s;
    const int g = s->Hq / s->Hkv, d = s->d;
    const size_t n = (size_t)s->n_max;
    double* x = (double*)malloc(n * sizeof(double));
    double* qrow = (double*)malloc((size_t)d * sizeof(double));
    double* acc = (double*)malloc((size_t)d * sizeof(double));
    if (!x || !qrow || !acc) {
        pthread_mutex_lock(&job->mu);
        job->status = ORACLE_NOMEM;
        pthread_mutex_unlock(&job->mu);
        free(x); free(qrow); free(acc);
        return NULL;
    }
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    for (;;) {
        pthread_mutex_lock(&job->mu);
        const int it = job->next_item++;
        pthread_mutex_unlock(&job->mu);
        if (it >= s->B * s->Hq) break;
        const int b = it / s->Hq, hq = it % s->Hq, h = hq / g;
        const int nb = job->lengths[b];
        const size_t kv_base = ((size_t)b * s->Hkv + h) * n * d;
        const size_t q_base = ((size_t)b * s->Hq + hq) * n * d;
        for (int i = 0; i < nb; ++i) {
            for (int c = 0; c < d; ++c) qrow[c] = load_elem(job->q, job->dtype, q_base + (size_t)i * d + c);
            double m = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                double dot = 0.0;
                for (int c = 0; c < d; ++c) dot += qrow[c] * load_elem(job->k, job->dtype, kv_base + (size_t)j * d + c);
                x[j] = dot * inv_sqrt_d;
                if (x[j] > m) m = x[j];
            }
            double l = 0.0;
            for (int j = 0; j <= i; ++j) {
                x[j] = exp(x[j] - m);
                l += x[j];
            }
            for (int c = 0; c < d; ++c) acc[c] = 0.0;
            for (int j = 0; j <= i; ++j) {
                const double p = x[j] / l;
                for (int c = 0; c < d; ++c) acc[c] += p * load_elem(job->v, job->dtype, kv_base + (size_t)j * d + c);
            }
            for (int c = 0; c < d; ++c) job->out[q_base + (size_t)i * d + c] = acc[c];
        }
        for (size_t i = (size_t)nb; i < n; ++i)
            for (int c = 0; c < d; ++c) job->out[q_base + i * d + c] = NAN;
    }
    free(x); free(qrow); free(acc);
    return NULL;
}

int oracle_prefill_attention(const oracle_shape* s, int dtype, const void* q, const void* k, const void* v,
                             const int32_t* lengths, double* out, int nthreads) {
    if (!s || !q || !k || !v || !lengths || !out) return ORACLE_INVALID;
    if (s->B < 1 || s->Hq < 1 || s->Hkv < 1 || s->Hq % s->Hkv != 0 || s->d < 1 || s->n_max < 1) return ORACLE_INVALID;
    for (int b = 0; b < s->B; ++b)
        if (lengths[b] < 1 || lengths[b] > s->n_max) return ORACLE_INVALID;
    prefill_job job;
    job.s = s; job.dtype = dtype; job.q = q; job.k = k; job.v = v; job.lengths = lengths; job.out = out;
    job.next_item = 0; job.status = ORACLE_OK;
    pthread_mutex_init(&job.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
    int started = 0;
    for (int i = 1; i < nthreads && th; ++i)
        if (pthread_create(&th[i], NULL, prefill_worker, &job) == 0) started = i; else break;
    prefill_worker(&job);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&job.mu);
    return job.status;
}
