/*
 * CPU oracle for the compressed sparse attention (CSA) decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Everything is computed in double precision from the caller's stored values
 * (bf16 or fp32 bit patterns, decoded exactly), one query at a time, in the
 * order the method states.  No blocking, fusion, streaming softmax or
 * selection algorithm: scores are a full loop, Top-K is a full sort, and
 * attention is one softmax over the union of the rows the query reads.
 *
 * Sources (pages of hw-native-sys/pypto-lib):
 *  - "Perf: skip redundant CSA scoring and fuse gather unpack", PR description:
 *    the indexer scores the ratio-4 compressed rows a query can see; when the
 *    visible rows fit Top-K, scoring and sorting are skipped and every visible
 *    row is taken, causal visibility retained; the indexer emits bounded
 *    Top-K indices.
 *  - "Fix: port the DeepSeek-V4 MoE, hc_pre and prefill fixes to DSpark", PR
 *    description: sparse CSA rows per query are bounded by
 *    WIN + min(max_visible_cmp, IDX_TOPK); reductions run in a fixed
 *    ascending order.
 *  - "Perf: fuse HCA merge, inverse RoPE, and packing", PR description: a raw
 *    (window) softmax stream and a compressed softmax stream are merged, then
 *    inverse RoPE is applied to the merged output.
 *  The indexer score itself is the DeepSeek lightning-indexer form,
 *  score_j = sum_h w_h * ReLU(q_idx[h] . k_idx[j]); the pages name the indexer
 *  but print no formula.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  visibility vis = floor((pos+1)/ratio); window = raw rows
 *  [max(0,pos-WIN+1), pos]; bypass when vis <= K; ties to the lower index;
 *  Top-K reported in ascending index order, -1 padded; softmax scale given by
 *  the caller; scores over all D dims, values are dims [0,V); inverse RoPE on
 *  output dims [V-R, V) with interleaved pairs, theta_i = base^(-2i/R),
 *  rotation by -pos*theta_i; HCA = every ratio-r2 row visible, no Top-K.
 *
 * Quantised indexer keys ("Fix: complete DeepSeek V4 TP CSA decode", PR
 * description: the indexer cache is a key pool plus a per-row scale pool):
 * with idx_dtype ORC_FP8_E4M3 a key element is one OCP FP8 E4M3 byte and the
 * key row is scale[row] times the decoded bytes; the score formula is
 * unchanged.  The element format is a reading (the pages name no format).
 *
 * Parity pins live in the tests; every function below is pinned there.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_FP8_E4M3 2

typedef struct {
    int32_t H, D, V, Hi, Di;
    int32_t ratio, topk, win, hca_ratio; /* hca_ratio 0 = no HCA stream */
    int32_t dtype;                       /* ORC_F32 or ORC_BF16 */
    double scale, rope_base;
    int32_t idx_dtype;                   /* 0: keys in dtype; ORC_FP8_E4M3: bytes + row scale */
} orc_cfg;

/* Host copies of one batch.  Pool row r of request b sits at
 * pool + (off[b] + r) * stride elements. */
typedef struct {
    int32_t B, S;
    const int32_t *ctx_len;
    const void *q;     /* [B,S,H,D]   */
    const void *q_idx; /* [B,S,Hi,Di] */
    const float *w;    /* [B,S,Hi]    */
    const void *raw;   const int64_t *raw_off; int64_t raw_stride;
    const void *cmp;   const int64_t *cmp_off; int64_t cmp_stride;
    const void *idx;   const int64_t *idx_off; int64_t idx_stride;
    const void *hca;   const int64_t *hca_off; int64_t hca_stride;
    const float *idx_scale; /* [rows] scale of each FP8 key row */
    /* paged pools: NULL tables = the contiguous layout above */
    const int32_t *raw_table, *cmp_table, *idx_table, *hca_table;
    int32_t raw_block, cmp_block, idx_block, hca_block, table_stride;
} orc_batch;

/* ------------------------------------------------------------------ */
/* storage decoding                                                    */

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static double orc_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double orc_load(const void *base, int32_t dtype, int64_t i)
{
    if (dtype == ORC_BF16)
        return orc_bf16_to_double(((const uint16_t *)base)[i]);
    return (double)((const float *)base)[i];
}

static void orc_load_vec(const void *base, int32_t dtype, int64_t first,
                         int64_t n, double *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = orc_load(base, dtype, first + i);
}

/* OCP FP8 E4M3 (the "fn" variant): bit 7 sign, bits 6..3 exponent e with
 * bias 7, bits 2..0 mantissa m.  e = 0: subnormal, m/8 * 2^(1-7); e = 15 and
 * m = 7: NaN (there is no infinity); otherwise (1 + m/8) * 2^(e-7). */
double orc_e4m3_to_double(uint8_t v)
{
    const int sign = v >> 7, e = (v >> 3) & 15, m = v & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Pool row of row r of request b: with a block table (a paged pool), entry
 * r / block of the request's table names the pool block that holds it, at
 * offset r % block; without one, the request's rows are consecutive from
 * off[b].  -1 when the block is unmapped (a negative entry) or past the
 * table.  (Paged pools: the pages' allocator-mapped cache pools, "Fix:
 * complete DeepSeek V4 TP CSA decode", PR description.) */
static int64_t orc_pool_row(const int32_t *table, int32_t block, int32_t tstride,
                            const int64_t *off, int32_t b, int64_t r)
{
    if (!table) return off[b] + r;
    if (r < 0 || r / block >= tstride) return -1;
    const int32_t pb = table[(int64_t)b * tstride + r / block];
    return pb < 0 ? -1 : (int64_t)pb * block + r % block;
}

/* Loads row `row` of a pool of width n, or zeros and *bad = 1 if row < 0. */
static void orc_load_row(const void *base, int32_t dtype, int64_t row, int64_t stride,
                         int64_t n, double *dst, int *bad)
{
    if (row < 0) {
        for (int64_t i = 0; i < n; ++i) dst[i] = 0.0;
        *bad = 1;
        return;
    }
    orc_load_vec(base, dtype, row * stride, n, dst);
}

/* Indexer key row `row` of the pool (absolute row index). */
static void orc_load_key_row(const orc_cfg *c, const orc_batch *bt, int64_t row, double *dst)
{
    if (c->idx_dtype == ORC_FP8_E4M3) {
        const uint8_t *p = (const uint8_t *)bt->idx + row * bt->idx_stride;
        const double sc = (double)bt->idx_scale[row];
        for (int32_t d = 0; d < c->Di; ++d)
            dst[d] = sc * orc_e4m3_to_double(p[d]);
    } else {
        orc_load_vec(bt->idx, c->dtype, row * bt->idx_stride, c->Di, dst);
    }
}

/* ------------------------------------------------------------------ */
/* (a) indexer score                                                   */

/* score_j = sum_{h ascending} w_h * max(0, sum_d qi[h,d] * k[j,d]). */
void orc_index_scores(int32_t Hi, int32_t Di, const double *qi,
                      const double *w, int32_t nrows, const double *k,
                      double *scores)
{
    for (int32_t j = 0; j < nrows; ++j) {
        double acc = 0.0;
        for (int32_t h = 0; h < Hi; ++h) {
            double dot = 0.0;
            for (int32_t d = 0; d < Di; ++d)
                dot += qi[(int64_t)h * Di + d] * k[(int64_t)j * Di + d];
            acc += w[h] * (dot > 0.0 ? dot : 0.0);
        }
        scores[j] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* (b) Top-K: full sort by (-score, index), keep K, report ascending.  */

typedef struct {
    double key;
    int32_t j;
} orc_pair;

static int orc_cmp_desc(const void *a, const void *b)
{
    const orc_pair *x = (const orc_pair *)a, *y = (const orc_pair *)b;
    if (x->key > y->key) return -1;
    if (x->key < y->key) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int orc_cmp_int(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Writes min(n, K) indices into idx (ascending), returns that count.
 * Scores must hold no NaN; -0.0 and +0.0 compare equal. */
int32_t orc_topk(const double *scores, int32_t n, int32_t K, int32_t *idx)
{
    int32_t cnt = n < K ? n : K;
    if (cnt <= 0) return 0;
    orc_pair *p = (orc_pair *)malloc(sizeof(orc_pair) * (size_t)n);
    for (int32_t j = 0; j < n; ++j) {
        p[j].key = scores[j];
        p[j].j = j;
    }
    qsort(p, (size_t)n, sizeof(orc_pair), orc_cmp_desc);
    for (int32_t i = 0; i < cnt; ++i) idx[i] = p[i].j;
    free(p);
    qsort(idx, (size_t)cnt, sizeof(int32_t), orc_cmp_int);
    return cnt;
}

/* ------------------------------------------------------------------ */
/* (d) softmax attention over a set of rows shared by all heads.      */

/* s[h,u] = scale * q[h,:D] . rows[u,:D];  p = softmax_u(s[h,:]);
 * o[h,v] = sum_u p[h,u] rows[u,v] for v < V;  lse[h] = log sum_u exp s[h,u].
 * With no rows, o = 0 and lse = -inf (an empty stream). */
void orc_attend(int32_t H, int32_t D, int32_t V, double scale,
                const double *q, int32_t nrows, const double *rows,
                double *o, double *lse)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(nrows > 0 ? nrows : 1));
    for (int32_t h = 0; h < H; ++h) {
        double *oh = o + (int64_t)h * V;
        for (int32_t v = 0; v < V; ++v) oh[v] = 0.0;
        if (nrows == 0) {
            lse[h] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int32_t u = 0; u < nrows; ++u) {
            double dot = 0.0;
            for (int32_t d = 0; d < D; ++d)
                dot += q[(int64_t)h * D + d] * rows[(int64_t)u * D + d];
            s[u] = scale * dot;
            if (s[u] > m) m = s[u];
        }
        double l = 0.0;
        for (int32_t u = 0; u < nrows; ++u) {
            s[u] = exp(s[u] - m);
            l += s[u];
        }
        for (int32_t u = 0; u < nrows; ++u) {
            double p = s[u] / l;
            for (int32_t v = 0; v < V; ++v)
                oh[v] += p * rows[(int64_t)u * D + v];
        }
        lse[h] = m + log(l);
    }
    free(s);
}

/* ------------------------------------------------------------------ */
/* inverse RoPE on the last R output dims [V-R, V), interleaved pairs. */

void orc_inverse_rope(int32_t H, int32_t V, int32_t R, double pos,
                      double base, double *o)
{
    for (int32_t h = 0; h < H; ++h) {
        double *x = o + (int64_t)h * V + (V - R);
        for (int32_t i = 0; i < R / 2; ++i) {
            double theta = pos * pow(base, -2.0 * (double)i / (double)R);
            double c = cos(theta), s = sin(theta);
            double x0 = x[2 * i], x1 = x[2 * i + 1];
            x[2 * i] = x0 * c + x1 * s;
            x[2 * i + 1] = -x0 * s + x1 * c;
        }
    }
}

/* ------------------------------------------------------------------ */
/* one query of the decode step                                        */

#define ORC_FORCE_SCORE 1 /* run scoring + sort even when vis <= K */

typedef struct {
    int32_t pos, vis, nwin, cnt, vis2, rows_used;
} orc_query_info;

/* Computes query (b, s).  out: [H*V] after inverse RoPE; lse: [H] of the
 * union softmax; idx: [K] ascending, -1 padded; info: counts. */
int orc_query(const orc_cfg *c, const orc_batch *bt, int32_t b, int32_t s,
              int32_t flags, double *out, double *lse, int32_t *idx,
              orc_query_info *info)
{
    const int32_t H = c->H, D = c->D, V = c->V, Hi = c->Hi, Di = c->Di;
    const int32_t K = c->topk;
    const int64_t qid = (int64_t)b * bt->S + s;
    const int32_t L = bt->ctx_len[b];
    const int32_t pos = L - bt->S + s;
    if (pos < 0) return -1;
    const int32_t vis = (pos + 1) / c->ratio;
    const int32_t nwin = (c->win < pos + 1) ? c->win : pos + 1;
    const int32_t vis2 = c->hca_ratio > 0 ? (pos + 1) / c->hca_ratio : 0;
    int bad = 0; /* a row the query needs lies in an unmapped block */

    /* (a)+(b): indexer score and Top-K, or the bypass */
    int32_t cnt;
    for (int32_t i = 0; i < K; ++i) idx[i] = -1;
    if (vis > K || (flags & ORC_FORCE_SCORE)) {
        double *qi = (double *)malloc(sizeof(double) * (size_t)Hi * Di);
        double *wv = (double *)malloc(sizeof(double) * (size_t)Hi);
        double *kr = (double *)malloc(sizeof(double) * (size_t)(vis > 0 ? vis : 1) * Di);
        double *sc = (double *)malloc(sizeof(double) * (size_t)(vis > 0 ? vis : 1));
        orc_load_vec(bt->q_idx, c->dtype, qid * Hi * Di, (int64_t)Hi * Di, qi);
        for (int32_t h = 0; h < Hi; ++h) wv[h] = (double)bt->w[qid * Hi + h];
        for (int32_t j = 0; j < vis; ++j) {
            const int64_t row = orc_pool_row(bt->idx_table, bt->idx_block, bt->table_stride,
                                             bt->idx_off, b, j);
            if (row < 0) {
                bad = 1;
                for (int32_t d = 0; d < Di; ++d) kr[(int64_t)j * Di + d] = 0.0;
            } else {
                orc_load_key_row(c, bt, row, kr + (int64_t)j * Di);
            }
        }
        orc_index_scores(Hi, Di, qi, wv, vis, kr, sc);
        cnt = orc_topk(sc, vis, K, idx);
        free(qi); free(wv); free(kr); free(sc);
    } else {
        cnt = vis;
        for (int32_t j = 0; j < vis; ++j) idx[j] = j;
    }

    /* (c): the rows this query reads, window first, then selected
     * compressed rows, then HCA rows; one union, no de-duplication. */
    const int32_t nrows = nwin + cnt + vis2;
    double *rows = (double *)malloc(sizeof(double) * (size_t)(nrows > 0 ? nrows : 1) * D);
    int32_t u = 0;
    for (int32_t r = pos - nwin + 1; r <= pos; ++r, ++u)
        orc_load_row(bt->raw, c->dtype,
                     orc_pool_row(bt->raw_table, bt->raw_block, bt->table_stride, bt->raw_off, b, r),
                     bt->raw_stride, D, rows + (int64_t)u * D, &bad);
    for (int32_t i = 0; i < cnt; ++i, ++u)
        orc_load_row(bt->cmp, c->dtype,
                     orc_pool_row(bt->cmp_table, bt->cmp_block, bt->table_stride, bt->cmp_off, b, idx[i]),
                     bt->cmp_stride, D, rows + (int64_t)u * D, &bad);
    for (int32_t r = 0; r < vis2; ++r, ++u)
        orc_load_row(bt->hca, c->dtype,
                     orc_pool_row(bt->hca_table, bt->hca_block, bt->table_stride, bt->hca_off, b, r),
                     bt->hca_stride, D, rows + (int64_t)u * D, &bad);

    /* (d): one softmax over the union, then inverse RoPE */
    double *qv = (double *)malloc(sizeof(double) * (size_t)H * D);
    orc_load_vec(bt->q, c->dtype, qid * H * D, (int64_t)H * D, qv);
    orc_attend(H, D, V, c->scale, qv, nrows, rows, out, lse);
    orc_inverse_rope(H, V, D - V, (double)pos, c->rope_base, out);
    free(qv);
    free(rows);

    if (info) {
        info->pos = pos;
        info->vis = vis;
        info->nwin = nwin;
        info->cnt = cnt;
        info->vis2 = vis2;
        info->rows_used = nrows;
    }
    return bad ? -2 : 0;
}

/* Scores of every visible row of query (b, s); returns vis. */
int32_t orc_query_scores(const orc_cfg *c, const orc_batch *bt, int32_t b,
                         int32_t s, double *scores)
{
    const int32_t Hi = c->Hi, Di = c->Di;
    const int64_t qid = (int64_t)b * bt->S + s;
    const int32_t pos = bt->ctx_len[b] - bt->S + s;
    const int32_t vis = (pos + 1) / c->ratio;
    double *qi = (double *)malloc(sizeof(double) * (size_t)Hi * Di);
    double *wv = (double *)malloc(sizeof(double) * (size_t)Hi);
    double *kr = (double *)malloc(sizeof(double) * (size_t)(vis > 0 ? vis : 1) * Di);
    orc_load_vec(bt->q_idx, c->dtype, qid * Hi * Di, (int64_t)Hi * Di, qi);
    for (int32_t h = 0; h < Hi; ++h) wv[h] = (double)bt->w[qid * Hi + h];
    int bad = 0;
    for (int32_t j = 0; j < vis; ++j) {
        const int64_t row = orc_pool_row(bt->idx_table, bt->idx_block, bt->table_stride,
                                         bt->idx_off, b, j);
        if (row < 0)
            bad = 1;
        else
            orc_load_key_row(c, bt, row, kr + (int64_t)j * Di);
    }
    if (!bad) orc_index_scores(Hi, Di, qi, wv, vis, kr, scores);
    free(qi); free(wv); free(kr);
    return bad ? -1 : vis;
}

/* ------------------------------------------------------------------ */
/* a list of queries, spread over threads                              */

typedef struct {
    const orc_cfg *c;
    const orc_batch *bt;
    const int32_t *qids;
    int32_t nq, flags, tid, nthreads;
    double *out, *lse;
    int32_t *idx;
    orc_query_info *info;
    int rc;
} orc_job;

static void *orc_worker(void *arg)
{
    orc_job *j = (orc_job *)arg;
    const orc_cfg *c = j->c;
    for (int32_t t = j->tid; t < j->nq; t += j->nthreads) {
        int32_t q = j->qids[t];
        int32_t b = q / j->bt->S, s = q % j->bt->S;
        int rc = orc_query(c, j->bt, b, s, j->flags,
                           j->out + (int64_t)t * c->H * c->V,
                           j->lse + (int64_t)t * c->H,
                           j->idx + (int64_t)t * c->topk,
                           j->info ? j->info + t : NULL);
        if (rc) j->rc = rc;
    }
    return NULL;
}

/* Runs the queries qids[0..nq) (flattened b*S+s) on nthreads threads.
 * Output slot t belongs to qids[t].  Returns 0, -1 on a bad query, or -2 if
 * a row a query needs lies in an unmapped block of a paged pool. */
int orc_decode(const orc_cfg *c, const orc_batch *bt, const int32_t *qids,
               int32_t nq, int32_t flags, int32_t nthreads, double *out,
               double *lse, int32_t *idx, orc_query_info *info)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nq) nthreads = nq > 0 ? nq : 1;
    orc_job *jobs = (orc_job *)calloc((size_t)nthreads, sizeof(orc_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int32_t t = 0; t < nthreads; ++t) {
        jobs[t] = (orc_job){c, bt, qids, nq, flags, t, nthreads, out, lse, idx, info, 0};
        if (nthreads == 1)
            orc_worker(&jobs[t]);
        else
            pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
    }
    int rc = 0;
    for (int32_t t = 0; t < nthreads; ++t) {
        if (nthreads > 1) pthread_join(th[t], NULL);
        if (jobs[t].rc) rc = jobs[t].rc;
    }
    free(jobs);
    free(th);
    return rc;
}
