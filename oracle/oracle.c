/*
 * oracle.c -- plain, slow CPU reference for the DeepSeek V4.1 attention hot path:
 * Indexer scores -> top-k -> sparse attention with an attention sink.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library.  It shares no code, header, table or
 * constant with the CUDA library and includes nothing from it.
 *
 * Sources (page title "DeepSeek V4.1", four pages of model source):
 *   [sel]   .../reuse-layers/attention/attend/selected  (mode=prefill)
 *   [read]  .../reindex-groups/reindex-layer/read-weights (mode=decode)
 *   [allow] .../source-layer/attention/attend/allowed  (mode=decode; same code as [sel])
 *
 * Precision: every floating-point accumulation is in double.  bf16 inputs are passed as
 * their 16-bit patterns and widened exactly (bf16 -> fp32 is a 16-bit shift, fp32 ->
 * double is exact).  Rows (one query each) are independent, so a fixed pool of POSIX
 * threads splits them; the arithmetic of a row does not depend on the thread count.
 *
 * Parity pins: every function below is pinned by the CPU tests (worked examples from
 * the pages, closed forms, brute force, library reductions).  No function is unpinned.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ helpers */

static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Run fn(ctx, row) for row in [0, n_rows) on up to n_threads POSIX threads. */
typedef void (*row_fn)(void *ctx, int64_t row);
typedef struct {
    row_fn fn;
    void *ctx;
    int64_t n_rows;
    int n_threads;
    int tid;
} worker_arg;

static void *worker_main(void *p) {
    worker_arg *a = (worker_arg *)p;
    for (int64_t r = a->tid; r < a->n_rows; r += a->n_threads) a->fn(a->ctx, r);
    return NULL;
}

static void parallel_rows(row_fn fn, void *ctx, int64_t n_rows, int n_threads) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((int64_t)n_threads > n_rows) n_threads = (int)(n_rows > 0 ? n_rows : 1);
    pthread_t th[256];
    worker_arg args[256];
    for (int i = 0; i < n_threads; ++i) {
        args[i].fn = fn;
        args[i].ctx = ctx;
        args[i].n_rows = n_rows;
        args[i].n_threads = n_threads;
        args[i].tid = i;
    }
    for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], NULL, worker_main, &args[i]);
    worker_main(&args[0]);
    for (int i = 1; i < n_threads; ++i) pthread_join(th[i], NULL);
}

/* --------------------------------------------------- window indices, lengths */

/*
 * [sel] get_window_topk_idxs(window_size, bsz, seqlen, start_pos).
 * Prefill (start_pos == 0): row t lists min(seqlen, W) slots starting at
 * max(0, t-W+1); any slot past t is -1 (before the sequence started).
 * Decode (start_pos > 0): one row listing the W ring slots oldest first,
 * slots (start_pos % W)+1 .. W-1 then 0 .. start_pos % W; a slot > start_pos is -1
 * (ring still filling).  Every batch row gets the same indices.
 * out: [bsz, rows, width] with rows = seqlen, width = min(seqlen, W) in prefill and
 * rows = 1, width = W in decode.  Returns width.
 */
int oracle_window_topk_idxs(int window_size, int bsz, int seqlen, int start_pos, int32_t *out) {
    int W = window_size;
    if (start_pos == 0) {
        int width = seqlen < W ? seqlen : W;
        for (int t = 0; t < seqlen; ++t) {
            int first = t - W + 1;
            if (first < 0) first = 0;
            for (int i = 0; i < width; ++i) {
                int idx = first + i;
                int32_t v = idx > t ? -1 : idx;
                for (int b = 0; b < bsz; ++b) out[((int64_t)b * seqlen + t) * width + i] = v;
            }
        }
        return width;
    }
    int oldest = start_pos % W + 1;
    for (int i = 0; i < W; ++i) {
        int idx = i < W - oldest ? oldest + i : i - (W - oldest);
        int32_t v = idx > start_pos ? -1 : idx;
        for (int b = 0; b < bsz; ++b) out[(int64_t)b * W + i] = v;
    }
    return W;
}

/* [read] Attention._compress_kv: compress_len = (start_pos + seqlen) // ratio. */
int oracle_compress_len(int start_pos, int seqlen, int ratio) { return (start_pos + seqlen) / ratio; }

/*
 * [sel] Indexer.forward: how many compressed positions query t sees.  Prefill uses
 * compress_lens[t] = (t+1) // ratio, decode end_pos // ratio with end_pos = start_pos+1;
 * both are (start_pos + t + 1) // ratio (group j becomes visible once the query has
 * passed the last token of its group, i.e. (j+1)*ratio <= start_pos+t+1).
 */
int oracle_visible(int start_pos, int t, int ratio) { return (start_pos + t + 1) / ratio; }

/* ------------------------------------------------------------ index scores */

typedef struct {
    const uint16_t *q;   /* [b, s, H, D] bf16 bits: index queries */
    const uint16_t *k;   /* [b, *, D] bf16 bits: index keys, batch stride k_bstride */
    int64_t k_bstride;   /* elements between batch rows of k */
    const uint16_t *w;   /* [b, s, H] bf16 bits: weights_proj output */
    double c;            /* index_head_dim^-0.5 * index_n_heads^-0.5 */
    const int32_t *start_pos;
    int s, H, D, n_cols, ratio;
    double *score;       /* [b, s, n_cols] */
} score_ctx;

/*
 * [sel] Indexer.forward:
 *   weights     = weights_proj(x) * (softmax_scale * n_heads^-0.5)
 *   index_score = einsum("bshd,btd->bsht", q, index_k)
 *   index_score = (relu(index_score) * weights).sum(over h)
 *   then positions the query cannot see are set to -inf.
 */
static void score_row(void *vctx, int64_t row) {
    score_ctx *x = (score_ctx *)vctx;
    int b = (int)(row / x->s), t = (int)(row % x->s);
    int vis = oracle_visible(x->start_pos[b], t, x->ratio);
    if (vis > x->n_cols) vis = x->n_cols;
    const uint16_t *qrow = x->q + row * x->H * x->D;
    const uint16_t *wrow = x->w + row * x->H;
    double *out = x->score + row * x->n_cols;
    double *qd = (double *)malloc(sizeof(double) * x->H * x->D);
    double *wd = (double *)malloc(sizeof(double) * x->H);
    for (int i = 0; i < x->H * x->D; ++i) qd[i] = bf16_bits_to_double(qrow[i]);
    for (int h = 0; h < x->H; ++h) wd[h] = bf16_bits_to_double(wrow[h]) * x->c;
    for (int j = 0; j < x->n_cols; ++j) {
        if (j >= vis) {
            out[j] = -INFINITY;
            continue;
        }
        const uint16_t *krow = x->k + (int64_t)b * x->k_bstride + (int64_t)j * x->D;
        double acc = 0.0;
        for (int h = 0; h < x->H; ++h) {
            double dot = 0.0;
            for (int e = 0; e < x->D; ++e) dot += qd[h * x->D + e] * bf16_bits_to_double(krow[e]);
            double r = dot > 0.0 ? dot : 0.0; /* relu */
            acc += r * wd[h];
        }
        out[j] = acc;
    }
    free(qd);
    free(wd);
}

void oracle_index_score(const uint16_t *q, const uint16_t *k, int64_t k_bstride, const uint16_t *w, double c,
                        const int32_t *start_pos, int b, int s, int H, int D, int n_cols, int ratio, double *score,
                        int n_threads) {
    score_ctx x = {q, k, k_bstride, w, c, start_pos, s, H, D, n_cols, ratio, score};
    parallel_rows(score_row, &x, (int64_t)b * s, n_threads);
}

/* ------------------------------------------------------------------- top-k */

typedef struct {
    double v;
    int32_t pos;
} scored_pos;

/* order: higher score first; equal scores -> lower position first */
static int by_score_desc(const void *a, const void *b) {
    const scored_pos *x = (const scored_pos *)a, *y = (const scored_pos *)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static int by_int_asc(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

typedef struct {
    const double *score; /* [b, s, n_cols] */
    const int32_t *start_pos;
    int s, n_cols, ratio, k;
    int32_t offset;
    int32_t *out;        /* [b, s, k] */
} topk_ctx;

/*
 * [sel] Indexer.forward, last three lines:
 *   topk = min(index_topk, end_pos // ratio)
 *   idxs = index_score.topk(topk).indices.sort()
 *   out  = where(idxs < compress_lens, idxs + offset, -1)
 * Written as a full sort of the visible positions by (score desc, position asc), the
 * first min(k, vis) kept, put back in position order, shifted by offset, and padded
 * with -1 to width k (the masked -inf columns the page's topk may pick become -1 and
 * sort after every visible position, so the padded row is the same set and order).
 */
static void topk_row(void *vctx, int64_t row) {
    topk_ctx *x = (topk_ctx *)vctx;
    int b = (int)(row / x->s), t = (int)(row % x->s);
    int vis = oracle_visible(x->start_pos[b], t, x->ratio);
    if (vis > x->n_cols) vis = x->n_cols;
    const double *sc = x->score + row * x->n_cols;
    int32_t *out = x->out + row * x->k;
    int m = vis < x->k ? vis : x->k;
    if (m < 0) m = 0;
    scored_pos *all = (scored_pos *)malloc(sizeof(scored_pos) * (vis > 0 ? vis : 1));
    for (int j = 0; j < vis; ++j) {
        all[j].v = sc[j];
        all[j].pos = j;
    }
    qsort(all, (size_t)vis, sizeof(scored_pos), by_score_desc);
    int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (m > 0 ? m : 1));
    for (int i = 0; i < m; ++i) sel[i] = all[i].pos;
    qsort(sel, (size_t)m, sizeof(int32_t), by_int_asc);
    for (int i = 0; i < x->k; ++i) out[i] = i < m ? sel[i] + x->offset : -1;
    free(all);
    free(sel);
}

void oracle_topk(const double *score, const int32_t *start_pos, int b, int s, int n_cols, int ratio, int k,
                 int32_t offset, int32_t *out, int n_threads) {
    topk_ctx x = {score, start_pos, s, n_cols, ratio, k, offset, out};
    parallel_rows(topk_row, &x, (int64_t)b * s, n_threads);
}

/* ------------------------------------------------- sparse attention + sink */

typedef struct {
    const uint16_t *q;    /* [b, s, h, d] */
    const uint16_t *kv1;  /* first KV source [b, n1, d], batch stride kv1_bstride */
    int64_t kv1_bstride;
    const uint16_t *kv2;  /* second KV source [b, n2, d] or NULL */
    int64_t kv2_bstride;
    int n1, n2;
    const float *sink;    /* [h] */
    const int32_t *idx;   /* [b, s, k] */
    double scale;
    int s, h, d, k;
    double *out;          /* [b, s, h, d] */
    double *lse;          /* [b, s, h] or NULL */
} attn_ctx;

/*
 * Row r of kv = cat([kv1, kv2], dim=1) ([sel] Attention.forward concatenates the window
 * KV and the compressed KV along the position axis).  NULL for indices that hold nothing.
 */
static const uint16_t *kv_row(const attn_ctx *x, int b, int32_t r) {
    if (r < 0) return NULL;
    if (r < x->n1) return x->kv1 + (int64_t)b * x->kv1_bstride + (int64_t)r * x->d;
    if (x->kv2 != NULL && r < x->n1 + x->n2)
        return x->kv2 + (int64_t)b * x->kv2_bstride + (int64_t)(r - x->n1) * x->d;
    return NULL; /* out of range: treated as masked */
}

/*
 * [sel] sparse_attn_kernel / sparse_attn: for each query and head,
 *   s_i = softmax_scale * q . kv[idx_i]         over slots with idx_i != -1
 *   o   = sum_i e^{s_i} kv[idx_i] / (sum_i e^{s_i} + e^{attn_sink[h]})
 * the same row serving as key and value; a query with no valid slot gets o = 0.
 * Computed exactly in double with the max M = max_i s_i factored out;
 * lse = M + ln(sum_i e^{s_i-M} + e^{sink-M}) (the log of the full denominator).
 */
static void attn_row(void *vctx, int64_t row) {
    attn_ctx *x = (attn_ctx *)vctx;
    int b = (int)(row / x->s);
    const int32_t *ids = x->idx + row * x->k;
    const uint16_t **rows = (const uint16_t **)malloc(sizeof(void *) * (x->k > 0 ? x->k : 1));
    double *logit = (double *)malloc(sizeof(double) * (x->k > 0 ? x->k : 1));
    double *acc = (double *)malloc(sizeof(double) * x->d);
    for (int i = 0; i < x->k; ++i) rows[i] = kv_row(x, b, ids[i]);
    for (int hh = 0; hh < x->h; ++hh) {
        const uint16_t *qv = x->q + (row * x->h + hh) * x->d;
        double *o = x->out + (row * x->h + hh) * x->d;
        double m = -INFINITY;
        int any = 0;
        for (int i = 0; i < x->k; ++i) {
            if (rows[i] == NULL) continue;
            double dot = 0.0;
            for (int e = 0; e < x->d; ++e) dot += bf16_bits_to_double(qv[e]) * bf16_bits_to_double(rows[i][e]);
            logit[i] = x->scale * dot;
            if (logit[i] > m) m = logit[i];
            any = 1;
        }
        if (!any) {
            for (int e = 0; e < x->d; ++e) o[e] = 0.0;
            if (x->lse) x->lse[row * x->h + hh] = -INFINITY;
            continue;
        }
        double z = exp((double)x->sink[hh] - m);
        for (int e = 0; e < x->d; ++e) acc[e] = 0.0;
        for (int i = 0; i < x->k; ++i) {
            if (rows[i] == NULL) continue;
            double p = exp(logit[i] - m);
            z += p;
            for (int e = 0; e < x->d; ++e) acc[e] += p * bf16_bits_to_double(rows[i][e]);
        }
        for (int e = 0; e < x->d; ++e) o[e] = acc[e] / z;
        if (x->lse) x->lse[row * x->h + hh] = m + log(z);
    }
    free(rows);
    free(logit);
    free(acc);
}

void oracle_sparse_attn(const uint16_t *q, const uint16_t *kv1, int64_t kv1_bstride, const uint16_t *kv2,
                        int64_t kv2_bstride, int n1, int n2, const float *sink, const int32_t *idx, double scale,
                        int b, int s, int h, int d, int k, double *out, double *lse, int n_threads) {
    attn_ctx x = {q, kv1, kv1_bstride, kv2, kv2_bstride, n1, n2, sink, idx, scale, s, h, d, k, out, lse};
    parallel_rows(attn_row, &x, (int64_t)b * s, n_threads);
}

/* ------------------------------------- dense windowed + compressed reference */

typedef struct {
    const uint16_t *q;    /* [b, s, h, d] */
    const uint16_t *win;  /* prefill: raw KV [b, s, d]; decode: ring [b, W, d] (position p in slot p % W) */
    int64_t win_bstride;
    const uint16_t *comp; /* compressed KV [b, *, d]; row j stands for positions j*ratio .. j*ratio+ratio-1 */
    int64_t comp_bstride;
    const int32_t *start_pos;
    const float *sink;
    double scale;
    int s, h, d, W, ratio;
    double *out;
} dense_ctx;

/*
 * Dense causal windowed attention with a sink, defined by positions alone (no index
 * lists): query t at position p = start_pos+t attends to the raw positions
 * max(0, p-W+1) .. p (the sliding window) and to every compressed group j with
 * (j+1)*ratio <= p+1 (a group is visible once the query passed its last token).
 * With index_topk >= the visible count the Indexer keeps every visible group, so the
 * sparse path must equal this.  In decode (s == 1) the raw window lives in the ring,
 * position p in slot p % W; in prefill (start_pos == 0) it is raw row p.
 */
static void dense_row(void *vctx, int64_t row) {
    dense_ctx *x = (dense_ctx *)vctx;
    int b = (int)(row / x->s), t = (int)(row % x->s);
    int p = x->start_pos[b] + t;
    int first = p - x->W + 1;
    if (first < 0) first = 0;
    int n_win = p - first + 1;
    int n_comp = (p + 1) / x->ratio;
    int n_all = n_win + n_comp;
    const uint16_t **rows = (const uint16_t **)malloc(sizeof(void *) * n_all);
    for (int i = 0; i < n_win; ++i) {
        int pos = first + i;
        int slot = x->start_pos[b] == 0 ? pos : pos % x->W;
        rows[i] = x->win + (int64_t)b * x->win_bstride + (int64_t)slot * x->d;
    }
    for (int j = 0; j < n_comp; ++j) rows[n_win + j] = x->comp + (int64_t)b * x->comp_bstride + (int64_t)j * x->d;
    double *logit = (double *)malloc(sizeof(double) * n_all);
    double *acc = (double *)malloc(sizeof(double) * x->d);
    for (int hh = 0; hh < x->h; ++hh) {
        const uint16_t *qv = x->q + (row * x->h + hh) * x->d;
        double m = -INFINITY;
        for (int i = 0; i < n_all; ++i) {
            double dot = 0.0;
            for (int e = 0; e < x->d; ++e) dot += bf16_bits_to_double(qv[e]) * bf16_bits_to_double(rows[i][e]);
            logit[i] = x->scale * dot;
            if (logit[i] > m) m = logit[i];
        }
        double z = exp((double)x->sink[hh] - m);
        for (int e = 0; e < x->d; ++e) acc[e] = 0.0;
        for (int i = 0; i < n_all; ++i) {
            double pr = exp(logit[i] - m);
            z += pr;
            for (int e = 0; e < x->d; ++e) acc[e] += pr * bf16_bits_to_double(rows[i][e]);
        }
        double *o = x->out + (row * x->h + hh) * x->d;
        for (int e = 0; e < x->d; ++e) o[e] = acc[e] / z;
    }
    free(rows);
    free(logit);
    free(acc);
}

void oracle_dense_attn(const uint16_t *q, const uint16_t *win, int64_t win_bstride, const uint16_t *comp,
                       int64_t comp_bstride, const int32_t *start_pos, const float *sink, double scale, int b, int s,
                       int h, int d, int W, int ratio, double *out, int n_threads) {
    dense_ctx x = {q, win, win_bstride, comp, comp_bstride, start_pos, sink, scale, s, h, d, W, ratio, out};
    parallel_rows(dense_row, &x, (int64_t)b * s, n_threads);
}
