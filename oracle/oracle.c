/*
 * oracle.c -- plain fp64 CPU oracle for one decode step of attention with a
 * KV append, grouped-query heads, an optional sliding window and a per-head
 * attention-sink logit, over three cache layouts (paged, ring, contiguous).
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library. The CUDA path shares no
 * code, header, table or helper with it, and never calls it.
 *
 * What is computed (SimpleLLM README, changes table, row "one decode-attention
 * kernel for sinks, sliding window, GQA and the KV append"; the paged cache
 * and the ring buffer come from the rows "paged KV cache for full-attention
 * layers" and "ring buffer for sliding-window layers" of the same table). The
 * pages print no formula, so the definition below is the plain reading:
 *
 *   for each active sequence b (seq_lens[b] = L > 0, the length *after* the
 *   new token is appended; the new token sits at position p = L - 1),
 *   each query head h, and KV head g = h / (Hq / Hkv)   (grouped-query):
 *     J      = positions j with lo <= j < L, lo = max(0, L - W) when a window
 *              W > 0 applies, else lo = 0        (window includes token p)
 *     s_j    = scale * sum_d q[b,h,d] * k_j[g,d]
 *     M      = max(sigma_h, max_j s_j)            (sigma_h = sink logit, or
 *                                                  -inf when there is none)
 *     out    = sum_j e^(s_j - M) v_j[g,:] / (e^(sigma_h - M) + sum_j e^(s_j - M))
 *   and out = 0 for an inactive sequence (L = 0).
 *
 * Token j < p is read from the cache through the layout's address map; token
 * p is k_new / v_new (when given) -- the append happens before attention.
 *
 * Layouts (element = bf16, given as raw 16-bit patterns):
 *   paged : k_cache[num_pages][Hkv][P][D]; token j of b lives in page
 *           block_table[b][j / P], slot j % P.
 *   ring  : k_cache[B][Hkv][W][D]; token j of b lives in cell j % W.
 *   contig: hist[B][Tmax][Hkv][D]; token j of b is hist[b][j] (includes p).
 *
 * Every bf16 input is widened exactly to double; all arithmetic is fp64 with
 * libm exp(). Work is split over (b, h) pairs across POSIX threads; each pair
 * is computed exactly as written above, no blocking or reordering.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_BAD_ARG (-1)
#define OR_BAD_INDEX (-2)
#define OR_NOMEM (-3)

static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* Layout descriptions: each maps (b, g, position j) to a key/value row. */

enum layout_kind { LAYOUT_PAGED = 0, LAYOUT_RING = 1, LAYOUT_CONTIG = 2 };

typedef struct {
    int kind;
    const uint16_t *q;      /* [B][Hq][D] */
    const double *q64;      /* [B][Hq][D] rotated queries in fp64, used instead of q when set */
    const uint16_t *k_new;  /* [B][Hkv][D] or NULL */
    const uint16_t *v_new;
    const uint16_t *k_src;  /* cache or history, per kind */
    const uint16_t *v_src;
    const int32_t *block_table; /* paged: [B][max_pages] */
    const int32_t *seq_lens;    /* [B] */
    const float *sinks;         /* [Hq] or NULL */
    int window;                 /* 0 = no window (paged / contig); ring capacity (ring) */
    double scale;
    int B, Hq, Hkv, D;
    int P, max_pages, num_pages; /* paged */
    int Tmax;                    /* contig */
    const int32_t *items;        /* NULL = every (b, h); else n_items pairs (b, h) */
    int n_items;
    double *out;                 /* [B][Hq][D] or [n_items][D] */
    int status;                  /* first error seen, 0 if none */
} problem;

/* Address of the key (or value, when v != 0) row of position j, KV head g,
 * sequence b, taken from the cache (j < p) or from k_new/v_new (j == p).
 * Returns NULL when the address map leaves the buffers (bad input). */
static const uint16_t *token_row(const problem *pr, int b, int g, int j, int v) {
    const int L = pr->seq_lens[b];
    const int D = pr->D, Hkv = pr->Hkv;
    if (j == L - 1 && pr->k_new != NULL && pr->kind != LAYOUT_CONTIG) {
        const uint16_t *src = v ? pr->v_new : pr->k_new;
        return src + ((size_t)b * Hkv + g) * D;
    }
    const uint16_t *base = v ? pr->v_src : pr->k_src;
    if (pr->kind == LAYOUT_PAGED) {
        int slot_in_table = j / pr->P;
        if (slot_in_table >= pr->max_pages) return NULL;
        int32_t page = pr->block_table[(size_t)b * pr->max_pages + slot_in_table];
        if (page < 0 || page >= pr->num_pages) return NULL;
        return base + (((size_t)page * Hkv + g) * pr->P + (size_t)(j % pr->P)) * D;
    }
    if (pr->kind == LAYOUT_RING) {
        int cell = j % pr->window;
        return base + (((size_t)b * Hkv + g) * pr->window + (size_t)cell) * D;
    }
    /* contig */
    if (j >= pr->Tmax) return NULL;
    return base + (((size_t)b * pr->Tmax + j) * Hkv + g) * D;
}

/* One (b, h) output row, straight from the definition in the file header. */
static int attend_one(const problem *pr, int b, int h, double *out) {
    const int D = pr->D;
    const int L = pr->seq_lens[b];
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L <= 0) return OR_OK; /* inactive slot: output 0 */

    const int G = pr->Hq / pr->Hkv;
    const int g = h / G;
    int W = 0;
    if (pr->kind == LAYOUT_RING) W = pr->window;            /* ring: window = capacity */
    else if (pr->window > 0) W = pr->window;                /* paged / contig windowed */
    const int lo = (W > 0 && L - W > 0) ? L - W : 0;
    const int n = L - lo;

    const uint16_t *qrow = pr->q + ((size_t)b * pr->Hq + h) * D;
    const double *q64row = pr->q64 ? pr->q64 + ((size_t)b * pr->Hq + h) * D : NULL;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s) return OR_NOMEM;

    const double sigma = pr->sinks ? (double)pr->sinks[h] : -INFINITY;
    double M = sigma;
    for (int i = 0; i < n; ++i) {
        const uint16_t *krow = token_row(pr, b, g, lo + i, 0);
        if (!krow) { free(s); return OR_BAD_INDEX; }
        double dot = 0.0;
        if (q64row)
            for (int d = 0; d < D; ++d) dot += q64row[d] * bf16_to_f64(krow[d]);
        else
            for (int d = 0; d < D; ++d) dot += bf16_to_f64(qrow[d]) * bf16_to_f64(krow[d]);
        s[i] = pr->scale * dot;
        if (s[i] > M) M = s[i];
    }
    double den = isinf(sigma) && sigma < 0 ? 0.0 : exp(sigma - M);
    for (int i = 0; i < n; ++i) {
        const uint16_t *vrow = token_row(pr, b, g, lo + i, 1);
        if (!vrow) { free(s); return OR_BAD_INDEX; }
        double w = exp(s[i] - M);
        den += w;
        for (int d = 0; d < D; ++d) out[d] += w * bf16_to_f64(vrow[d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
    free(s);
    return OR_OK;
}

typedef struct {
    problem *pr;
    int tid, nthreads;
    int status;
} worker_arg;

static void *worker(void *p) {
    worker_arg *a = (worker_arg *)p;
    problem *pr = a->pr;
    const int total = pr->items ? pr->n_items : pr->B * pr->Hq;
    for (int w = a->tid; w < total; w += a->nthreads) {
        int b, h;
        if (pr->items) { b = pr->items[2 * w]; h = pr->items[2 * w + 1]; }
        else { b = w / pr->Hq; h = w % pr->Hq; }
        if (b < 0 || b >= pr->B || h < 0 || h >= pr->Hq) { a->status = OR_BAD_ARG; continue; }
        int st = attend_one(pr, b, h, pr->out + (size_t)w * pr->D);
        if (st != OR_OK && a->status == OR_OK) a->status = st;
    }
    return NULL;
}

static int run(problem *pr, int nthreads) {
    if (pr->B < 0 || pr->Hq <= 0 || pr->Hkv <= 0 || pr->D <= 0 || pr->Hq % pr->Hkv != 0)
        return OR_BAD_ARG;
    if ((!pr->q && !pr->q64) || !pr->seq_lens || !pr->out) return OR_BAD_ARG;
    if ((pr->k_new == NULL) != (pr->v_new == NULL)) return OR_BAD_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    worker_arg args[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        args[t].pr = pr; args[t].tid = t; args[t].nthreads = nthreads; args[t].status = OR_OK;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, &args[t]) != 0) break;
        started = t;
    }
    /* threads that failed to start: run their share here */
    for (int t = started + 1; t < nthreads; ++t) worker(&args[t]);
    worker(&args[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    int st = OR_OK;
    for (int t = 0; t < nthreads; ++t) if (args[t].status != OR_OK) { st = args[t].status; break; }
    return st;
}

/* ------------------------------------------------------------------ */
/* Public entry points.                                                */

int oracle_decode_paged(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                        const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_table, const int32_t *seq_lens, const float *sinks,
                        int window, double scale, double *out,
                        int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                        const int32_t *items, int n_items, int nthreads) {
    if (page_size <= 0 || max_pages <= 0 || num_pages <= 0 || window < 0 || !block_table)
        return OR_BAD_ARG;
    problem pr;
    memset(&pr, 0, sizeof pr);
    pr.kind = LAYOUT_PAGED;
    pr.q = q; pr.k_new = k_new; pr.v_new = v_new; pr.k_src = k_cache; pr.v_src = v_cache;
    pr.block_table = block_table; pr.seq_lens = seq_lens; pr.sinks = sinks;
    pr.window = window; pr.scale = scale; pr.B = B; pr.Hq = Hq; pr.Hkv = Hkv; pr.D = D;
    pr.P = page_size; pr.max_pages = max_pages; pr.num_pages = num_pages;
    pr.items = items; pr.n_items = n_items; pr.out = out;
    return run(&pr, nthreads);
}

int oracle_decode_ring(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                       const uint16_t *k_cache, const uint16_t *v_cache,
                       const int32_t *seq_lens, const float *sinks,
                       int window, double scale, double *out, int B, int Hq, int Hkv, int D,
                       const int32_t *items, int n_items, int nthreads) {
    if (window <= 0) return OR_BAD_ARG;
    problem pr;
    memset(&pr, 0, sizeof pr);
    pr.kind = LAYOUT_RING;
    pr.q = q; pr.k_new = k_new; pr.v_new = v_new; pr.k_src = k_cache; pr.v_src = v_cache;
    pr.seq_lens = seq_lens; pr.sinks = sinks; pr.window = window; pr.scale = scale;
    pr.B = B; pr.Hq = Hq; pr.Hkv = Hkv; pr.D = D;
    pr.items = items; pr.n_items = n_items; pr.out = out;
    return run(&pr, nthreads);
}

int oracle_decode_contig(const uint16_t *q, const uint16_t *hist_k, const uint16_t *hist_v,
                         const int32_t *seq_lens, int Tmax, const float *sinks,
                         int window, double scale, double *out, int B, int Hq, int Hkv, int D,
                         const int32_t *items, int n_items, int nthreads) {
    if (window < 0 || Tmax < 0) return OR_BAD_ARG;
    problem pr;
    memset(&pr, 0, sizeof pr);
    pr.kind = LAYOUT_CONTIG;
    pr.q = q; pr.k_src = hist_k; pr.v_src = hist_v;
    pr.seq_lens = seq_lens; pr.Tmax = Tmax; pr.sinks = sinks; pr.window = window;
    pr.scale = scale; pr.B = B; pr.Hq = Hq; pr.Hkv = Hkv; pr.D = D;
    pr.items = items; pr.n_items = n_items; pr.out = out;
    return run(&pr, nthreads);
}

/* Append (bit copy) of the new token of every active sequence into a paged
 * cache: position p = L - 1 goes to page block_table[b][p / P], slot p % P. */
int oracle_kv_append_paged(const uint16_t *k_new, const uint16_t *v_new,
                           uint16_t *k_cache, uint16_t *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           int B, int Hkv, int D, int page_size, int max_pages, int num_pages) {
    if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens) return OR_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        if (L <= 0) continue;
        int p = L - 1;
        if (p / page_size >= max_pages) return OR_BAD_INDEX;
        int32_t page = block_table[(size_t)b * max_pages + p / page_size];
        if (page < 0 || page >= num_pages) return OR_BAD_INDEX;
        for (int g = 0; g < Hkv; ++g) {
            size_t dst = (((size_t)page * Hkv + g) * page_size + (size_t)(p % page_size)) * D;
            size_t src = ((size_t)b * Hkv + g) * D;
            memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * (size_t)D);
            memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * (size_t)D);
        }
    }
    return OR_OK;
}

/* Append into a ring of capacity W: position p goes to cell p % W. */
int oracle_kv_append_ring(const uint16_t *k_new, const uint16_t *v_new,
                          uint16_t *k_cache, uint16_t *v_cache, const int32_t *seq_lens,
                          int window, int B, int Hkv, int D) {
    if (!k_new || !v_new || !k_cache || !v_cache || !seq_lens || window <= 0) return OR_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        if (L <= 0) continue;
        int cell = (L - 1) % window;
        for (int g = 0; g < Hkv; ++g) {
            size_t dst = (((size_t)b * Hkv + g) * window + (size_t)cell) * D;
            size_t src = ((size_t)b * Hkv + g) * D;
            memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * (size_t)D);
            memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * (size_t)D);
        }
    }
    return OR_OK;
}

/* Materialise the first n[b] tokens of a contiguous history hist[B][Tmax][Hkv][D]
 * into a paged cache through the block table. Other cells are left untouched. */
int oracle_scatter_paged(const uint16_t *hist_k, const uint16_t *hist_v, const int32_t *n_tokens,
                         int Tmax, const int32_t *block_table, uint16_t *k_cache, uint16_t *v_cache,
                         int B, int Hkv, int D, int page_size, int max_pages, int num_pages) {
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < n_tokens[b]; ++j) {
            if (j >= Tmax || j / page_size >= max_pages) return OR_BAD_INDEX;
            int32_t page = block_table[(size_t)b * max_pages + j / page_size];
            if (page < 0 || page >= num_pages) return OR_BAD_INDEX;
            for (int g = 0; g < Hkv; ++g) {
                size_t dst = (((size_t)page * Hkv + g) * page_size + (size_t)(j % page_size)) * D;
                size_t src = (((size_t)b * Tmax + j) * Hkv + g) * D;
                memcpy(k_cache + dst, hist_k + src, sizeof(uint16_t) * (size_t)D);
                memcpy(v_cache + dst, hist_v + src, sizeof(uint16_t) * (size_t)D);
            }
        }
    }
    return OR_OK;
}

/* Materialise the ring state after n[b] tokens: tokens max(0, n - W) .. n - 1
 * sit in cells j % W; older tokens have been overwritten. */
int oracle_scatter_ring(const uint16_t *hist_k, const uint16_t *hist_v, const int32_t *n_tokens,
                        int Tmax, int window, uint16_t *k_cache, uint16_t *v_cache,
                        int B, int Hkv, int D) {
    if (window <= 0) return OR_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        int n = n_tokens[b];
        int lo = n - window > 0 ? n - window : 0;
        for (int j = lo; j < n; ++j) {
            if (j >= Tmax) return OR_BAD_INDEX;
            for (int g = 0; g < Hkv; ++g) {
                size_t dst = (((size_t)b * Hkv + g) * window + (size_t)(j % window)) * D;
                size_t src = (((size_t)b * Tmax + j) * Hkv + g) * D;
                memcpy(k_cache + dst, hist_k + src, sizeof(uint16_t) * (size_t)D);
                memcpy(v_cache + dst, hist_v + src, sizeof(uint16_t) * (size_t)D);
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Rotary position embedding of the new token (SimpleLLM README, changes
 * table, row "RoPE as one fused kernel at every batch size"). The pages give
 * no formula; the reading is the rotate-half form used by gpt-oss: for
 * i < D/2 the pair (x_i, x_{i+D/2}) of a query or key vector at position pos
 * is rotated by the table angle of (pos, i):
 *     x_i'       = x_i c - x_{i+D/2} s
 *     x_{i+D/2}' = x_{i+D/2} c + x_i s,        c = cos[pos][i], s = sin[pos][i]
 * with the cos/sin tables (fp32, [max_position][D/2]) supplied by the caller,
 * so any frequency scaling lives in the tables. pos = L - 1 for the new token;
 * cached keys are stored already rotated; values are not rotated.
 *
 * Queries are rotated exactly (fp64). The new key is stored in a bf16 cache, so
 * its rotation decides bits: it is computed the way the kernel computes it --
 * each product and the difference/sum rounded to fp32 (no fused multiply-add),
 * then rounded to bf16 to nearest, ties to even. */

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static void rope_row_f64(const uint16_t *x, const float *c, const float *sn, int D, double *out) {
    const int h = D / 2;
    for (int i = 0; i < h; ++i) {
        const double x1 = bf16_to_f64(x[i]), x2 = bf16_to_f64(x[i + h]);
        out[i] = x1 * (double)c[i] - x2 * (double)sn[i];
        out[i + h] = x2 * (double)c[i] + x1 * (double)sn[i];
    }
}

static void rope_row_bf16(const uint16_t *x, const float *c, const float *sn, int D, uint16_t *out) {
    const int h = D / 2;
    for (int i = 0; i < h; ++i) {
        const float x1 = bf16_to_f32(x[i]), x2 = bf16_to_f32(x[i + h]);
        const float a = x1 * c[i], b = x2 * sn[i];
        const float e = x2 * c[i], f = x1 * sn[i];
        out[i] = f32_to_bf16_rne(a - b);
        out[i + h] = f32_to_bf16_rne(e + f);
    }
}

/* Rotated queries, fp64, [B][Hq][D]; rows of inactive slots are left zero. */
int oracle_rope_q64(const uint16_t *q, const int32_t *seq_lens, const float *rope_cos,
                    const float *rope_sin, int max_position, int B, int Hq, int D, double *out) {
    if (!q || !seq_lens || !rope_cos || !rope_sin || !out || D % 2 || max_position <= 0)
        return OR_BAD_ARG;
    const int h = D / 2;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b];
        for (int hq = 0; hq < Hq; ++hq) {
            double *o = out + ((size_t)b * Hq + hq) * D;
            if (L <= 0) { for (int d = 0; d < D; ++d) o[d] = 0.0; continue; }
            if (L - 1 >= max_position) return OR_BAD_INDEX;
            const size_t row = (size_t)(L - 1) * h;
            rope_row_f64(q + ((size_t)b * Hq + hq) * D, rope_cos + row, rope_sin + row, D, o);
        }
    }
    return OR_OK;
}

/* Rotated new keys as stored in the cache, bf16 bits, [B][Hkv][D]. */
int oracle_rope_k(const uint16_t *k_new, const int32_t *seq_lens, const float *rope_cos,
                  const float *rope_sin, int max_position, int B, int Hkv, int D, uint16_t *out) {
    if (!k_new || !seq_lens || !rope_cos || !rope_sin || !out || D % 2 || max_position <= 0)
        return OR_BAD_ARG;
    const int h = D / 2;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b];
        for (int g = 0; g < Hkv; ++g) {
            const size_t off = ((size_t)b * Hkv + g) * D;
            if (L <= 0) { memcpy(out + off, k_new + off, sizeof(uint16_t) * (size_t)D); continue; }
            if (L - 1 >= max_position) return OR_BAD_INDEX;
            const size_t row = (size_t)(L - 1) * h;
            rope_row_bf16(k_new + off, rope_cos + row, rope_sin + row, D, out + off);
        }
    }
    return OR_OK;
}

/* Decode steps with the fused RoPE: rotate q (fp64) and k_new (bf16, as stored), then
 * append and attend exactly as oracle_decode_paged / oracle_decode_ring. */
static int rope_inputs(const uint16_t *q, const uint16_t *k_new, const int32_t *seq_lens,
                       const float *rope_cos, const float *rope_sin, int max_position, int B, int Hq,
                       int Hkv, int D, double **q64, uint16_t **krot) {
    *q64 = (double *)malloc(sizeof(double) * (size_t)B * Hq * D + 1);
    *krot = k_new ? (uint16_t *)malloc(sizeof(uint16_t) * (size_t)B * Hkv * D + 1) : NULL;
    if (!*q64 || (k_new && !*krot)) return OR_NOMEM;
    int st = oracle_rope_q64(q, seq_lens, rope_cos, rope_sin, max_position, B, Hq, D, *q64);
    if (st == OR_OK && k_new)
        st = oracle_rope_k(k_new, seq_lens, rope_cos, rope_sin, max_position, B, Hkv, D, *krot);
    return st;
}

int oracle_decode_paged_rope(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                             const uint16_t *k_cache, const uint16_t *v_cache,
                             const int32_t *block_table, const int32_t *seq_lens, const float *sinks,
                             const float *rope_cos, const float *rope_sin, int max_position,
                             int window, double scale, double *out,
                             int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                             const int32_t *items, int n_items, int nthreads) {
    if (page_size <= 0 || max_pages <= 0 || num_pages <= 0 || window < 0 || !block_table)
        return OR_BAD_ARG;
    double *q64 = NULL;
    uint16_t *krot = NULL;
    int st = rope_inputs(q, k_new, seq_lens, rope_cos, rope_sin, max_position, B, Hq, Hkv, D, &q64, &krot);
    if (st == OR_OK) {
        problem pr;
        memset(&pr, 0, sizeof pr);
        pr.kind = LAYOUT_PAGED;
        pr.q = q; pr.q64 = q64; pr.k_new = krot; pr.v_new = v_new; pr.k_src = k_cache; pr.v_src = v_cache;
        pr.block_table = block_table; pr.seq_lens = seq_lens; pr.sinks = sinks;
        pr.window = window; pr.scale = scale; pr.B = B; pr.Hq = Hq; pr.Hkv = Hkv; pr.D = D;
        pr.P = page_size; pr.max_pages = max_pages; pr.num_pages = num_pages;
        pr.items = items; pr.n_items = n_items; pr.out = out;
        st = run(&pr, nthreads);
    }
    free(q64);
    free(krot);
    return st;
}

int oracle_decode_ring_rope(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                            const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *seq_lens, const float *sinks,
                            const float *rope_cos, const float *rope_sin, int max_position,
                            int window, double scale, double *out, int B, int Hq, int Hkv, int D,
                            const int32_t *items, int n_items, int nthreads) {
    if (window <= 0) return OR_BAD_ARG;
    double *q64 = NULL;
    uint16_t *krot = NULL;
    int st = rope_inputs(q, k_new, seq_lens, rope_cos, rope_sin, max_position, B, Hq, Hkv, D, &q64, &krot);
    if (st == OR_OK) {
        problem pr;
        memset(&pr, 0, sizeof pr);
        pr.kind = LAYOUT_RING;
        pr.q = q; pr.q64 = q64; pr.k_new = krot; pr.v_new = v_new; pr.k_src = k_cache; pr.v_src = v_cache;
        pr.seq_lens = seq_lens; pr.sinks = sinks; pr.window = window; pr.scale = scale;
        pr.B = B; pr.Hq = Hq; pr.Hkv = Hkv; pr.D = D;
        pr.items = items; pr.n_items = n_items; pr.out = out;
        st = run(&pr, nthreads);
    }
    free(q64);
    free(krot);
    return st;
}

/* ------------------------------------------------------------------ */
/* fp8 KV cache (reading of "quantised KV pages": the pages name quantisation
 * only as a topic). Every cached K or V row of one token and one KV head is
 * stored as 64 OCP e4m3 codes (the FN variant: sign, 4 exponent bits with bias
 * 7, 3 mantissa bits, no infinities, largest finite 448, NaN = 0x7F / 0xFF)
 * and one fp32 scale; its value is decode(code) * scale.
 * Quantising a row when it is appended: amax = max |x_d| (x widened exactly
 * from bf16), scale = amax / 448 in fp32 (scale = 1 when amax = 0), code_d =
 * the e4m3 value nearest to x_d / scale (fp32 division), ties to even,
 * saturating at +-448. The kernel takes the same fp32 decisions.
 * Layout: the cache is an array of blocks, one per P = 16 tokens of one KV head,
 * each 2PD + 8P bytes: K codes [P][D] (row per token), V codes transposed [D][P],
 * K scales [P] and V scales [P] as fp32 in native byte order. Paged: the block of
 * (page, g) is number page * Hkv + g, slot j % P. Ring of capacity W (a multiple
 * of P): cell c = j % W lives in block (b * Hkv + g) * (W / P) + c / P, slot c % P. */

static size_t blk8_bytes(int P, int D) { return 2 * (size_t)P * D + 8 * (size_t)P; }

static float f32_at(const uint8_t *p) { float f; memcpy(&f, p, sizeof f); return f; }
static void f32_put(uint8_t *p, float f) { memcpy(p, &f, sizeof f); }

/* block number holding position j of (b, g), and its slot; -1 for a bad page */
static long long blk8_of(int ring, int b, int g, int j, int Hkv, int P, int W, const int32_t *block_table,
                         int max_pages, int num_pages, int *slot) {
    if (!ring) {
        if (j / P >= max_pages) return -1;
        const int32_t page = block_table[(size_t)b * max_pages + j / P];
        if (page < 0 || page >= num_pages) return -1;
        *slot = j % P;
        return (long long)page * Hkv + g;
    }
    const int cell = j % W;
    *slot = cell % P;
    return ((long long)b * Hkv + g) * (W / P) + cell / P;
}

static double e4m3_decode(uint8_t c) {
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* nearest e4m3 value to f (ties to even mantissa), saturating at 448; f finite */
static uint8_t e4m3_encode(float f) {
    if (f != f) return 0x7F;
    const uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7E;
    /* candidates are k * 2^(e-3) on the grid of the binade of a (subnormal grid 2^-9) */
    int ex;
    frexp(a, &ex);                 /* a = frac * 2^ex, frac in [0.5, 1) */
    int e_unb = ex - 1;            /* a in [2^e_unb, 2^(e_unb+1)) */
    if (e_unb < -6) e_unb = -6;    /* subnormal range shares the grid of binade -6 */
    const double step = ldexp(1.0, e_unb - 3);
    double k = floor(a / step);
    const double rem = a - k * step;
    if (rem > step / 2 || (rem == step / 2 && fmod(k, 2.0) == 1.0)) k += 1.0;
    const double v = k * step;     /* may reach the next binade: still representable */
    if (v >= 448.0) return sign | 0x7E;
    if (v == 0.0) return sign;
    int ev;
    frexp(v, &ev);
    int eu = ev - 1;
    if (eu < -6) { /* subnormal: v = m * 2^-9 */
        return sign | (uint8_t)(v / ldexp(1.0, -9));
    }
    const int mant = (int)((v / ldexp(1.0, eu) - 1.0) * 8.0 + 0.5);
    return sign | (uint8_t)(((eu + 7) << 3) | mant);
}

/* quantise one row of D bf16 values: codes[D] and its scale */
static void quantise_row(const uint16_t *x, int D, uint8_t *codes, float *scale_out) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        const float v = fabsf(bf16_to_f32(x[d]));
        if (v > amax) amax = v;
    }
    const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int d = 0; d < D; ++d) codes[d] = e4m3_encode(bf16_to_f32(x[d]) / scale);
    *scale_out = scale;
}

int oracle_e4m3_decode(const uint8_t *codes, int n, double *out) {
    for (int i = 0; i < n; ++i) out[i] = e4m3_decode(codes[i]);
    return OR_OK;
}

int oracle_e4m3_encode(const float *x, int n, uint8_t *out) {
    for (int i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
    return OR_OK;
}

/* rows [n][D] bf16 -> codes [n][D], scales [n] */
int oracle_quantise_rows(const uint16_t *x, int n, int D, uint8_t *codes, float *scales) {
    for (int i = 0; i < n; ++i) quantise_row(x + (size_t)i * D, D, codes + (size_t)i * D, scales + i);
    return OR_OK;
}

typedef struct {
    int ring;                    /* 0 paged, 1 ring */
    const uint16_t *q;
    const uint16_t *k_new, *v_new; /* bf16 [B][Hkv][D], quantised on append, or NULL */
    const uint8_t *blocks;       /* the cache blocks */
    const int32_t *block_table, *seq_lens;
    const float *sinks;
    int window; double scale;
    int B, Hq, Hkv, D, P, max_pages, num_pages;
    const int32_t *items; int n_items;
    double *out;
    const double *q64;           /* rotated queries [B][Hq][D] in fp64 (the RoPE steps), or NULL */
} problem8;

/* dequantised key and value rows of position j (cache or, for j = L-1, the quantised new token) */
static int token_rows8(const problem8 *pr, int b, int g, int j, double *k, double *v) {
    const int L = pr->seq_lens[b], D = pr->D;
    if (j == L - 1 && pr->k_new) {
        uint8_t ck[256], cv[256];
        float sk, sv;
        if (D > 256) return OR_BAD_ARG;
        quantise_row(pr->k_new + ((size_t)b * pr->Hkv + g) * D, D, ck, &sk);
        quantise_row(pr->v_new + ((size_t)b * pr->Hkv + g) * D, D, cv, &sv);
        for (int d = 0; d < D; ++d) { k[d] = e4m3_decode(ck[d]) * sk; v[d] = e4m3_decode(cv[d]) * sv; }
        return OR_OK;
    }
    const int P = pr->P;
    int slot = 0;
    const long long bi = blk8_of(pr->ring, b, g, j, pr->Hkv, P, pr->window, pr->block_table, pr->max_pages,
                                 pr->num_pages, &slot);
    if (bi < 0) return OR_BAD_INDEX;
    const uint8_t *blk = pr->blocks + (size_t)bi * blk8_bytes(P, D);
    const double sk = f32_at(blk + 2 * (size_t)P * D + 4 * (size_t)slot);
    const double sv = f32_at(blk + 2 * (size_t)P * D + 4 * (size_t)(P + slot));
    for (int d = 0; d < D; ++d) {
        k[d] = e4m3_decode(blk[(size_t)slot * D + d]) * sk;
        v[d] = e4m3_decode(blk[(size_t)P * D + (size_t)d * P + slot]) * sv;
    }
    return OR_OK;
}

static int attend_one8(const problem8 *pr, int b, int h, double *out) {
    const int D = pr->D, L = pr->seq_lens[b];
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L <= 0) return OR_OK;
    const int g = h / (pr->Hq / pr->Hkv);
    const int W = pr->ring ? pr->window : pr->window;
    const int lo = (W > 0 && L - W > 0) ? L - W : 0, n = L - lo;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *kv = (double *)malloc(sizeof(double) * 2 * (size_t)D);
    if (!s || !kv) { free(s); free(kv); return OR_NOMEM; }
    const uint16_t *qrow = pr->q + ((size_t)b * pr->Hq + h) * D;
    const double *q64 = pr->q64 ? pr->q64 + ((size_t)b * pr->Hq + h) * D : NULL;
    const double sigma = pr->sinks ? (double)pr->sinks[h] : -INFINITY;
    double M = sigma;
    int st = OR_OK;
    for (int i = 0; i < n && st == OR_OK; ++i) {
        st = token_rows8(pr, b, g, lo + i, kv, kv + D);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (q64 ? q64[d] : bf16_to_f64(qrow[d])) * kv[d];
        s[i] = pr->scale * dot;
        if (s[i] > M) M = s[i];
    }
    double den = isinf(sigma) && sigma < 0 ? 0.0 : exp(sigma - M);
    for (int i = 0; i < n && st == OR_OK; ++i) {
        st = token_rows8(pr, b, g, lo + i, kv, kv + D);
        const double w = exp(s[i] - M);
        den += w;
        for (int d = 0; d < D; ++d) out[d] += w * kv[D + d];
    }
    if (st == OR_OK) for (int d = 0; d < D; ++d) out[d] /= den;
    free(s); free(kv);
    return st;
}

typedef struct { problem8 *pr; int tid, nthreads, status; } worker8_arg;

static void *worker8(void *p) {
    worker8_arg *a = (worker8_arg *)p;
    problem8 *pr = a->pr;
    const int total = pr->items ? pr->n_items : pr->B * pr->Hq;
    for (int w = a->tid; w < total; w += a->nthreads) {
        int b = pr->items ? pr->items[2 * w] : w / pr->Hq;
        int h = pr->items ? pr->items[2 * w + 1] : w % pr->Hq;
        if (b < 0 || b >= pr->B || h < 0 || h >= pr->Hq) { a->status = OR_BAD_ARG; continue; }
        int st = attend_one8(pr, b, h, pr->out + (size_t)w * pr->D);
        if (st != OR_OK && a->status == OR_OK) a->status = st;
    }
    return NULL;
}

static int run8(problem8 *pr, int nthreads) {
    if (pr->B < 0 || pr->Hq <= 0 || pr->Hkv <= 0 || pr->Hq % pr->Hkv || pr->D <= 0 || pr->D > 256)
        return OR_BAD_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    worker8_arg args[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) { args[t].pr = pr; args[t].tid = t; args[t].nthreads = nthreads; args[t].status = OR_OK; }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker8, &args[t]) != 0) break;
        started = t;
    }
    for (int t = started + 1; t < nthreads; ++t) worker8(&args[t]);
    worker8(&args[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t) if (args[t].status != OR_OK) return args[t].status;
    return OR_OK;
}

int oracle_decode_paged_fp8(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                            const uint8_t *blocks, const int32_t *block_table, const int32_t *seq_lens,
                            const float *sinks, int window, double scale, double *out,
                            int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                            const int32_t *items, int n_items, int nthreads) {
    if (!q || !blocks || !block_table || !seq_lens || !out || page_size <= 0 || max_pages <= 0 ||
        num_pages <= 0 || window < 0 || ((k_new == NULL) != (v_new == NULL)))
        return OR_BAD_ARG;
    problem8 pr = {0, q, k_new, v_new, blocks, block_table, seq_lens, sinks,
                   window, scale, B, Hq, Hkv, D, page_size, max_pages, num_pages, items, n_items, out};
    return run8(&pr, nthreads);
}

int oracle_decode_ring_fp8(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                           const uint8_t *blocks, const int32_t *seq_lens, const float *sinks, int window,
                           double scale, double *out, int B, int Hq, int Hkv, int D,
                           const int32_t *items, int n_items, int nthreads) {
    if (!q || !blocks || !seq_lens || !out || window <= 0 || window % 16 != 0 ||
        ((k_new == NULL) != (v_new == NULL)))
        return OR_BAD_ARG;
    problem8 pr = {1, q, k_new, v_new, blocks, NULL, seq_lens, sinks,
                   window, scale, B, Hq, Hkv, D, 16, 0, 0, items, n_items, out};
    return run8(&pr, nthreads);
}

/* fp8 cache with the fused RoPE: q is rotated to position L - 1 exactly (fp64) and the new
 * key is rotated as it is stored (bf16, rope_row_bf16) BEFORE it is quantised; then the step
 * is oracle_decode_paged_fp8 / oracle_decode_ring_fp8 on those inputs. */
static int decode_fp8_rope(int ring, const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                           const uint8_t *blocks, const int32_t *block_table, const int32_t *seq_lens,
                           const float *sinks, const float *rope_cos, const float *rope_sin,
                           int max_position, int window, double scale, double *out, int B, int Hq, int Hkv,
                           int D, int page_size, int max_pages, int num_pages, const int32_t *items,
                           int n_items, int nthreads) {
    double *q64 = NULL;
    uint16_t *krot = NULL;
    int st = rope_inputs(q, k_new, seq_lens, rope_cos, rope_sin, max_position, B, Hq, Hkv, D, &q64, &krot);
    if (st == OR_OK) {
        problem8 pr = {ring, q, krot, v_new, blocks, block_table, seq_lens, sinks,
                       window, scale, B, Hq, Hkv, D, page_size, max_pages, num_pages, items, n_items, out,
                       q64};
        st = run8(&pr, nthreads);
    }
    free(q64);
    free(krot);
    return st;
}

int oracle_decode_paged_fp8_rope(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                                 const uint8_t *blocks, const int32_t *block_table, const int32_t *seq_lens,
                                 const float *sinks, const float *rope_cos, const float *rope_sin,
                                 int max_position, int window, double scale, double *out, int B, int Hq,
                                 int Hkv, int D, int page_size, int max_pages, int num_pages,
                                 const int32_t *items, int n_items, int nthreads) {
    if (!q || !blocks || !block_table || !seq_lens || !out || page_size <= 0 || max_pages <= 0 ||
        num_pages <= 0 || window < 0 || ((k_new == NULL) != (v_new == NULL)))
        return OR_BAD_ARG;
    return decode_fp8_rope(0, q, k_new, v_new, blocks, block_table, seq_lens, sinks, rope_cos, rope_sin,
                           max_position, window, scale, out, B, Hq, Hkv, D, page_size, max_pages, num_pages,
                           items, n_items, nthreads);
}

int oracle_decode_ring_fp8_rope(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                                const uint8_t *blocks, const int32_t *seq_lens, const float *sinks,
                                const float *rope_cos, const float *rope_sin, int max_position, int window,
                                double scale, double *out, int B, int Hq, int Hkv, int D,
                                const int32_t *items, int n_items, int nthreads) {
    if (!q || !blocks || !seq_lens || !out || window <= 0 || window % 16 != 0 ||
        ((k_new == NULL) != (v_new == NULL)))
        return OR_BAD_ARG;
    return decode_fp8_rope(1, q, k_new, v_new, blocks, NULL, seq_lens, sinks, rope_cos, rope_sin,
                           max_position, window, scale, out, B, Hq, Hkv, D, 16, 0, 0, items, n_items,
                           nthreads);
}

/* Write token rows (bf16 [n][Hkv][D] per sequence b at positions pos[b] .. ) quantised into an
 * fp8 cache: the append of the new tokens (positions L-1), or the materialisation of a history. */
static int put8(int ring, uint8_t *blocks, int b, int g, int j, const uint16_t *krow, const uint16_t *vrow,
                int Hkv, int D, int P, int W, const int32_t *block_table, int max_pages, int num_pages) {
    uint8_t ck[256], cv[256];
    float sk, sv;
    int slot = 0;
    const long long bi = blk8_of(ring, b, g, j, Hkv, P, W, block_table, max_pages, num_pages, &slot);
    if (bi < 0) return OR_BAD_INDEX;
    quantise_row(krow, D, ck, &sk);
    quantise_row(vrow, D, cv, &sv);
    uint8_t *blk = blocks + (size_t)bi * blk8_bytes(P, D);
    for (int d = 0; d < D; ++d) {
        blk[(size_t)slot * D + d] = ck[d];
        blk[(size_t)P * D + (size_t)d * P + slot] = cv[d];
    }
    f32_put(blk + 2 * (size_t)P * D + 4 * (size_t)slot, sk);
    f32_put(blk + 2 * (size_t)P * D + 4 * (size_t)(P + slot), sv);
    return OR_OK;
}

int oracle_kv_append_fp8(const uint16_t *k_new, const uint16_t *v_new, uint8_t *blocks,
                         const int32_t *block_table /* NULL = ring */, const int32_t *seq_lens, int window,
                         int B, int Hkv, int D, int page_size, int max_pages, int num_pages) {
    if (D > 256 || (!block_table && (window <= 0 || window % page_size != 0))) return OR_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b];
        if (L <= 0) continue;
        for (int g = 0; g < Hkv; ++g) {
            const size_t src = ((size_t)b * Hkv + g) * D;
            const int st = put8(block_table == NULL, blocks, b, g, L - 1, k_new + src, v_new + src, Hkv, D,
                                page_size, window, block_table, max_pages, num_pages);
            if (st != OR_OK) return st;
        }
    }
    return OR_OK;
}

/* Materialise the first n[b] tokens of hist [B][Tmax][Hkv][D] into an fp8 cache (paged when a
 * block table is given, else the ring state of capacity `window`). */
int oracle_scatter_fp8(const uint16_t *hist_k, const uint16_t *hist_v, const int32_t *n_tokens, int Tmax,
                       const int32_t *block_table, int window, uint8_t *blocks, int B, int Hkv, int D,
                       int page_size, int max_pages, int num_pages) {
    if (D > 256 || (!block_table && (window <= 0 || window % page_size != 0))) return OR_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        const int n = n_tokens[b];
        const int lo = (!block_table && n - window > 0) ? n - window : 0;
        for (int j = lo; j < n; ++j) {
            if (j >= Tmax) return OR_BAD_INDEX;
            for (int g = 0; g < Hkv; ++g) {
                const size_t src = (((size_t)b * Tmax + j) * Hkv + g) * D;
                const int st = put8(block_table == NULL, blocks, b, g, j, hist_k + src, hist_v + src, Hkv, D,
                                    page_size, window, block_table, max_pages, num_pages);
                if (st != OR_OK) return st;
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Several query tokens per sequence in one step (reading of the chapters "Chunked
 * Prefill" and "Speculative Decoding" named in the teaching repo's table "The files",
 * page "Run it locally": both run attention for a run of new tokens over the cached
 * history, each new token seeing the history and the new tokens before it).
 *
 *   n = q_lens[b] (T when q_lens is NULL) new tokens, at positions base .. L-1 with
 *   L = seq_lens[b] and base = L - n (n <= T, n <= L). Query row (t, h), t < n, sits at
 *   p = base + t and attends the positions j with lo <= j <= p (causal), lo = max(0,
 *   p - W + 1) when a window W > 0 applies (always for the ring), else 0. Position
 *   j >= base is new token j - base (k_new / v_new [B][T][Hkv][D]); j < base comes from
 *   the cache. Rows t >= n, and every row of an inactive slot (L = 0), are zero.
 *   q / out are [B][T][Hq][D].
 *
 * The cache holds the history before this step: the ring of capacity W holds positions
 * max(0, base - W) .. base - 1 (cell j % W). The n new tokens are appended afterwards
 * (oracle_kv_append_multi); the ring's early queries still see the cells that the later
 * new tokens overwrite, so the append cannot come first. */

typedef struct {
    int ring;
    const uint16_t *q, *k_new, *v_new, *k_cache, *v_cache;
    const int32_t *block_table, *seq_lens, *q_lens;
    const float *sinks;
    int window; double scale;
    int B, T, Hq, Hkv, D, P, max_pages, num_pages;
    double *out;
    const double *q64;  /* rotated queries [B][T][Hq][D] in fp64, or NULL: q as given */
} problemM;

static int q_count(const int32_t *q_lens, int T, int b) { return q_lens ? q_lens[b] : T; }

/* key (v = 0) or value (v = 1) row of position j for (b, g); NULL for a bad page */
static const uint16_t *rowM(const problemM *pr, int b, int g, int j, int v) {
    const int L = pr->seq_lens[b], base = L - q_count(pr->q_lens, pr->T, b), D = pr->D;
    if (j >= base) {
        const int t = j - base;
        return (v ? pr->v_new : pr->k_new) + (((size_t)b * pr->T + t) * pr->Hkv + g) * D;
    }
    const uint16_t *cache = v ? pr->v_cache : pr->k_cache;
    if (pr->ring) {
        const int cell = j % pr->window;
        return cache + (((size_t)b * pr->Hkv + g) * pr->window + cell) * D;
    }
    if (j / pr->P >= pr->max_pages) return NULL;
    const int32_t page = pr->block_table[(size_t)b * pr->max_pages + j / pr->P];
    if (page < 0 || page >= pr->num_pages) return NULL;
    return cache + (((size_t)page * pr->Hkv + g) * pr->P + j % pr->P) * D;
}

static int attend_oneM(const problemM *pr, int b, int t, int h, double *out) {
    const int D = pr->D, L = pr->seq_lens[b], n = q_count(pr->q_lens, pr->T, b);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L <= 0 || t >= n) return OR_OK;
    const int g = h / (pr->Hq / pr->Hkv);
    const int p = L - n + t;
    const int W = pr->window;
    const int lo = (W > 0 && p - W + 1 > 0) ? p - W + 1 : 0;
    const int cnt = p - lo + 1;
    double *s = (double *)malloc(sizeof(double) * (size_t)cnt);
    if (!s) return OR_NOMEM;
    const size_t qoff = (((size_t)b * pr->T + t) * pr->Hq + h) * D;
    const uint16_t *qrow = pr->q + qoff;
    const double *q64 = pr->q64 ? pr->q64 + qoff : NULL;
    const double sigma = pr->sinks ? (double)pr->sinks[h] : -INFINITY;
    double M = sigma;
    for (int i = 0; i < cnt; ++i) {
        const uint16_t *krow = rowM(pr, b, g, lo + i, 0);
        if (!krow) { free(s); return OR_BAD_INDEX; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (q64 ? q64[d] : bf16_to_f64(qrow[d])) * bf16_to_f64(krow[d]);
        s[i] = pr->scale * dot;
        if (s[i] > M) M = s[i];
    }
    double den = isinf(sigma) && sigma < 0 ? 0.0 : exp(sigma - M);
    for (int i = 0; i < cnt; ++i) {
        const uint16_t *vrow = rowM(pr, b, g, lo + i, 1);
        const double w = exp(s[i] - M);
        den += w;
        for (int d = 0; d < D; ++d) out[d] += w * bf16_to_f64(vrow[d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
    free(s);
    return OR_OK;
}

typedef struct { problemM *pr; int tid, nthreads, status; } workerM_arg;

static void *workerM(void *arg) {
    workerM_arg *a = (workerM_arg *)arg;
    problemM *pr = a->pr;
    const long long total = (long long)pr->B * pr->T * pr->Hq;
    for (long long w = a->tid; w < total; w += a->nthreads) {
        const int h = (int)(w % pr->Hq), t = (int)((w / pr->Hq) % pr->T), b = (int)(w / ((long long)pr->Hq * pr->T));
        const int st = attend_oneM(pr, b, t, h, pr->out + (size_t)w * pr->D);
        if (st != OR_OK && a->status == OR_OK) a->status = st;
    }
    return NULL;
}

static int check_counts(const int32_t *seq_lens, const int32_t *q_lens, int B, int T) {
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b], n = q_count(q_lens, T, b);
        if (L < 0 || n < 0 || n > T || (L > 0 && n > L)) return OR_BAD_ARG;
    }
    return OR_OK;
}

static int decode_multi_q64(int ring, const uint16_t *q, const double *q64_in, const uint16_t *k_new,
                            const uint16_t *v_new, const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_lens,
                            const float *sinks, int window, double scale, double *out, int B, int T, int Hq,
                            int Hkv, int D, int page_size, int max_pages, int num_pages, int nthreads) {
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !seq_lens || !out || B < 0 || T <= 0 || Hq <= 0 ||
        Hkv <= 0 || Hq % Hkv || D <= 0 || window < 0 || (ring && window <= 0) ||
        (!ring && (!block_table || page_size <= 0 || max_pages <= 0 || num_pages <= 0)))
        return OR_BAD_ARG;
    if (check_counts(seq_lens, q_lens, B, T) != OR_OK) return OR_BAD_ARG;
    problemM pr = {ring, q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, q_lens, sinks, window, scale,
                   B, T, Hq, Hkv, D, page_size, max_pages, num_pages, out, q64_in};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    workerM_arg args[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) { args[t].pr = &pr; args[t].tid = t; args[t].nthreads = nthreads; args[t].status = OR_OK; }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, workerM, &args[t]) != 0) break;
        started = t;
    }
    for (int t = started + 1; t < nthreads; ++t) workerM(&args[t]);
    workerM(&args[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t) if (args[t].status != OR_OK) return args[t].status;
    return OR_OK;
}

int oracle_decode_multi(int ring, const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                        const uint16_t *k_cache, const uint16_t *v_cache, const int32_t *block_table,
                        const int32_t *seq_lens, const int32_t *q_lens, const float *sinks, int window,
                        double scale, double *out, int B, int T, int Hq, int Hkv, int D, int page_size,
                        int max_pages, int num_pages, int nthreads) {
    return decode_multi_q64(ring, q, NULL, k_new, v_new, k_cache, v_cache, block_table, seq_lens, q_lens, sinks,
                            window, scale, out, B, T, Hq, Hkv, D, page_size, max_pages, num_pages, nthreads);
}

/* Several query tokens with the rotary embedding (the rotate-half form of the one-token
 * steps above, at each new token's own position): query row (t, h) and new key (t, g),
 * t < n, are rotated to position p = L - n + t. q64 gets the exact rotation of the query
 * (fp64); qrot (if given) the query as the bf16 model holds it after the rotation, and krot
 * the key as it is stored: fp32 products and sum or difference, rounded to bf16 nearest
 * even. Rows t >= n are left as they are (zero in q64; copied into qrot and krot). */
int oracle_rope_multi(const uint16_t *q, const uint16_t *k_new, const int32_t *seq_lens, const int32_t *q_lens,
                      const float *rope_cos, const float *rope_sin, int max_position, int B, int T, int Hq,
                      int Hkv, int D, double *q64, uint16_t *qrot, uint16_t *krot) {
    if (!q || !seq_lens || !rope_cos || !rope_sin || !q64 || (k_new && !krot) || D % 2 || max_position <= 0 ||
        B < 0 || T <= 0)
        return OR_BAD_ARG;
    if (check_counts(seq_lens, q_lens, B, T) != OR_OK) return OR_BAD_ARG;
    const int h = D / 2;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b], n = q_count(q_lens, T, b);
        for (int t = 0; t < T; ++t) {
            const int active = L > 0 && t < n;
            const int p = L - n + t;
            if (active && p >= max_position) return OR_BAD_INDEX;
            const size_t row = active ? (size_t)p * h : 0;
            for (int hq = 0; hq < Hq; ++hq) {
                const size_t off = (((size_t)b * T + t) * Hq + hq) * D;
                if (active) rope_row_f64(q + off, rope_cos + row, rope_sin + row, D, q64 + off);
                else for (int d = 0; d < D; ++d) q64[off + d] = 0.0;
                if (!qrot) continue;
                if (active) rope_row_bf16(q + off, rope_cos + row, rope_sin + row, D, qrot + off);
                else memcpy(qrot + off, q + off, sizeof(uint16_t) * (size_t)D);
            }
            if (!k_new) continue;
            for (int g = 0; g < Hkv; ++g) {
                const size_t off = (((size_t)b * T + t) * Hkv + g) * D;
                if (active) rope_row_bf16(k_new + off, rope_cos + row, rope_sin + row, D, krot + off);
                else memcpy(krot + off, k_new + off, sizeof(uint16_t) * (size_t)D);
            }
        }
    }
    return OR_OK;
}

/* The several-token step with the rotary embedding: rotate (oracle_rope_multi), then attend
 * exactly as oracle_decode_multi with the rotated queries and keys, both as the bf16 model
 * holds them (the query rounded to bf16 like the stored key). */
int oracle_decode_multi_rope(int ring, const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                             const uint16_t *k_cache, const uint16_t *v_cache, const int32_t *block_table,
                             const int32_t *seq_lens, const int32_t *q_lens, const float *sinks,
                             const float *rope_cos, const float *rope_sin, int max_position, int window,
                             double scale, double *out, int B, int T, int Hq, int Hkv, int D, int page_size,
                             int max_pages, int num_pages, int nthreads) {
    if (!k_new) return OR_BAD_ARG;
    double *q64 = (double *)malloc(sizeof(double) * (size_t)B * T * Hq * D + 1);
    uint16_t *qrot = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)B * T * Hq * D + 1);
    uint16_t *krot = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)B * T * Hkv * D + 1);
    int st = (q64 && qrot && krot) ? OR_OK : OR_NOMEM;
    if (st == OR_OK)
        st = oracle_rope_multi(q, k_new, seq_lens, q_lens, rope_cos, rope_sin, max_position, B, T, Hq, Hkv, D,
                               q64, qrot, krot);
    if (st == OR_OK)
        st = decode_multi_q64(ring, qrot, NULL, krot, v_new, k_cache, v_cache, block_table, seq_lens, q_lens,
                              sinks, window, scale, out, B, T, Hq, Hkv, D, page_size, max_pages, num_pages,
                              nthreads);
    free(q64);
    free(qrot);
    free(krot);
    return st;
}

/* The append of a multi-token step: new token t < n of b goes to position L - n + t (paged:
 * its page and slot; ring of capacity W: cell (L - n + t) % W). */
int oracle_kv_append_multi(int ring, const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_cache,
                           uint16_t *v_cache, const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *q_lens, int window, int B, int T, int Hkv, int D, int page_size,
                           int max_pages, int num_pages) {
    if (!k_new || !v_new || !k_cache || !v_cache || !seq_lens || (ring && window <= 0) ||
        (!ring && (!block_table || page_size <= 0 || max_pages <= 0)))
        return OR_BAD_ARG;
    if (check_counts(seq_lens, q_lens, B, T) != OR_OK) return OR_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b], n = q_count(q_lens, T, b);
        if (L <= 0) continue;
        for (int t = 0; t < n; ++t) {
            const int pos = L - n + t;
            for (int g = 0; g < Hkv; ++g) {
                size_t dst;
                if (ring) {
                    dst = (((size_t)b * Hkv + g) * window + pos % window) * D;
                } else {
                    if (pos / page_size >= max_pages) return OR_BAD_INDEX;
                    const int32_t page = block_table[(size_t)b * max_pages + pos / page_size];
                    if (page < 0 || page >= num_pages) return OR_BAD_INDEX;
                    dst = (((size_t)page * Hkv + g) * page_size + pos % page_size) * D;
                }
                const size_t src = (((size_t)b * T + t) * Hkv + g) * D;
                memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * (size_t)D);
                memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * (size_t)D);
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Several query tokens per sequence over an fp8 cache: the several-token step above
 * (positions, causal and window bounds, counts, zero rows) with every key and value row
 * taken as the fp8 cache holds it -- history rows dequantised from their blocks, and the new
 * token j - base quantised exactly as its append stores it (quantise_row) and dequantised. */
typedef struct {
    int ring;
    const uint16_t *q, *k_new, *v_new;
    const uint8_t *blocks;
    const int32_t *block_table, *seq_lens, *q_lens;
    const float *sinks;
    int window; double scale;
    int B, T, Hq, Hkv, D, P, max_pages, num_pages;
    double *out;
} problemM8;

static int rowsM8(const problemM8 *pr, int b, int g, int j, double *k, double *v) {
    const int L = pr->seq_lens[b], n = q_count(pr->q_lens, pr->T, b), base = L - n, D = pr->D, P = pr->P;
    if (j >= base) {
        uint8_t ck[256], cv[256];
        float sk, sv;
        const size_t src = (((size_t)b * pr->T + (j - base)) * pr->Hkv + g) * D;
        quantise_row(pr->k_new + src, D, ck, &sk);
        quantise_row(pr->v_new + src, D, cv, &sv);
        for (int d = 0; d < D; ++d) { k[d] = e4m3_decode(ck[d]) * sk; v[d] = e4m3_decode(cv[d]) * sv; }
        return OR_OK;
    }
    int slot = 0;
    const long long bi = blk8_of(pr->ring, b, g, j, pr->Hkv, P, pr->window, pr->block_table, pr->max_pages,
                                 pr->num_pages, &slot);
    if (bi < 0) return OR_BAD_INDEX;
    const uint8_t *blk = pr->blocks + (size_t)bi * blk8_bytes(P, D);
    const double sk = f32_at(blk + 2 * (size_t)P * D + 4 * (size_t)slot);
    const double sv = f32_at(blk + 2 * (size_t)P * D + 4 * (size_t)(P + slot));
    for (int d = 0; d < D; ++d) {
        k[d] = e4m3_decode(blk[(size_t)slot * D + d]) * sk;
        v[d] = e4m3_decode(blk[(size_t)P * D + (size_t)d * P + slot]) * sv;
    }
    return OR_OK;
}

static int attend_oneM8(const problemM8 *pr, int b, int t, int h, double *out) {
    const int D = pr->D, L = pr->seq_lens[b], n = q_count(pr->q_lens, pr->T, b);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L <= 0 || t >= n) return OR_OK;
    const int g = h / (pr->Hq / pr->Hkv);
    const int p = L - n + t;
    const int W = pr->window;
    const int lo = (W > 0 && p - W + 1 > 0) ? p - W + 1 : 0;
    const int cnt = p - lo + 1;
    double *s = (double *)malloc(sizeof(double) * (size_t)cnt);
    double *kv = (double *)malloc(sizeof(double) * 2 * (size_t)D);
    if (!s || !kv) { free(s); free(kv); return OR_NOMEM; }
    const uint16_t *qrow = pr->q + (((size_t)b * pr->T + t) * pr->Hq + h) * D;
    const double sigma = pr->sinks ? (double)pr->sinks[h] : -INFINITY;
    double M = sigma;
    int st = OR_OK;
    for (int i = 0; i < cnt && st == OR_OK; ++i) {
        st = rowsM8(pr, b, g, lo + i, kv, kv + D);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_f64(qrow[d]) * kv[d];
        s[i] = pr->scale * dot;
        if (s[i] > M) M = s[i];
    }
    double den = isinf(sigma) && sigma < 0 ? 0.0 : exp(sigma - M);
    for (int i = 0; i < cnt && st == OR_OK; ++i) {
        st = rowsM8(pr, b, g, lo + i, kv, kv + D);
        const double w = exp(s[i] - M);
        den += w;
        for (int d = 0; d < D; ++d) out[d] += w * kv[D + d];
    }
    if (st == OR_OK) for (int d = 0; d < D; ++d) out[d] /= den;
    free(s); free(kv);
    return st;
}

typedef struct { problemM8 *pr; int tid, nthreads, status; } workerM8_arg;

static void *workerM8(void *arg) {
    workerM8_arg *a = (workerM8_arg *)arg;
    problemM8 *pr = a->pr;
    const long long total = (long long)pr->B * pr->T * pr->Hq;
    for (long long w = a->tid; w < total; w += a->nthreads) {
        const int h = (int)(w % pr->Hq), t = (int)((w / pr->Hq) % pr->T), b = (int)(w / ((long long)pr->Hq * pr->T));
        const int st = attend_oneM8(pr, b, t, h, pr->out + (size_t)w * pr->D);
        if (st != OR_OK && a->status == OR_OK) a->status = st;
    }
    return NULL;
}

int oracle_decode_multi_fp8(int ring, const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                            const uint8_t *blocks, const int32_t *block_table, const int32_t *seq_lens,
                            const int32_t *q_lens, const float *sinks, int window, double scale, double *out,
                            int B, int T, int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                            int nthreads) {
    if (!q || !k_new || !v_new || !blocks || !seq_lens || !out || B < 0 || T <= 0 || Hq <= 0 || Hkv <= 0 ||
        Hq % Hkv || D <= 0 || D > 256 || window < 0 || page_size <= 0 ||
        (ring && (window <= 0 || window % page_size != 0)) ||
        (!ring && (!block_table || max_pages <= 0 || num_pages <= 0)))
        return OR_BAD_ARG;
    if (check_counts(seq_lens, q_lens, B, T) != OR_OK) return OR_BAD_ARG;
    problemM8 pr = {ring, q, k_new, v_new, blocks, block_table, seq_lens, q_lens, sinks, window, scale,
                    B, T, Hq, Hkv, D, page_size, max_pages, num_pages, out};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    workerM8_arg args[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) { args[t].pr = &pr; args[t].tid = t; args[t].nthreads = nthreads; args[t].status = OR_OK; }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, workerM8, &args[t]) != 0) break;
        started = t;
    }
    for (int t = started + 1; t < nthreads; ++t) workerM8(&args[t]);
    workerM8(&args[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t) if (args[t].status != OR_OK) return args[t].status;
    return OR_OK;
}

/* The append of a several-token step into an fp8 cache: new token t < n of b, quantised, to
 * position L - n + t (ring: cell (L - n + t) % W, written in order, so the last W survive). */
int oracle_kv_append_multi_fp8(int ring, const uint16_t *k_new, const uint16_t *v_new, uint8_t *blocks,
                               const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_lens,
                               int window, int B, int T, int Hkv, int D, int page_size, int max_pages,
                               int num_pages) {
    if (!k_new || !v_new || !blocks || !seq_lens || D > 256 || page_size <= 0 ||
        (ring && (window <= 0 || window % page_size != 0)) || (!ring && (!block_table || max_pages <= 0)))
        return OR_BAD_ARG;
    if (check_counts(seq_lens, q_lens, B, T) != OR_OK) return OR_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b], n = q_count(q_lens, T, b);
        if (L <= 0) continue;
        for (int t = 0; t < n; ++t)
            for (int g = 0; g < Hkv; ++g) {
                const size_t src = (((size_t)b * T + t) * Hkv + g) * D;
                const int st = put8(ring, blocks, b, g, L - n + t, k_new + src, v_new + src, Hkv, D, page_size,
                                    window, block_table, max_pages, num_pages);
                if (st != OR_OK) return st;
            }
    }
    return OR_OK;
}
