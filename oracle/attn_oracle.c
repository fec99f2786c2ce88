/*
 * attn_oracle.c -- plain fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA path is
 * checked against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the CUDA library, and it never calls into it.
 *
 * What it computes (the plain definition, no blocking, fusion or reordering):
 *
 *   S[i][j] = scale * sum_t q[i][t] * k[j][t]                (fp64, full Sq x Skv)
 *   S[i][j] = -inf  if causal and j > i + (Skv - Sq)          (bottom-right alignment)
 *   S[i][j] = -inf  if a window W > 0 is set and n_sink <= j <= i + (Skv - Sq) - W
 *                   (sliding window of the last W positions up to the query's
 *                   own, plus the first n_sink positions always visible)
 *   m_i     = max_j S[i][j]
 *   l_i     = sum_j exp(S[i][j] - m_i)
 *   P[i][j] = exp(S[i][j] - m_i) / l_i
 *   O[i]    = sum_j P[i][j] * v[j]
 *   LSE_i   = m_i + ln(l_i)                                    (natural log)
 *   A row with no admissible key gives O = 0, LSE = -inf.
 *
 * Sources:
 *  - "60 . r57 -- FA KV staging double buffering (REVERTED)", section 2.3:
 *    online softmax (running max, rescale by exp(m_old - m_new) at every KV
 *    tile boundary) is a re-grouping of this same sum, so the plain definition
 *    is the exact result it approximates only by rounding order.
 *  - "STAGE_D.md -- FMHA Kernel Development", "Kernel Output": O from
 *    P = exp(S*scale - row_max), LSE from ln(row_sum) plus the row max; the
 *    page mixes a base-2 max with a natural log, and this oracle takes LSE in
 *    natural units throughout (LSE = ln sum_j exp(S_ij)).
 *  - "STAGE_D.md -- FMHA Kernel Development", D3-D5: a length mask on the
 *    sliding-window branch, a causal mask on it, and a merge of the window
 *    branch with a sink branch through their LSEs.  Here both branches are
 *    one key set: the window of the last W positions and the first n_sink
 *    positions, under the causal mask (the merge of two disjoint key sets
 *    through their LSEs is exactly the softmax over their union).
 *  - "66 . D2: explicit K+V register staging", section 3.2: the decode split
 *    body walks rows [lo, hi) of one sequence for one KV head, with score
 *    s = (q . k) * scale and the running max / running sum / running O update.
 *    Here each split is computed by the plain definition over [lo, hi).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - causal alignment when Sq != Skv: bottom-right (query i sits at key
 *    position i + Skv - Sq); equals top-left when Sq == Skv.
 *  - GQA head mapping: kv head of query head hq is hq / (Hq / Hkv).
 *  - split-KV partials are normalised within their split:
 *      part_o_s = sum_{j in split} exp(S_j - lse_s) v_j,  lse_s = ln sum exp(S_j)
 *    so that the merge needs only (part_o, part_lse):
 *      M = max_s lse_s,  w_s = exp(lse_s - M),
 *      O = sum_s w_s part_o_s / sum_s w_s,   LSE = M + ln sum_s w_s.
 *    Empty splits have lse = -inf, part_o = 0 and are skipped by the merge.
 *  - split rule: chunk_b = max(ceil(L_b / n_splits), min_rows_per_split),
 *    split s covers [s*chunk_b, min(L_b, (s+1)*chunk_b)); a split whose start
 *    is >= L_b is empty.
 *
 * Layouts (row-major, contiguous):
 *   prefill  q, o : [B][Sq][Hq][d]      k, v : [B][Skv][Hkv][d]    lse : [B][Hq][Sq]
 *   decode   q, o : [B][Hq][d]          kc, vc : [B][Lmax][Hkv][d] kv_lens : [B]
 *            part_o : [B][Hq][n_splits][d]   part_lse : [B][Hq][n_splits]   lse : [B][Hq]
 * All floating-point arrays are fp64.  Callers widen bf16 inputs to fp64
 * exactly before calling.
 *
 * Threads: work is split over (b, hq) pairs with POSIX threads; nthreads <= 0
 * means "all online cores".  Each (b, hq) is computed by exactly one thread in
 * the same order, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

/* ------------------------------------------------------------------------ */
/* threading helper: run fn(ctx, item) for item in [0, n_items)              */
/* ------------------------------------------------------------------------ */
typedef void (*item_fn)(void* ctx, long item);

typedef struct {
    item_fn fn;
    void* ctx;
    long n_items;
    long next; /* guarded by mu */
    pthread_mutex_t mu;
} pool_t;

static void* pool_worker(void* arg) {
    pool_t* p = (pool_t*)arg;
    for (;;) {
        long it;
        pthread_mutex_lock(&p->mu);
        it = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (it >= p->n_items) break;
        p->fn(p->ctx, it);
    }
    return NULL;
}

int oracle_num_cores(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void run_items(item_fn fn, void* ctx, long n_items, int nthreads) {
    pool_t p;
    int t, nt;
    pthread_t* th;
    if (nthreads <= 0) nthreads = oracle_num_cores();
    nt = nthreads;
    if (nt > n_items) nt = (int)(n_items > 0 ? n_items : 1);
    p.fn = fn;
    p.ctx = ctx;
    p.n_items = n_items;
    p.next = 0;
    pthread_mutex_init(&p.mu, NULL);
    if (nt <= 1) {
        pool_worker(&p);
        pthread_mutex_destroy(&p.mu);
        return;
    }
    th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th) { /* fall back to the calling thread */
        pool_worker(&p);
        pthread_mutex_destroy(&p.mu);
        return;
    }
    for (t = 0; t < nt; ++t) pthread_create(&th[t], NULL, pool_worker, &p);
    for (t = 0; t < nt; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&p.mu);
}

/* ------------------------------------------------------------------------ */
/* one query row against keys [j0, j1): the plain definition                 */
/* ------------------------------------------------------------------------ */
/* Scores s[j - j0] for admissible keys; inadmissible keys (j > jmax) get -inf.
 * Writes o_row[d] and returns lse through *lse_out.  s is caller scratch of
 * length (j1 - j0). */
static void softmax_row(const double* q_row, const double* k_base, const double* v_base,
                        long kv_row_stride, int d, int j0, int j1, int jmax, int jlo, int nsink,
                        double scale, double* s, double* o_row, double* lse_out) {
    int j, t;
    double m = -INFINITY, l = 0.0;
    /* step 1-2: scores with mask (keys past jmax; keys before jlo except sinks) */
    for (j = j0; j < j1; ++j) {
        if (j > jmax) {
            s[j - j0] = -INFINITY;
            continue;
        }
        if (j < jlo && j >= nsink) {
            s[j - j0] = -INFINITY;
            continue;
        }
        const double* k_row = k_base + (long)j * kv_row_stride;
        double dot = 0.0;
        for (t = 0; t < d; ++t) dot += q_row[t] * k_row[t];
        s[j - j0] = scale * dot;
    }
    /* step 3: row max and row sum */
    for (j = j0; j < j1; ++j)
        if (s[j - j0] > m) m = s[j - j0];
    for (t = 0; t < d; ++t) o_row[t] = 0.0;
    if (m == -INFINITY) { /* no admissible key */
        *lse_out = -INFINITY;
        return;
    }
    for (j = j0; j < j1; ++j) l += exp(s[j - j0] - m);
    /* step 4: O = sum_j P_j v_j with P_j = exp(s_j - m) / l */
    for (j = j0; j < j1; ++j) {
        double p;
        const double* v_row;
        if (s[j - j0] == -INFINITY) continue;
        p = exp(s[j - j0] - m) / l;
        v_row = v_base + (long)j * kv_row_stride;
        for (t = 0; t < d; ++t) o_row[t] += p * v_row[t];
    }
    *lse_out = m + log(l);
}

/* ------------------------------------------------------------------------ */
/* prefill: full score matrix per (b, hq)                                    */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v;
    int B, Hq, Hkv, Sq, Skv, d, causal;
    int window, n_sink; /* window <= 0: no window */
    double scale;
    double *o, *lse;
    int err;
} sdpa_ctx;

static void sdpa_item(void* vctx, long item) {
    sdpa_ctx* c = (sdpa_ctx*)vctx;
    int b = (int)(item / c->Hq), hq = (int)(item % c->Hq);
    int G = c->Hq / c->Hkv, hk = hq / G;
    int i, j, t;
    long q_row_stride = (long)c->Hq * c->d;
    long kv_row_stride = (long)c->Hkv * c->d;
    /* the full Sq x Skv score matrix, materialised */
    double* S = (double*)malloc(sizeof(double) * (size_t)c->Sq * (size_t)c->Skv);
    if (!S) {
        c->err = ORACLE_ENOMEM;
        return;
    }
    const double* qb = c->q + (long)b * c->Sq * q_row_stride + (long)hq * c->d;
    const double* kb = c->k + (long)b * c->Skv * kv_row_stride + (long)hk * c->d;
    const double* vb = c->v + (long)b * c->Skv * kv_row_stride + (long)hk * c->d;
    /* S = scale * Q K^T, then the causal mask */
    for (i = 0; i < c->Sq; ++i) {
        const double* q_row = qb + (long)i * q_row_stride;
        for (j = 0; j < c->Skv; ++j) {
            double dot = 0.0;
            const double* k_row = kb + (long)j * kv_row_stride;
            for (t = 0; t < c->d; ++t) dot += q_row[t] * k_row[t];
            S[(long)i * c->Skv + j] = c->scale * dot;
            if (c->causal && j > i + (c->Skv - c->Sq)) S[(long)i * c->Skv + j] = -INFINITY;
            if (c->window > 0 && j >= c->n_sink && j <= i + (c->Skv - c->Sq) - c->window)
                S[(long)i * c->Skv + j] = -INFINITY;
        }
    }
    /* softmax row by row, O = P V, LSE = m + ln l */
    for (i = 0; i < c->Sq; ++i) {
        double* Srow = S + (long)i * c->Skv;
        double* o_row = c->o + ((long)b * c->Sq + i) * q_row_stride + (long)hq * c->d;
        double m = -INFINITY, l = 0.0;
        for (j = 0; j < c->Skv; ++j)
            if (Srow[j] > m) m = Srow[j];
        for (t = 0; t < c->d; ++t) o_row[t] = 0.0;
        if (m == -INFINITY) {
            c->lse[((long)b * c->Hq + hq) * c->Sq + i] = -INFINITY;
            continue;
        }
        for (j = 0; j < c->Skv; ++j) l += exp(Srow[j] - m);
        for (j = 0; j < c->Skv; ++j) {
            double p;
            const double* v_row;
            if (Srow[j] == -INFINITY) continue;
            p = exp(Srow[j] - m) / l;
            v_row = vb + (long)j * kv_row_stride;
            for (t = 0; t < c->d; ++t) o_row[t] += p * v_row[t];
        }
        c->lse[((long)b * c->Hq + hq) * c->Sq + i] = m + log(l);
    }
    free(S);
}

static int check_dims(int B, int Hq, int Hkv, int d) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return 0;
    if (Hq % Hkv != 0) return 0;
    return 1;
}

/* Exact SDPA forward (prefill shape).  Returns 0 or a negative error. */
int oracle_sdpa(const double* q, const double* k, const double* v, int B, int Hq, int Hkv, int Sq,
                int Skv, int d, int causal, double scale, double* o, double* lse, int nthreads) {
    sdpa_ctx c;
    if (!check_dims(B, Hq, Hkv, d) || Sq < 0 || Skv < 0) return ORACLE_EINVAL;
    if (B == 0 || Sq == 0) return ORACLE_OK;
    if (!q || !o || !lse || (Skv > 0 && (!k || !v))) return ORACLE_EINVAL;
    c.q = q; c.k = k; c.v = v;
    c.B = B; c.Hq = Hq; c.Hkv = Hkv; c.Sq = Sq; c.Skv = Skv; c.d = d; c.causal = causal;
    c.window = 0; c.n_sink = 0;
    c.scale = scale; c.o = o; c.lse = lse; c.err = ORACLE_OK;
    run_items(sdpa_item, &c, (long)B * Hq, nthreads);
    return c.err;
}

/* Causal attention over a sliding window of the last `window` positions (the
 * query's own included) plus the first n_sink positions.  window >= 1,
 * n_sink >= 0.  Returns 0 or a negative error. */
int oracle_sdpa_window(const double* q, const double* k, const double* v, int B, int Hq, int Hkv,
                       int Sq, int Skv, int d, int window, int n_sink, double scale, double* o,
                       double* lse, int nthreads) {
    sdpa_ctx c;
    if (!check_dims(B, Hq, Hkv, d) || Sq < 0 || Skv < 0 || window < 1 || n_sink < 0)
        return ORACLE_EINVAL;
    if (B == 0 || Sq == 0) return ORACLE_OK;
    if (!q || !o || !lse || (Skv > 0 && (!k || !v))) return ORACLE_EINVAL;
    c.q = q; c.k = k; c.v = v;
    c.B = B; c.Hq = Hq; c.Hkv = Hkv; c.Sq = Sq; c.Skv = Skv; c.d = d; c.causal = 1;
    c.window = window; c.n_sink = n_sink;
    c.scale = scale; c.o = o; c.lse = lse; c.err = ORACLE_OK;
    run_items(sdpa_item, &c, (long)B * Hq, nthreads);
    return c.err;
}

/* ------------------------------------------------------------------------ */
/* prefill, selected rows only: each (b, hq, i) row computed independently   */
/* from its own score row (used to check single rows of full-size runs)      */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v;
    int B, Hq, Hkv, Sq, Skv, d, causal;
    int window, n_sink; /* window <= 0: no window */
    double scale;
    const int* rows; /* n x 3: (b, hq, i) */
    double *o, *lse; /* n x d, n */
    int err;
} rows_ctx;

static void rows_item(void* vctx, long item) {
    rows_ctx* c = (rows_ctx*)vctx;
    int b = c->rows[3 * item], hq = c->rows[3 * item + 1], i = c->rows[3 * item + 2];
    int G = c->Hq / c->Hkv, hk = hq / G;
    long q_row_stride = (long)c->Hq * c->d, kv_row_stride = (long)c->Hkv * c->d;
    int jmax = c->causal ? i + (c->Skv - c->Sq) : c->Skv - 1;
    int jlo = c->window > 0 ? i + (c->Skv - c->Sq) - c->window + 1 : 0;
    double* s;
    if (b < 0 || b >= c->B || hq < 0 || hq >= c->Hq || i < 0 || i >= c->Sq) {
        c->err = ORACLE_EINVAL;
        return;
    }
    s = (double*)malloc(sizeof(double) * (size_t)(c->Skv > 0 ? c->Skv : 1));
    if (!s) {
        c->err = ORACLE_ENOMEM;
        return;
    }
    softmax_row(c->q + ((long)b * c->Sq + i) * q_row_stride + (long)hq * c->d,
                c->k + (long)b * c->Skv * kv_row_stride + (long)hk * c->d,
                c->v + (long)b * c->Skv * kv_row_stride + (long)hk * c->d, kv_row_stride, c->d, 0,
                c->Skv, jmax, jlo, c->n_sink, c->scale, s, c->o + item * c->d, &c->lse[item]);
    free(s);
}

int oracle_sdpa_rows(const double* q, const double* k, const double* v, int B, int Hq, int Hkv,
                     int Sq, int Skv, int d, int causal, double scale, const int* rows, int n_rows,
                     double* o, double* lse, int nthreads) {
    rows_ctx c;
    if (!check_dims(B, Hq, Hkv, d) || Sq < 0 || Skv < 0 || n_rows < 0) return ORACLE_EINVAL;
    if (n_rows == 0) return ORACLE_OK;
    if (!q || !k || !v || !rows || !o || !lse) return ORACLE_EINVAL;
    c.q = q; c.k = k; c.v = v;
    c.B = B; c.Hq = Hq; c.Hkv = Hkv; c.Sq = Sq; c.Skv = Skv; c.d = d; c.causal = causal;
    c.window = 0; c.n_sink = 0;
    c.scale = scale; c.rows = rows; c.o = o; c.lse = lse; c.err = ORACLE_OK;
    run_items(rows_item, &c, n_rows, nthreads);
    return c.err;
}

/* Selected rows of oracle_sdpa_window. */
int oracle_sdpa_window_rows(const double* q, const double* k, const double* v, int B, int Hq,
                            int Hkv, int Sq, int Skv, int d, int window, int n_sink, double scale,
                            const int* rows, int n_rows, double* o, double* lse, int nthreads) {
    rows_ctx c;
    if (!check_dims(B, Hq, Hkv, d) || Sq < 0 || Skv < 0 || n_rows < 0 || window < 1 || n_sink < 0)
        return ORACLE_EINVAL;
    if (n_rows == 0) return ORACLE_OK;
    if (!q || !k || !v || !rows || !o || !lse) return ORACLE_EINVAL;
    c.q = q; c.k = k; c.v = v;
    c.B = B; c.Hq = Hq; c.Hkv = Hkv; c.Sq = Sq; c.Skv = Skv; c.d = d; c.causal = 1;
    c.window = window; c.n_sink = n_sink;
    c.scale = scale; c.rows = rows; c.o = o; c.lse = lse; c.err = ORACLE_OK;
    run_items(rows_item, &c, n_rows, nthreads);
    return c.err;
}

/* ------------------------------------------------------------------------ */
/* decode: split rule, per-split partials, merge, and the unsplit result     */
/* ------------------------------------------------------------------------ */
/* Split s of a sequence of length L: chunk = max(ceil(L / n_splits), min_rows),
 * rows [s*chunk, min(L, (s+1)*chunk)); empty (lo == hi) when s*chunk >= L. */
int oracle_split_bounds(int L, int n_splits, int min_rows, int s, int* lo, int* hi) {
    long chunk, a, e;
    if (L < 0 || n_splits < 1 || min_rows < 0 || s < 0 || s >= n_splits || !lo || !hi)
        return ORACLE_EINVAL;
    chunk = ((long)L + n_splits - 1) / n_splits;
    if (chunk < min_rows) chunk = min_rows;
    if (chunk < 1) chunk = 1;
    a = (long)s * chunk;
    e = a + chunk;
    if (a > L) a = L;
    if (e > L) e = L;
    *lo = (int)a;
    *hi = (int)e;
    return ORACLE_OK;
}

typedef struct {
    const double *q, *kc, *vc;
    const int* kv_lens;
    int B, Hq, Hkv, d, Lmax, n_splits, min_rows;
    double scale;
    double *part_o, *part_lse; /* split outputs (may be NULL in unsplit mode) */
    double *o, *lse;           /* unsplit outputs (may be NULL in split mode) */
    int err;
} dec_ctx;

static void dec_split_item(void* vctx, long item) {
    dec_ctx* c = (dec_ctx*)vctx;
    int b = (int)(item / c->Hq), hq = (int)(item % c->Hq);
    int G = c->Hq / c->Hkv, hk = hq / G, s, L = c->kv_lens[b];
    long kv_row_stride = (long)c->Hkv * c->d;
    const double* q_row = c->q + ((long)b * c->Hq + hq) * c->d;
    const double* kb = c->kc + (long)b * c->Lmax * kv_row_stride + (long)hk * c->d;
    const double* vb = c->vc + (long)b * c->Lmax * kv_row_stride + (long)hk * c->d;
    double* sc = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    if (!sc) {
        c->err = ORACLE_ENOMEM;
        return;
    }
    for (s = 0; s < c->n_splits; ++s) {
        int lo, hi;
        long idx = ((long)b * c->Hq + hq) * c->n_splits + s;
        oracle_split_bounds(L, c->n_splits, c->min_rows, s, &lo, &hi);
        /* an empty split: lo == hi gives m = -inf -> O = 0, lse = -inf */
        softmax_row(q_row, kb, vb, kv_row_stride, c->d, lo, hi, hi - 1, lo, 0, c->scale, sc,
                    c->part_o + idx * c->d, &c->part_lse[idx]);
    }
    free(sc);
}

static void dec_full_item(void* vctx, long item) {
    dec_ctx* c = (dec_ctx*)vctx;
    int b = (int)(item / c->Hq), hq = (int)(item % c->Hq);
    int G = c->Hq / c->Hkv, hk = hq / G, L = c->kv_lens[b];
    long kv_row_stride = (long)c->Hkv * c->d;
    double* sc = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    if (!sc) {
        c->err = ORACLE_ENOMEM;
        return;
    }
    softmax_row(c->q + ((long)b * c->Hq + hq) * c->d,
                c->kc + (long)b * c->Lmax * kv_row_stride + (long)hk * c->d,
                c->vc + (long)b * c->Lmax * kv_row_stride + (long)hk * c->d, kv_row_stride, c->d,
                0, L, L - 1, 0, 0, c->scale, sc, c->o + ((long)b * c->Hq + hq) * c->d,
                &c->lse[(long)b * c->Hq + hq]);
    free(sc);
}

static int check_lens(const int* kv_lens, int B, int Lmax) {
    int b;
    for (b = 0; b < B; ++b)
        if (kv_lens[b] < 0 || kv_lens[b] > Lmax) return 0;
    return 1;
}

/* Per-split partials of one-token decode (split-KV). */
int oracle_decode_split(const double* q, const double* kc, const double* vc, const int* kv_lens,
                        int B, int Hq, int Hkv, int d, int Lmax, double scale, int n_splits,
                        int min_rows, double* part_o, double* part_lse, int nthreads) {
    dec_ctx c;
    if (!check_dims(B, Hq, Hkv, d) || Lmax < 0 || n_splits < 1 || min_rows < 0)
        return ORACLE_EINVAL;
    if (B == 0) return ORACLE_OK;
    if (!q || !kc || !vc || !kv_lens || !part_o || !part_lse) return ORACLE_EINVAL;
    if (!check_lens(kv_lens, B, Lmax)) return ORACLE_EINVAL;
    memset(&c, 0, sizeof(c));
    c.q = q; c.kc = kc; c.vc = vc; c.kv_lens = kv_lens;
    c.B = B; c.Hq = Hq; c.Hkv = Hkv; c.d = d; c.Lmax = Lmax; c.n_splits = n_splits;
    c.min_rows = min_rows; c.scale = scale; c.part_o = part_o; c.part_lse = part_lse;
    run_items(dec_split_item, &c, (long)B * Hq, nthreads);
    return c.err;
}

/* Unsplit one-token decode: the plain definition over rows [0, L_b). */
int oracle_decode(const double* q, const double* kc, const double* vc, const int* kv_lens, int B,
                  int Hq, int Hkv, int d, int Lmax, double scale, double* o, double* lse,
                  int nthreads) {
    dec_ctx c;
    if (!check_dims(B, Hq, Hkv, d) || Lmax < 0) return ORACLE_EINVAL;
    if (B == 0) return ORACLE_OK;
    if (!q || !kc || !vc || !kv_lens || !o || !lse) return ORACLE_EINVAL;
    if (!check_lens(kv_lens, B, Lmax)) return ORACLE_EINVAL;
    memset(&c, 0, sizeof(c));
    c.q = q; c.kc = kc; c.vc = vc; c.kv_lens = kv_lens;
    c.B = B; c.Hq = Hq; c.Hkv = Hkv; c.d = d; c.Lmax = Lmax; c.scale = scale;
    c.o = o; c.lse = lse;
    run_items(dec_full_item, &c, (long)B * Hq, nthreads);
    return c.err;
}

/* LSE-weighted merge of split partials (the split-combine step). */
int oracle_merge(const double* part_o, const double* part_lse, int B, int Hq, int n_splits, int d,
                 double* o, double* lse) {
    int b, hq, s, t;
    if (B < 0 || Hq <= 0 || n_splits < 1 || d <= 0) return ORACLE_EINVAL;
    if (B == 0) return ORACLE_OK;
    if (!part_o || !part_lse || !o || !lse) return ORACLE_EINVAL;
    for (b = 0; b < B; ++b) {
        for (hq = 0; hq < Hq; ++hq) {
            long row = (long)b * Hq + hq;
            const double* pl = part_lse + row * n_splits;
            const double* po = part_o + row * n_splits * d;
            double* orow = o + row * d;
            double M = -INFINITY, wsum = 0.0;
            for (s = 0; s < n_splits; ++s)
                if (pl[s] > M) M = pl[s];
            for (t = 0; t < d; ++t) orow[t] = 0.0;
            if (M == -INFINITY) { /* every split empty */
                lse[row] = -INFINITY;
                continue;
            }
            for (s = 0; s < n_splits; ++s) {
                double w;
                if (pl[s] == -INFINITY) continue; /* empty split: not read */
                w = exp(pl[s] - M);
                wsum += w;
                for (t = 0; t < d; ++t) orow[t] += w * po[(long)s * d + t];
            }
            for (t = 0; t < d; ++t) orow[t] /= wsum;
            lse[row] = M + log(wsum);
        }
    }
    return ORACLE_OK;
}
