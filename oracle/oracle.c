/*
 * CPU oracle for dynamic top-k sparse attention — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow and direct: every function below writes out the definition of
 * one step of the method in fp64 loops, with the C library's qsort as the only
 * library primitive. Only the tests, the smoke check and the benchmark's CPU
 * baseline may load this code; the product path never does. It shares no code,
 * header or constant with the CUDA library.
 *
 * Passages followed (page, section):
 *  - mhpq.cn/news/1098205 (untitled long-context write-up), section 2.2: the
 *    low-rank scorer, scores = q_low . k_low^T * d_proj^-0.5.
 *  - same page, section 3.2: topk over the scores (sorted, as torch.topk's
 *    default), top_k = min(top_k, seq_len), masked positions set to -inf before
 *    selection; gather of the selected K/V, logits * head_dim^-0.5, softmax,
 *    weighted sum of V.
 *  - "Attention机制优化：原理、挑战与工程实践" (bjdmk.com.cn), section 1.1:
 *    scaled dot-product attention softmax(Q K^T / sqrt(d_k)) V.
 *  - mhpq.cn/news/1098205, section 2.2 (the scorer class): q_low and k_low
 *    come from bias-free linear layers d_model -> d_proj applied to each
 *    head's query and key, q_low = q_proj(query), i.e. x . W^T with W in a
 *    linear layer's [d_proj][d_model] layout.
 *  - nxmr.cn/news/163144 (global vs local attention), section 2.2: a local
 *    window is a radius w around the query, i.e. keys |i - j| <= w, clipped at
 *    the sequence ends; "Attention机制改进：稀疏注意力应用" (yongjin360.com),
 *    section 性能收益与硬件适配: the same band as a boolean mask.
 *
 * Readings where the pages are silent:
 *  - ties in the selection go to the lower key index; the output is ordered by
 *    (score descending, index ascending);
 *  - a row with fewer valid keys than k selects all of them and pads the rest
 *    with index -1 / score -inf;
 *  - causal masking is bottom-right aligned: query i of Tq may see key j of Tk
 *    iff j <= i + (Tk - Tq);
 *  - the score is the fp64 dot product rounded once to fp32, then multiplied
 *    by the fp32 scale in fp32;
 *  - an attention row whose index list holds no valid key outputs zeros;
 *    entries equal to -1 are skipped, repeated entries count once per entry.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    float s;
    int64_t j;
} scored_key;

/* Order: larger score first; equal scores, smaller key index first. */
static int by_score_desc_index_asc(const void* pa, const void* pb) {
    const scored_key* a = (const scored_key*)pa;
    const scored_key* b = (const scored_key*)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    if (a->j < b->j) return -1;
    if (a->j > b->j) return 1;
    return 0;
}

/* ---------------------------------------------------------------- threads */

typedef void (*row_fn)(void* ctx, int64_t r);

typedef struct {
    row_fn fn;
    void* ctx;
    int64_t lo, hi;
} span;

static void* run_span(void* p) {
    span* s = (span*)p;
    for (int64_t r = s->lo; r < s->hi; ++r) s->fn(s->ctx, r);
    return NULL;
}

/* Runs fn(ctx, r) for r in [0, n) on up to nthreads threads, contiguous spans. */
static void for_rows(row_fn fn, void* ctx, int64_t n, int nthreads) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)n;
    pthread_t th[256];
    int started[256];
    span sp[256];
    int64_t per = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        sp[t].fn = fn;
        sp[t].ctx = ctx;
        sp[t].lo = (int64_t)t * per < n ? (int64_t)t * per : n;
        sp[t].hi = sp[t].lo + per < n ? sp[t].lo + per : n;
        started[t] = 0;
        if (t > 0 && sp[t].lo < sp[t].hi)
            started[t] = pthread_create(&th[t], NULL, run_span, &sp[t]) == 0;
    }
    run_span(&sp[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t])
            pthread_join(th[t], NULL);
        else
            run_span(&sp[t]); /* thread creation failed: run the span here */
    }
}

/* ------------------------------------------------------------ score + topk */

typedef struct {
    const double* q_rows; /* [n, P] */
    const int64_t* qpos;  /* [n] absolute query position i in [0, Tq) */
    const double* k_low;  /* [Tk, P] */
    int64_t Tq, Tk;
    int P, k, causal;
    float scale;
    int32_t* idx_out;     /* [n, k] */
    float* score_out;     /* [n, k] or NULL */
} topk_ctx;

/* Number of keys query i may select (bottom-right causal alignment). */
static int64_t valid_count(int64_t i, int64_t Tq, int64_t Tk, int causal) {
    if (!causal) return Tk;
    int64_t last = i + (Tk - Tq); /* largest admissible key index */
    if (last < 0) return 0;
    return last + 1 < Tk ? last + 1 : Tk;
}

static void topk_row(void* vctx, int64_t r) {
    topk_ctx* c = (topk_ctx*)vctx;
    const double* q = c->q_rows + r * c->P;
    int64_t nv = valid_count(c->qpos[r], c->Tq, c->Tk, c->causal);
    scored_key* all = (scored_key*)malloc(sizeof(scored_key) * (size_t)(nv > 0 ? nv : 1));
    for (int64_t j = 0; j < nv; ++j) {
        const double* kr = c->k_low + j * c->P;
        double acc = 0.0;
        for (int p = 0; p < c->P; ++p) acc += q[p] * kr[p];
        float s = (float)acc;
        s = s * c->scale;
        all[j].s = s;
        all[j].j = j;
    }
    qsort(all, (size_t)nv, sizeof(scored_key), by_score_desc_index_asc);
    int64_t keff = nv < c->k ? nv : c->k;
    int32_t* io = c->idx_out + r * c->k;
    float* so = c->score_out ? c->score_out + r * c->k : NULL;
    for (int64_t t = 0; t < c->k; ++t) {
        if (t < keff) {
            io[t] = (int32_t)all[t].j;
            if (so) so[t] = all[t].s;
        } else {
            io[t] = -1;
            if (so) so[t] = -INFINITY;
        }
    }
    free(all);
}

/*
 * Exact per-row top-k of the low-rank scores for n query rows of one head.
 * scale <= 0 selects the default d_proj^-0.5 (rounded to fp32).
 */
int oracle_topk_rows(const double* q_rows, const int64_t* qpos, int64_t n, const double* k_low,
                     int64_t Tq, int64_t Tk, int P, int k, int causal, float scale,
                     int32_t* idx_out, float* score_out, int nthreads) {
    if (!q_rows || !qpos || !k_low || !idx_out || n < 0 || Tk < 0 || P < 1 || k < 1) return 1;
    topk_ctx c;
    c.q_rows = q_rows;
    c.qpos = qpos;
    c.k_low = k_low;
    c.Tq = Tq;
    c.Tk = Tk;
    c.P = P;
    c.k = k;
    c.causal = causal;
    c.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)P));
    c.idx_out = idx_out;
    c.score_out = score_out;
    for_rows(topk_row, &c, n, nthreads);
    return 0;
}

/* ------------------------------------------------------------ scores only */

typedef struct {
    const double* q_rows; /* [n, P] */
    const int64_t* qpos;  /* [n] */
    const double* k_low;  /* [Tk, P] */
    int64_t Tq, Tk;
    int P, causal;
    float scale;
    float* out;           /* [n, Tk] */
} scores_ctx;

static void scores_row(void* vctx, int64_t r) {
    scores_ctx* c = (scores_ctx*)vctx;
    const double* q = c->q_rows + r * c->P;
    int64_t nv = valid_count(c->qpos[r], c->Tq, c->Tk, c->causal);
    float* o = c->out + r * c->Tk;
    for (int64_t j = 0; j < c->Tk; ++j) {
        if (j >= nv) {
            o[j] = -INFINITY; /* masked: never selectable */
            continue;
        }
        const double* kr = c->k_low + j * c->P;
        double acc = 0.0;
        for (int p = 0; p < c->P; ++p) acc += q[p] * kr[p];
        float s = (float)acc;
        o[j] = s * c->scale;
    }
}

/*
 * The low-rank scorer alone (mhpq.cn/news/1098205, section 2.2):
 * S[r, j] = fp32(q_low[r] . k_low[j]) * scale for the keys query qpos[r] may
 * see, -inf for the masked ones (section 3.2, note 3). scale <= 0 selects
 * d_proj^-0.5 rounded to fp32.
 */
int oracle_scores_rows(const double* q_rows, const int64_t* qpos, int64_t n, const double* k_low,
                       int64_t Tq, int64_t Tk, int P, int causal, float scale, float* out,
                       int nthreads) {
    if (!q_rows || !qpos || !k_low || !out || n < 0 || Tk < 0 || P < 1) return 1;
    scores_ctx c;
    c.q_rows = q_rows;
    c.qpos = qpos;
    c.k_low = k_low;
    c.Tq = Tq;
    c.Tk = Tk;
    c.P = P;
    c.causal = causal;
    c.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)P));
    c.out = out;
    for_rows(scores_row, &c, n, nthreads);
    return 0;
}

/* ---------------------------------------------------------------- attend */

/* softmax(q . K_t * scale) weighted sum of V_t over the listed keys, fp64. */
static void attend(const double* q, const double* K, const double* V, int D, const int64_t* keys,
                   int64_t m, double scale, double* logits, double* o) {
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (m == 0) return;
    double mx = -INFINITY;
    for (int64_t t = 0; t < m; ++t) {
        const double* kr = K + keys[t] * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * kr[d];
        logits[t] = acc * scale;
        if (logits[t] > mx) mx = logits[t];
    }
    double den = 0.0;
    for (int64_t t = 0; t < m; ++t) {
        double w = exp(logits[t] - mx);
        logits[t] = w;
        den += w;
    }
    for (int64_t t = 0; t < m; ++t) {
        const double* vr = V + keys[t] * D;
        double w = logits[t] / den;
        for (int d = 0; d < D; ++d) o[d] += w * vr[d];
    }
}

typedef struct {
    const double* q_rows; /* [n, D] */
    const double* K;      /* [Tk, D] */
    const double* V;      /* [Tk, D] */
    int64_t Tk;
    int D, k;
    const int32_t* idx;   /* [n, k] */
    double scale;
    double* O;            /* [n, D] */
    int64_t bad;          /* out-of-range entries seen (counted, skipped) */
    pthread_mutex_t mu;
} attn_ctx;

static void attn_row(void* vctx, int64_t r) {
    attn_ctx* c = (attn_ctx*)vctx;
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)c->k);
    double* lg = (double*)malloc(sizeof(double) * (size_t)c->k);
    int64_t m = 0, bad = 0;
    for (int t = 0; t < c->k; ++t) {
        int32_t j = c->idx[r * c->k + t];
        if (j == -1) continue;
        if (j < -1 || (int64_t)j >= c->Tk) {
            bad++;
            continue;
        }
        keys[m++] = j;
    }
    attend(c->q_rows + r * c->D, c->K, c->V, c->D, keys, m, c->scale, lg, c->O + r * c->D);
    if (bad) {
        pthread_mutex_lock(&c->mu);
        c->bad += bad;
        pthread_mutex_unlock(&c->mu);
    }
    free(keys);
    free(lg);
}

/*
 * Attention of n query rows of one head over the keys their index lists name.
 * scale <= 0 selects head_dim^-0.5. Returns the number of out-of-range
 * entries (they are skipped), or -1 on bad arguments.
 */
int64_t oracle_attn_rows(const double* q_rows, int64_t n, const double* K, const double* V, int64_t Tk,
                         int D, const int32_t* idx, int k, double scale, double* O, int nthreads) {
    if (!q_rows || !K || !V || !idx || !O || n < 0 || D < 1 || k < 1) return -1;
    attn_ctx c;
    c.q_rows = q_rows;
    c.K = K;
    c.V = V;
    c.Tk = Tk;
    c.D = D;
    c.k = k;
    c.idx = idx;
    c.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)D);
    c.O = O;
    c.bad = 0;
    pthread_mutex_init(&c.mu, NULL);
    for_rows(attn_row, &c, n, nthreads);
    pthread_mutex_destroy(&c.mu);
    return c.bad;
}

/* ---------------------------------------------------------------- window */

typedef struct {
    const double* q_rows; /* [n, D] */
    const int64_t* qpos;  /* [n] */
    const double* K;
    const double* V;
    int64_t T;
    int D, wl, wr;
    double scale;
    double* O;
} win_ctx;

static void win_row(void* vctx, int64_t r) {
    win_ctx* c = (win_ctx*)vctx;
    int64_t i = c->qpos[r];
    int64_t lo = i - c->wl < 0 ? 0 : i - c->wl;
    int64_t hi = i + c->wr > c->T - 1 ? c->T - 1 : i + c->wr;
    int64_t m = hi >= lo ? hi - lo + 1 : 0;
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(m > 0 ? m : 1));
    double* lg = (double*)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
    for (int64_t t = 0; t < m; ++t) keys[t] = lo + t;
    attend(c->q_rows + r * c->D, c->K, c->V, c->D, keys, m, c->scale, lg, c->O + r * c->D);
    free(keys);
    free(lg);
}

/*
 * Sliding-window attention of n query rows of one head: query i attends keys
 * j with i - wl <= j <= i + wr, clipped to [0, T). scale <= 0: head_dim^-0.5.
 */
int oracle_window_rows(const double* q_rows, const int64_t* qpos, int64_t n, const double* K,
                       const double* V, int64_t T, int D, int wl, int wr, double scale, double* O,
                       int nthreads) {
    if (!q_rows || !qpos || !K || !V || !O || n < 0 || D < 1 || wl < 0 || wr < 0) return 1;
    win_ctx c;
    c.q_rows = q_rows;
    c.qpos = qpos;
    c.K = K;
    c.V = V;
    c.T = T;
    c.D = D;
    c.wl = wl;
    c.wr = wr;
    c.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)D);
    c.O = O;
    for_rows(win_row, &c, n, nthreads);
    return 0;
}

/*
 * Low-rank projection of the scorer: out[r][p] = sum_c x[r][c] * W[p][c] in
 * fp64, for rows r < n, p < P (W is a linear layer's weight, [P][d_model];
 * no bias). Rounding to the output precision is the caller's.
 */
typedef struct {
    const double* x;
    const double* W;
    int64_t dm;
    int P;
    double* out;
} proj_ctx;

static void proj_row(void* vctx, int64_t r) {
    proj_ctx* c = (proj_ctx*)vctx;
    const double* xr = c->x + r * c->dm;
    for (int p = 0; p < c->P; ++p) {
        const double* wp = c->W + (int64_t)p * c->dm;
        double acc = 0.0;
        for (int64_t cc = 0; cc < c->dm; ++cc) acc += xr[cc] * wp[cc];
        c->out[r * c->P + p] = acc;
    }
}

int oracle_project_rows(const double* x, const double* W, int64_t n, int64_t dm, int P,
                        double* out, int nthreads) {
    if (!x || !W || !out || n < 0 || dm < 1 || P < 1) return 1;
    proj_ctx c;
    c.x = x;
    c.W = W;
    c.dm = dm;
    c.P = P;
    c.out = out;
    for_rows(proj_row, &c, n, nthreads);
    return 0;
}

/* --------------------------------------------------------------- backward */

/*
 * Backward of the sparse attention under the straight-through estimator of
 * mhpq.cn/news/1098205, section 2.3: the forward keeps its hard top-k; in the
 * backward the selected (query, key) pairs pass their gradients exactly as the
 * attention over those keys would, the keys a row did not select get nothing
 * from it, and the scorer receives, for every selected pair, the gradient of
 * that pair's attention logit (the route "through the attention weights of the
 * selected positions"), zero for the pairs not selected.
 *
 * Row i with selected keys j_0 .. j_{m-1} (entries -1 skipped, repeated entries
 * counted once per entry, as in the forward), logits l_t = scale * Q_i . K_{j_t},
 * p = softmax(l), O_i = sum_t p_t V_{j_t}, and the incoming gradient dO_i:
 *   dp_t  = dO_i . V_{j_t}
 *   delta = sum_t p_t dp_t
 *   dl_t  = p_t (dp_t - delta)              (softmax backward)
 *   dQ_i  = scale * sum_t dl_t K_{j_t}
 *   dK_j += scale * dl_t Q_i,   dV_j += p_t dO_i   for each (i, t) with j_t = j
 *   dS[i][t] = dl_t  (0 in skipped slots)
 */
typedef struct {
    const double* q_rows; /* [n, D] */
    const double* K;      /* [Tk, D] */
    const double* V;      /* [Tk, D] */
    const double* dO;     /* [n, D] */
    int64_t Tk;
    int D, k;
    const int32_t* idx;   /* [n, k] */
    double scale;
    double* dQ;           /* [n, D] */
    double* dS;           /* [n, k] */
    double* prob;         /* [n, k] softmax weights, 0 in skipped slots */
    int64_t bad;
    pthread_mutex_t mu;
} bwd_ctx;

/* Key of slot t of row r, or -1 when the slot is skipped (-1 or out of range). */
static int64_t slot_key(const int32_t* idx, int k, int64_t Tk, int64_t r, int t) {
    const int32_t j = idx[r * k + t];
    return (j >= 0 && (int64_t)j < Tk) ? (int64_t)j : -1;
}

static double dot(const double* a, const double* b, int D) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += a[d] * b[d];
    return acc;
}

static void bwd_row(void* vctx, int64_t r) {
    bwd_ctx* c = (bwd_ctx*)vctx;
    const int k = c->k, D = c->D;
    const double* q = c->q_rows + r * D;
    const double* go = c->dO + r * D;
    double* dq = c->dQ + r * D;
    double* ds = c->dS + r * k;
    double* p = c->prob + r * k;
    int64_t bad = 0, m = 0;
    double mx = -INFINITY;
    for (int t = 0; t < k; ++t) {
        ds[t] = 0.0;
        p[t] = 0.0;
        const int64_t j = slot_key(c->idx, k, c->Tk, r, t);
        if (j < 0) {
            if (c->idx[r * k + t] != -1) bad++;
            continue;
        }
        p[t] = c->scale * dot(q, c->K + j * D, D); /* the logit, for now */
        if (p[t] > mx) mx = p[t];
        m++;
    }
    for (int d = 0; d < D; ++d) dq[d] = 0.0;
    if (m > 0) {
        double den = 0.0;
        for (int t = 0; t < k; ++t) {
            if (slot_key(c->idx, k, c->Tk, r, t) < 0) continue;
            p[t] = exp(p[t] - mx);
            den += p[t];
        }
        double delta = 0.0;
        for (int t = 0; t < k; ++t) {
            const int64_t j = slot_key(c->idx, k, c->Tk, r, t);
            if (j < 0) continue;
            p[t] /= den;
            ds[t] = dot(go, c->V + j * D, D); /* dp_t, for now */
            delta += p[t] * ds[t];
        }
        for (int t = 0; t < k; ++t) {
            const int64_t j = slot_key(c->idx, k, c->Tk, r, t);
            if (j < 0) continue;
            ds[t] = p[t] * (ds[t] - delta);
            for (int d = 0; d < D; ++d) dq[d] += c->scale * ds[t] * c->K[j * D + d];
        }
    }
    if (bad) {
        pthread_mutex_lock(&c->mu);
        c->bad += bad;
        pthread_mutex_unlock(&c->mu);
    }
}

/*
 * Gradients of n query rows of one head: dQ [n, D], dK and dV [Tk, D] (set
 * here: zero, then the sum over every row and slot that selected the key), and
 * dS [n, k], the gradient the straight-through estimator hands to each selected
 * pair's score. scale <= 0 selects head_dim^-0.5. Returns the number of
 * out-of-range entries (skipped), or -1 on bad arguments.
 */
int64_t oracle_attn_bwd_rows(const double* q_rows, int64_t n, const double* K, const double* V,
                             int64_t Tk, int D, const int32_t* idx, int k, double scale,
                             const double* dO, double* dQ, double* dK, double* dV, double* dS,
                             int nthreads) {
    if (!q_rows || !K || !V || !idx || !dO || !dQ || !dK || !dV || !dS || n < 0 || Tk < 0 ||
        D < 1 || k < 1)
        return -1;
    bwd_ctx c;
    c.q_rows = q_rows;
    c.K = K;
    c.V = V;
    c.dO = dO;
    c.Tk = Tk;
    c.D = D;
    c.k = k;
    c.idx = idx;
    c.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)D);
    c.dQ = dQ;
    c.dS = dS;
    c.prob = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)k);
    if (!c.prob) return -1;
    c.bad = 0;
    pthread_mutex_init(&c.mu, NULL);
    for_rows(bwd_row, &c, n, nthreads);
    pthread_mutex_destroy(&c.mu);
    /* the key-side sums, one row and slot at a time */
    for (int64_t e = 0; e < Tk * D; ++e) {
        dK[e] = 0.0;
        dV[e] = 0.0;
    }
    for (int64_t r = 0; r < n; ++r) {
        for (int t = 0; t < k; ++t) {
            const int64_t j = slot_key(idx, k, Tk, r, t);
            if (j < 0) continue;
            for (int d = 0; d < D; ++d) {
                dK[j * D + d] += c.scale * dS[r * k + t] * q_rows[r * D + d];
                dV[j * D + d] += c.prob[r * k + t] * dO[r * D + d];
            }
        }
    }
    free(c.prob);
    return c.bad;
}

/*
 * The scorer's gradients under the same estimator: the score of a selected
 * pair, S = scale * q_low_i . k_low_j (mhpq.cn/news/1098205, section 2.2),
 * receives dS[i][t], and a pair not selected receives nothing, so
 *   dq_low_i  = scale * sum_t dS[i][t] k_low_{j_t}
 *   dk_low_j += scale * dS[i][t] q_low_i   for each (i, t) with j_t = j.
 * q_low [n, P], k_low [Tk, P], idx and dS [n, k]; dq_low [n, P] and dk_low
 * [Tk, P] are set here. scale <= 0 selects d_proj^-0.5 rounded to fp32 (the
 * factor the forward scores use). Returns 0, or 1 on bad arguments.
 */
int oracle_scorer_bwd_rows(const double* q_low, int64_t n, const double* k_low, int64_t Tk, int P,
                           const int32_t* idx, int k, double scale, const double* dS,
                           double* dq_low, double* dk_low) {
    if (!q_low || !k_low || !idx || !dS || !dq_low || !dk_low || n < 0 || Tk < 0 || P < 1 || k < 1)
        return 1;
    const double s = scale > 0.0 ? scale : (double)(float)(1.0 / sqrt((double)P));
    for (int64_t e = 0; e < n * P; ++e) dq_low[e] = 0.0;
    for (int64_t e = 0; e < Tk * P; ++e) dk_low[e] = 0.0;
    for (int64_t r = 0; r < n; ++r) {
        for (int t = 0; t < k; ++t) {
            const int64_t j = slot_key(idx, k, Tk, r, t);
            if (j < 0) continue;
            const double g = s * dS[r * k + t];
            for (int p = 0; p < P; ++p) {
                dq_low[r * P + p] += g * k_low[j * P + p];
                dk_low[j * P + p] += g * q_low[r * P + p];
            }
        }
    }
    return 0;
}
