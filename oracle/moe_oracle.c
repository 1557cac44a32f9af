/*
 * moe_oracle.c -- plain fp64 CPU oracle of one MoE layer (see moe_oracle.h).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the GPU product path.
 *
 * What pins each function to something other than itself (CPU test-suite):
 *   oracle_logits      numpy fp64 matmul x @ Wg.T on tiny shapes; bias shifts
 *                      every column by exactly bias[e]
 *   oracle_select      brute-force enumeration of all C(E,K) subsets on tiny E;
 *                      constructed exact ties (duplicate gate rows, -0/+0);
 *                      torch.topk on tie-free rows
 *   oracle_weights     sum of weights = 1; K = 1 gives 1; torch.softmax /
 *                      torch.sigmoid on the selected logits
 *   oracle_offsets,
 *   oracle_place       the 8-token t0..t7 -> e0/e1/e2 worked example of the
 *                      contiguous paradigm reproduced exactly; offsets are the
 *                      prefix sum of counts; perm_src / inv_perm are mutual
 *                      inverses (permute then un-permute is the identity)
 *   oracle_expert_*    E = 1, K = 1 reduces to a dense FFN (numpy matmuls);
 *                      silu(0) = 0, silu(g) -> g for large g
 *   oracle_combine     identical experts make the output routing-independent;
 *                      identity experts give out = x
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread.
 * No FMA contraction, no fast-math: every sum is the plain left-to-right
 * double-precision sum.
 */
#define _POSIX_C_SOURCE 200809L
#include "moe_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    if (n < 1) n = 1;
    if (n > 256) n = 256;
    return (int)n;
}

/* ---------------------------------------------------------------------------
 * A minimal parallel-for: [0, n) is cut into nthreads contiguous ranges and
 * each range runs body(ctx, begin, end) on its own thread.  The split changes
 * only which thread computes a result, never the arithmetic of any result.
 * ------------------------------------------------------------------------- */
typedef void (*range_fn)(void* ctx, int64_t begin, int64_t end);
typedef struct { range_fn fn; void* ctx; int64_t begin, end; } range_job;

static void* run_range(void* p) {
    range_job* j = (range_job*)p;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void* ctx) {
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (n <= 0) return;
    if ((int64_t)nthreads > n) nthreads = (int)n;
    if (nthreads <= 1) { fn(ctx, 0, n); return; }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    range_job* jobs = (range_job*)malloc(sizeof(range_job) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].fn = fn;
        jobs[i].ctx = ctx;
        jobs[i].begin = n * i / nthreads;
        jobs[i].end = n * (i + 1) / nthreads;
        if (i == 0) continue; /* range 0 runs on the calling thread */
        if (pthread_create(&th[i], NULL, run_range, &jobs[i]) != 0) {
            /* could not start a thread: run its range here instead */
            run_range(&jobs[i]);
            jobs[i].fn = NULL;
        }
    }
    run_range(&jobs[0]);
    for (int i = 1; i < nthreads; ++i)
        if (jobs[i].fn != NULL) pthread_join(th[i], NULL);
    free(th);
    free(jobs);
}

/* ---------------------------------------------------------------------------
 * O1 router logits: L = x Wg^T (+ bias).
 * ------------------------------------------------------------------------- */
typedef struct {
    const uint16_t *x, *wg;
    const double* bias;
    int64_t D, E;
    double* L;
} logits_ctx;

static void logits_rows(void* p, int64_t t0, int64_t t1) {
    logits_ctx* c = (logits_ctx*)p;
    for (int64_t t = t0; t < t1; ++t) {
        for (int64_t e = 0; e < c->E; ++e) {
            double s = 0.0;
            for (int64_t d = 0; d < c->D; ++d)
                s += oracle_bf16_to_f64(c->x[t * c->D + d]) *
                     oracle_bf16_to_f64(c->wg[e * c->D + d]);
            if (c->bias) s += c->bias[e];
            c->L[t * c->E + e] = s;
        }
    }
}

void oracle_logits(const uint16_t* x, const uint16_t* wg, const double* bias,
                   int64_t N, int64_t D, int64_t E, double* L, int nthreads) {
    logits_ctx c = {x, wg, bias, D, E, L};
    parallel_for(N, nthreads, logits_rows, &c);
}

/* ---------------------------------------------------------------------------
 * O2 top-K: order experts by (logit desc, index asc); keep the first K.
 * "a comes before b" is a strict total order, so the result is unique.
 * -0.0 and +0.0 compare equal and fall through to the index.
 * ------------------------------------------------------------------------- */
static int comes_before(double va, int64_t ia, double vb, int64_t ib) {
    if (va > vb) return 1;
    if (va < vb) return 0;
    return ia < ib;
}

int oracle_select(const double* L, int64_t N, int64_t E, int64_t K, int32_t* ids) {
    if (K < 1 || K > E) return -1;
    for (int64_t t = 0; t < N; ++t) {
        const double* row = L + t * E;
        /* selection by repeated "best remaining": pick k is the expert that
           comes first among those not yet picked */
        char* taken = (char*)calloc((size_t)E, 1);
        for (int64_t k = 0; k < K; ++k) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || comes_before(row[e], e, row[best], best)) best = e;
            }
            taken[best] = 1;
            ids[t * K + k] = (int32_t)best;
        }
        free(taken);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * O3 weights over the K selected logits.
 * ------------------------------------------------------------------------- */
void oracle_weights(const double* L, const int32_t* ids, int64_t N, int64_t E,
                    int64_t K, int mode, double* w) {
    for (int64_t t = 0; t < N; ++t) {
        const double* row = L + t * E;
        const int32_t* id = ids + t * K;
        double* wt = w + t * K;
        double sum = 0.0;
        if (mode == ORACLE_SCORE_SOFTMAX_TOPK) {
            double top = row[id[0]]; /* the largest selected logit */
            for (int64_t k = 0; k < K; ++k) {
                wt[k] = exp(row[id[k]] - top);
                sum += wt[k];
            }
        } else {
            for (int64_t k = 0; k < K; ++k) {
                wt[k] = 1.0 / (1.0 + exp(-row[id[k]]));
                sum += wt[k];
            }
        }
        if (sum > 0.0) {
            for (int64_t k = 0; k < K; ++k) wt[k] = wt[k] / sum;
        } else {
            for (int64_t k = 0; k < K; ++k) wt[k] = 1.0 / (double)K;
        }
    }
}

/* ---------------------------------------------------------------------------
 * O4 offsets = exclusive prefix sum of per-expert counts.
 * ------------------------------------------------------------------------- */
int oracle_offsets(const int32_t* ids, int64_t N, int64_t K, int64_t E, int32_t* offsets) {
    int64_t* count = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t i = 0; i < N * K; ++i) {
        if (ids[i] < 0 || ids[i] >= E) { free(count); return -1; }
        count[ids[i]] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = (int32_t)(offsets[e] + count[e]);
    free(count);
    return 0;
}

/* ---------------------------------------------------------------------------
 * O5 stable placement in (t, k) order.
 * ------------------------------------------------------------------------- */
int oracle_place(const int32_t* ids, const int32_t* offsets, int64_t N, int64_t K,
                 int64_t E, int32_t* perm_src, int32_t* inv_perm) {
    int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t t = 0; t < N; ++t) {
        for (int64_t k = 0; k < K; ++k) {
            int32_t e = ids[t * K + k];
            if (e < 0 || e >= E) { free(fill); return -1; }
            int64_t r = offsets[e] + fill[e];
            fill[e] += 1;
            perm_src[r] = (int32_t)t;
            inv_perm[t * K + k] = (int32_t)r;
        }
    }
    free(fill);
    return 0;
}

void oracle_gather_rows(const uint16_t* x, const int32_t* perm_src, int64_t rows,
                        int64_t D, uint16_t* x_perm) {
    for (int64_t r = 0; r < rows; ++r)
        memcpy(x_perm + r * D, x + (int64_t)perm_src[r] * D, sizeof(uint16_t) * (size_t)D);
}

/* ---------------------------------------------------------------------------
 * O6 expert FFN.
 * ------------------------------------------------------------------------- */
static double silu(double g) { return g / (1.0 + exp(-g)); }

/* One element h[r][j] (up) or y[r][d] (down) is one plain dot product over
 * the reduction index in increasing order; xr / hr are the input rows already
 * converted (exactly) to double. */
static double up_element(const double* xr, const uint16_t* w1, const uint16_t* w3,
                         int64_t D, int64_t j, int act) {
    double g = 0.0;
    for (int64_t d = 0; d < D; ++d) g += oracle_bf16_to_f64(w1[j * D + d]) * xr[d];
    if (act != ORACLE_ACT_SWIGLU) return silu(g);
    double u = 0.0;
    for (int64_t d = 0; d < D; ++d) u += oracle_bf16_to_f64(w3[j * D + d]) * xr[d];
    return silu(g) * u;
}

static double down_element(const double* hr, const uint16_t* w2, int64_t Dff, int64_t d) {
    double s = 0.0;
    for (int64_t j = 0; j < Dff; ++j) s += oracle_bf16_to_f64(w2[d * Dff + j]) * hr[j];
    return s;
}

static double* rows_to_f64(const uint16_t* rows, int64_t R, int64_t W) {
    double* out = (double*)malloc(sizeof(double) * (size_t)(R * W > 0 ? R * W : 1));
    for (int64_t i = 0; i < R * W; ++i) out[i] = oracle_bf16_to_f64(rows[i]);
    return out;
}

/* Work items are output elements (row-major), so a call with few rows still
 * spreads over every thread. */
typedef struct {
    const double* xf;
    const uint16_t *w1, *w3;
    int64_t D, Dff;
    int act;
    double* h;
} up_ctx;

static void up_items(void* p, int64_t i0, int64_t i1) {
    up_ctx* c = (up_ctx*)p;
    for (int64_t i = i0; i < i1; ++i) {
        const int64_t r = i / c->Dff, j = i % c->Dff;
        c->h[i] = up_element(c->xf + r * c->D, c->w1, c->w3, c->D, j, c->act);
    }
}

void oracle_expert_up(const uint16_t* xrows, int64_t R, const uint16_t* w1,
                      const uint16_t* w3, int64_t D, int64_t Dff, int act,
                      double* h, int nthreads) {
    double* xf = rows_to_f64(xrows, R, D);
    up_ctx c = {xf, w1, w3, D, Dff, act, h};
    parallel_for(R * Dff, nthreads, up_items, &c);
    free(xf);
}

typedef struct {
    const double* hf;
    const uint16_t* w2;
    int64_t D, Dff;
    double* y;
} down_ctx;

static void down_items(void* p, int64_t i0, int64_t i1) {
    down_ctx* c = (down_ctx*)p;
    for (int64_t i = i0; i < i1; ++i) {
        const int64_t r = i / c->D, d = i % c->D;
        c->y[i] = down_element(c->hf + r * c->Dff, c->w2, c->Dff, d);
    }
}

void oracle_expert_down(const double* h, int64_t R, const uint16_t* w2, int64_t D,
                        int64_t Dff, double* y, int nthreads) {
    down_ctx c = {h, w2, D, Dff, y};
    parallel_for(R * D, nthreads, down_items, &c);
}

void oracle_expert_down_bf16(const uint16_t* h, int64_t R, const uint16_t* w2,
                             int64_t D, int64_t Dff, double* y, int nthreads) {
    double* hf = rows_to_f64(h, R, Dff);
    down_ctx c = {hf, w2, D, Dff, y};
    parallel_for(R * D, nthreads, down_items, &c);
    free(hf);
}

/* All experts: one row of x_perm at a time, each with its own expert's
 * weights.  Parallel over rows; each row's arithmetic is the per-expert one. */
typedef struct {
    const uint16_t *x_perm, *w1, *w3, *w2;
    const int32_t* offsets;
    int64_t E, D, Dff;
    int act;
    double *h, *y;
} grouped_ctx;

static void grouped_rows(void* p, int64_t r0, int64_t r1) {
    grouped_ctx* c = (grouped_ctx*)p;
    double* xr = (double*)malloc(sizeof(double) * (size_t)c->D);
    double* hrow = (double*)malloc(sizeof(double) * (size_t)c->Dff);
    int64_t e = 0;
    for (int64_t r = r0; r < r1; ++r) {
        while (e < c->E && r >= c->offsets[e + 1]) ++e; /* expert owning row r */
        const uint16_t* w1e = c->w1 + e * c->Dff * c->D;
        const uint16_t* w3e = c->w3 ? c->w3 + e * c->Dff * c->D : NULL;
        const uint16_t* w2e = c->w2 + e * c->D * c->Dff;
        for (int64_t d = 0; d < c->D; ++d) xr[d] = oracle_bf16_to_f64(c->x_perm[r * c->D + d]);
        for (int64_t j = 0; j < c->Dff; ++j) hrow[j] = up_element(xr, w1e, w3e, c->D, j, c->act);
        if (c->h) memcpy(c->h + r * c->Dff, hrow, sizeof(double) * (size_t)c->Dff);
        for (int64_t d = 0; d < c->D; ++d) c->y[r * c->D + d] = down_element(hrow, w2e, c->Dff, d);
    }
    free(xr);
    free(hrow);
}

void oracle_grouped_ffn(const uint16_t* x_perm, const int32_t* offsets, int64_t E,
                        const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                        int64_t D, int64_t Dff, int act, double* h, double* y,
                        int nthreads) {
    grouped_ctx c = {x_perm, w1, (act == ORACLE_ACT_SWIGLU) ? w3 : NULL, w2,
                     offsets, E, D, Dff, act, h, y};
    parallel_for((int64_t)offsets[E], nthreads, grouped_rows, &c);
}

/* ---------------------------------------------------------------------------
 * O7 combine.
 * ------------------------------------------------------------------------- */
void oracle_combine(const double* y, const int32_t* inv_perm, const double* w,
                    int64_t N, int64_t D, int64_t K, double* out) {
    for (int64_t t = 0; t < N; ++t) {
        for (int64_t d = 0; d < D; ++d) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += w[t * K + k] * y[(int64_t)inv_perm[t * K + k] * D + d];
            out[t * D + d] = s;
        }
    }
}

/* ---------------------------------------------------------------------------
 * The whole layer.
 * ------------------------------------------------------------------------- */
int oracle_layer(const uint16_t* x, const uint16_t* wg, const double* bias,
                 const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                 int64_t N, int64_t D, int64_t E, int64_t K, int64_t Dff,
                 int mode, int act, double* L, int32_t* ids, double* w,
                 int32_t* offsets, int32_t* perm_src, int32_t* inv_perm,
                 double* out, int nthreads) {
    if (N < 0 || D < 1 || E < 1 || K < 1 || K > E || Dff < 1) return -1;
    int64_t A = N * K;
    double* logits = L ? L : (double*)malloc(sizeof(double) * (size_t)(N * E > 0 ? N * E : 1));
    uint16_t* x_perm = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(A * D > 0 ? A * D : 1));
    double* y = (double*)malloc(sizeof(double) * (size_t)(A * D > 0 ? A * D : 1));
    int rc = 0;
    oracle_logits(x, wg, bias, N, D, E, logits, nthreads);            /* O1 */
    rc |= oracle_select(logits, N, E, K, ids);                        /* O2 */
    oracle_weights(logits, ids, N, E, K, mode, w);                    /* O3 */
    rc |= oracle_offsets(ids, N, K, E, offsets);                      /* O4 */
    if (rc == 0) {
        rc |= oracle_place(ids, offsets, N, K, E, perm_src, inv_perm); /* O5 */
        oracle_gather_rows(x, perm_src, A, D, x_perm);
        oracle_grouped_ffn(x_perm, offsets, E, w1, w3, w2, D, Dff, act, NULL, y,
                           nthreads);                                 /* O6 */
        oracle_combine(y, inv_perm, w, N, D, K, out);                 /* O7 */
    }
    if (!L) free(logits);
    free(x_perm);
    free(y);
    return rc;
}

/* ---------------------------------------------------------------------------
 * Routing statistics: EMA of per-expert fractions, KL to uniform, bias step.
 * ------------------------------------------------------------------------- */
double oracle_routing_stats(const int32_t* offsets, int64_t E, double decay, double step,
                            double* ema, double* bias) {
    const double total = (double)offsets[E];
    if (total <= 0.0) return 0.0;
    double sum = 0.0;
    for (int64_t e = 0; e < E; ++e) {
        const double frac = (double)(offsets[e + 1] - offsets[e]) / total;
        ema[e] = decay * ema[e] + (1.0 - decay) * frac;
        sum += ema[e];
    }
    double kl = 0.0;
    for (int64_t e = 0; e < E; ++e) {
        const double f = ema[e] / sum;
        kl += f * log(f * (double)E + 1e-9);
        if (bias) bias[e] += step * ((double)E * f - 1.0);
    }
    return kl;
}

/* ---------------------------------------------------------------------------
 * Paradigm B: padded placement and the weighted sum over kept assignments.
 * ------------------------------------------------------------------------- */
int oracle_place_padded(const int32_t* ids, int64_t N, int64_t K, int64_t E, int64_t C,
                        int32_t* slot, int32_t* kept) {
    if (C < 0) return -1;
    for (int64_t e = 0; e < E; ++e) kept[e] = 0;
    for (int64_t t = 0; t < N; ++t) {
        for (int64_t k = 0; k < K; ++k) {
            const int32_t e = ids[t * K + k];
            if (e < 0 || e >= E) return -1;
            if (kept[e] < C) {
                slot[t * K + k] = (int32_t)(e * C + kept[e]);
                kept[e] += 1;
            } else {
                slot[t * K + k] = -1;
            }
        }
    }
    return 0;
}

void oracle_combine_kept(const double* y, const int32_t* slot, const double* w, int64_t N,
                         int64_t D, int64_t K, double* out) {
    for (int64_t t = 0; t < N; ++t) {
        for (int64_t d = 0; d < D; ++d) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const int32_t r = slot[t * K + k];
                if (r >= 0) s += w[t * K + k] * y[(int64_t)r * D + d];
            }
            out[t * D + d] = s;
        }
    }
}
