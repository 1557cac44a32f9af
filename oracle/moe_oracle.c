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
 *   oracle_e4m3_*      every code decoded by hand from the format's definition
 *                      and against torch.float8_e4m3fn; every bf16 value in
 *                      range encoded against torch's cast; hand-computed ties,
 *                      subnormals and saturation
 *   oracle_f64_to_bf16 torch's float -> bf16 rounding on float inputs; a
 *                      double-rounding case computed by hand; overflow, subnormal
 *   oracle_quant_rows  the scale rule at hand-computed amax values; scaled row
 *                      maxima in (224, 448]; representable rows round-trip
 *                      exactly; the e4m3 error bound on every element
 *   oracle_*_e4m3      on e4m3-representable operands the FP8 GEMMs equal the
 *                      bf16 oracle exactly (same sums in the same order)
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
 * FP8 (e4m3) experts.
 * ------------------------------------------------------------------------- */
double oracle_e4m3_decode(uint8_t c) {
    const int sign = (c >> 7) & 1, ex = (c >> 3) & 15, man = c & 7;
    double mag;
    if (ex == 15 && man == 7) return NAN;               /* the only NaN codes */
    if (ex == 0) mag = ldexp((double)man / 8.0, -6);    /* subnormal */
    else mag = ldexp(1.0 + (double)man / 8.0, ex - 7);  /* normal */
    return sign ? -mag : mag;
}

/* Decoded values of all 256 codes (g_e4m3[0..126] are the finite
 * non-negative ones, strictly increasing in the code). */
static double g_e4m3[256];
static pthread_once_t g_e4m3_once = PTHREAD_ONCE_INIT;
static void e4m3_table_init(void) {
    for (int c = 0; c < 256; ++c) g_e4m3[c] = oracle_e4m3_decode((uint8_t)c);
}

uint8_t oracle_e4m3_encode(double v) {
    pthread_once(&g_e4m3_once, e4m3_table_init);
    const double a = fabs(v);
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (a >= g_e4m3[126]) return (uint8_t)(sign | 126); /* saturate at 448 */
    /* lo = the largest code whose value is <= a (bisection on the table) */
    int lo = 0, hi = 126;
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (g_e4m3[mid] <= a) lo = mid; else hi = mid;
    }
    /* a lies in [value(lo), value(lo+1)): take the nearer, ties to the even code */
    const double dlo = a - g_e4m3[lo], dhi = g_e4m3[lo + 1] - a;
    int c = lo;
    if (dhi < dlo || (dhi == dlo && ((lo + 1) & 1) == 0)) c = lo + 1;
    return (uint8_t)(sign | c);
}

void oracle_e4m3_encode_array(const double* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

uint16_t oracle_f64_to_bf16(double v) {
    if (v != v) return 0x7fc0;
    const uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    const double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a = m 2^e with m in [0.5, 1): leading bit 2^(e-1) */
    int lsb = (e - 1) - 7;        /* weight of the 8th significant bit */
    if (lsb < -133) lsb = -133;   /* below 2^-126 the spacing is fixed (subnormals) */
    const double r = ldexp(nearbyint(ldexp(a, -lsb)), lsb); /* ties to even */
    const float f = (float)r;     /* exact, or +inf past the largest bf16 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

int oracle_e4m3_scale_exp(double amax) {
    int k = -126;
    if (!(amax > 0.0)) return k;
    while (amax > ldexp(448.0, k)) ++k;
    return k;
}

typedef struct {
    const uint16_t* src;
    int64_t cols;
    uint8_t* q;
    float* scale;
} quant_ctx;

static void quant_rows_range(void* p, int64_t r0, int64_t r1) {
    quant_ctx* c = (quant_ctx*)p;
    for (int64_t r = r0; r < r1; ++r) {
        const uint16_t* row = c->src + r * c->cols;
        double amax = 0.0;
        for (int64_t j = 0; j < c->cols; ++j) {
            const double a = fabs(oracle_bf16_to_f64(row[j]));
            if (a > amax) amax = a;
        }
        const int k = oracle_e4m3_scale_exp(amax);
        c->scale[r] = (float)ldexp(1.0, k);
        for (int64_t j = 0; j < c->cols; ++j)
            c->q[r * c->cols + j] = oracle_e4m3_encode(ldexp(oracle_bf16_to_f64(row[j]), -k));
    }
}

void oracle_quant_rows_e4m3(const uint16_t* src, int64_t rows, int64_t cols, uint8_t* q,
                            float* scale, int nthreads) {
    quant_ctx c = {src, cols, q, scale};
    parallel_for(rows, nthreads, quant_rows_range, &c);
}

void oracle_dequant_rows_e4m3(const uint8_t* q, const float* scale, int64_t rows, int64_t cols,
                              double* out) {
    pthread_once(&g_e4m3_once, e4m3_table_init);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < cols; ++j)
            out[r * cols + j] = g_e4m3[q[r * cols + j]] * (double)scale[r];
}

/* One output of the FP8 GEMMs: a plain dot product of a dequantised weight
 * row with an already dequantised activation row, in increasing index order. */
static double dot_e4m3_row(const uint8_t* wq, double ws, const double* act, int64_t n) {
    pthread_once(&g_e4m3_once, e4m3_table_init);
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += (g_e4m3[wq[i]] * ws) * act[i];
    return s;
}

static double up_element_e4m3(const double* xr, const uint8_t* w1q, const float* s1,
                              const uint8_t* w3q, const float* s3, int64_t D, int64_t j, int act) {
    const double g = dot_e4m3_row(w1q + j * D, (double)s1[j], xr, D);
    if (act != ORACLE_ACT_SWIGLU) return silu(g);
    const double u = dot_e4m3_row(w3q + j * D, (double)s3[j], xr, D);
    return silu(g) * u;
}

typedef struct {
    const double* xf;
    const uint8_t *w1q, *w3q;
    const float *s1, *s3;
    int64_t D, Dff;
    int act;
    double* h;
} up8_ctx;

static void up8_items(void* p, int64_t i0, int64_t i1) {
    up8_ctx* c = (up8_ctx*)p;
    for (int64_t i = i0; i < i1; ++i) {
        const int64_t r = i / c->Dff, j = i % c->Dff;
        c->h[i] = up_element_e4m3(c->xf + r * c->D, c->w1q, c->s1, c->w3q, c->s3, c->D, j, c->act);
    }
}

void oracle_expert_up_e4m3(const uint8_t* xq, const float* sx, int64_t R, const uint8_t* w1q,
                           const float* s1, const uint8_t* w3q, const float* s3, int64_t D,
                           int64_t Dff, int act, double* h, int nthreads) {
    double* xf = (double*)malloc(sizeof(double) * (size_t)(R * D > 0 ? R * D : 1));
    oracle_dequant_rows_e4m3(xq, sx, R, D, xf);
    up8_ctx c = {xf, w1q, (act == ORACLE_ACT_SWIGLU) ? w3q : NULL, s1,
                 (act == ORACLE_ACT_SWIGLU) ? s3 : NULL, D, Dff, act, h};
    parallel_for(R * Dff, nthreads, up8_items, &c);
    free(xf);
}

typedef struct {
    const double* hf;
    const uint8_t* w2q;
    const float* s2;
    int64_t D, Dff;
    double* y;
} down8_ctx;

static void down8_items(void* p, int64_t i0, int64_t i1) {
    down8_ctx* c = (down8_ctx*)p;
    for (int64_t i = i0; i < i1; ++i) {
        const int64_t r = i / c->D, d = i % c->D;
        c->y[i] = dot_e4m3_row(c->w2q + d * c->Dff, (double)c->s2[d], c->hf + r * c->Dff, c->Dff);
    }
}

void oracle_expert_down_e4m3(const uint8_t* hq, const float* sh, int64_t R, const uint8_t* w2q,
                             const float* s2, int64_t D, int64_t Dff, double* y, int nthreads) {
    double* hf = (double*)malloc(sizeof(double) * (size_t)(R * Dff > 0 ? R * Dff : 1));
    oracle_dequant_rows_e4m3(hq, sh, R, Dff, hf);
    down8_ctx c = {hf, w2q, s2, D, Dff, y};
    parallel_for(R * D, nthreads, down8_items, &c);
    free(hf);
}

typedef struct {
    const uint8_t* xq;
    const float* sx;
    const int32_t* offsets;
    int64_t E, D, Dff;
    const uint8_t *w1q, *w3q, *w2q;
    const float *s1, *s3, *s2;
    int act;
    double* h;
    uint16_t* hb;
    uint8_t* hq;
    float* sh;
    double* y;
} grouped8_ctx;

static void grouped8_rows(void* p, int64_t r0, int64_t r1) {
    grouped8_ctx* c = (grouped8_ctx*)p;
    const int64_t D = c->D, Dff = c->Dff;
    double* xr = (double*)malloc(sizeof(double) * (size_t)D);
    double* hrow = (double*)malloc(sizeof(double) * (size_t)Dff);
    uint16_t* hbrow = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)Dff);
    uint8_t* hqrow = (uint8_t*)malloc((size_t)Dff);
    double* hdq = (double*)malloc(sizeof(double) * (size_t)Dff);
    int64_t e = 0;
    for (int64_t r = r0; r < r1; ++r) {
        while (e < c->E && r >= c->offsets[e + 1]) ++e; /* expert owning row r */
        const uint8_t* w1e = c->w1q + e * Dff * D;
        const uint8_t* w3e = c->w3q ? c->w3q + e * Dff * D : NULL;
        const uint8_t* w2e = c->w2q + e * D * Dff;
        const float* s1e = c->s1 + e * Dff;
        const float* s3e = c->s3 ? c->s3 + e * Dff : NULL;
        const float* s2e = c->s2 + e * D;
        oracle_dequant_rows_e4m3(c->xq + r * D, c->sx + r, 1, D, xr);
        for (int64_t j = 0; j < Dff; ++j) {
            hrow[j] = up_element_e4m3(xr, w1e, s1e, w3e, s3e, D, j, c->act);
            hbrow[j] = oracle_f64_to_bf16(hrow[j]);
        }
        float shr;
        quant_ctx qc = {hbrow, Dff, hqrow, &shr};
        quant_rows_range(&qc, 0, 1);
        oracle_dequant_rows_e4m3(hqrow, &shr, 1, Dff, hdq);
        for (int64_t d = 0; d < D; ++d) c->y[r * D + d] = dot_e4m3_row(w2e + d * Dff, (double)s2e[d], hdq, Dff);
        if (c->h) memcpy(c->h + r * Dff, hrow, sizeof(double) * (size_t)Dff);
        if (c->hb) memcpy(c->hb + r * Dff, hbrow, sizeof(uint16_t) * (size_t)Dff);
        if (c->hq) memcpy(c->hq + r * Dff, hqrow, (size_t)Dff);
        if (c->sh) c->sh[r] = shr;
    }
    free(xr);
    free(hrow);
    free(hbrow);
    free(hqrow);
    free(hdq);
}

void oracle_grouped_ffn_e4m3(const uint8_t* xq_perm, const float* sx_perm, const int32_t* offsets,
                             int64_t E, const uint8_t* w1q, const float* s1, const uint8_t* w3q,
                             const float* s3, const uint8_t* w2q, const float* s2, int64_t D,
                             int64_t Dff, int act, double* h, uint16_t* hb, uint8_t* hq,
                             float* sh, double* y, int nthreads) {
    const int swiglu = (act == ORACLE_ACT_SWIGLU);
    grouped8_ctx c = {xq_perm, sx_perm, offsets, E, D, Dff, w1q, swiglu ? w3q : NULL, w2q,
                      s1, swiglu ? s3 : NULL, s2, act, h, hb, hq, sh, y};
    parallel_for((int64_t)offsets[E], nthreads, grouped8_rows, &c);
}

int oracle_layer_e4m3(const uint16_t* x, const uint16_t* wg, const double* bias,
                      const uint8_t* w1q, const float* s1, const uint8_t* w3q, const float* s3,
                      const uint8_t* w2q, const float* s2, int64_t N, int64_t D, int64_t E,
                      int64_t K, int64_t Dff, int mode, int act, double* L, int32_t* ids, double* w,
                      int32_t* offsets, int32_t* perm_src, int32_t* inv_perm, double* out,
                      int nthreads) {
    if (N < 0 || D < 1 || E < 1 || K < 1 || K > E || Dff < 1) return -1;
    const int64_t A = N * K;
    double* logits = L ? L : (double*)malloc(sizeof(double) * (size_t)(N * E > 0 ? N * E : 1));
    uint8_t* xq = (uint8_t*)malloc((size_t)(N * D > 0 ? N * D : 1));
    float* sx = (float*)malloc(sizeof(float) * (size_t)(N > 0 ? N : 1));
    uint8_t* xq_perm = (uint8_t*)malloc((size_t)(A * D > 0 ? A * D : 1));
    float* sx_perm = (float*)malloc(sizeof(float) * (size_t)(A > 0 ? A : 1));
    double* y = (double*)malloc(sizeof(double) * (size_t)(A * D > 0 ? A * D : 1));
    int rc = 0;
    oracle_logits(x, wg, bias, N, D, E, logits, nthreads);            /* O1 */
    rc |= oracle_select(logits, N, E, K, ids);                        /* O2 */
    oracle_weights(logits, ids, N, E, K, mode, w);                    /* O3 */
    rc |= oracle_offsets(ids, N, K, E, offsets);                      /* O4 */
    if (rc == 0) {
        rc |= oracle_place(ids, offsets, N, K, E, perm_src, inv_perm); /* O5 */
        oracle_quant_rows_e4m3(x, N, D, xq, sx, nthreads);            /* tokens -> e4m3 */
        for (int64_t r = 0; r < A; ++r) {
            memcpy(xq_perm + r * D, xq + (int64_t)perm_src[r] * D, (size_t)D);
            sx_perm[r] = sx[perm_src[r]];
        }
        oracle_grouped_ffn_e4m3(xq_perm, sx_perm, offsets, E, w1q, s1, w3q, s3, w2q, s2, D, Dff,
                                act, NULL, NULL, NULL, NULL, y, nthreads); /* O6 */
        oracle_combine(y, inv_perm, w, N, D, K, out);                 /* O7 */
    }
    if (!L) free(logits);
    free(xq);
    free(sx);
    free(xq_perm);
    free(sx_perm);
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
