/*
 * moe_oracle.h -- plain, slow, fp64 CPU oracle of one MoE layer's forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The GPU product path
 * never calls it, never links it, and shares no code with it.
 *
 * Every function is the plain definition of one step of the layer, evaluated
 * in double precision from bf16 inputs (each bf16 value converts exactly to
 * double).  Nothing is blocked, fused or reordered beyond the definition.
 *
 * Sources (page title, section):
 *   [Z]  "MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im)
 *        - 起手 "MoE 到底为什么难": the layer's dataflow figure
 *        - 第一层 "Router 与 Top-K 的算法细节": gate, top-K + softmax over the
 *          K selected, and the DeepSeek sigmoid + renormalise variant
 *        - 第二层 "Fused MoE Kernel 的两种范式", 范式 A Step 1-3: contiguous
 *          permutation, expert_offsets, per-expert two-GEMM FFN, un-permute
 *          with router weights
 *   [Y]  "MoE 大规模分布式推理工程实战：从 All-to-All 通信到动态专家放置"
 *        (ybb.press), 4.1 "Router 辅助损失的工程化实现": bias-free
 *        Linear(hidden, E) gate, additive per-expert bias before top-K
 *
 * Conventions: row-major contiguous arrays; bf16 arrays are raw uint16 bits.
 * Parity pins for each function live in the CPU test-suite; the header of
 * moe_oracle.c lists which property pins which function.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_SCORE_SOFTMAX_TOPK = 0, ORACLE_SCORE_SIGMOID_NORM = 1 };
enum { ORACLE_ACT_SILU = 0, ORACLE_ACT_SWIGLU = 1 };

/* Exact bf16 -> double conversion (bf16 is the top half of an IEEE binary32). */
double oracle_bf16_to_f64(uint16_t b);

/* O1 router logits [Z 第一层; Y 4.1]:
 *   L[t,e] = sum_d x[t,d] * Wg[e,d]  (+ bias[e] when bias != NULL).
 * x [N,D] bf16, wg [E,D] bf16, bias [E] double or NULL, L [N,E] double.
 * nthreads <= 0 uses every online core. */
void oracle_logits(const uint16_t* x, const uint16_t* wg, const double* bias,
                   int64_t N, int64_t D, int64_t E, double* L, int nthreads);

/* O2 top-K selection [Z 第一层 torch.topk]: per row, the K experts that come
 * first when ordered by (logit descending, expert index ascending), written in
 * that order.  Sigmoid mode selects on the logits too: sigmoid is monotone, so
 * the selected set and order are the same as on sigmoid(L).
 * L [N,E] double, ids [N,K] int32.  Returns 0, or -1 if K is not in 1..E. */
int oracle_select(const double* L, int64_t N, int64_t E, int64_t K, int32_t* ids);

/* O3 routing weights [Z 第一层]: with L_1 .. L_K the selected logits in order,
 *   softmax mode: w_k = exp(L_k - L_1) / sum_j exp(L_j - L_1)
 *   sigmoid mode: s_k = 1 / (1 + exp(-L_k)),  w_k = s_k / sum_j s_j
 *                 (uniform 1/K if every s_j underflows to 0).
 * L [N,E] double, ids [N,K] int32, w [N,K] double. */
void oracle_weights(const double* L, const int32_t* ids, int64_t N, int64_t E,
                    int64_t K, int mode, double* w);

/* O4 expert_offsets [Z 第二层 范式 A Step 1]: count[e] = #{(t,k): ids[t,k]=e},
 * offsets[0] = 0, offsets[e+1] = offsets[e] + count[e].  offsets has E+1
 * entries.  Returns 0, or -1 if an id is outside 0..E-1. */
int oracle_offsets(const int32_t* ids, int64_t N, int64_t K, int64_t E, int32_t* offsets);

/* O5 stable placement [Z 第二层 范式 A Step 1]: assignments are visited in
 * token order t = 0..N-1 and, within a token, k = 0..K-1; each goes to the
 * next free row of its expert's segment:
 *   r = offsets[e] + fill[e]++;  perm_src[r] = t;  inv_perm[t,k] = r.
 * perm_src [N*K], inv_perm [N,K].  Returns 0, or -1 on a bad id. */
int oracle_place(const int32_t* ids, const int32_t* offsets, int64_t N, int64_t K,
                 int64_t E, int32_t* perm_src, int32_t* inv_perm);

/* Row gather of the permuted token buffer: x_perm[r,:] = x[perm_src[r],:]
 * (bit copy of bf16 rows).  x [N,D], x_perm [rows,D]. */
void oracle_gather_rows(const uint16_t* x, const int32_t* perm_src, int64_t rows,
                        int64_t D, uint16_t* x_perm);

/* O6a expert FFN, first GEMM + activation [Z 第二层 范式 A Step 2]:
 * for the R rows of one expert,
 *   g = W1 x,  SwiGLU: h = silu(g) * (W3 x);  SiLU: h = silu(g),
 *   silu(g) = g / (1 + exp(-g)).
 * xrows [R,D] bf16, w1/w3 [Dff,D] bf16 (w3 ignored for SiLU), h [R,Dff] double. */
void oracle_expert_up(const uint16_t* xrows, int64_t R, const uint16_t* w1,
                      const uint16_t* w3, int64_t D, int64_t Dff, int act,
                      double* h, int nthreads);

/* O6b expert FFN, second GEMM [Z 第二层 范式 A Step 2]: y = W2 h.
 * h [R,Dff] double, w2 [D,Dff] bf16, y [R,D] double. */
void oracle_expert_down(const double* h, int64_t R, const uint16_t* w2, int64_t D,
                        int64_t Dff, double* y, int nthreads);

/* Same as oracle_expert_down with h given as bf16 (used to check the second
 * GEMM in isolation on the exact bf16 activations a GPU run produced). */
void oracle_expert_down_bf16(const uint16_t* h, int64_t R, const uint16_t* w2,
                             int64_t D, int64_t Dff, double* y, int nthreads);

/* O6 over all experts: rows offsets[e]..offsets[e+1]-1 of x_perm use expert e's
 * weights w1[e], w3[e] ([E,Dff,D]) and w2[e] ([E,D,Dff]).
 * h [rows,Dff] double (may be NULL to skip keeping it), y [rows,D] double. */
void oracle_grouped_ffn(const uint16_t* x_perm, const int32_t* offsets, int64_t E,
                        const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                        int64_t D, int64_t Dff, int act, double* h, double* y,
                        int nthreads);

/* O7 un-permute + weighted sum [Z 第二层 范式 A Step 3; 起手 dataflow]:
 *   out[t,:] = sum_{k=0}^{K-1} w[t,k] * y[inv_perm[t,k], :].
 * y [rows,D] double, inv_perm [N,K], w [N,K] double, out [N,D] double. */
void oracle_combine(const double* y, const int32_t* inv_perm, const double* w,
                    int64_t N, int64_t D, int64_t K, double* out);

/* The whole layer O1..O7 on one set of inputs.  Every intermediate is fp64.
 * Outputs: ids [N,K], w [N,K], offsets [E+1], perm_src [N*K], inv_perm [N,K],
 * out [N,D] double.  L (optional, [N,E]) receives the logits when non-NULL.
 * Returns 0, or -1 on bad arguments. */
int oracle_layer(const uint16_t* x, const uint16_t* wg, const double* bias,
                 const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                 int64_t N, int64_t D, int64_t E, int64_t K, int64_t Dff,
                 int mode, int act, double* L, int32_t* ids, double* w,
                 int32_t* offsets, int32_t* perm_src, int32_t* inv_perm,
                 double* out, int nthreads);

/* Padded placement, paradigm B ("MoE 推理完整机制", 第二层 范式 B: every
 * expert gets a fixed capacity C of rows; tokens beyond it are dropped):
 * assignments are visited in token order t = 0..N-1, k = 0..K-1, and each
 * takes the next free row of its expert's block while one is left,
 *   fill[e] < C:  slot[t,k] = e*C + fill[e]++;   otherwise slot[t,k] = -1.
 * kept[e] = rows used in expert e's block (min(count, C)).  Returns 0, or -1
 * on a bad id or C < 0. */
int oracle_place_padded(const int32_t* ids, int64_t N, int64_t K, int64_t E, int64_t C,
                        int32_t* slot, int32_t* kept);

/* Weighted sum over the kept assignments only:
 *   out[t,:] = sum_{k : slot[t,k] >= 0} w[t,k] * y[slot[t,k], :].
 * (Paradigm B; with no dropped slot this is oracle_combine.) */
void oracle_combine_kept(const double* y, const int32_t* slot, const double* w, int64_t N,
                         int64_t D, int64_t K, double* out);

/* Routing statistics and the online bias update ("MoE 大规模分布式推理工程实战",
 * 4.1 Router 辅助损失的工程化实现: _update_load_balance_stats, then
 * load_balance_loss), in that order, from one batch's expert_offsets:
 *   frac[e] = (offsets[e+1] - offsets[e]) / offsets[E]
 *   ema[e]  = decay * ema[e] + (1 - decay) * frac[e]          (in place)
 *   f[e]    = ema[e] / sum_j ema[j]
 *   kl      = sum_e f[e] * log(f[e] * E + 1e-9)       (f against uniform 1/E)
 *   bias[e] += step * (E * f[e] - 1)                  (when bias != NULL)
 * A batch with no assignments (offsets[E] == 0) changes nothing and gives
 * kl = 0.  Returns kl. */
double oracle_routing_stats(const int32_t* offsets, int64_t E, double decay, double step,
                            double* ema, double* bias);

/* Number of threads a call with nthreads <= 0 would use. */
int oracle_default_threads(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ORACLE_H */
