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

/* ---------------------------------------------------------------------------
 * FP8 expert GEMMs ("MoE 推理完整机制", 第四层 DeepGEMM & MegaMoE: FP8 expert
 * weights; 第三层 DeepEP: FP8 token hidden states halve the bytes moved).
 * The pages name the format only; the reading taken here: e4m3 codes with one
 * power-of-two scale per row -- per output channel for a weight matrix, per
 * token (or per permuted row) for activations -- so that the contraction is a
 * plain FP8 dot product and the scales are exact factors outside it.
 * ------------------------------------------------------------------------- */

/* e4m3 (the "fn" variant): sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (m/8 * 2^-6); no infinities; codes
 * 0x7f / 0xff are NaN; the largest finite magnitude is 448 (code 0x7e). */
double oracle_e4m3_decode(uint8_t c);

/* The e4m3 code nearest to v, ties to the code with an even mantissa, and
 * magnitudes beyond 448 saturate to +-448; the sign of v is kept (so a value
 * that rounds to zero keeps its sign).  v must not be NaN. */
uint8_t oracle_e4m3_encode(double v);
void oracle_e4m3_encode_array(const double* v, int64_t n, uint8_t* out);

/* v rounded to bf16 (8 significant bits, binary32 exponent range), to nearest
 * with ties to even, in one rounding from the exact double; returns the bits. */
uint16_t oracle_f64_to_bf16(double v);

/* Row scale exponent: the smallest integer k >= -126 with amax <= 448 * 2^k
 * (amax == 0 gives -126). */
int oracle_e4m3_scale_exp(double amax);

/* Per-row quantisation of a bf16 matrix [rows, cols]: for row r,
 *   amax = max_c |src[r,c]|,  k = oracle_e4m3_scale_exp(amax),
 *   scale[r] = 2^k,  q[r,c] = oracle_e4m3_encode(src[r,c] * 2^-k).
 * src * 2^-k is exact, so q is the one rounding of the method. */
void oracle_quant_rows_e4m3(const uint16_t* src, int64_t rows, int64_t cols, uint8_t* q,
                            float* scale, int nthreads);

/* Dequantised values: out[r,c] = decode(q[r,c]) * scale[r] (exact). */
void oracle_dequant_rows_e4m3(const uint8_t* q, const float* scale, int64_t rows, int64_t cols,
                              double* out);

/* FP8 expert FFN, first GEMM + activation, for the R rows of one expert:
 * the definition of oracle_expert_up on the dequantised operands
 *   x^[r,d] = decode(xq[r,d]) sx[r],  W1^[j,d] = decode(w1q[j,d]) s1[j]  (W3 alike).
 * xq [R,D], sx [R], w1q/w3q [Dff,D], s1/s3 [Dff]; h [R,Dff] double. */
void oracle_expert_up_e4m3(const uint8_t* xq, const float* sx, int64_t R, const uint8_t* w1q,
                           const float* s1, const uint8_t* w3q, const float* s3, int64_t D,
                           int64_t Dff, int act, double* h, int nthreads);

/* FP8 second GEMM: y[r,d] = sum_j W2^[d,j] h^[r,j] with
 *   h^[r,j] = decode(hq[r,j]) sh[r],  W2^[d,j] = decode(w2q[d,j]) s2[d].
 * hq [R,Dff], sh [R], w2q [D,Dff], s2 [D]; y [R,D] double. */
void oracle_expert_down_e4m3(const uint8_t* hq, const float* sh, int64_t R, const uint8_t* w2q,
                             const float* s2, int64_t D, int64_t Dff, double* y, int nthreads);

/* FP8 FFN over all experts (rows offsets[e]..offsets[e+1]-1 belong to expert
 * e; w1q/w3q [E,Dff,D], s1/s3 [E,Dff], w2q [E,D,Dff], s2 [E,D]).  Per row:
 *   h  = the first GEMM + activation on the dequantised operands (fp64),
 *   hb = h rounded to bf16,
 *   hq, sh = per-row quantisation of hb,
 *   y  = the second GEMM on hq, sh.
 * Any of h, hb, hq, sh may be NULL; y [rows,D] double is required. */
void oracle_grouped_ffn_e4m3(const uint8_t* xq_perm, const float* sx_perm, const int32_t* offsets,
                             int64_t E, const uint8_t* w1q, const float* s1, const uint8_t* w3q,
                             const float* s3, const uint8_t* w2q, const float* s2, int64_t D,
                             int64_t Dff, int act, double* h, uint16_t* hb, uint8_t* hq,
                             float* sh, double* y, int nthreads);

/* The whole layer with FP8 experts: routing O1..O5 exactly as oracle_layer
 * (bf16 router), then xq, sx = per-row quantisation of x (one scale per
 * token), rows gathered in placement order with their token's scale, the FP8
 * FFN above, and the combine O7 in fp64.  Returns 0, or -1 on bad arguments. */
int oracle_layer_e4m3(const uint16_t* x, const uint16_t* wg, const double* bias,
                      const uint8_t* w1q, const float* s1, const uint8_t* w3q, const float* s3,
                      const uint8_t* w2q, const float* s2, int64_t N, int64_t D, int64_t E,
                      int64_t K, int64_t Dff, int mode, int act, double* L, int32_t* ids, double* w,
                      int32_t* offsets, int32_t* perm_src, int32_t* inv_perm, double* out,
                      int nthreads);

/* Number of threads a call with nthreads <= 0 would use. */
int oracle_default_threads(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ORACLE_H */
