/*
 * moe.h -- C ABI of a single-GPU Mixture-of-Experts layer for GB300 (sm_103a).
 *
 * The layer, as "MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切"
 * (zoe.im) states it in its opening dataflow figure (起手 "MoE 到底为什么难"):
 * N tokens of width D are scored by a router, each token picks its top-K of E
 * experts, tokens are regrouped by expert, every expert runs a two-GEMM FFN on
 * its rows, and the results return to token order as a router-weighted sum.
 * The five compute entry points follow the split that page's vLLM modular
 * kernel paragraph describes (prepare = route + permute, fused_experts =
 * grouped FFN, finalize = combine), plus the whole layer in one call.
 *
 * Conventions for every entry point
 *   - Plain pointers, no CUDA or framework types.  Tensors are row-major and
 *     contiguous.  moe_bf16 holds raw IEEE bfloat16 bits.
 *   - Every tensor pointer, including the workspace, is a DEVICE pointer of
 *     the current CUDA device and must be 16-byte aligned.  The caller owns
 *     every buffer: inputs, outputs and workspace.  The library allocates no
 *     device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work and return without synchronising, except
 *     moe_read_device_error.
 *   - `ws` / `ws_bytes`: caller-allocated scratch of at least
 *     moe_workspace_size(<op>, ...) bytes.  Its first 256 bytes are a header
 *     holding the device error word; the header must be zeroed once before
 *     first use (moe_clear_device_error does that) and is never cleared by the
 *     compute calls, so a device error stays visible until cleared.
 *   - Host-side validation returns MOE_ERR_INVALID_ARG (bad sizes, NULL
 *     required pointers, misalignment), MOE_ERR_WORKSPACE (ws_bytes too small)
 *     or MOE_ERR_UNSUPPORTED (a valid combination this build does not run).
 *     Nothing is enqueued when validation fails.  A failed launch returns
 *     MOE_ERR_CUDA.  moe_last_error_detail() describes the last failure of
 *     the calling thread.
 *   - Problems seen on the device (an expert id outside 0..E-1, a row index
 *     outside the permuted buffer, a pipeline wait that exceeded its time
 *     limit) never trap: the kernel skips the access or abandons the tile,
 *     records the problem in the workspace's error word and returns.  Read it
 *     with moe_read_device_error.
 *   - N = 0 (or total_rows = 0) is a valid no-op returning MOE_OK.
 *
 * Size limits checked by every call: 1 <= K <= E, E <= 1024, K <= 32,
 * D and D_ffn positive multiples of 64, N >= 0, N*K < 2^31, rows*D < 2^40.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16; /* raw bfloat16 bits */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_UNSUPPORTED = 2,
    MOE_ERR_WORKSPACE = 3,
    MOE_ERR_CUDA = 4,
    MOE_ERR_DEVICE_BOUNDS = 5,
    MOE_ERR_DEVICE_TIMEOUT = 6
} moe_status;

/* Router score functions ("MoE 推理完整机制", 第一层 Router 与 Top-K):
 *   SOFTMAX_TOPK  -- top-K of the logits, then softmax over those K only;
 *   SIGMOID_NORM  -- DeepSeek variant: sigmoid of each logit, top-K, then
 *                    divide by the sum of the K selected sigmoids. */
typedef enum { MOE_SCORE_SOFTMAX_TOPK = 0, MOE_SCORE_SIGMOID_NORM = 1 } moe_score_mode;

/* Expert FFN activation:
 *   SILU    -- y = W2 silu(W1 x)                (w3 unused, may be NULL)
 *   SWIGLU  -- y = W2 (silu(W1 x) * (W3 x))     (gate W1, up W3, down W2) */
typedef enum { MOE_ACT_SILU = 0, MOE_ACT_SWIGLU = 1 } moe_act;

/* Bytes of workspace an operation needs.  `op` is one of "route", "permute",
 * "route_permute", "ffn", "combine", "layer".  Returns 0 for an unknown op or
 * invalid sizes.  Arguments a given op does not use are ignored (pass 0):
 *   route   N, D, E (fp32 split-K partial logits)
 *   permute N, E    (per-block expert histograms)
 *   route_permute N, D, E (both of the above)
 *   ffn     N = total_rows of the permuted buffer, D, E, Dff (fp32 split-K
 *           partials, used when the call is too small to fill the GPU)
 *   combine -       (header only)
 *   layer   N, D, E, K, Dff (every intermediate of moe_layer_forward)
 *   layer_e4m3  the same for moe_layer_forward_e4m3 (0 unless D and Dff are
 *           multiples of 128)
 * The sizes do not depend on the device. */
size_t moe_workspace_size(const char* op, int N, int D, int E, int K, int Dff);

/* Router: logits, top-K selection and routing weights.
 * ("MoE 推理完整机制", 第一层: logits = x W_gate^T from a bias-free
 * Linear(D -> E); torch.topk then softmax over the K selected, or the DeepSeek
 * sigmoid + renormalise variant; "MoE 大规模分布式推理工程实战", 4.1: an
 * optional per-expert bias added to the logits before top-K.)
 *   x         [N,D]  bf16 tokens
 *   w_gate    [E,D]  bf16 gate weight (nn.Linear layout)
 *   bias      [E]    fp32 or NULL; added to every row's logits before
 *                    selection and used in the weights
 *   topk_ids  [N,K]  int32 out: selected experts ordered by (logit desc,
 *                    expert index asc); equal logits -> lower index first
 *   topk_w    [N,K]  fp32 out: routing weights, summing to 1 per token
 *   logits_out[N,E]  fp32 out or NULL: the biased fp32 logits the selection
 *                    used (for parity checks)
 * Logits accumulate in fp32 on the tensor cores; when the token tiles alone
 * would leave SMs idle the reduction over D is split and the fp32 partials
 * are summed in a fixed order, so results are deterministic on a device. */
moe_status moe_route(const moe_bf16* x, const moe_bf16* w_gate, const float* bias,
                     int N, int D, int E, int K, int mode,
                     int32_t* topk_ids, float* topk_w, float* logits_out,
                     void* ws, size_t ws_bytes, void* stream);

/* Permutation into contiguous per-expert segments ("MoE 推理完整机制",
 * 第二层 范式 A Step 1): per-expert counts, expert_offsets = their exclusive
 * prefix sum, then a stable scatter -- assignment (t,k) goes to row
 *   r = expert_offsets[e] + #{(t',k') before (t,k) in token-major order with e}
 * so each segment lists its tokens in ascending order.
 *   topk_ids       [N,K]     int32 in (ids outside 0..E-1 are skipped and
 *                            flagged MOE_ERR_DEVICE_BOUNDS)
 *   expert_offsets [E+1]     int32 out; expert_offsets[E] = N*K
 *   perm_src       [N*K]     int32 out: token of each permuted row
 *   inv_perm       [N,K]     int32 out: permuted row of each (t,k)
 *   x_perm         [N*K,D]   bf16 out: x_perm[r] = x[perm_src[r]] (bit copy) */
moe_status moe_permute(const moe_bf16* x, const int32_t* topk_ids, int N, int D, int E, int K,
                       int32_t* expert_offsets, int32_t* perm_src, int32_t* inv_perm,
                       moe_bf16* x_perm, void* ws, size_t ws_bytes, void* stream);

/* The permutation's indices only (expert_offsets, perm_src, inv_perm as in
 * moe_permute) without the row copy: for moe_grouped_ffn_gathered, which
 * reads the token rows through perm_src.  Workspace as for "permute". */
moe_status moe_permute_indices(const int32_t* topk_ids, int N, int E, int K, int32_t* expert_offsets,
                               int32_t* perm_src, int32_t* inv_perm, void* ws, size_t ws_bytes,
                               void* stream);

/* moe_route followed by moe_permute, as one call: the "prepare" stage of the
 * prepare / fused_experts / finalize split ("MoE 推理完整机制", 第二层
 * "vLLM 的 Fused MoE Modular Kernel"), i.e. 第一层 top-K and weights, then
 * 第二层 范式 A Step 1.  Arguments and outputs as for the two calls.  A
 * decode-sized call (up to 8 tokens, N*K <= 256) selects the top-K and
 * permutes in a single launch (MOE_FUSED_ROUTE_PERMUTE=0 in the environment
 * turns that off); the results are bit for bit those of the two calls.
 *   ws  moe_workspace_size("route_permute", N, D, E, K, 0) bytes
 * Errors as for moe_route and moe_permute. */
moe_status moe_route_permute(const moe_bf16* x, const moe_bf16* w_gate, const float* bias,
                             int N, int D, int E, int K, int mode,
                             int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                             int32_t* perm_src, int32_t* inv_perm, moe_bf16* x_perm,
                             void* ws, size_t ws_bytes, void* stream);

/* moe_permute without a caller workspace.  The pages have no counterpart:
 * this exists for callers that cannot allocate device memory when they run
 * the layer -- runtimes that plan every buffer in advance and forbid
 * allocation during execution (for example the enqueue step of a plugin in a
 * pre-built inference engine), or code that must not risk the device-wide
 * synchronisation a cudaMalloc can cause.  It computes exactly what
 * moe_permute computes, with the same arguments minus the workspace.
 *   - Scratch lives in a fixed array of device global memory owned by the
 *     library: 1,048,576 int32 (4 MiB), held on every GPU that loads the
 *     library until the process exits.  A call needs E * ceil(N/16) + E of
 *     them; larger calls return MOE_ERR_UNSUPPORTED (detail in
 *     moe_last_error_detail) and enqueue nothing.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: calls after a cudaDeviceReset are not supported.
 *   - Sizes are validated exactly as moe_permute validates them
 *     (MOE_ERR_INVALID_ARG), before the scratch limit.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; calls whose kernels overlap on the GPU (different streams
 *     without ordering between them) race on it and give wrong results.
 *   - There is no error word: ids outside 0..E-1 are skipped, their inv_perm
 *     entry is -1 and expert_offsets[E] counts only the valid assignments. */
moe_status moe_permute_static_scratch(const moe_bf16* x, const int32_t* topk_ids, int N, int D,
                                      int E, int K, int32_t* expert_offsets, int32_t* perm_src,
                                      int32_t* inv_perm, moe_bf16* x_perm, void* stream);

/* Grouped expert FFN ("MoE 推理完整机制", 第二层 范式 A Step 2 and
 * "关键 kernel：Grouped GEMM"): one persistent launch per GEMM covers every
 * expert's ragged segment; expert e owns rows expert_offsets[e] ..
 * expert_offsets[e+1]-1 of x_perm.
 *   GEMM1 + activation: h = silu(x W1_e^T) * (x W3_e^T)  (SiLU: silu(x W1_e^T))
 *   GEMM2:              y = h W2_e^T
 * fp32 accumulation on the tensor cores; h and y_perm are rounded to bf16.
 *   x_perm         [total_rows,D]   bf16
 *   expert_offsets [E+1]            int32, non-decreasing, offsets[0] = 0,
 *                                   offsets[E] = total_rows
 *   w1, w3         [E,Dff,D]        bf16 (w3 NULL allowed only for SILU)
 *   w2             [E,D,Dff]        bf16
 *   h              [total_rows,Dff] bf16 out (intermediate activations)
 *   y_perm         [total_rows,D]   bf16 out
 * Decode-sized SwiGLU calls (at most 32 rows per touched expert, from 16 rows
 * total) run both GEMMs in one persistent cooperative launch ("MoE 推理完整机制",
 * 第四层 MegaMoE): identical results, fewer launches.  MOE_FUSED_DECODE=0 in
 * the environment turns it off, =1 uses it at any decode size. */
moe_status moe_grouped_ffn(const moe_bf16* x_perm, const int32_t* expert_offsets, int total_rows,
                           const moe_bf16* w1, const moe_bf16* w3, const moe_bf16* w2,
                           int E, int D, int Dff, int act,
                           moe_bf16* h, moe_bf16* y_perm, void* ws, size_t ws_bytes,
                           void* stream);

/* moe_grouped_ffn with the permutation fused into GEMM1's operand load
 * ("MoE 推理完整机制", 第二层 "优化亮点": the permute is one scatter/gather
 * pass over HBM; here that pass is folded into the GEMM): row r of the
 * permuted buffer is token perm_src[r] of x [N,D], copied straight into the
 * GEMM's shared-memory tile, so no x_perm is written or read.  Results are
 * bit-identical to moe_permute + moe_grouped_ffn.  perm_src entries outside
 * 0..N-1 are skipped and flagged MOE_ERR_DEVICE_BOUNDS.  Other arguments and
 * the workspace as in moe_grouped_ffn.  Measured on GB300 it is slower than
 * the separate copy (the 16-byte row copies in the operand load cannot keep
 * enough bytes in flight while the weights stream from HBM). */
moe_status moe_grouped_ffn_gathered(const moe_bf16* x, int N, const int32_t* perm_src,
                                    const int32_t* expert_offsets, int total_rows, const moe_bf16* w1,
                                    const moe_bf16* w3, const moe_bf16* w2, int E, int D, int Dff, int act,
                                    moe_bf16* h, moe_bf16* y_perm, void* ws, size_t ws_bytes,
                                    void* stream);

/* Un-permute and weighted sum ("MoE 推理完整机制", 第二层 范式 A Step 3):
 *   out[t,:] = bf16( sum_{k=0..K-1} topk_w[t,k] * y_perm[inv_perm[t,k], :] )
 * summed in fp32 in k order, rounded once to bf16 (nearest-even).
 *   y_perm [N*K,D] bf16, inv_perm [N,K] int32 (entries outside 0..N*K-1 are
 *   skipped and flagged), topk_w [N,K] fp32, out [N,D] bf16. */
moe_status moe_combine(const moe_bf16* y_perm, const int32_t* inv_perm, const float* topk_w,
                       int N, int D, int K, moe_bf16* out, void* ws, size_t ws_bytes,
                       void* stream);

/* The whole layer: route -> permute -> grouped FFN -> combine, all on
 * `stream`, every intermediate inside `ws` (size moe_workspace_size("layer")).
 * With MOE_GATHER=1 in the environment the permutation runs fused into GEMM1
 * (moe_permute_indices + moe_grouped_ffn_gathered, identical results, x_perm
 * left unwritten); the default is the row copy, which is faster on GB300.
 *
 * Decode batches of up to 4 tokens (bf16 experts, and e4m3 ones in
 * moe_layer_forward_e4m3) with N*K <= 64 and E <= 256 run as ONE cooperative
 * launch ("MoE 推理完整机制", 第四层 "DeepGEMM 的 MegaMoE Kernel": the decode
 * step's expert work as one persistent kernel): router logits, top-K,
 * placement, GEMM1 + activation, GEMM2 and the combine, phases separated by
 * two grid barriers whose words live in the workspace header (bytes
 * 128..255).  Both GEMMs run on the tensor cores (mma.sync) with the weight
 * rows as the 16-row operand and the expert's token rows as the 8 columns,
 * reading the weights in 32-byte pieces: w1, w3, w2 (and w1q, w3q, w2q) must
 * start on a 32-byte boundary, which every tensor allocation does, else the
 * call runs the chain of launches.  Every intermediate is written as by the chain of
 * launches; routing, placement and x_perm are bit-identical to it, h /
 * y_perm / out agree within bf16 rounding (the GEMM sums run in another
 * order).  The token limits are where the one launch measured faster on
 * GB300 (Qwen3-shaped layer).  MOE_LAYER_DECODE=0 selects the chain of
 * launches, MOE_LAYER_DECODE_MAX_N=n (<= 8) sets the token limit,
 * MOE_LAYER_DECODE_L2_MB (default 64) bounds the W2 bytes prefetched into L2
 * during GEMM1, and MOE_LAYER_DECODE_W2_SMEM=1 stages each CTA's W2 rows in
 * shared memory instead (where they fit).  A barrier wait that runs out
 * records MOE_ERR_DEVICE_TIMEOUT; clear the header (moe_clear_device_error)
 * before the next call on that workspace.
 *
 * Argument meanings as above; out [N,D] bf16.  No host synchronisation. */
moe_status moe_layer_forward(const moe_bf16* x, const moe_bf16* w_gate, const float* bias,
                             const moe_bf16* w1, const moe_bf16* w3, const moe_bf16* w2,
                             int N, int D, int E, int K, int Dff, int mode, int act,
                             moe_bf16* out, void* ws, size_t ws_bytes, void* stream);

/* ---- Paradigm B: fixed capacity per expert ("MoE 推理完整机制", 第二层
 * 范式 B (Padded): every expert gets the same number of rows, `capacity`;
 * assignments beyond it are dropped; the padded buffer is one uniform batched
 * FFN).  Expert e owns rows e*capacity .. e*capacity+capacity-1, filled with
 * its assignments in token order (t, then k); an assignment that finds its
 * expert's block full is dropped: slot = -1, and it adds nothing to its
 * token's output (the kept weights are not renormalised).  Unused rows of a
 * block are zero.  The FFN step is moe_grouped_ffn with expert_offsets[e] =
 * e*capacity and total_rows = E*capacity. */

/* ceil(capacity_factor * N * K / E) -- the page's capacity_per_expert with
 * capacity_factor 1.5 -- or -1 on invalid arguments. */
int moe_capacity(int N, int E, int K, float capacity_factor);

/* Workspace bytes for "permute", "combine" or "layer" of the padded paradigm
 * (0 on invalid sizes). */
size_t moe_workspace_size_padded(const char* op, int N, int D, int E, int K, int Dff, int capacity);

/* Padded placement.  Outputs: expert_offsets [E+1] (= e*capacity), kept [E]
 * (rows used per block, min(count, capacity)), slot [N,K] (row of each
 * assignment or -1), x_pad [E*capacity, D] (token rows, zero padding).
 * Expert ids outside 0..E-1 are skipped (slot -1) and flagged. */
moe_status moe_permute_padded(const moe_bf16* x, const int32_t* topk_ids, int N, int D, int E, int K,
                              int capacity, int32_t* expert_offsets, int32_t* kept, int32_t* slot,
                              moe_bf16* x_pad, void* ws, size_t ws_bytes, void* stream);

/* out[t,:] = bf16( sum over k with slot[t,k] >= 0 of topk_w[t,k] * y_pad[slot[t,k], :] ),
 * fp32 in k order.  slot -1 = dropped (no error); other rows outside
 * 0..E*capacity-1 are skipped and flagged. */
moe_status moe_combine_padded(const moe_bf16* y_pad, const int32_t* slot, const float* topk_w, int N,
                              int D, int K, int E, int capacity, moe_bf16* out, void* ws,
                              size_t ws_bytes, void* stream);

/* The whole layer in the padded paradigm (route -> padded placement ->
 * grouped FFN over the E*capacity rows -> combine of the kept assignments). */
moe_status moe_layer_forward_padded(const moe_bf16* x, const moe_bf16* w_gate, const float* bias,
                                    const moe_bf16* w1, const moe_bf16* w3, const moe_bf16* w2,
                                    int N, int D, int E, int K, int Dff, int mode, int act,
                                    int capacity, moe_bf16* out, void* ws, size_t ws_bytes,
                                    void* stream);

/* Byte offsets of moe_layer_forward_padded's intermediates in its workspace:
 * topk_ids, topk_w, expert_offsets, kept, slot, x_pad, h, y_pad. */
int moe_layer_padded_workspace_layout(int N, int D, int E, int K, int Dff, int capacity,
                                      size_t offsets_out[8]);

/* ---- FP8 experts ("MoE 推理完整机制", 第四层 DeepGEMM & MegaMoE: FP8 expert
 * weights; 第三层 (DeepEP): token hidden states moved in FP8 at half the
 * bytes).  The pages fix no format or scaling; this library uses e4m3 codes
 * (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest finite 448,
 * no infinities) with one power-of-two fp32 scale per ROW:
 *   scale = 2^k, k = the smallest integer >= -126 with max|row| <= 448 * 2^k,
 *   code  = e4m3(x * 2^-k), round to nearest even, saturating at +-448.
 * A weight matrix row is one output channel (W1/W3: [E*Dff] rows of D codes,
 * W2: [E*D] rows of Dff codes); activations have one scale per token (x) or
 * per permuted row (h).  The GEMMs run on the tensor cores in e4m3 with fp32
 * accumulation (tcgen05 kind::f8f6f4) and multiply each accumulator by its
 * row's and column's scales, which are exact factors.  The router stays bf16.
 * D and Dff must be multiples of 128 for every e4m3 call. */

/* Per-row e4m3 quantisation of a bf16 matrix [rows, cols] (cols a positive
 * multiple of 16): q [rows, cols] uint8 codes, scale [rows] fp32 (2^k as
 * above).  Used once for the expert weights (a [E,Dff,D] tensor is rows =
 * E*Dff, cols = D) and by the e4m3 layer for tokens and hidden activations. */
moe_status moe_quantize_e4m3(const moe_bf16* src, long long rows, int cols, uint8_t* q, float* scale,
                             void* stream);

/* moe_permute on e4m3 token rows (D codes each; D a multiple of 128).  The
 * token scales stay in token order: row r of xq_perm uses x_scale[perm_src[r]]. */
moe_status moe_permute_e4m3(const uint8_t* xq, const int32_t* topk_ids, int N, int D, int E, int K,
                            int32_t* expert_offsets, int32_t* perm_src, int32_t* inv_perm,
                            uint8_t* xq_perm, void* ws, size_t ws_bytes, void* stream);

/* Grouped expert FFN with e4m3 operands; workspace as moe_workspace_size("ffn").
 *   xq_perm        [total_rows,D]   e4m3 codes
 *   x_scale        fp32: scale of row r is x_scale[x_scale_index[r]], or
 *                  x_scale[r] when x_scale_index is NULL (pass perm_src and the
 *                  per-token scales of moe_quantize_e4m3 on x)
 *   w1q, w3q       [E,Dff,D] e4m3, w1_scale/w3_scale [E,Dff] fp32
 *                  (w3q, w3_scale may be NULL for SILU)
 *   w2q            [E,D,Dff] e4m3, w2_scale [E,D] fp32
 *   h              [total_rows,Dff] bf16 out: silu(g)*u (or silu(g)), with
 *                  g = sum_d x^ W1^ over the dequantised operands, in fp32
 *   hq, h_scale    [total_rows,Dff] e4m3 / [total_rows] fp32 out: h quantised
 *                  per row (the second GEMM's input)
 *   y_perm         [total_rows,D]   bf16 out
 * With MOE_FUSED_DECODE=1 decode-sized SwiGLU calls run GEMM1, the h
 * quantisation and GEMM2 in one persistent launch (bit-identical outputs);
 * the default is the separate launches, which measured faster on GB300. */
moe_status moe_grouped_ffn_e4m3(const uint8_t* xq_perm, const float* x_scale, const int32_t* x_scale_index,
                                const int32_t* expert_offsets, int total_rows, const uint8_t* w1q,
                                const float* w1_scale, const uint8_t* w3q, const float* w3_scale,
                                const uint8_t* w2q, const float* w2_scale, int E, int D, int Dff, int act,
                                moe_bf16* h, uint8_t* hq, float* h_scale, moe_bf16* y_perm, void* ws,
                                size_t ws_bytes, void* stream);

/* moe_grouped_ffn_e4m3 with the permutation fused into GEMM1: row r reads
 * token perm_src[r] of xq [N,D] (codes) and its scale x_scale[perm_src[r]]. */
moe_status moe_grouped_ffn_e4m3_gathered(const uint8_t* xq, const float* x_scale, int N,
                                         const int32_t* perm_src, const int32_t* expert_offsets,
                                         int total_rows, const uint8_t* w1q, const float* w1_scale,
                                         const uint8_t* w3q, const float* w3_scale, const uint8_t* w2q,
                                         const float* w2_scale, int E, int D, int Dff, int act, moe_bf16* h,
                                         uint8_t* hq, float* h_scale, moe_bf16* y_perm, void* ws,
                                         size_t ws_bytes, void* stream);

/* The whole layer with e4m3 experts: bf16 router -> per-token e4m3 tokens ->
 * permutation of the codes -> e4m3 grouped FFN -> bf16 combine.  Workspace
 * moe_workspace_size("layer_e4m3", N, D, E, K, Dff).  Decode batches (up to
 * 4 tokens by default) run as one launch, as moe_layer_forward describes;
 * the token codes, their scales and their permutation are bit-identical to
 * the chain's, h is quantised by the same row rule before GEMM2. */
moe_status moe_layer_forward_e4m3(const moe_bf16* x, const moe_bf16* w_gate, const float* bias,
                                  const uint8_t* w1q, const float* w1_scale, const uint8_t* w3q,
                                  const float* w3_scale, const uint8_t* w2q, const float* w2_scale, int N,
                                  int D, int E, int K, int Dff, int mode, int act, moe_bf16* out, void* ws,
                                  size_t ws_bytes, void* stream);

/* Byte offsets of moe_layer_forward_e4m3's intermediates in its workspace:
 * topk_ids, topk_w, expert_offsets, perm_src, inv_perm, xq, x_scale, xq_perm,
 * h, hq, h_scale, y_perm.  0 on success, -1 on invalid sizes. */
int moe_layer_e4m3_workspace_layout(int N, int D, int E, int K, int Dff, size_t offsets_out[12]);

/* Number of kernels moe_layer_forward_e4m3 launches, or -1 on invalid sizes. */
int moe_layer_launches_e4m3(int N, int D, int E, int K, int Dff, int act);

/* On-GPU routing statistics and the online bias step ("MoE 大规模分布式推理
 * 工程实战", 4.1 Router 辅助损失的工程化实现), from one batch's expert_offsets:
 *   frac[e] = (expert_offsets[e+1] - expert_offsets[e]) / expert_offsets[E]
 *   ema[e]  = decay * ema[e] + (1 - decay) * frac[e]              (in place)
 *   f[e]    = ema[e] / sum_j ema[j]
 *   *kl_out = sum_e f[e] * log(E * f[e] + 1e-9)    (KL of f to uniform)
 *   bias[e] += bias_step * (E * f[e] - 1)           (when bias != NULL)
 * The page prints bias_step = +0.1; a negative step lowers the bias of
 * experts that receive more than their share (the balancing direction).
 * `bias` can be the router bias moe_route adds.  A batch without assignments
 * changes nothing.  ema [E], bias [E] fp32 device arrays; kl_out fp32 or
 * NULL.  Needs no workspace; enqueues one kernel on `stream`. */
moe_status moe_routing_stats(const int32_t* expert_offsets, int E, float decay, float bias_step,
                             float* ema, float* bias, float* kl_out, void* stream);

/* Number of kernels moe_layer_forward (capacity < 0) or
 * moe_layer_forward_padded (capacity >= 0) launches for these sizes on the
 * current device (with weights on 32-byte boundaries), or -1 on invalid
 * sizes. */
int moe_layer_launches(int N, int D, int E, int K, int Dff, int act, int capacity);

/* Byte offsets of the layer's intermediates inside its workspace, so a caller
 * can inspect them after moe_layer_forward (order: topk_ids, topk_w,
 * expert_offsets, perm_src, inv_perm, x_perm, h, y_perm).  Returns 0 on
 * success, -1 on invalid sizes. */
int moe_layer_workspace_layout(int N, int D, int E, int K, int Dff, size_t offsets_out[8]);

/* Synchronises `stream`, then returns MOE_OK, MOE_ERR_DEVICE_BOUNDS or
 * MOE_ERR_DEVICE_TIMEOUT from the workspace's error word (timeout wins when
 * both are set), or MOE_ERR_CUDA if the stream reported an error. */
moe_status moe_read_device_error(const void* ws, void* stream);

/* Zeroes the workspace header (error word and debug flags) on `stream`. */
moe_status moe_clear_device_error(void* ws, void* stream);

/* Test hook: stores `flags` in the workspace header.  Bit 0 makes the next
 * grouped-GEMM launch withhold its first operand load so the consumer's wait
 * runs out (bounded) and the call records MOE_ERR_DEVICE_TIMEOUT; in the
 * one-launch decode layer, CTA 0 leaves before its first grid-barrier
 * arrival and the other CTAs' barrier waits run out the same way. */
moe_status moe_set_debug_flags(void* ws, uint32_t flags, void* stream);

const char* moe_status_string(moe_status s);

/* Human-readable detail of the calling thread's last failed call. */
const char* moe_last_error_detail(void);

/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
