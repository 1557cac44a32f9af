// common.h -- constants and internal launch interfaces shared by the host API
// (moe_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#include <utility>

namespace moe {

// ---- launches ----
// Every kernel of the library is launched with programmatic stream
// serialisation: the next kernel on the stream may start its prologue while
// this one drains, and waits (griddepcontrol.wait) before reading anything an
// earlier kernel wrote.  MOE_PDL=0 turns it off.
inline bool pdl_enabled() {
    static const bool on = [] {
        const char* f = getenv("MOE_PDL");
        return f == nullptr || atoi(f) != 0;
    }();
    return on;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- workspace header (first 256 bytes of every workspace) ----
//   word 0: device error bits (atomicOr), word 1: debug flags (test hooks),
//   bytes 128..135: the decode layer's grid-barrier arrival count (64-bit)
constexpr size_t kWsHeaderBytes = 256;
constexpr size_t kWsBarrierCount = 128;
constexpr uint32_t MOE_DEVERR_BOUNDS = 1u;
constexpr uint32_t MOE_DEVERR_TIMEOUT = 2u;
constexpr uint32_t MOE_DBG_WITHHOLD_FIRST_LOAD = 1u;

// Longest any pipeline wait may take before the kernel gives up (1 s).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// ---- GEMM tiling ----
constexpr int kBM = 128;       // rows per tile (MMA M)
constexpr int kBK = 64;        // bf16 K per pipeline stage: one 128-byte swizzle row
constexpr int kRowBytes = 128; // bytes of K per stage and tile row, for either operand type

// Operand type of the grouped GEMMs.  A pipeline stage always holds one
// 128-byte swizzle row of K per tile row: 64 bf16 or 128 e4m3 values; one MMA
// instruction consumes 32 bytes of K (16 bf16 / 32 e4m3).
template <bool FP8>
struct OpType {
    static constexpr int KB = FP8 ? 128 : 64;    // K elements per stage
    static constexpr int KSTEP = FP8 ? 32 : 16;  // K elements per MMA instruction
    static constexpr int MMAS = kRowBytes / 32;  // MMA instructions per stage
};

enum EpiKind : int {
    EPI_STORE_BF16 = 0,   // y = acc                          -> bf16
    EPI_SILU_BF16 = 1,    // h = silu(acc)                    -> bf16
    EPI_SWIGLU_BF16 = 2,  // h = silu(acc[:BN/2])*acc[BN/2:]  -> bf16 (B = W1 half | W3 half)
    EPI_F32 = 3,          // raw fp32 accumulator (split-K partial), one B operand
    EPI_F32_DUAL = 4      // raw fp32 accumulator, B = W1 half | W3 half (split-K GEMM1)
};

// Everything a grouped-GEMM launch needs besides its tensor maps.
struct GemmArgs {
    const int32_t* group_offsets;  // [G+1] row offsets of each group; nullptr = one group of M rows
    int G;                         // number of groups (experts)
    int M;                         // rows of A (all groups)
    int n_out;                     // output columns per group (the tile count is derived from it)
    int k_dim;                     // reduction length (multiple of 64)
    int b_rows_per_group;          // rows of the B operand per group in its 2-D view
    int splits;                    // split-K factor >= 1: split s sums k-blocks
                                   // [s*nkb/splits, (s+1)*nkb/splits)
    void* out;                     // bf16 output, or fp32 partials for the EPI_F32 kinds
    long long ldo;                 // output row stride in elements
    long long split_stride;        // elements between the fp32 slabs of consecutive splits
    uint32_t* err;                 // workspace error word
    const uint32_t* dbg;           // workspace debug flags
    // e4m3 operands only (unused for bf16): every output is
    //   acc[r][c] * row_scale[r'] * col_scale[g * b_rows_per_group + c]
    // with r' = row_scale_idx ? row_scale_idx[r] : r (r = row of A, i.e. of
    // the output); for the SwiGLU kinds the up half uses col_scale_up (W3).
    const float* row_scale;
    const int32_t* row_scale_idx;
    const float* col_scale;
    const float* col_scale_up;
    // gathered A (the permutation fused into GEMM1's operand load): row r of
    // A is row a_src_rows[r] of a_src (a_src_n rows, a_src_ld bytes apart),
    // copied into the swizzled tile by the producer warp; tmA is not read.
    const void* a_src;
    const int32_t* a_src_rows;
    long long a_src_ld;
    int a_src_n;
    // mixed CTA-pair kernel only: experts with 1 .. cold_rows rows run as
    // weight-streaming tiles (0: every expert runs 256-row tiles)
    int cold_rows;
    // CTA-pair kernels: m-tiles per raster band (0: the default, 8)
    int band;
};

// ---- internal launchers (return cudaError_t of the launch) ----
// Grouped GEMM with tensor maps prepared by the host.  tmB2 (the W3 operand)
// is read only by the dual-B kinds.  bn = N tile width.
cudaError_t launch_grouped_gemm(int epi, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                const CUtensorMap& tmB2, const GemmArgs& a, int grid,
                                cudaStream_t st);

// The same on CTA pairs (256 x 256 tiles, tcgen05 cta_group::2) for
// EPI_SWIGLU_BF16 / EPI_STORE_BF16 with bn = 256 and no split; the B maps
// have 128-row boxes.  tiles_ub bounds the number of pair tiles.
cudaError_t launch_grouped_gemm_pair(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                     const CUtensorMap& tmB2, const GemmArgs& a, long long tiles_ub,
                                     cudaStream_t st);

// The CTA-pair GEMM with hot experts (more than a.cold_rows rows) on 256-row
// pair tiles, heaviest expert first, and cold experts (1 .. a.cold_rows rows)
// on weight-streaming tiles (weights as the MMA's M, 32 tokens as its N)
// spread evenly among them.  bf16 operands, EPI_SWIGLU_BF16 / EPI_STORE_BF16,
// up to 256 groups, K a multiple of 256.  All maps view their matrix as
// {64 elements, rows, k-blocks}: hot tiles read tmA (A) and tmB / tmB2 (W1 or
// W, and W3) in 128-row x 2-k-block boxes; cold tiles read tmT (A) in 16-row
// x 4-k-block boxes and tmW / tmW2 in 128-row x 4-k-block boxes.
cudaError_t launch_grouped_gemm_pair_mixed(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                           const CUtensorMap& tmB2, const CUtensorMap& tmT,
                                           const CUtensorMap& tmW, const CUtensorMap& tmW2, const GemmArgs& a,
                                           long long tiles_ub, cudaStream_t st);

// The same with operand roles swapped for few rows per expert (decode):
// the weights are the 128-row MMA operand, the tokens the BT-row one
// (bt = 16 or 32).  tmW: weights with 64-row (SwiGLU GEMM1, W1; tmW2 = W3)
// or 128-row boxes; tmX: activations with BT-row boxes.
cudaError_t launch_grouped_gemm_swap(int epi, int bt, const CUtensorMap& tmW, const CUtensorMap& tmW2,
                                     const CUtensorMap& tmX, const GemmArgs& a, int grid, cudaStream_t st);

// The three grouped GEMMs above with e4m3 operands (tcgen05 kind::f8f6f4) and
// the per-row / per-column scales of GemmArgs; tensor maps over uint8 data
// with 128-element boxes; k_dim a multiple of 128.
cudaError_t launch_grouped_gemm_e4m3(int epi, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                     const CUtensorMap& tmB2, const GemmArgs& a, int grid, cudaStream_t st);
cudaError_t launch_grouped_gemm_pair_e4m3(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                          const CUtensorMap& tmB2, const GemmArgs& a, long long tiles_ub,
                                          cudaStream_t st);
cudaError_t launch_grouped_gemm_swap_e4m3(int epi, int bt, const CUtensorMap& tmW, const CUtensorMap& tmW2,
                                          const CUtensorMap& tmX, const GemmArgs& a, int grid, cudaStream_t st);

// GEMM1 with the permutation fused into its operand load: the A rows (the
// token rows of the swapped kernel) are gathered through GemmArgs::a_src*
// instead of read by TMA; bf16 or e4m3 operands.  Kinds: the GEMM1 epilogues
// (SwiGLU, SiLU, and the fp32 partials of a split).
cudaError_t launch_grouped_gemm_gather(bool e4m3, int epi, int bn, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                                       const GemmArgs& a, int grid, cudaStream_t st);
cudaError_t launch_grouped_gemm_pair_gather(bool e4m3, int epi, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                                            const GemmArgs& a, long long tiles_ub, cudaStream_t st);
cudaError_t launch_grouped_gemm_swap_gather(bool e4m3, int epi, int bt, const CUtensorMap& tmW,
                                            const CUtensorMap& tmW2, const GemmArgs& a, int grid, cudaStream_t st);

// The whole bf16 SwiGLU grouped FFN of a decode-sized call in one persistent
// cooperative launch (GEMM1 + SwiGLU and GEMM2, split partials summed by the
// last split of each tile, GEMM2 items of an expert waiting until its h is
// complete).  Tensor maps: W1, W3 ([E*Dff, D], 64-row boxes), x_perm
// ([M, D], BT-row boxes), W2 ([E*D, Dff], 128-row boxes), h ([M, Dff],
// BT-row boxes).  The counters must be zero at launch.
struct FusedFfnArgs {
    const int32_t* group_offsets;  // [G+1]
    int G, M, D, Dff;
    int splits1, splits2;          // k-splits of GEMM1 (over D) and GEMM2 (over Dff)
    float* part1;                  // [splits1][M][2*Dff] fp32: tile n at columns n*128 (gate 64 | up 64)
    float* part2;                  // [splits2][M][D] fp32
    uint16_t* h;                   // [M][Dff] bf16 out (GEMM2's input)
    uint16_t* y;                   // [M][D] bf16 out
    int* tile_cnt1;                // [tiles1_cap] splits finished per GEMM1 tile
    int* tile_cnt2;                // [tiles2_cap] splits finished per GEMM2 tile
    int* expert_done;              // [G] GEMM1 tiles of h written per expert
    int tiles1_cap, tiles2_cap;
    uint32_t* err;
    const uint32_t* dbg;
    // e4m3 operands only (null otherwise)
    const float* x_scale;          // token scales: per row of the permuted codes, or
    const int32_t* x_scale_idx;    //   per token, indexed through x_scale_idx[row] when given
    const float* s1;               // [G*Dff] W1 row scales
    const float* s3;               // [G*Dff] W3 row scales
    const float* s2;               // [G*D] W2 row scales
    uint8_t* hq;                   // [M][Dff] e4m3 codes of h (GEMM2's input)
    float* h_scale;                // [M] their row scales
    uint32_t* h_amax;              // [M] max |h| bf16 bits per row, zero at launch
    int* quant_done;               // [G] token tiles of hq written per expert, zero at launch
    int xs_rows;                   // M: token scales staged in shared memory; 0: read from x_scale
};
cudaError_t launch_ffn_fused_decode(bool e4m3, int bt, const CUtensorMap* maps, const FusedFfnArgs& a, int grid,
                                    cudaStream_t st);
// `rows` when that many token scales fit in shared memory beside the pipeline, else 0.
int ffn_fused_decode_xs_rows(int bt, int G, int rows);
// CTAs that can be resident at once (the cooperative launch's grid limit).
int ffn_fused_decode_max_grid(bool e4m3, int bt, int G, int xs_rows);

// The whole bf16 layer of a small decode batch in one persistent cooperative
// launch of one CTA per SM (layer_decode.cu): router logits, top-K and
// placement, GEMM1 + activation and GEMM2 + combine, phases separated by two
// grid barriers whose words live in the workspace header.
constexpr int kLayerDecodeMaxN = 8;      // tokens: a token has at most this many rows in any expert
constexpr int kLayerDecodeMaxRows = 64;  // assignments N * K
constexpr int kLayerDecodeMaxE = 256;    // experts
struct LayerDecodeArgs {
    const uint16_t* x;       // [N][D]
    const uint16_t* wg;      // [E][D]
    const float* bias;       // [E] or null
    const uint16_t* w1;      // [E][Dff][D]
    const uint16_t* w3;      // [E][Dff][D], null: SiLU (no W3)
    const uint16_t* w2;      // [E][D][Dff]
    int N, D, E, K, Dff, mode;
    float* logits;           // [N][E] fp32 scratch
    int32_t* ids;            // the layer's intermediates, as the separate kernels write them
    float* w;
    int32_t* offsets;
    int32_t* perm_src;
    int32_t* inv_perm;
    uint16_t* x_perm;
    uint16_t* h;
    uint16_t* y_perm;
    uint16_t* out;           // [N][D]
    uint32_t* err;
    const uint32_t* dbg;
    unsigned long long* bar; // grid-barrier arrivals: grows by the grid size per barrier
    long long l2_prefetch_max;  // W2 of the chosen experts is prefetched into L2 when at most this many bytes
    int w2_smem;             // 1: each CTA's W2 rows are TMA-copied into shared memory during GEMM1
    // e4m3 experts (fp8 = 1; w1/w3/w2 unused): weight codes and their per-row
    // scales; the kernel quantises x and h per row and writes their codes
    // and scales (the e4m3 layer's intermediates; x_perm holds no rows)
    int fp8;
    const uint8_t* w1q;      // [E][Dff][D]
    const uint8_t* w3q;      // [E][Dff][D] or null
    const uint8_t* w2q;      // [E][D][Dff]
    const float* s1;         // [E*Dff]
    const float* s3;         // [E*Dff] or null
    const float* s2;         // [E*D]
    uint8_t* xq;             // [N][D]
    float* x_scale;          // [N]
    uint8_t* xq_perm;        // [N*K][D]
    uint8_t* hq;             // [N*K][Dff]
    float* h_scale;          // [N*K]
};
// Byte offsets of the kernel's dynamic shared memory (host and device),
// relative to its first 1024-byte boundary (the kernel rounds its base up;
// `total` includes that slack).  With w2_smem the W2 rows of each expert slot
// are a 16-row, 128-byte-swizzled TMA box of every 64-column block (the
// layout ldmatrix reads without bank conflicts), and h is staged in bf16.
constexpr int kLayerDecodeW2Rows = 16;   // W2 rows per staged slot (the MMA's M)
struct LayerDecodeSmem {
    size_t logits, off, xh, y, part, g1, w2, total;
};
__host__ __device__ inline size_t layer_decode_up16(size_t v) { return (v + 15) & ~static_cast<size_t>(15); }
__host__ __device__ inline LayerDecodeSmem layer_decode_smem(int N, int D, int E, int K, int Dff, int grid,
                                                              bool w2_smem, bool fp8 = false) {
    LayerDecodeSmem s;
    size_t o = 0;
    const int tmax = N * K < E ? N * K : E;
    const int esize = fp8 ? 1 : 2;
    s.w2 = o;                                         // staged W2 [slot][Dff*esize/128][16 rows][128 B]
    if (w2_smem) o += static_cast<size_t>(tmax) * kLayerDecodeW2Rows * Dff * esize;
    s.logits = o;                                     // scores [N][E] fp32
    o = layer_decode_up16(o + static_cast<size_t>(N) * E * 4);
    s.off = o;                                        // [E + 1] expert_offsets
    o = layer_decode_up16(o + static_cast<size_t>(E + 1) * 4);
    // x rows [N][D] bf16 (e4m3: their codes), later h rows [N*K][Dff] bf16
    // (e4m3: codes)
    s.xh = o;
    const size_t xb = static_cast<size_t>(N) * D * (fp8 ? 1 : 2);
    const size_t hb = static_cast<size_t>(N) * K * Dff * (fp8 ? 1 : 2);
    o = layer_decode_up16(o + (xb > hb ? xb : hb));
    s.y = o;                                          // y of the CTA's columns [N*K][nd] (bf16)
    const int pairs = (D / 2 + grid - 1) / grid;
    o = layer_decode_up16(o + static_cast<size_t>(N) * K * 2 * pairs * 2);
    s.part = o;                                       // staged GEMM2 partial tiles [max(16, slots)][16][8] fp32
    if (w2_smem) o += static_cast<size_t>(tmax > 16 ? tmax : 16) * kLayerDecodeW2Rows * 8 * 4;
    // tensor-core GEMV partial sums [16 warps][2 tiles][2][16 rows][nr] fp32
    // (nr = N rounded up to a power of two)
    s.g1 = o;
    const int nr = N <= 1 ? 1 : (N <= 2 ? 2 : (N <= 4 ? 4 : 8));
    o += static_cast<size_t>(16) * 2 * 2 * kLayerDecodeW2Rows * nr * 4;
    s.total = o + 1024;
    return s;
}
// tm_w2: W2 viewed {64, E*D rows, Dff/64} with {64, 16, Dff/64} swizzled boxes (read with w2_smem only).
cudaError_t launch_layer_decode(const LayerDecodeArgs& a, const CUtensorMap& tm_w2, int grid, cudaStream_t st);
// The launch's grid (one CTA per SM, 0 when the sizes do not fit) and
// whether the CTAs' W2 columns fit in shared memory (*w2_smem).  e4m3
// experts need D and D_ffn multiples of 128.
int layer_decode_plan(int N, int D, int E, int K, int Dff, bool swiglu, bool fp8, int* w2_smem);

// Per-row e4m3 quantisation of a bf16 matrix [rows, cols] (cols % 8 == 0):
// scale[r] = 2^k with k the smallest integer >= -126 such that
// max|src[r,:]| <= 448 * 2^k, q[r,c] = e4m3_rn_satfinite(src[r,c] * 2^-k).
cudaError_t launch_quant_rows_e4m3(const uint16_t* src, long long rows, int cols, uint8_t* q, float* scale,
                                   cudaStream_t st);

// Router logits of up to kSmallRouteMaxN tokens (D <= 8192) on the CUDA cores:
// logits [N][E] fp32 = x [N][D] . W_gate [E][D] (bf16), one CTA per expert.
constexpr int kSmallRouteMaxN = 32;
cudaError_t launch_route_logits_small(const uint16_t* x, const uint16_t* wg, int N, int D, int E, float* logits,
                                      cudaStream_t st);

// Router top-K over fp32 logit partials [splits][N][ldp] (summed in split
// order, + bias): ids, weights, optional logits export.
cudaError_t launch_route_topk(const float* partial, int splits, long long split_stride, int ldp,
                              const float* bias, int N, int E, int K, int mode, float* logits_out,
                              int32_t* ids, float* w, uint32_t* err, cudaStream_t st);

constexpr int kFusedRoutePermuteMax = 256;  // assignments of the fused top-K + permute launch

// route_topk and the permutation (expert_offsets, perm_src, inv_perm, the
// row copy x -> x_perm) of a call with N * K <= 256 in one launch of `grid`
// CTAs (each computes the whole routing; CTA 0 stores it; they share the row
// copy).  Same bits as launch_route_topk followed by launch_permute.
cudaError_t launch_route_topk_permute(const float* partial, int splits, long long split_stride, int ldp,
                                      const float* bias, int N, int E, int K, int mode, float* logits_out,
                                      int32_t* ids, float* w, const uint16_t* x, int D, int32_t* offsets,
                                      int32_t* perm_src, int32_t* inv_perm, uint16_t* x_perm, int grid,
                                      uint32_t* err, cudaStream_t st);

// Split-K reductions of the grouped FFN: partials [splits][rows][ldp] fp32.
//   swiglu: h[r][c] = bf16(silu(sum g) * sum u), g/u at tile-interleaved columns
//           (tile n of width bn holds g for columns n*bn/2.. then u)
//   store:  y[r][c] = bf16(sum p), or bf16(silu(sum p)) with silu = true
cudaError_t launch_ffn_reduce_swiglu(const float* partial, int splits, long long split_stride, int ldp,
                                     int rows, int Dff, int bn, uint16_t* h, cudaStream_t st);
cudaError_t launch_ffn_reduce_store(const float* partial, int splits, long long split_stride, int ldp,
                                    int rows, int ncols, bool silu, uint16_t* y, cudaStream_t st);

// Permutation (histogram -> scan -> stable scatter + row copy).
constexpr int kPermTokensPerBlock = 16;
size_t permute_scratch_bytes(int N, int E);
cudaError_t launch_permute(const uint16_t* x, const int32_t* ids, int N, int D, int E, int K,
                           int32_t* offsets, int32_t* perm_src, int32_t* inv_perm,
                           uint16_t* x_perm, int32_t* scratch, uint32_t* err, cudaStream_t st);

// Paradigm B: fixed blocks of C rows per expert, drops past C (slot -1).
cudaError_t launch_permute_padded(const uint16_t* x, const int32_t* ids, int N, int D, int E, int K, int C,
                                  int32_t* pad_offsets, int32_t* kept, int32_t* slot, uint16_t* x_pad,
                                  int32_t* scratch, uint32_t* err, cudaStream_t st);

cudaError_t launch_pad_offsets(int E, int C, int32_t* pad_offsets, int32_t* kept, cudaStream_t st);

// Combine with an explicit row count; allow_dropped treats row -1 as an
// assignment dropped at capacity (no error, no contribution).
cudaError_t launch_combine_rows(const uint16_t* y_perm, const int32_t* inv_perm, const float* w, int N, int D,
                                int K, long long rows, bool allow_dropped, uint16_t* out, uint32_t* err,
                                cudaStream_t st);

// Combine (gather K rows, weight, fp32 sum in k order, bf16 store).
cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* inv_perm, const float* w, int N,
                           int D, int K, uint16_t* out, uint32_t* err, cudaStream_t st);

// Routing statistics: EMA of expert fractions, KL to uniform, bias step.
cudaError_t launch_routing_stats(const int32_t* offsets, int E, float decay, float step, float* ema, float* bias,
                                 float* kl_out, cudaStream_t st);

// Sets the text moe_last_error_detail() returns on the calling thread.
void set_error_detail(const char* msg);
// moe_permute's size checks: a moe_status value (0 = ok; the detail message
// is recorded on failure).
int check_permute_sizes(int N, int D, int E, int K);

}  // namespace moe
