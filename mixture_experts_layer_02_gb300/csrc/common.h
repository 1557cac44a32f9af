// common.h -- constants and internal launch interfaces shared by the host API
// (moe_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// ---- workspace header (first 256 bytes of every workspace) ----
//   word 0: device error bits (atomicOr), word 1: debug flags (test hooks)
constexpr size_t kWsHeaderBytes = 256;
constexpr uint32_t MOE_DEVERR_BOUNDS = 1u;
constexpr uint32_t MOE_DEVERR_TIMEOUT = 2u;
constexpr uint32_t MOE_DBG_WITHHOLD_FIRST_LOAD = 1u;

// Longest any pipeline wait may take before the kernel gives up (1 s).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// ---- GEMM tiling ----
constexpr int kBM = 128;  // rows per tile (MMA M)
constexpr int kBK = 64;   // K per pipeline stage: one 128-byte swizzle atom of bf16

enum EpiKind : int {
    EPI_STORE_BF16 = 0,  // y = acc                        -> bf16
    EPI_SILU_BF16 = 1,   // h = silu(acc)                  -> bf16
    EPI_SWIGLU_BF16 = 2, // h = silu(acc[:BN/2])*acc[BN/2:] -> bf16 (BN/2 outputs)
    EPI_ROUTER = 3       // logits -> top-K ids + weights (fp32)
};

// Everything a grouped-GEMM launch needs besides its tensor maps.
struct GemmArgs {
    const int32_t* group_offsets;  // [G+1] row offsets of each group; nullptr = one group of M rows
    int G;                         // number of groups (experts)
    int M;                         // rows when group_offsets == nullptr
    int n_out;                     // output columns per group
    int k_dim;                     // reduction length (multiple of 64)
    int b_rows_per_group;          // rows of the B operand per group in its 2-D view
    void* out;                     // output base (bf16 for FFN epilogues)
    long long ldo;                 // output row stride in elements
    uint32_t* err;                 // workspace error word
    const uint32_t* dbg;           // workspace debug flags
    // router epilogue
    const float* bias;             // [E] or nullptr
    int E, K, mode;
    int32_t* topk_ids;
    float* topk_w;
    float* logits_out;             // [N,E] or nullptr
};

// ---- internal launchers (return cudaError_t of the launch) ----
// Grouped GEMM with tensor maps prepared by the host.  tmB2 is used only by
// the SwiGLU epilogue (the W3 operand).  bn = N tile width.
cudaError_t launch_grouped_gemm(int epi, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                const CUtensorMap& tmB2, const GemmArgs& a, int grid,
                                cudaStream_t st);
size_t gemm_smem_bytes(int epi, int bn, int G);
int gemm_stages(int epi, int bn);

// Permutation (histogram -> scan -> stable scatter + row copy).
constexpr int kPermTokensPerBlock = 16;
size_t permute_scratch_bytes(int N, int E);
cudaError_t launch_permute(const uint16_t* x, const int32_t* ids, int N, int D, int E, int K,
                           int32_t* offsets, int32_t* perm_src, int32_t* inv_perm,
                           uint16_t* x_perm, int32_t* scratch, uint32_t* err, cudaStream_t st);

// Combine (gather K rows, weight, fp32 sum in k order, bf16 store).
cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* inv_perm, const float* w, int N,
                           int D, int K, uint16_t* out, uint32_t* err, cudaStream_t st);

// Sets the text moe_last_error_detail() returns on the calling thread.
void set_error_detail(const char* msg);

}  // namespace moe
