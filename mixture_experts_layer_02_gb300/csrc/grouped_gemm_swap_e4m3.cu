// grouped_gemm_swap_e4m3.cu -- e4m3 instantiations of the swapped-operand
// grouped GEMM (kernel in grouped_gemm_swap.cuh): FP8 decode-sized calls.
#include "grouped_gemm_swap.cuh"

namespace moe {

#define MOE_SWAP8_CASE(E_, B_) \
    if (epi == E_ && bt == B_) return swap_launch<E_, B_, true>(tmW, tmW2, tmX, a, grid, st);

cudaError_t launch_grouped_gemm_swap_e4m3(int epi, int bt, const CUtensorMap& tmW, const CUtensorMap& tmW2,
                                          const CUtensorMap& tmX, const GemmArgs& a, int grid, cudaStream_t st) {
    MOE_SWAP8_CASE(EPI_SWIGLU_BF16, 16)
    MOE_SWAP8_CASE(EPI_SWIGLU_BF16, 32)
    MOE_SWAP8_CASE(EPI_SILU_BF16, 16)
    MOE_SWAP8_CASE(EPI_SILU_BF16, 32)
    MOE_SWAP8_CASE(EPI_STORE_BF16, 16)
    MOE_SWAP8_CASE(EPI_STORE_BF16, 32)
    MOE_SWAP8_CASE(EPI_F32, 16)
    MOE_SWAP8_CASE(EPI_F32, 32)
    MOE_SWAP8_CASE(EPI_F32_DUAL, 16)
    MOE_SWAP8_CASE(EPI_F32_DUAL, 32)
    return cudaErrorInvalidValue;
}

}  // namespace moe
