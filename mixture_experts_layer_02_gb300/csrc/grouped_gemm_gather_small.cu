// grouped_gemm_gather_small.cu -- the CTA-pair and swapped-operand grouped
// GEMMs with gathered token rows (kernels in grouped_gemm_2sm.cuh and
// grouped_gemm_swap.cuh), bf16 and e4m3.
#include "grouped_gemm_2sm.cuh"
#include "grouped_gemm_swap.cuh"

namespace moe {

cudaError_t launch_grouped_gemm_pair_gather(bool e4m3, int epi, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                                            const GemmArgs& a, long long tiles_ub, cudaStream_t st) {
    if (epi != EPI_SWIGLU_BF16) return cudaErrorInvalidValue;  // pair GEMM1 runs SwiGLU only
    return e4m3 ? pair_launch<EPI_SWIGLU_BF16, true, true>(tmB, tmB, tmB2, a, tiles_ub, st)
                : pair_launch<EPI_SWIGLU_BF16, false, true>(tmB, tmB, tmB2, a, tiles_ub, st);
}

#define MOE_SWAPG_CASE(E_, B_)                                                                \
    if (epi == E_ && bt == B_)                                                                \
        return e4m3 ? swap_launch<E_, B_, true, true>(tmW, tmW2, tmW, a, grid, st)           \
                    : swap_launch<E_, B_, false, true>(tmW, tmW2, tmW, a, grid, st);

cudaError_t launch_grouped_gemm_swap_gather(bool e4m3, int epi, int bt, const CUtensorMap& tmW,
                                            const CUtensorMap& tmW2, const GemmArgs& a, int grid, cudaStream_t st) {
    MOE_SWAPG_CASE(EPI_SWIGLU_BF16, 16)
    MOE_SWAPG_CASE(EPI_SWIGLU_BF16, 32)
    MOE_SWAPG_CASE(EPI_SILU_BF16, 16)
    MOE_SWAPG_CASE(EPI_SILU_BF16, 32)
    MOE_SWAPG_CASE(EPI_F32, 16)
    MOE_SWAPG_CASE(EPI_F32, 32)
    MOE_SWAPG_CASE(EPI_F32_DUAL, 16)
    MOE_SWAPG_CASE(EPI_F32_DUAL, 32)
    return cudaErrorInvalidValue;
}

}  // namespace moe
