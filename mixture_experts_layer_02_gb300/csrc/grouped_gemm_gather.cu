// grouped_gemm_gather.cu -- bf16 instantiations of the one-CTA grouped GEMM
// with a gathered A operand (kernel in grouped_gemm.cuh): GEMM1 reading the
// token rows through the permutation instead of a permuted copy.
#include "grouped_gemm.cuh"

namespace moe {

#define MOE_GATHER_CASE(E_, B_) \
    if (epi == E_ && bn == B_) return launch_t<E_, B_, false, true>(tmB, tmB, tmB2, a, grid, st);

cudaError_t launch_grouped_gemm_gather_bf16(int epi, int bn, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                                            const GemmArgs& a, int grid, cudaStream_t st) {
    MOE_GATHER_CASE(EPI_SWIGLU_BF16, 256)
    MOE_GATHER_CASE(EPI_SWIGLU_BF16, 128)
    MOE_GATHER_CASE(EPI_SWIGLU_BF16, 64)
    MOE_GATHER_CASE(EPI_SILU_BF16, 256)
    MOE_GATHER_CASE(EPI_SILU_BF16, 128)
    MOE_GATHER_CASE(EPI_SILU_BF16, 64)
    MOE_GATHER_CASE(EPI_F32, 256)
    MOE_GATHER_CASE(EPI_F32, 128)
    MOE_GATHER_CASE(EPI_F32, 64)
    MOE_GATHER_CASE(EPI_F32_DUAL, 256)
    MOE_GATHER_CASE(EPI_F32_DUAL, 128)
    MOE_GATHER_CASE(EPI_F32_DUAL, 64)
    return cudaErrorInvalidValue;
}

cudaError_t launch_grouped_gemm_gather_e4m3(int epi, int bn, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                                            const GemmArgs& a, int grid, cudaStream_t st);

cudaError_t launch_grouped_gemm_gather(bool e4m3, int epi, int bn, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                                       const GemmArgs& a, int grid, cudaStream_t st) {
    return e4m3 ? launch_grouped_gemm_gather_e4m3(epi, bn, tmB, tmB2, a, grid, st)
                : launch_grouped_gemm_gather_bf16(epi, bn, tmB, tmB2, a, grid, st);
}

}  // namespace moe
