// grouped_gemm_gather_e4m3.cu -- e4m3 instantiations of the one-CTA grouped
// GEMM with a gathered A operand (kernel in grouped_gemm.cuh).
#include "grouped_gemm.cuh"

namespace moe {

#define MOE_GATHER8_CASE(E_, B_) \
    if (epi == E_ && bn == B_) return launch_t<E_, B_, true, true>(tmB, tmB, tmB2, a, grid, st);

cudaError_t launch_grouped_gemm_gather_e4m3(int epi, int bn, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                                            const GemmArgs& a, int grid, cudaStream_t st) {
    MOE_GATHER8_CASE(EPI_SWIGLU_BF16, 256)
    MOE_GATHER8_CASE(EPI_SWIGLU_BF16, 128)
    MOE_GATHER8_CASE(EPI_SWIGLU_BF16, 64)
    MOE_GATHER8_CASE(EPI_SILU_BF16, 256)
    MOE_GATHER8_CASE(EPI_SILU_BF16, 128)
    MOE_GATHER8_CASE(EPI_SILU_BF16, 64)
    MOE_GATHER8_CASE(EPI_F32, 256)
    MOE_GATHER8_CASE(EPI_F32, 128)
    MOE_GATHER8_CASE(EPI_F32, 64)
    MOE_GATHER8_CASE(EPI_F32_DUAL, 256)
    MOE_GATHER8_CASE(EPI_F32_DUAL, 128)
    MOE_GATHER8_CASE(EPI_F32_DUAL, 64)
    return cudaErrorInvalidValue;
}

}  // namespace moe
