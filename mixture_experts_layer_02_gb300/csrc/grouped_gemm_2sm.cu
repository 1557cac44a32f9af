// grouped_gemm_2sm.cu -- bf16 instantiations of the CTA-pair grouped GEMM
// (kernel in grouped_gemm_2sm.cuh).
#include "grouped_gemm_2sm.cuh"

namespace moe {

cudaError_t launch_grouped_gemm_pair(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                     const CUtensorMap& tmB2, const GemmArgs& a, long long tiles_ub,
                                     cudaStream_t st) {
    if (epi == EPI_SWIGLU_BF16) return pair_launch<EPI_SWIGLU_BF16, false>(tmA, tmB, tmB2, a, tiles_ub, st);
    if (epi == EPI_STORE_BF16) return pair_launch<EPI_STORE_BF16, false>(tmA, tmB, tmB2, a, tiles_ub, st);
    return cudaErrorInvalidValue;
}

}  // namespace moe
