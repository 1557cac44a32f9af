// grouped_gemm_2sm_mixed.cu -- bf16 instantiations of the CTA-pair grouped
// GEMM with hot (256-row) and cold (weight-streaming) tiles in one launch
// (kernel in grouped_gemm_2sm_mixed.cuh).
#include "grouped_gemm_2sm_mixed.cuh"

namespace moe {

cudaError_t launch_grouped_gemm_pair_mixed(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                           const CUtensorMap& tmB2, const CUtensorMap& tmT,
                                           const CUtensorMap& tmW, const CUtensorMap& tmW2, const GemmArgs& a,
                                           long long tiles_ub, cudaStream_t st) {
    if (epi == EPI_SWIGLU_BF16)
        return pair_mixed_launch<EPI_SWIGLU_BF16>(tmA, tmB, tmB2, tmT, tmW, tmW2, a, tiles_ub, st);
    if (epi == EPI_STORE_BF16)
        return pair_mixed_launch<EPI_STORE_BF16>(tmA, tmB, tmB2, tmT, tmW, tmW2, a, tiles_ub, st);
    return cudaErrorInvalidValue;
}

}  // namespace moe
