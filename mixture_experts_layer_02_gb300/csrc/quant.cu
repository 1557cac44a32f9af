// quant.cu -- per-row e4m3 quantisation of bf16 matrices: the expert weights
// (once, offline), the tokens before the permutation and the FFN's hidden
// activations before the second GEMM.  This is the FP8 path of "MoE 推理完整机制：
// 从 Router 到 Expert Parallelism 的一切" (zoe.im), 第四层 DeepGEMM & MegaMoE (FP8
// expert weights) and 第三层 (DeepEP: FP8 token hidden states halve the bytes
// moved); the pages fix no scaling rule, and the one used here is one
// power-of-two scale per row:
//   k = the smallest integer >= -126 with max|row| <= 448 * 2^k,
//   scale = 2^k,  q = e4m3(round to nearest even, saturating)(x * 2^-k).
// x * 2^-k is exact in fp32, so the e4m3 rounding is the only one, and the
// scale is an exact factor wherever it is applied.
//
// One warp per row: a first pass finds max|x| on the raw bits (for bf16 the
// magnitude order is the integer order of bits & 0x7fff), a second pass
// (rows are at most tens of KB, so it hits L2) converts eight values per lane
// and stores 8 bytes per lane, coalesced.
#include <cuda_fp8.h>

#include <algorithm>

#include "device.cuh"

namespace moe {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
    // the first component goes to the low byte
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kQuantThreads)
quant_rows_e4m3_kernel(const uint16_t* __restrict__ src, long long rows, int cols, uint8_t* __restrict__ q,
                       float* __restrict__ scale) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int chunks = cols >> 3;  // 8 bf16 = 16 bytes
    for (long long r = w0; r < rows; r += nw) {
        const uint4* row = reinterpret_cast<const uint4*>(src + r * cols);
        uint32_t m = 0;
        for (int c = lane; c < chunks; c += 32) {
            const uint4 v = row[c];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        // amax = (1 + f) 2^e with bf16 exponent field ef and 7-bit fraction:
        // 448 = 1.75 * 2^8, so k = e - 8 when f <= 0.75 (fraction <= 0x60), else e - 7
        const int ef = static_cast<int>(m >> 7), frac = static_cast<int>(m & 0x7fu);
        const int k = (ef == 0) ? -126 : max(-126, ef - 127 - 8 + (frac > 0x60 ? 1 : 0));
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);  // 2^-k
        if (lane == 0) scale[r] = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
        uint2* qrow = reinterpret_cast<uint2*>(q + r * cols);
        for (int c = lane; c < chunks; c += 32) {
            const uint4 v = row[c];
            const uint32_t p0 = fp8x2(bf16_lo(v.x) * inv, bf16_hi(v.x) * inv);
            const uint32_t p1 = fp8x2(bf16_lo(v.y) * inv, bf16_hi(v.y) * inv);
            const uint32_t p2 = fp8x2(bf16_lo(v.z) * inv, bf16_hi(v.z) * inv);
            const uint32_t p3 = fp8x2(bf16_lo(v.w) * inv, bf16_hi(v.w) * inv);
            qrow[c] = make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
        }
    }
    pdl_trigger();
}

cudaError_t launch_quant_rows_e4m3(const uint16_t* src, long long rows, int cols, uint8_t* q, float* scale,
                                   cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    constexpr int rows_per_block = kQuantThreads / 32;
    const long long need = (rows + rows_per_block - 1) / rows_per_block;
    const int grid = static_cast<int>(std::min<long long>(need, static_cast<long long>(nsm) * 8));
    return launch_kernel(quant_rows_e4m3_kernel, dim3(grid), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
}

}  // namespace moe
