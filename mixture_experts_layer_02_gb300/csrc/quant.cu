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
// Every row is read from HBM once and held in registers: rows of up to 2048
// values by one warp (up to 8 16-byte chunks per lane, eight rows per CTA in
// flight), rows of up to 16384 values by one 256-thread CTA (up to 8 chunks
// per thread).  max|x| comes from the raw bits (for bf16 the magnitude order
// is the integer order of bits & 0x7fff), then eight conversions and one
// 8-byte store per chunk, coalesced.  Longer rows: one warp per row and a
// second pass that re-reads the row.
#include <algorithm>

#include "quant.cuh"

namespace moe {

constexpr int kQuantThreads = 256;

template <int V>
__global__ void __launch_bounds__(kQuantThreads)
quant_rows_reg_kernel(const uint16_t* __restrict__ src, long long rows, int cols, uint8_t* __restrict__ q,
                      float* __restrict__ scale) {
    __shared__ uint32_t s_max[kQuantThreads / 32];
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunks = cols >> 3;  // 8 bf16 = 16 bytes
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint4* row = reinterpret_cast<const uint4*>(src + r * cols);
        uint4 v[V];
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int c = threadIdx.x + i * kQuantThreads;
            v[i] = (c < chunks) ? row[c] : make_uint4(0, 0, 0, 0);
            m = max(m, absmax8(v[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) s_max[warp] = m;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < kQuantThreads / 32; ++w) m = max(m, s_max[w]);
        __syncthreads();  // s_max is rewritten for the next row
        const int k = scale_exp_of(m);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);  // 2^-k
        if (threadIdx.x == 0) scale[r] = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
        uint2* qrow = reinterpret_cast<uint2*>(q + r * cols);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int c = threadIdx.x + i * kQuantThreads;
            if (c < chunks) qrow[c] = to_e4m3x8(v[i], inv);
        }
    }
    pdl_trigger();
}

template <int V>
__global__ void __launch_bounds__(kQuantThreads)
quant_rows_warp_kernel(const uint16_t* __restrict__ src, long long rows, int cols, uint8_t* __restrict__ q,
                       float* __restrict__ scale) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int chunks = cols >> 3;
    for (long long r = w0; r < rows; r += nw) {
        const uint4* row = reinterpret_cast<const uint4*>(src + r * cols);
        uint4 v[V];
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int c = lane + i * 32;
            v[i] = (c < chunks) ? row[c] : make_uint4(0, 0, 0, 0);
            m = max(m, absmax8(v[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int k = scale_exp_of(m);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);  // 2^-k
        if (lane == 0) scale[r] = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
        uint2* qrow = reinterpret_cast<uint2*>(q + r * cols);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int c = lane + i * 32;
            if (c < chunks) qrow[c] = to_e4m3x8(v[i], inv);
        }
    }
    pdl_trigger();
}

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
        for (int c = lane; c < chunks; c += 32) m = max(m, absmax8(row[c]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int k = scale_exp_of(m);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);  // 2^-k
        if (lane == 0) scale[r] = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
        uint2* qrow = reinterpret_cast<uint2*>(q + r * cols);
        for (int c = lane; c < chunks; c += 32) qrow[c] = to_e4m3x8(row[c], inv);
    }
    pdl_trigger();
}

cudaError_t launch_quant_rows_e4m3(const uint16_t* src, long long rows, int cols, uint8_t* q, float* scale,
                                   cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    constexpr int rows_per_block = kQuantThreads / 32;
    const long long warp_grid = std::min<long long>((rows + rows_per_block - 1) / rows_per_block,
                                                    static_cast<long long>(nsm) * 8);
    const int wg = static_cast<int>(warp_grid);
    const int vw = (cols / 8 + 31) / 32;  // chunks per lane, one row per warp
    switch (vw) {
        case 1: return launch_kernel(quant_rows_warp_kernel<1>, dim3(wg), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 2: return launch_kernel(quant_rows_warp_kernel<2>, dim3(wg), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 3:
        case 4: return launch_kernel(quant_rows_warp_kernel<4>, dim3(wg), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 5:
        case 6:
        case 7:
        case 8: return launch_kernel(quant_rows_warp_kernel<8>, dim3(wg), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        default: break;
    }
    const int v = (cols / 8 + kQuantThreads - 1) / kQuantThreads;  // chunks per thread, one row per CTA
    const int grid_rows = static_cast<int>(std::min<long long>(rows, static_cast<long long>(nsm) * 8));
    switch (v) {
        case 1: return launch_kernel(quant_rows_reg_kernel<1>, dim3(grid_rows), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 2: return launch_kernel(quant_rows_reg_kernel<2>, dim3(grid_rows), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 3: return launch_kernel(quant_rows_reg_kernel<3>, dim3(grid_rows), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 4: return launch_kernel(quant_rows_reg_kernel<4>, dim3(grid_rows), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 5: return launch_kernel(quant_rows_reg_kernel<5>, dim3(grid_rows), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 6: return launch_kernel(quant_rows_reg_kernel<6>, dim3(grid_rows), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 7: return launch_kernel(quant_rows_reg_kernel<7>, dim3(grid_rows), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        case 8: return launch_kernel(quant_rows_reg_kernel<8>, dim3(grid_rows), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
        default: break;
    }
    return launch_kernel(quant_rows_e4m3_kernel, dim3(wg), dim3(kQuantThreads), 0, st, src, rows, cols, q, scale);
}

}  // namespace moe
