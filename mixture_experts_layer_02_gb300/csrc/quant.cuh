// quant.cuh -- device helpers of the per-row e4m3 quantisation (see quant.cu
// for the rule): magnitude maxima on raw bf16 bits, the power-of-two scale
// exponent, and eight bf16 values converted to e4m3 codes.  Shared by the
// quantisation kernels and the fused decode FFN.
#pragma once

#include <cuda_fp8.h>

#include "device.cuh"

namespace moe {

__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
    // the first component goes to the low byte
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t absmax8(const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
    return m;
}

// k from the bf16 bits of the row maximum: amax = (1 + f) 2^e with exponent
// field ef and 7-bit fraction; 448 = 1.75 * 2^8, so k = e - 8 when f <= 0.75
// (fraction <= 0x60), else e - 7; rows below 2^-126 (and zero rows) get -126.
__device__ __forceinline__ int scale_exp_of(uint32_t m) {
    const int ef = static_cast<int>(m >> 7), frac = static_cast<int>(m & 0x7fu);
    return (ef == 0) ? -126 : max(-126, ef - 127 - 8 + (frac > 0x60 ? 1 : 0));
}

__device__ __forceinline__ uint2 to_e4m3x8(const uint4& v, float inv) {
    const uint32_t p0 = fp8x2(bf16_lo(v.x) * inv, bf16_hi(v.x) * inv);
    const uint32_t p1 = fp8x2(bf16_lo(v.y) * inv, bf16_hi(v.y) * inv);
    const uint32_t p2 = fp8x2(bf16_lo(v.z) * inv, bf16_hi(v.z) * inv);
    const uint32_t p3 = fp8x2(bf16_lo(v.w) * inv, bf16_hi(v.w) * inv);
    return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
}

}  // namespace moe
