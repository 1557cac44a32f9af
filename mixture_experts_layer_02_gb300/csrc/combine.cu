// combine.cu -- un-permute and router-weighted sum.
//
// "MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im), 第二层
// 范式 A Step 3 and the opening dataflow figure: expert outputs go back to the
// original token order and are summed with the router weights,
//   out[t,:] = sum_k w[t,k] * y_perm[inv_perm[t,k], :].
// The sum runs in fp32 in k order (one fused multiply-add per term) and is
// rounded once to bf16 (nearest-even), so the result does not depend on the
// launch shape.
//
// Work item = (token, slice of D); a warp owns one item and moves 16-byte
// chunks: per chunk, K independent row loads, fp32 accumulate, one 16-byte
// store.  For small N the row is cut into slices so enough warps are in
// flight to keep HBM busy.
#include "device.cuh"

namespace moe {

constexpr int kCombThreads = 256;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <int KMAX>  // K <= KMAX
__global__ void __launch_bounds__(kCombThreads)
combine_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ inv_perm,
               const float* __restrict__ w, int N, int D, int K, int nslices, long long rows,
               bool allow_dropped, uint16_t* __restrict__ out, uint32_t* err) {
    const int lane = threadIdx.x & 31;
    const long long item = static_cast<long long>(blockIdx.x) * (kCombThreads / 32) + (threadIdx.x >> 5);
    pdl_wait();
    if (item >= static_cast<long long>(N) * nslices) return;
    const int t = static_cast<int>(item / nslices);
    const int s = static_cast<int>(item - static_cast<long long>(t) * nslices);
    const int cpr = D / 8;
    const int per = (cpr + nslices - 1) / nslices;
    const int c0 = s * per;
    const int c1 = min(cpr, c0 + per);

    // lane k holds assignment k's row and weight
    int my_r = -1;
    float my_w = 0.0f;
    if (lane < K) {
        my_r = inv_perm[static_cast<long long>(t) * K + lane];
        my_w = w[static_cast<long long>(t) * K + lane];
        if (my_r < 0 || my_r >= rows) {
            // row -1 marks an assignment dropped at capacity (paradigm B)
            if (s == 0 && !(allow_dropped && my_r == -1)) record_error(err, MOE_DEVERR_BOUNDS);
            my_r = -1;
        }
    }
    int rk[KMAX];
    float wk[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        rk[k] = __shfl_sync(0xffffffffu, my_r, k);
        wk[k] = __shfl_sync(0xffffffffu, my_w, k);
    }
    for (int c = c0 + lane; c < c1; c += 32) {
        // all K row loads in flight, then the fp32 sum in k order
        uint4 v[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
            if (k < K && rk[k] >= 0)
                v[k] = __ldg(reinterpret_cast<const uint4*>(y + static_cast<long long>(rk[k]) * D) + c);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            if (k < K && rk[k] >= 0) {
                float f[8];
                bf16x8_to_f32(v[k], f);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(wk[k], f[i], acc[i]);
            }
        }
        reinterpret_cast<uint4*>(out + static_cast<long long>(t) * D)[c] =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                       pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
    pdl_trigger();
}

cudaError_t launch_combine_rows(const uint16_t* y_perm, const int32_t* inv_perm, const float* w, int N, int D,
                                int K, long long rows, bool allow_dropped, uint16_t* out, uint32_t* err,
                                cudaStream_t st) {
    // enough warps for ~8 per SM-slot even at tiny N; a slice keeps >= 32 chunks
    const int cpr = D / 8;
    const long long target_warps = 152LL * 64;
    int nslices = static_cast<int>((target_warps + N - 1) / N);
    nslices = max(1, min(nslices, cpr / 32));
    const long long items = static_cast<long long>(N) * nslices;
    const int warps_per_cta = kCombThreads / 32;
    const long long grid = (items + warps_per_cta - 1) / warps_per_cta;
    const unsigned g = static_cast<unsigned>(grid);
    auto kern = (K <= 2) ? combine_kernel<2> : (K <= 8) ? combine_kernel<8> : combine_kernel<32>;
    return launch_kernel(kern, dim3(g), dim3(kCombThreads), 0, st, y_perm, inv_perm, w, N, D, K, nslices, rows,
                         allow_dropped, out, err);
}

cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* inv_perm, const float* w, int N,
                           int D, int K, uint16_t* out, uint32_t* err, cudaStream_t st) {
    return launch_combine_rows(y_perm, inv_perm, w, N, D, K, static_cast<long long>(N) * K, false, out, err, st);
}

}  // namespace moe
