// route_reduce.cu -- the small kernels that follow a split-K GEMM.
//
// route_topk: router top-K and weights ("MoE 推理完整机制：从 Router 到 Expert
// Parallelism 的一切" (zoe.im), 第一层 "Router 与 Top-K 的算法细节": top-K of
// the logits, softmax over the K selected only, or the DeepSeek variant --
// sigmoid of each logit, then divide by the sum over the K selected; the
// per-expert bias of "MoE 大规模分布式推理工程实战" (ybb.press), 4.1 is added
// to the logits before selection).  One warp per token (topk_token in
// route_common.cuh); lanes 0..K-1 store the ids and weights.
//
// route_topk_permute: route_topk and the permutation of a decode-sized call
// (at most 256 assignments) in one launch, below.
//
// route_logits_small: the router logits of a decode-sized call (N <= 32) on
// the CUDA cores.  The tensor-core GEMM's fixed pipeline latency dominates a
// product of a few token rows with W_gate; here one CTA per expert loads its
// W_gate row once, spread over all threads (16-byte loads), and forms every
// token's dot product in a fixed order (small_logits_expert), so the logits
// are deterministic; route_topk reads them as a single split.
//
// ffn_reduce_*: sum the k-split partials of a grouped-FFN GEMM in split order
// and apply the epilogue (SwiGLU or plain) to bf16.
#include <math.h>

#include "route_common.cuh"

namespace moe {

constexpr int kTopkWarps = 8;

template <int J>
__global__ void __launch_bounds__(kTopkWarps * 32)
route_topk_kernel(const float* __restrict__ partial, int splits, long long split_stride, int ldp,
                  const float* __restrict__ bias, int N, int E, int K, int mode,
                  float* __restrict__ logits_out, int32_t* __restrict__ ids, float* __restrict__ w,
                  uint32_t* err) {
    const int lane = threadIdx.x & 31;
    const long long t = static_cast<long long>(blockIdx.x) * kTopkWarps + (threadIdx.x >> 5);
    pdl_wait();
    if (t >= N) return;
    int pick;
    float weight;
    bool bad;
    topk_token<J>(partial, splits, split_stride, ldp, bias, t, E, K, mode, logits_out, lane, &pick, &weight, &bad);
    if (bad && lane == 0) record_error(err, MOE_DEVERR_BOUNDS);
    if (lane < K) {
        ids[t * K + lane] = pick;
        w[t * K + lane] = weight;
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// route_topk_permute: top-K, weights and the permutation of a decode-sized
// call (at most kFusedRoutePermute assignments) in one launch
// ("MoE 推理完整机制" 第一层 top-K and weights, then 第二层 范式 A Step 1:
// per-expert counts, their exclusive prefix sum expert_offsets, the stable
// placement in (t, k) order and the token-row copy).  Every CTA computes the
// whole routing of the call in shared memory (the host uses it for up to 8
// tokens: one warp each); CTA 0 stores ids, weights, expert_offsets, perm_src and
// inv_perm, and the CTAs share the row copy (permuted row r by CTA
// r mod gridDim.x).  Bits identical to route_topk + the permutation kernels.
// ---------------------------------------------------------------------------
constexpr int kFusedRoutePermute = kFusedRoutePermuteMax;

template <int J>
__global__ void __launch_bounds__(kTopkWarps * 32)
route_topk_permute_kernel(const float* __restrict__ partial, int splits, long long split_stride, int ldp,
                          const float* __restrict__ bias, int N, int E, int K, int mode,
                          float* __restrict__ logits_out, int32_t* __restrict__ ids, float* __restrict__ w,
                          const uint16_t* __restrict__ x, int D, int32_t* __restrict__ offsets,
                          int32_t* __restrict__ perm_src, int32_t* __restrict__ inv_perm,
                          uint16_t* __restrict__ x_perm, uint32_t* err) {
    __shared__ int s_id[kFusedRoutePermute];   // the call's assignments in (t, k) order
    __shared__ int s_src[kFusedRoutePermute];  // token of each permuted row
    extern __shared__ int s_cnt[];             // [E + 1]: counts, then the first free row of each expert
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int A = N * K;
    const bool writer = blockIdx.x == 0;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) s_cnt[e] = 0;
    pdl_wait();
    __syncthreads();
    // 1. top-K of every token (warp per token), as route_topk_kernel
    bool any_bad = false;
    for (int t = warp; t < N; t += kTopkWarps) {
        int pick;
        float weight;
        bool bad;
        topk_token<J>(partial, splits, split_stride, ldp, bias, t, E, K, mode, writer ? logits_out : nullptr, lane,
                      &pick, &weight, &bad);
        any_bad |= bad;
        if (lane < K) {
            s_id[t * K + lane] = pick;
            if (pick >= 0) atomicAdd(&s_cnt[pick], 1);
            if (writer) {
                ids[static_cast<long long>(t) * K + lane] = pick;
                w[static_cast<long long>(t) * K + lane] = weight;
            }
        }
    }
    if (writer && any_bad && lane == 0) record_error(err, MOE_DEVERR_BOUNDS);
    __syncthreads();
    // 2. exclusive prefix of the counts (expert_offsets) and 3. the stable
    // placement in (t, k) order, by warp 0
    if (warp == 0)
        place_rows_warp(s_id, A, K, E, s_cnt, s_src, nullptr, nullptr, writer, offsets, perm_src, inv_perm, lane);
    __syncthreads();
    // 4. the row copy: permuted row r <- token s_src[r], 16-byte chunks
    const int rows = x_perm ? s_cnt[E] : 0;  // no copy for an index-only permutation
    const int chunks = D / 8;
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<long long>(s_src[r]) * D);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<long long>(r) * D);
        for (int c = threadIdx.x; c < chunks; c += blockDim.x) dst[c] = src[c];
    }
    pdl_trigger();
}

// One CTA per expert (blockIdx.x), kSmallRouteThreads threads.
__global__ void __launch_bounds__(kSmallRouteThreads)
route_logits_small_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wg, int N, int D, int E,
                          float* __restrict__ logits) {
    __shared__ float s_part[kSmallRouteThreads / 32][kSmallRouteMaxN];
    pdl_wait();
    small_logits_expert(x, wg, N, D, E, static_cast<int>(blockIdx.x), static_cast<int>(threadIdx.x), s_part, logits,
                        [] { __syncthreads(); });
    pdl_trigger();
}

cudaError_t launch_route_logits_small(const uint16_t* x, const uint16_t* wg, int N, int D, int E, float* logits,
                                      cudaStream_t st) {
    if (N > kSmallRouteMaxN || D / 8 > kSmallRouteThreads * kSmallRouteMaxChunks) return cudaErrorInvalidValue;
    return launch_kernel(route_logits_small_kernel, dim3(E), dim3(kSmallRouteThreads), 0, st, x, wg, N, D, E, logits);
}

cudaError_t launch_route_topk(const float* partial, int splits, long long split_stride, int ldp,
                              const float* bias, int N, int E, int K, int mode, float* logits_out,
                              int32_t* ids, float* w, uint32_t* err, cudaStream_t st) {
    const int grid = (N + kTopkWarps - 1) / kTopkWarps;
    const int threads = kTopkWarps * 32;
#define MOE_TOPK_CASE(J_)                                                                            \
    if (E <= 32 * J_)                                                                                \
        return launch_kernel(route_topk_kernel<J_>, dim3(grid), dim3(threads), 0, st, partial, splits, \
                             split_stride, ldp, bias, N, E, K, mode, logits_out, ids, w, err);
    MOE_TOPK_CASE(1)
    MOE_TOPK_CASE(2)
    MOE_TOPK_CASE(4)
    MOE_TOPK_CASE(8)
    MOE_TOPK_CASE(16)
    MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_route_topk_permute(const float* partial, int splits, long long split_stride, int ldp,
                                      const float* bias, int N, int E, int K, int mode, float* logits_out,
                                      int32_t* ids, float* w, const uint16_t* x, int D, int32_t* offsets,
                                      int32_t* perm_src, int32_t* inv_perm, uint16_t* x_perm, int grid,
                                      uint32_t* err, cudaStream_t st) {
    if (static_cast<long long>(N) * K > kFusedRoutePermute || grid < 1) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(E + 1) * sizeof(int);
    const int threads = kTopkWarps * 32;
#define MOE_TOPK_PERM_CASE(J_)                                                                                 \
    if (E <= 32 * J_)                                                                                          \
        return launch_kernel(route_topk_permute_kernel<J_>, dim3(grid), dim3(threads), smem, st, partial, splits, \
                             split_stride, ldp, bias, N, E, K, mode, logits_out, ids, w, x, D, offsets, perm_src,   \
                             inv_perm, x_perm, err);
    MOE_TOPK_PERM_CASE(1)
    MOE_TOPK_PERM_CASE(2)
    MOE_TOPK_PERM_CASE(4)
    MOE_TOPK_PERM_CASE(8)
    MOE_TOPK_PERM_CASE(16)
    MOE_TOPK_PERM_CASE(32)
#undef MOE_TOPK_PERM_CASE
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// grouped-FFN split-K reductions; one thread per 4 output columns of a row
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
ffn_reduce_swiglu_kernel(const float* __restrict__ partial, int splits, long long split_stride, int ldp,
                         int rows, int Dff, int half, uint16_t* __restrict__ h) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int q = Dff / 4;
    pdl_wait();
    if (i >= static_cast<long long>(rows) * q) return;
    const long long r = i / q;
    const int c = static_cast<int>(i - r * q) * 4;
    const int tile = c / half, j = c - tile * half;          // half = BN/2, a multiple of 4
    const float* g = partial + r * ldp + static_cast<long long>(tile) * 2 * half + j;
    float4 gs = *reinterpret_cast<const float4*>(g);
    float4 us = *reinterpret_cast<const float4*>(g + half);
    for (int sp = 1; sp < splits; ++sp) {
        const float4 a = *reinterpret_cast<const float4*>(g + sp * split_stride);
        const float4 b = *reinterpret_cast<const float4*>(g + sp * split_stride + half);
        gs.x += a.x; gs.y += a.y; gs.z += a.z; gs.w += a.w;
        us.x += b.x; us.y += b.y; us.z += b.z; us.w += b.w;
    }
    uint2 o;
    o.x = pack_bf16x2(silu_f32(gs.x) * us.x, silu_f32(gs.y) * us.y);
    o.y = pack_bf16x2(silu_f32(gs.z) * us.z, silu_f32(gs.w) * us.w);
    *reinterpret_cast<uint2*>(h + r * Dff + c) = o;
    pdl_trigger();
}

__global__ void __launch_bounds__(256)
ffn_reduce_store_kernel(const float* __restrict__ partial, int splits, long long split_stride, int ldp,
                        int rows, int ncols, bool silu, uint16_t* __restrict__ y) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int q = ncols / 4;
    pdl_wait();
    if (i >= static_cast<long long>(rows) * q) return;
    const long long r = i / q;
    const int c = static_cast<int>(i - r * q) * 4;
    const float* p = partial + r * ldp + c;
    float4 s = *reinterpret_cast<const float4*>(p);
    for (int sp = 1; sp < splits; ++sp) {
        const float4 a = *reinterpret_cast<const float4*>(p + sp * split_stride);
        s.x += a.x; s.y += a.y; s.z += a.z; s.w += a.w;
    }
    if (silu) {
        s.x = silu_f32(s.x); s.y = silu_f32(s.y); s.z = silu_f32(s.z); s.w = silu_f32(s.w);
    }
    uint2 o;
    o.x = pack_bf16x2(s.x, s.y);
    o.y = pack_bf16x2(s.z, s.w);
    *reinterpret_cast<uint2*>(y + r * ncols + c) = o;
    pdl_trigger();
}

cudaError_t launch_ffn_reduce_swiglu(const float* partial, int splits, long long split_stride, int ldp,
                                     int rows, int Dff, int bn, uint16_t* h, cudaStream_t st) {
    const long long items = static_cast<long long>(rows) * (Dff / 4);
    const long long grid = (items + 255) / 256;
    if (grid == 0) return cudaSuccess;
    return launch_kernel(ffn_reduce_swiglu_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, partial,
                         splits, split_stride, ldp, rows, Dff, bn / 2, h);
}

cudaError_t launch_ffn_reduce_store(const float* partial, int splits, long long split_stride, int ldp,
                                    int rows, int ncols, bool silu, uint16_t* y, cudaStream_t st) {
    const long long items = static_cast<long long>(rows) * (ncols / 4);
    const long long grid = (items + 255) / 256;
    if (grid == 0) return cudaSuccess;
    return launch_kernel(ffn_reduce_store_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, partial,
                         splits, split_stride, ldp, rows, ncols, silu, y);
}

// ---------------------------------------------------------------------------
// Routing statistics and the online bias step ("MoE 大规模分布式推理工程实战"
// (ybb.press), 4.1 Router 辅助损失的工程化实现: the EMA of per-expert
// assignment fractions, then the KL of the normalised EMA to uniform and the
// dynamic-bias update).  One CTA, thread e = expert e; sums are a fixed-order
// tree over shared memory, so the result is deterministic.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_sum_1024(float v, float* sh) {
    sh[threadIdx.x] = v;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
        __syncthreads();
    }
    const float r = sh[0];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(1024)
routing_stats_kernel(const int32_t* __restrict__ offsets, int E, float decay, float step, float* __restrict__ ema,
                     float* __restrict__ bias, float* __restrict__ kl_out) {
    __shared__ float sh[1024];
    pdl_wait();
    const int e = threadIdx.x;
    const int total = offsets[E];
    if (total <= 0) {  // no assignments: nothing changes
        if (e == 0 && kl_out) *kl_out = 0.0f;
        pdl_trigger();
        return;
    }
    float m = 0.0f;
    if (e < E) {
        const float frac = static_cast<float>(offsets[e + 1] - offsets[e]) / static_cast<float>(total);
        m = decay * ema[e] + (1.0f - decay) * frac;
        ema[e] = m;
    }
    const float sum = block_sum_1024(m, sh);
    float kl = 0.0f;
    if (e < E) {
        const float f = m / sum;
        kl = f * logf(f * static_cast<float>(E) + 1e-9f);
        if (bias) bias[e] += step * (static_cast<float>(E) * f - 1.0f);
    }
    kl = block_sum_1024(kl, sh);
    if (e == 0 && kl_out) *kl_out = kl;
    pdl_trigger();
}

cudaError_t launch_routing_stats(const int32_t* offsets, int E, float decay, float step, float* ema, float* bias,
                                 float* kl_out, cudaStream_t st) {
    int threads = 32;
    while (threads < E) threads <<= 1;  // power of two for the tree sum
    return launch_kernel(routing_stats_kernel, dim3(1), dim3(threads), 0, st, offsets, E, decay, step, ema, bias,
                         kl_out);
}

}  // namespace moe
