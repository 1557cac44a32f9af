// route_reduce.cu -- the small kernels that follow a split-K GEMM.
//
// route_topk: router top-K and weights ("MoE 推理完整机制：从 Router 到 Expert
// Parallelism 的一切" (zoe.im), 第一层 "Router 与 Top-K 的算法细节": top-K of
// the logits, softmax over the K selected only, or the DeepSeek variant --
// sigmoid of each logit, then divide by the sum over the K selected; the
// per-expert bias of "MoE 大规模分布式推理工程实战" (ybb.press), 4.1 is added
// to the logits before selection).  One warp per token:
//   1. each lane owns experts e = lane + 32 j and forms logit[e] as the sum of
//      the GEMM's k-split partials in split order, plus bias[e] (fp32);
//   2. K rounds of a warp arg-max under the order (value desc, index asc):
//      every lane proposes its best expert that comes after the previous
//      pick, a butterfly of shuffles agrees on the winner;
//   3. lanes 0..K-1 compute the weights of the K picks and store ids/weights.
//
// route_topk_permute: route_topk and the permutation of a decode-sized call
// (at most 256 assignments) in one launch, below.
//
// route_logits_small: the router logits of a decode-sized call (N <= 32) on
// the CUDA cores.  The tensor-core GEMM's fixed pipeline latency dominates a
// product of a few token rows with W_gate; here one CTA per expert loads its
// W_gate row once, spread over all threads (16-byte loads), and forms every
// token's dot product in a fixed order, so the logits are deterministic;
// route_topk reads them as a single split.
//
// ffn_reduce_*: sum the k-split partials of a grouped-FFN GEMM in split order
// and apply the epilogue (SwiGLU or plain) to bf16.
#include <math.h>

#include "device.cuh"

namespace moe {

constexpr int kTopkWarps = 8;

// (va, ia) comes before (vb, ib): larger value first, lower index on ties.
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// One token's routing, by one warp: lanes 0..K-1 return pick `lane` (its
// expert id, -1 only for NaN logits, and its weight); *bad is set when a pick
// is not a valid expert.  Shared by route_topk_kernel and the fused decode
// route + permute kernel, so both give the same bits.
template <int J>  // logits per lane: E <= 32 * J
__device__ __forceinline__ void topk_token(const float* __restrict__ partial, int splits, long long split_stride,
                                           int ldp, const float* __restrict__ bias, long long t, int E, int K,
                                           int mode, float* __restrict__ logits_out, int lane, int* pick,
                                           float* weight, bool* bad_out) {
    // logit[e] = split 0 + split 1 + ... in split order.  The loads of SG
    // splits for all J experts of the lane are issued before any of them is
    // summed, so a warp waits about once per SG splits, not once per expert.
    constexpr int SG = (32 / J > 16) ? 16 : 32 / J;
    float v[J];
#pragma unroll
    for (int j = 0; j < J; ++j) v[j] = 0.0f;
    const float* prow = partial + t * ldp + lane;
    for (int s0 = 0; s0 < splits; s0 += SG) {
        float pv[SG][J];
#pragma unroll
        for (int g = 0; g < SG; ++g)
#pragma unroll
            for (int j = 0; j < J; ++j)
                pv[g][j] = (s0 + g < splits && lane + 32 * j < E) ? prow[(s0 + g) * split_stride + 32 * j] : 0.0f;
#pragma unroll
        for (int g = 0; g < SG; ++g)
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (s0 + g < splits) v[j] = (s0 + g == 0) ? pv[g][j] : v[j] + pv[g][j];
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        if (e < E) {
            if (bias) v[j] += bias[e];
            if (logits_out) logits_out[t * E + e] = v[j];
        } else {
            v[j] = -INFINITY;
        }
    }
    float prev_v = INFINITY;
    int prev_i = -1;
    float my_v = 0.0f;   // lane k keeps pick k
    int my_i = -1;
    for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            if (e < E && before(prev_v, prev_i, v[j], e) && before(v[j], e, bv, bi)) {
                bv = v[j];
                bi = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (before(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == k) {
            my_v = bv;
            my_i = bi;
        }
        prev_v = bv;
        prev_i = bi;
    }
    const bool bad = (lane < K) && (my_i < 0 || my_i >= E);  // only with NaN logits
    *bad_out = __any_sync(0xffffffffu, bad);
    // weights over the K picks
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    float s = 0.0f;
    if (lane < K) s = (mode == 0) ? expf(my_v - top) : 1.0f / (1.0f + expf(-my_v));
    float sum = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    *pick = bad ? -1 : my_i;
    *weight = (sum > 0.0f) ? s / sum : 1.0f / static_cast<float>(K);
}

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
    // 2. exclusive prefix of the counts (warp 0), expert_offsets
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = (e < E) ? s_cnt[e] : 0;
            int v = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            const int excl = carry + v - c;
            if (e < E) {
                s_cnt[e] = excl;
                if (writer) offsets[e] = excl;
            }
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) {
            s_cnt[E] = carry;  // rows placed (assignments with a valid expert)
            if (writer) offsets[E] = carry;
        }
        // 3. stable placement in (t, k) order, 32 assignments at a time
        const unsigned lt = (1u << lane) - 1u;
        for (int base = 0; base < A; base += 32) {
            const int i = base + lane;
            const int e = (i < A) ? s_id[i] : -1;
            const bool ok = e >= 0;
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1 - lane);
            const int r = ok ? s_cnt[e] + __popc(peers & lt) : -1;
            __syncwarp();
            if (ok && __popc(peers & lt) == 0) s_cnt[e] += __popc(peers);
            __syncwarp();
            if (i < A) {
                if (ok) s_src[r] = i / K;
                if (writer) {
                    inv_perm[i] = r;
                    if (ok) perm_src[r] = i / K;
                }
            }
        }
    }
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

constexpr int kSmallRouteThreads = 256;
constexpr int kSmallRouteMaxChunks = 4;  // 16-byte chunks of a W_gate row per thread: D <= 8192

// One CTA per expert e: thread t holds chunks c = t + 256 i of W_gate row e
// (8 bf16 each, loaded once) and, 8 tokens at a time, forms its part of each
// token's dot product in element order; lanes are summed by a butterfly of
// shuffles, the 8 warps in warp order.
__global__ void __launch_bounds__(kSmallRouteThreads)
route_logits_small_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wg, int N, int D, int E,
                          float* __restrict__ logits) {
    __shared__ float s_part[kSmallRouteThreads / 32][kSmallRouteMaxN];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x;
    const int chunks = D / 8;
    pdl_wait();
    uint4 wv[kSmallRouteMaxChunks];
    const uint4* wrow = reinterpret_cast<const uint4*>(wg + static_cast<long long>(e) * D);
#pragma unroll
    for (int i = 0; i < kSmallRouteMaxChunks; ++i) {
        const int c = threadIdx.x + i * kSmallRouteThreads;
        wv[i] = (c < chunks) ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0);
    }
    for (int n0 = 0; n0 < N; n0 += 8) {
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = 0.0f;
#pragma unroll
        for (int i = 0; i < kSmallRouteMaxChunks; ++i) {
            const int c = threadIdx.x + i * kSmallRouteThreads;
            if (c < chunks) {
                uint4 xv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (n0 + u < N) xv[u] = __ldg(reinterpret_cast<const uint4*>(x + static_cast<long long>(n0 + u) * D) + c);
                const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (n0 + u < N) {
                        const uint32_t xx[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
                        float sacc = acc[u];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            sacc = fmaf(__uint_as_float(xx[k] << 16), __uint_as_float(ww[k] << 16), sacc);
                            sacc = fmaf(__uint_as_float(xx[k] & 0xffff0000u), __uint_as_float(ww[k] & 0xffff0000u), sacc);
                        }
                        acc[u] = sacc;
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            float v = acc[u];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0 && n0 + u < N) s_part[warp][n0 + u] = v;
        }
    }
    __syncthreads();
    if (threadIdx.x < N) {
        float v = 0.0f;
#pragma unroll
        for (int w8 = 0; w8 < kSmallRouteThreads / 32; ++w8) v += s_part[w8][threadIdx.x];
        logits[static_cast<long long>(threadIdx.x) * E + e] = v;
    }
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
