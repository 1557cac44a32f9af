// route_common.cuh -- routing arithmetic shared by the router kernels
// (route_reduce.cu) and the one-launch decode layer (layer_decode.cu), so that
// every path forms the same logits, picks the same experts with the same
// weights and places the assignments in the same rows, bit for bit.
//
// "MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im):
//   第一层 "Router 与 Top-K 的算法细节" -- logits = x . W_gate, top-K of the
//     logits, softmax over the K selected only, or (DeepSeek) sigmoid of each
//     selected logit divided by their sum;
//   第二层 范式 A Step 1 -- per-expert counts, their exclusive prefix sum
//     (expert_offsets) and the stable placement of assignment (t, k) in
//     (t, k) order inside its expert's segment.
// The per-expert bias of "MoE 大规模分布式推理工程实战" (ybb.press), 4.1 is
// added to the logits before selection.
#pragma once

#include <math.h>

#include "device.cuh"

namespace moe {

// (va, ia) comes before (vb, ib): larger value first, lower index on ties.
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// One token's routing, by one warp: lanes 0..K-1 return pick `lane` (its
// expert id, -1 only for NaN logits, and its weight); *bad is set when a pick
// is not a valid expert.
//   1. each lane owns experts e = lane + 32 j and forms logit[e] as the sum of
//      the k-split partials in split order, plus bias[e] (fp32);
//   2. K rounds of a warp arg-max under the order (value desc, index asc):
//      every lane proposes its best expert that comes after the previous
//      pick, a butterfly of shuffles agrees on the winner;
//   3. lanes 0..K-1 compute the weights of the K picks.
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

// ---------------------------------------------------------------------------
// Router logits of a decode-sized call on the CUDA cores: one group of
// kSmallRouteThreads threads forms expert e's logits for all N tokens.
// Thread `tid` of the group holds chunks c = tid + 256 i of W_gate row e
// (8 bf16 each, loaded once) and, 8 tokens at a time, forms its part of each
// token's dot product in element order; lanes are summed by a butterfly of
// shuffles, the group's 8 warps in warp order.  `sync` is the group's
// barrier; s_part is the group's [8][kSmallRouteMaxN] scratch.  Threads
// 0..N-1 of the group store logits[t][e].
// ---------------------------------------------------------------------------
constexpr int kSmallRouteThreads = 256;
constexpr int kSmallRouteMaxChunks = 4;  // 16-byte chunks of a W_gate row per thread: D <= 8192

template <typename Sync>
__device__ __forceinline__ void small_logits_expert(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wg,
                                                    int N, int D, int E, int e, int tid,
                                                    float (*s_part)[kSmallRouteMaxN], float* __restrict__ logits,
                                                    Sync sync) {
    const int lane = tid & 31, warp = tid >> 5;
    const int chunks = D / 8;
    uint4 wv[kSmallRouteMaxChunks];
    const uint4* wrow = reinterpret_cast<const uint4*>(wg + static_cast<long long>(e) * D);
#pragma unroll
    for (int i = 0; i < kSmallRouteMaxChunks; ++i) {
        const int c = tid + i * kSmallRouteThreads;
        wv[i] = (c < chunks) ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0);
    }
    for (int n0 = 0; n0 < N; n0 += 8) {
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = 0.0f;
#pragma unroll
        for (int i = 0; i < kSmallRouteMaxChunks; ++i) {
            const int c = tid + i * kSmallRouteThreads;
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
    sync();
    if (tid < N) {
        float v = 0.0f;
#pragma unroll
        for (int w8 = 0; w8 < kSmallRouteThreads / 32; ++w8) v += s_part[w8][tid];
        logits[static_cast<long long>(tid) * E + e] = v;
    }
}

// ---------------------------------------------------------------------------
// The permutation indices of a small call, by one warp, from the experts of
// its A assignments in (t, k) order (s_id, -1 = not a valid expert) and their
// counts (s_cnt[0..E-1]):
//   - s_cnt[e] becomes the exclusive prefix (expert_offsets), s_cnt[E] the
//     rows placed; s_off (optional) keeps a copy of the offsets;
//   - assignment i = t*K + k of expert e takes row offsets[e] + (the number of
//     earlier assignments of e), 32 assignments at a time; s_src[row] = t and
//     s_inv[i] (optional) = row, or -1 for an invalid expert; s_cnt[e] ends
//     as offsets[e + 1].
// With `writer`, the offsets, perm_src and inv_perm also go to global memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void place_rows_warp(const int* s_id, int A, int K, int E, int* s_cnt, int* s_src,
                                                int* s_off, int* s_inv, bool writer, int32_t* offsets,
                                                int32_t* perm_src, int32_t* inv_perm, int lane) {
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
            if (s_off) s_off[e] = excl;
            if (writer) offsets[e] = excl;
        }
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) {
        s_cnt[E] = carry;  // rows placed (assignments with a valid expert)
        if (s_off) s_off[E] = carry;
        if (writer) offsets[E] = carry;
    }
    __syncwarp();
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
            if (s_inv) s_inv[i] = r;
            if (writer) {
                inv_perm[i] = r;
                if (ok) perm_src[r] = i / K;
            }
        }
    }
}

}  // namespace moe
