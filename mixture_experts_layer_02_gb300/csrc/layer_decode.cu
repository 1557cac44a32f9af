// layer_decode.cu -- the whole MoE layer of a small decode batch (up to
// kLayerDecodeMaxN tokens) in one persistent cooperative launch.
//
// "MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im):
// 第一层 (router logits, top-K, weights), 第二层 范式 A Steps 1-3 (placement,
// one FFN per expert, weighted combine in token order), and 第四层 "DeepGEMM
// 的 MegaMoE Kernel": the expert computation of a decode step as one
// persistent kernel instead of a chain of launches.
//
// A decode step of a few tokens moves tens of MB of expert weights and
// almost nothing else; a chain of five launches pays each launch's fill and
// drain on that short stream.  Here every CTA (one per SM) runs four phases,
// separated by two grid barriers:
//
//   1. router logits: expert e's logits for all N tokens by a group of 256
//      threads (small_logits_expert, the same arithmetic as
//      route_logits_small_kernel), two groups per CTA;
//   -- grid barrier 1 --
//   2. routing: every CTA reads the N x E logits and computes the routing
//      itself, spread over all its threads (one warp walking the experts
//      serially would take microseconds): each (token, expert) counts the
//      experts that come before it in the order (score desc, index asc), and
//      rank k < K makes it pick k -- topk_token's picks; the weights use
//      topk_token's arithmetic; one block scan of the per-expert counts gives
//      expert_offsets and the touched experts; assignment i takes row
//      offsets[e] + (earlier assignments of e).  Same bits as the separate
//      kernels; CTA 0 stores them; CTAs share the x_perm row copy.  As soon
//      as the picks are known (before the weights and the placement), each
//      CTA starts bulk copies of the W2 rows its phase 4 will read into its
//      shared memory (when they fit: one token) or asks L2 to prefetch them,
//      so that the W2 stream runs under GEMM1's;
//   3. GEMM1 + activation: one warp per (expert, f) item, f < D_ffn, each
//      CTA a contiguous range of items: the warp streams W1[e][f] (and
//      W3[e][f]) through registers with 16-byte loads, forms the dot products
//      with the expert's token rows (<= N, from shared memory) in fp32 with
//      paired fused multiply-adds, reduces across lanes and stores
//      h[row][f] = bf16(silu(g) * u) (SwiGLU) or bf16(silu(g)) (SiLU);
//   -- grid barrier 2 --
//   4. GEMM2 + combine: CTA b owns output columns [d0, d1) of every row.
//      It stages h (all rows, as fp32) in shared memory, forms y_perm[row][d] =
//      bf16(sum_f h[row][f] W2[e][d][f]) for its columns, then
//      out[t][d] = bf16(sum_k w[t,k] * y_perm[inv_perm[t,k]][d]) in k order
//      (fp32 fused multiply-adds from 0, as combine_kernel).
//
// At these sizes the GEMMs are matrix-vector products (at most N rows per
// expert), so they run on the CUDA cores with fp32 accumulation: the bound
// is the weight stream, which 16 warps of 16-byte loads per SM keep at HBM
// speed.  Routing, placement and the combine give the bits of the separate
// kernels; h and y round the same quantities to bf16 but sum in another
// order than the tensor-core GEMMs.
//
// The grid barriers count arrivals in one 64-bit word of the workspace
// header, which grows by the grid size per barrier and is never reset: each
// CTA reads it once at the start (rounded down to a multiple of the grid
// size, it is the launch's base), then at barrier k adds 1 with release
// semantics and waits (acquire loads) until it reaches base + k * grid, so
// no per-call clearing is needed and a barrier costs one fire-and-forget add
// and the polls.  Every wait is
// bounded (kWaitLimitNs); on expiry the CTA records MOE_DEVERR_TIMEOUT, waits
// (bounded) for its own bulk copies and returns.
#include "route_common.cuh"

namespace moe {

constexpr int kLdThreads = 512;
constexpr int kLdWarps = kLdThreads / 32;
constexpr uint32_t kLdBulkBytes = 32768;  // largest single W2 bulk copy

// 16-byte chunks per lane and operand in flight in GEMM1 for NR = the most
// rows an expert can have (N rounded up to a power of two): fewer as the
// per-row accumulators take registers.
template <int NR>
struct LdCfg {
    static constexpr int B1 = NR <= 2 ? 8 : 4;
    // GEMM2: W2 columns per item, sharing each loaded chunk of the expert's h rows
    static constexpr int G2 = NR <= 1 ? 8 : (NR <= 2 ? 4 : (NR <= 4 ? 2 : 1));
};


__device__ __forceinline__ void bf16x8_f32(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// 8 bf16 (one 16-byte chunk) -> 4 float2 pairs (element 2i, 2i + 1)
__device__ __forceinline__ void bf16x8_f32x2(const uint4& v, float2 (&f)[4]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

__device__ __forceinline__ uint16_t bf16_rn_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// One GEMM2 item: columns dd0 .. dd0 + ncol of the CTA's, for the ne rows of
// one expert starting at row r0.  Per 16-byte chunk c of D_ffn (lane-strided)
// the item loads the rows' h (fp32, shared memory) once and the ncol W2 rows'
// chunk (rows Dff apart from `w`, in shared memory when SMEM, else global),
// and accumulates with paired fused multiply-adds; then a butterfly per
// (column, row) and lane 0 stores y (bf16) to s_y and y_perm.
struct G2Item {
    int r0, ne, dd0, ncol;
};
template <int NR, bool SMEM>
__device__ __forceinline__ void gemm2_item(const G2Item& g, const uint4* __restrict__ w, const float* __restrict__ s_hf,
                                           int Dff, int lane, uint16_t* s_y, int nd, uint16_t* __restrict__ y_perm,
                                           int D, int d0) {
    constexpr int C = LdCfg<NR>::G2;
    const int chunks2 = Dff / 8;
    float2 acc[C][NR];
#pragma unroll
    for (int j = 0; j < C; ++j)
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[j][r] = make_float2(0.0f, 0.0f);
    for (int c = lane; c < chunks2; c += 32) {
        uint4 wv[C];
#pragma unroll
        for (int j = 0; j < C; ++j)
            if (j < g.ncol) wv[j] = SMEM ? w[j * chunks2 + c] : __ldg(w + j * chunks2 + c);
        // h chunk of row r (fp32 pairs); held across the C columns when C > 1
        auto h_chunk = [&](int r, float2 (&hf)[4]) {
            const float4* hp = reinterpret_cast<const float4*>(s_hf + static_cast<size_t>(g.r0 + r) * Dff + c * 8);
            const float4 ha = hp[0], hb = hp[1];
            hf[0] = make_float2(ha.x, ha.y);
            hf[1] = make_float2(ha.z, ha.w);
            hf[2] = make_float2(hb.x, hb.y);
            hf[3] = make_float2(hb.z, hb.w);
        };
        constexpr int HR = C > 1 ? NR : 1;
        float2 hf[HR][4];
        if (C > 1) {
#pragma unroll
            for (int r = 0; r < HR; ++r)
                if (r < g.ne) h_chunk(r, hf[r]);
        }
#pragma unroll
        for (int j = 0; j < C; ++j) {
            if (j < g.ncol) {
                float2 wf[4];
                bf16x8_f32x2(wv[j], wf);
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    if (r < g.ne) {
                        float2 hr[4];
                        if (C > 1) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) hr[i] = hf[r < HR ? r : 0][i];
                        } else {
                            h_chunk(r, hr);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[j][r] = __ffma2_rn(hr[i], wf[i], acc[j][r]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < C; ++j)
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            if (j < g.ncol && r < g.ne) {
                const float y = warp_sum(acc[j][r].x + acc[j][r].y);
                if (lane == 0) {
                    const uint16_t yb = bf16_rn_bits(y);
                    s_y[(g.r0 + r) * nd + g.dd0 + j] = yb;
                    y_perm[static_cast<long long>(g.r0 + r) * D + d0 + g.dd0 + j] = yb;
                }
            }
        }
}

// Grid-wide barrier over the CTAs of a cooperative launch.  Thread 0 adds 1
// to the arrival count with release semantics (the CTA's writes, ordered
// before it by __syncthreads, become visible to whoever acquires the count)
// and polls the count with acquire loads until it reaches *s_base + past_base, bounded
// by kWaitLimitNs.  `withhold` (test hook) makes this CTA leave without
// arriving.  Returns false when the CTA must stop.
__device__ __forceinline__ bool grid_barrier(unsigned long long* count, const unsigned long long* s_base,
                                             unsigned long long past_base, uint32_t* err, volatile int* s_abort,
                                             bool withhold) {
    __syncthreads();
    if (threadIdx.x == 0) {
        if (withhold) {
            *s_abort = 1;
        } else {
            const unsigned long long target = *s_base + past_base;
            red_add_release_gpu(count, 1ull);
            if (ld_acquire_gpu_u64(count) < target) {
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire_gpu_u64(count) < target) {
                    if (globaltimer_ns() - t0 > kWaitLimitNs) {
                        record_error(err, MOE_DEVERR_TIMEOUT);
                        *s_abort = 1;
                        break;
                    }
                }
            }
        }
    }
    __syncthreads();
    return *s_abort == 0;
}

template <bool SWIGLU, int NR>
__global__ void __launch_bounds__(kLdThreads, 1) layer_decode_kernel(const LayerDecodeArgs a) {
    constexpr int kLdBatch1 = LdCfg<NR>::B1;
    extern __shared__ __align__(16) unsigned char ld_smem[];
    __shared__ float s_part[2][kSmallRouteThreads / 32][kSmallRouteMaxN];
    __shared__ int s_id[kLayerDecodeMaxRows];       // expert of assignment t*K+k (-1: none)
    __shared__ float s_w[kLayerDecodeMaxRows];      // its weight
    __shared__ int s_src[kLayerDecodeMaxRows];      // token of each permuted row
    __shared__ int s_inv[kLayerDecodeMaxRows];      // row of each assignment (-1: none)
    __shared__ int s_touched[kLayerDecodeMaxRows];  // experts with rows, ascending
    __shared__ int s_wsum[kLdWarps];                // block scan: inclusive warp totals
    __shared__ int s_T;
    __shared__ volatile int s_abort;
    __shared__ __align__(8) uint64_t s_w2bar;       // W2 bulk copies landed
    __shared__ unsigned long long s_bar_base;       // the barrier count when this launch began

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = a.N, D = a.D, E = a.E, K = a.K, Dff = a.Dff, A = N * K;
    const int G = gridDim.x, b = blockIdx.x;
    const bool writer = b == 0;
    const LayerDecodeSmem L = layer_decode_smem(N, D, E, K, Dff, G, a.w2_smem != 0);
    float* s_v = reinterpret_cast<float*>(ld_smem + L.logits);   // scores: logit + bias [N][E]
    int* s_cnt = reinterpret_cast<int*>(ld_smem + L.cnt);
    int* s_off = reinterpret_cast<int*>(ld_smem + L.off);
    uint4* s_x = reinterpret_cast<uint4*>(ld_smem + L.xh);      // x rows, bf16 (phases 1-3)
    float* s_hf = reinterpret_cast<float*>(ld_smem + L.xh);     // h rows, fp32 (phase 4)
    uint16_t* s_y = reinterpret_cast<uint16_t*>(ld_smem + L.y);
    uint16_t* s_w2 = reinterpret_cast<uint16_t*>(ld_smem + L.w2);

    if (tid == 0) {
        s_abort = 0;
        mbar_init(&s_w2bar, 1);
        fence_barrier_init();
    }
    for (int e = tid; e <= E; e += kLdThreads) s_cnt[e] = 0;
    for (int i = tid; i < A; i += kLdThreads) s_id[i] = -1;
    pdl_wait();
    // every launch on the workspace passes both barriers, so the count is a
    // multiple of the grid size when it starts; CTAs already at barrier 1 add
    // less than one grid size
    if (tid == 0) s_bar_base = ld_relaxed_gpu_u64(a.bar) / G * G;
    const bool withhold = writer && a.dbg && (*a.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD);
    const int chunks = D / 8;  // 16-byte chunks of an x / W1 / W3 row
    for (int i = tid; i < N * chunks; i += kLdThreads) s_x[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);

    // ---- 1. router logits, expert e by thread group grp (named barrier 1 + grp)
    {
        const int grp = tid / kSmallRouteThreads, gtid = tid % kSmallRouteThreads;
        for (int e = b + grp * G; e < E; e += 2 * G) {
            small_logits_expert(a.x, a.wg, N, D, E, e, gtid, s_part[grp], a.logits,
                                [grp] { named_barrier_sync(1 + grp, kSmallRouteThreads); });
            named_barrier_sync(1 + grp, kSmallRouteThreads);  // s_part is reused
        }
    }
    if (!grid_barrier(a.bar, &s_bar_base, G, a.err, &s_abort, withhold)) return;

    // ---- 2. routing in every CTA, spread over all its threads
    for (int i = tid; i < N * E; i += kLdThreads) {
        float v = ld_cg_f32(a.logits + i);
        if (a.bias) v += a.bias[i % E];   // the score route_topk forms: logit + bias
        s_v[i] = v;
    }
    __syncthreads();
    // 2a. rank of (token t, expert e) among t's scores that are not NaN, in the
    //     order (score desc, index asc), counted by four lanes over a quarter of
    //     the experts each: rank k < K makes e pick k (the picks of topk_token)
    {
        const int total = N * E * 4;
        for (int base = warp * 32; base < total; base += kLdThreads) {
            const int i = base + lane;
            const int te = i >> 2, t = te / E, e = te - t * E;
            const float ve = i < total ? s_v[te] : 0.0f;
            const bool mine = i < total && ve == ve;
            int cnt = 0;
            if (mine) {
                const float* vt = s_v + t * E;
                for (int e2 = i & 3; e2 < E; e2 += 4) cnt += before(vt[e2], e2, ve, e) ? 1 : 0;
            }
            cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
            cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
            if (mine && (i & 3) == 0 && cnt < K) s_id[t * K + cnt] = e;
        }
    }
    __syncthreads();
    // 2b. the experts that received assignments, in order of first appearance
    //     among the picks (t, k): the slots of the GEMM items and W2 copies
    if (warp == 0) {
        int n = 0;
        for (int base = 0; base < A; base += 32) {
            const int i = base + lane;
            const int e = i < A ? s_id[i] : -1;
            bool first = e >= 0;
            for (int i2 = 0; i2 < i && first; ++i2) first = s_id[i2] != e;
            const unsigned m = __ballot_sync(0xffffffffu, first);
            if (first) s_touched[n + __popc(m & ((1u << lane) - 1u))] = e;
            n += __popc(m);
        }
        if (lane == 0) s_T = n;
    }
    __syncthreads();
    const int T = s_T;
    // the CTA's output columns (pairs of columns, spread evenly over the CTAs)
    const int P = D / 2;
    const int d0 = 2 * static_cast<int>(static_cast<long long>(b) * P / G);
    const int nd = 2 * static_cast<int>(static_cast<long long>(b + 1) * P / G) - d0;
    // W2 rows of the CTA's columns: expert slot i holds W2[e][d0 .. d0+nd) (contiguous)
    const uint32_t w2_bytes = static_cast<uint32_t>(nd) * Dff * 2;
    const bool staged = a.w2_smem && nd > 0 && T > 0;
    // GEMM1 items of this CTA: a contiguous range, so warp 15 has no more than the others
    const int U1 = T * Dff;
    const int u_lo = static_cast<int>(static_cast<long long>(U1) * b / G);
    const int u_hi = static_cast<int>(static_cast<long long>(U1) * (b + 1) / G);
    if (staged) {
        if (tid == kLdThreads - 32) {  // lane 0 of warp 15 issues the bulk copies
            mbar_arrive_expect_tx(&s_w2bar, w2_bytes * T);
            for (int i = 0; i < T; ++i) {
                const char* src =
                    reinterpret_cast<const char*>(a.w2 + (static_cast<long long>(s_touched[i]) * D + d0) * Dff);
                char* dst = reinterpret_cast<char*>(s_w2) + static_cast<size_t>(i) * w2_bytes;
                for (uint32_t o = 0; o < w2_bytes; o += kLdBulkBytes)
                    bulk_load_1d(dst + o, src + o, min(kLdBulkBytes, w2_bytes - o), &s_w2bar);
            }
        }
    } else if (tid < T && nd > 0 && static_cast<long long>(T) * D * Dff * 2 <= a.l2_prefetch_max) {
        l2_prefetch_bulk(a.w2 + (static_cast<long long>(s_touched[tid]) * D + d0) * Dff, w2_bytes);
    }
    // GEMM1 item u = (expert slot, f), one warp each (issuing the loads of
    // the first item here, under the rest of the routing, measured slower:
    // warps stall at the load issue and hold up the routing's barriers)
    const uint64_t pol = l2_policy_evict_first();
    uint4 v1[kLdBatch1], v3[kLdBatch1];
    const uint4* p1 = nullptr;
    const uint4* p3 = nullptr;
    auto item_rows = [&](int uu) {  // W1 (and W3) row of item uu
        const int slot = uu / Dff, f = uu - slot * Dff;
        const long long row = static_cast<long long>(s_touched[slot]) * Dff + f;
        p1 = reinterpret_cast<const uint4*>(a.w1 + row * D);
        p3 = SWIGLU ? reinterpret_cast<const uint4*>(a.w3 + row * D) : p1;
    };
    auto load_batch = [&](int c0) {  // chunks c0 + lane + 32 j of both rows
#pragma unroll
        for (int j = 0; j < kLdBatch1; ++j) {
            const int c = c0 + lane + 32 * j;
            if (c < chunks) {
                v1[j] = ld_stream_v4(p1 + c, pol);
                if (SWIGLU) v3[j] = ld_stream_v4(p3 + c, pol);
            }
        }
    };

    // 2c. weights of each token's picks, one warp per token, with topk_token's
    //     arithmetic (a pick that stayed -1 has score -inf)
    bool any_bad = false;
    for (int t = warp; t < N; t += kLdWarps) {
        const int pk = lane < K ? s_id[t * K + lane] : -1;
        const float my_v = pk >= 0 ? s_v[t * E + pk] : -INFINITY;
        const float top = __shfl_sync(0xffffffffu, my_v, 0);
        float sc = 0.0f;
        if (lane < K) sc = (a.mode == 0) ? expf(my_v - top) : 1.0f / (1.0f + expf(-my_v));
        float sum = sc;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        const float weight = (sum > 0.0f) ? sc / sum : 1.0f / static_cast<float>(K);
        any_bad |= __any_sync(0xffffffffu, lane < K && pk < 0);
        if (lane < K) {
            s_w[t * K + lane] = weight;
            if (pk >= 0) atomicAdd(&s_cnt[pk], 1);
            if (writer) {
                a.ids[t * K + lane] = pk;
                a.w[t * K + lane] = weight;
            }
        }
    }
    if (writer && any_bad && lane == 0) record_error(a.err, MOE_DEVERR_BOUNDS);
    __syncthreads();
    // 2d. expert_offsets: one block scan of the per-expert counts
    {
        const int c = tid < E ? s_cnt[tid] : 0;
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) s_wsum[warp] = inc;
        __syncthreads();
        if (warp == 0) {
            int wv = lane < kLdWarps ? s_wsum[lane] : 0;
#pragma unroll
            for (int o = 1; o < kLdWarps; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, wv, o);
                if (lane >= o) wv += y;
            }
            if (lane < kLdWarps) s_wsum[lane] = wv;
        }
        __syncthreads();
        const int excl = (warp > 0 ? s_wsum[warp - 1] : 0) + inc - c;
        if (tid < E) {
            s_off[tid] = excl;
            if (writer) a.offsets[tid] = excl;
        }
        if (tid == 0) {
            const int tot = s_wsum[kLdWarps - 1];
            s_off[E] = tot;  // rows placed (assignments with a valid expert)
            if (writer) a.offsets[E] = tot;
        }
    }
    __syncthreads();
    // 2e. stable placement: assignment i of expert e takes row offsets[e] + the
    //     number of earlier assignments of e
    if (tid < A) {
        const int e = s_id[tid];
        int r = -1;
        if (e >= 0) {
            r = s_off[e];
            for (int i2 = 0; i2 < tid; ++i2) r += s_id[i2] == e ? 1 : 0;
            s_src[r] = tid / K;
        }
        s_inv[tid] = r;
        if (writer) {
            a.inv_perm[tid] = r;
            if (r >= 0) a.perm_src[r] = tid / K;
        }
    }
    __syncthreads();
    const int rows = s_off[E];
    for (int r = b; r < rows; r += G) {
        uint4* dst = reinterpret_cast<uint4*>(a.x_perm + static_cast<long long>(r) * D);
        for (int c = tid; c < chunks; c += kLdThreads) dst[c] = s_x[s_src[r] * chunks + c];
    }

    // ---- 3. GEMM1 + activation
    for (int u = u_lo + warp; u < u_hi; u += kLdWarps) {
        item_rows(u);
        load_batch(0);
        const int slot = u / Dff, f = u - slot * Dff;
        const int e = s_touched[slot], r0 = s_off[e], ne = s_off[e + 1] - r0;
        float2 ag[NR], au[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) ag[r] = au[r] = make_float2(0.0f, 0.0f);
        for (int c0 = 0; c0 < chunks; c0 += 32 * kLdBatch1) {
            if (c0 > 0) load_batch(c0);
#pragma unroll
            for (int j = 0; j < kLdBatch1; ++j) {
                const int c = c0 + lane + 32 * j;
                if (c < chunks) {
                    float2 w1f[4], w3f[4];
                    bf16x8_f32x2(v1[j], w1f);
                    if (SWIGLU) bf16x8_f32x2(v3[j], w3f);
#pragma unroll
                    for (int r = 0; r < NR; ++r) {
                        if (r < ne) {
                            float2 xf[4];
                            bf16x8_f32x2(s_x[s_src[r0 + r] * chunks + c], xf);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                ag[r] = __ffma2_rn(xf[i], w1f[i], ag[r]);
                                if (SWIGLU) au[r] = __ffma2_rn(xf[i], w3f[i], au[r]);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            if (r < ne) {
                const float g = warp_sum(ag[r].x + ag[r].y);
                const float up = SWIGLU ? warp_sum(au[r].x + au[r].y) : 1.0f;
                if (lane == 0)
                    a.h[static_cast<long long>(r0 + r) * Dff + f] =
                        bf16_rn_bits(SWIGLU ? silu_f32(g) * up : silu_f32(g));
            }
        }
    }
    if (!grid_barrier(a.bar, &s_bar_base, 2ull * G, a.err, &s_abort, false)) {
        if (staged && tid == 0) {  // the bulk copies write this CTA's shared memory: let them land first
            volatile int keep_waiting = 0;
            mbar_wait(&s_w2bar, 0, &keep_waiting, a.err);
        }
        return;
    }

    // ---- 4. GEMM2 for columns [d0, d0 + nd) of every row, then the combine
    const int chunks2 = Dff / 8;  // 16-byte chunks of an h / W2 row
    for (int i = tid; i < rows * chunks2; i += kLdThreads) {  // h rows as fp32
        float2 hv[4];
        bf16x8_f32x2(ld_cg_v4(reinterpret_cast<const uint4*>(a.h) + i), hv);
        float4* dst = reinterpret_cast<float4*>(s_hf + static_cast<size_t>(i) * 8);
        dst[0] = make_float4(hv[0].x, hv[0].y, hv[1].x, hv[1].y);
        dst[1] = make_float4(hv[2].x, hv[2].y, hv[3].x, hv[3].y);
    }
    if (staged && tid == 0 && !mbar_wait(&s_w2bar, 0, &s_abort, a.err)) {
        volatile int keep_waiting = 0;  // timed out: wait once more for the copies before leaving
        mbar_wait(&s_w2bar, 0, &keep_waiting, a.err);
    }
    __syncthreads();
    if (s_abort) return;
    // item = (expert slot, up to kG2Cols consecutive columns of the CTA's);
    // the W2 rows come from shared memory (staged) or global memory
    const int per_slot = (nd + LdCfg<NR>::G2 - 1) / LdCfg<NR>::G2;
    const uint4* s_w2v = reinterpret_cast<const uint4*>(s_w2);
    for (int it = warp; it < T * per_slot; it += kLdWarps) {
        const int slot = it / per_slot, dd0 = (it - slot * per_slot) * LdCfg<NR>::G2;
        const int e = s_touched[slot];
        G2Item g{s_off[e], s_off[e + 1] - s_off[e], dd0, min(LdCfg<NR>::G2, nd - dd0)};
        if (staged)
            gemm2_item<NR, true>(g, s_w2v + (slot * nd + dd0) * chunks2, s_hf, Dff, lane, s_y, nd, a.y_perm, D, d0);
        else
            gemm2_item<NR, false>(g, reinterpret_cast<const uint4*>(a.w2 + (static_cast<long long>(e) * D + d0 + dd0) * Dff),
                                  s_hf, Dff, lane, s_y, nd, a.y_perm, D, d0);
    }
    __syncthreads();
    // combine: out[t][d0 + 2p .. +1], fp32 fused multiply-adds in k order
    const int np = nd / 2;
    for (int i = tid; i < N * np; i += kLdThreads) {
        const int t = i / np, c = 2 * (i - t * np);
        float acc0 = 0.0f, acc1 = 0.0f;
        for (int k = 0; k < K; ++k) {
            const int r = s_inv[t * K + k];
            if (r >= 0) {
                const float wk = s_w[t * K + k];
                acc0 = fmaf(wk, __uint_as_float(static_cast<uint32_t>(s_y[r * nd + c]) << 16), acc0);
                acc1 = fmaf(wk, __uint_as_float(static_cast<uint32_t>(s_y[r * nd + c + 1]) << 16), acc1);
            }
        }
        *reinterpret_cast<uint32_t*>(a.out + static_cast<long long>(t) * D + d0 + c) = pack_bf16x2(acc0, acc1);
    }
    pdl_trigger();
}

template <bool SWIGLU, int NR>
static cudaError_t ld_launch(const LayerDecodeArgs& a, int grid, size_t smem, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(layer_decode_kernel<SWIGLU, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // CTAs wait on each other at the grid barriers: all resident (cooperative)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kLdThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, layer_decode_kernel<SWIGLU, NR>, a);
}

template <bool SWIGLU>
static cudaError_t ld_dispatch(const LayerDecodeArgs& a, int grid, size_t smem, cudaStream_t st) {
    if (a.N <= 1) return ld_launch<SWIGLU, 1>(a, grid, smem, st);
    if (a.N <= 2) return ld_launch<SWIGLU, 2>(a, grid, smem, st);
    if (a.N <= 4) return ld_launch<SWIGLU, 4>(a, grid, smem, st);
    return ld_launch<SWIGLU, 8>(a, grid, smem, st);
}

cudaError_t launch_layer_decode(const LayerDecodeArgs& a, int grid, cudaStream_t st) {
    if (a.N < 1 || a.N > kLayerDecodeMaxN || a.N * a.K > kLayerDecodeMaxRows || a.E > kLayerDecodeMaxE ||
        grid < 1 || a.D / 8 > kSmallRouteThreads * kSmallRouteMaxChunks)
        return cudaErrorInvalidValue;
    const size_t smem = layer_decode_smem(a.N, a.D, a.E, a.K, a.Dff, grid, a.w2_smem != 0).total;
    return a.w3 ? ld_dispatch<true>(a, grid, smem, st) : ld_dispatch<false>(a, grid, smem, st);
}

int layer_decode_plan(int N, int D, int E, int K, int Dff, bool swiglu, int* w2_smem) {
    int dev = 0, nsm = 0, optin = 0;
    *w2_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    // the kernel's static shared memory is about 3.4 KB
    const size_t limit = static_cast<size_t>(optin) - 4096;
    if (layer_decode_smem(N, D, E, K, Dff, nsm, false).total > limit) return 0;
    *w2_smem = layer_decode_smem(N, D, E, K, Dff, nsm, true).total <= limit ? 1 : 0;
    // 512 threads of at most 128 registers and this shared memory: one CTA per SM
    return nsm;
}

}  // namespace moe
