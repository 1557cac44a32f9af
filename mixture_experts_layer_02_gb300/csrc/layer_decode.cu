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
//      rank k < K makes it pick k -- topk_token's picks.  Then, at once on
//      disjoint warps: expert_offsets[e] = the valid picks of experts below
//      e, the row of pick i = that count for its expert + the earlier picks
//      of its expert, each token's weights with topk_token's arithmetic, and
//      the experts that received rows (the work slots).  Same bits as the
//      separate kernels; CTA 0 stores them; CTAs share the x_perm row copy.
//      Each CTA then starts bulk copies of the W2 rows its phase 4 will read
//      into its shared memory (when they fit: one token) or asks L2 to
//      prefetch them, so that the W2 stream runs under GEMM1's;
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

// 3-D tiled TMA load global -> shared (this CTA), completion on `bar`.
__device__ __forceinline__ void tma_load_3d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// d[16 x 8] += a[16 x 16] . b[16 x 8], bf16 operands, fp32 accumulators (warp-wide)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9},"
        " {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// One GEMM2 item: columns dd0 .. dd0 + ncol of the CTA's, for the ne rows of
// one expert starting at row r0.  Per 16-byte chunk c of D_ffn (lane-strided)
// the item loads the rows' h (fp32, shared memory) once and the ncol W2 rows'
// chunk (rows Dff apart from `w`, global memory),
// and accumulates with paired fused multiply-adds; then a butterfly per
// (column, row) and lane 0 stores y (bf16) to s_y and y_perm.
struct G2Item {
    int r0, ne, dd0, ncol;
};
template <int NR>
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
            if (j < g.ncol) wv[j] = __ldg(w + j * chunks2 + c);
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
__global__ void __launch_bounds__(kLdThreads, 1)
layer_decode_kernel(const LayerDecodeArgs a, const __grid_constant__ CUtensorMap tmW2) {
    constexpr int kLdBatch1 = LdCfg<NR>::B1;
    extern __shared__ __align__(16) unsigned char ld_smem[];
    __shared__ float s_part[2][kSmallRouteThreads / 32][kSmallRouteMaxN];
    __shared__ int s_id[kLayerDecodeMaxRows];       // expert of assignment t*K+k (-1: none)
    __shared__ float s_w[kLayerDecodeMaxRows];      // its weight
    __shared__ int s_src[kLayerDecodeMaxRows];      // token of each permuted row
    __shared__ int s_inv[kLayerDecodeMaxRows];      // row of each assignment (-1: none)
    __shared__ int s_touched[kLayerDecodeMaxRows];  // experts with rows, ascending
    __shared__ int s_T;
    __shared__ volatile int s_abort;
    __shared__ __align__(8) uint64_t s_w2bar;       // W2 bulk copies landed
    __shared__ unsigned long long s_bar_base;       // the barrier count when this launch began

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = a.N, D = a.D, E = a.E, K = a.K, Dff = a.Dff, A = N * K;
    const int G = gridDim.x, b = blockIdx.x;
    const bool writer = b == 0;
    const LayerDecodeSmem L = layer_decode_smem(N, D, E, K, Dff, G, a.w2_smem != 0);
    unsigned char* sm = ld_smem + ((1024u - (smem_u32(ld_smem) & 1023u)) & 1023u);  // 128-byte swizzle atoms
    float* s_v = reinterpret_cast<float*>(sm + L.logits);   // scores: logit + bias [N][E]
    int* s_off = reinterpret_cast<int*>(sm + L.off);
    uint4* s_x = reinterpret_cast<uint4*>(sm + L.xh);      // x rows, bf16 (phases 1-3); staged: h rows, bf16
    float* s_hf = reinterpret_cast<float*>(sm + L.xh);     // h rows, fp32 (phase 4, not staged)
    uint16_t* s_y = reinterpret_cast<uint16_t*>(sm + L.y);
    float* s_tile = reinterpret_cast<float*>(sm + L.part);  // GEMM2 partial tiles (staged)
    uint16_t* s_w2 = reinterpret_cast<uint16_t*>(sm + L.w2);

    if (tid == 0) {
        s_abort = 0;
        mbar_init(&s_w2bar, 1);
        fence_barrier_init();
        if (a.w2_smem) tma_prefetch_desc(&tmW2);
    }
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
                if ((E & 3) == 0) {  // lane part p reads the groups of four scores q = p, p + 4, ...
                    const float4* vt4 = reinterpret_cast<const float4*>(vt);
                    for (int q = i & 3; q < (E >> 2); q += 4) {
                        const float4 f = vt4[q];
                        const int e2 = q * 4;
                        cnt += (before(f.x, e2, ve, e) ? 1 : 0) + (before(f.y, e2 + 1, ve, e) ? 1 : 0) +
                               (before(f.z, e2 + 2, ve, e) ? 1 : 0) + (before(f.w, e2 + 3, ve, e) ? 1 : 0);
                    }
                } else {
                    for (int e2 = i & 3; e2 < E; e2 += 4) cnt += before(vt[e2], e2, ve, e) ? 1 : 0;
                }
            }
            cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
            cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
            if (mine && (i & 3) == 0 && cnt < K) s_id[t * K + cnt] = e;
        }
    }
    __syncthreads();
    // 2b. the rest of the routing at once, on disjoint warps, from the picks
    //     (direct counts over the at most 64 assignments instead of scans):
    //       threads e < E:          expert_offsets[e] = valid picks of experts below e;
    //       warps 8-9, thread i < A: the row of assignment i = valid picks of experts
    //                                below its expert + earlier picks of its expert;
    //       warps 10-13:            each token's weights (topk_token's arithmetic);
    //       warp 14:                the experts that received rows in order of first
    //                                appearance (the work slots), and the row count
    if (tid < E) {
        int off = 0;
        for (int i = 0; i < A; ++i) {
            const int v = s_id[i];
            off += (v >= 0 && v < tid) ? 1 : 0;
        }
        s_off[tid] = off;
        if (writer) a.offsets[tid] = off;
    } else if (warp >= 8 && warp < 10) {
        const int i = tid - 256;
        if (i < A) {
            const int e = s_id[i];
            int r = -1;
            if (e >= 0) {
                r = 0;
                for (int i2 = 0; i2 < A; ++i2) {
                    const int v = s_id[i2];
                    r += ((v >= 0 && v < e) || (i2 < i && v == e)) ? 1 : 0;
                }
                s_src[r] = i / K;
            }
            s_inv[i] = r;
            if (writer) {
                a.inv_perm[i] = r;
                if (r >= 0) a.perm_src[r] = i / K;
            }
        }
    } else if (warp >= 10 && warp < 14) {
        bool any_bad = false;
        for (int t = warp - 10; t < N; t += 4) {
            const int pk = lane < K ? s_id[t * K + lane] : -1;
            const float my_v = pk >= 0 ? s_v[t * E + pk] : -INFINITY;  // a pick that stayed -1 scores -inf
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
                if (writer) {
                    a.ids[t * K + lane] = pk;
                    a.w[t * K + lane] = weight;
                }
            }
        }
        if (writer && any_bad && lane == 0) record_error(a.err, MOE_DEVERR_BOUNDS);
    } else if (warp == 14) {
        int n = 0, valid = 0;
        for (int base = 0; base < A; base += 32) {
            const int i = base + lane;
            const int e = i < A ? s_id[i] : -1;
            bool first = e >= 0;
            for (int i2 = 0; i2 < i && first; ++i2) first = s_id[i2] != e;
            const unsigned m = __ballot_sync(0xffffffffu, first);
            if (first) s_touched[n + __popc(m & ((1u << lane) - 1u))] = e;
            n += __popc(m);
            valid += __popc(__ballot_sync(0xffffffffu, e >= 0));
        }
        if (lane == 0) {
            s_T = n;
            s_off[E] = valid;  // rows placed (assignments with a valid expert)
            if (writer) a.offsets[E] = valid;
        }
    }
    __syncthreads();
    const int T = s_T, rows = s_off[E];
    // the CTA's output columns (pairs of columns, spread evenly over the CTAs)
    const int P = D / 2;
    // (32-bit arithmetic: the host admits only sizes with N*K*D_ffn*grid and
    // D/2*grid below 2^31; a 64-bit division here cost about a microsecond)
    const int d0 = 2 * static_cast<int>(static_cast<unsigned>(b) * P / G);
    const int nd = 2 * static_cast<int>(static_cast<unsigned>(b + 1) * P / G) - d0;
    // W2 rows of the CTA's columns: W2[e][d0 .. d0+nd) (contiguous; staged as a 16-row box)
    const uint32_t w2_bytes = static_cast<uint32_t>(nd) * Dff * 2;
    const bool staged = a.w2_smem && nd > 0 && T > 0;
    // GEMM1 items of this CTA: a contiguous range, so warp 15 has no more than the others
    const int U1 = T * Dff;
    const int u_lo = static_cast<int>(static_cast<unsigned>(U1) * b / G);
    const int u_hi = static_cast<int>(static_cast<unsigned>(U1) * (b + 1) / G);
    if (staged) {
        if (tid == kLdThreads - 32) {  // lane 0 of warp 15 issues one 16-row box per expert slot
            const uint32_t box = static_cast<uint32_t>(kLayerDecodeW2Rows) * Dff * 2;
            mbar_arrive_expect_tx(&s_w2bar, box * T);
            for (int i = 0; i < T; ++i)
                tma_load_3d(&tmW2, &s_w2bar, reinterpret_cast<char*>(s_w2) + static_cast<size_t>(i) * box, 0,
                            s_touched[i] * D + d0, 0);
        }
    } else if (tid < T && nd > 0 && static_cast<long long>(T) * D * Dff * 2 <= a.l2_prefetch_max) {
        l2_prefetch_bulk(a.w2 + (static_cast<long long>(s_touched[tid]) * D + d0) * Dff, w2_bytes);
    }
    for (int r = b; r < rows; r += G) {
        uint4* dst = reinterpret_cast<uint4*>(a.x_perm + static_cast<long long>(r) * D);
        for (int c = tid; c < chunks; c += kLdThreads) dst[c] = s_x[s_src[r] * chunks + c];
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
    if (staged) {  // h rows in bf16: the MMA's B operand
        for (int i = tid; i < rows * chunks2; i += kLdThreads)
            s_x[i] = ld_cg_v4(reinterpret_cast<const uint4*>(a.h) + i);
    } else {  // h rows as fp32 for the CUDA-core items
        for (int i = tid; i < rows * chunks2; i += kLdThreads) {
            float2 hv[4];
            bf16x8_f32x2(ld_cg_v4(reinterpret_cast<const uint4*>(a.h) + i), hv);
            float4* dst = reinterpret_cast<float4*>(s_hf + static_cast<size_t>(i) * 8);
            dst[0] = make_float4(hv[0].x, hv[0].y, hv[1].x, hv[1].y);
            dst[1] = make_float4(hv[2].x, hv[2].y, hv[3].x, hv[3].y);
        }
    }
    if (staged && tid == 0 && !mbar_wait(&s_w2bar, 0, &s_abort, a.err)) {
        volatile int keep_waiting = 0;  // timed out: wait once more for the copies before leaving
        mbar_wait(&s_w2bar, 0, &keep_waiting, a.err);
    }
    __syncthreads();
    if (s_abort) return;
    if (staged) {
        // Tensor cores: per expert slot, D[16 W2 rows][8 token rows] = W2 slice
        // . h^T over D_ffn, in kparts k-ranges (one warp each, mma.sync
        // m16n8k16 bf16 -> fp32, operands read with ldmatrix from the
        // swizzled W2 box and the bf16 h rows); the partial tiles are summed
        // in k-range order.  Token rows past the expert's own read its first
        // row; their outputs are not used.
        const int kparts = T < kLdWarps ? kLdWarps / T : 1;  // k-ranges per slot: at most max(16, T) tiles
        const int ksteps = Dff / 16;
        const uint32_t w2s = smem_u32(s_w2), hs = smem_u32(s_x);
        for (int it = warp; it < T * kparts; it += kLdWarps) {
            const int slot = it / kparts, kp = it - slot * kparts;
            const int e = s_touched[slot], r0 = s_off[e], ne = s_off[e + 1] - r0;
            const int k_lo = ksteps * kp / kparts, k_hi = ksteps * (kp + 1) / kparts;
            // ldmatrix row addresses: A (x4) rows (m & 1) * 8 + lane & 7 at k-chunk m >> 1, m = lane >> 3;
            // B (x2) token row lane & 7 at k-chunk (lane >> 3) & 1
            const int arow = ((lane >> 3) & 1) * 8 + (lane & 7), akc = lane >> 4;
            const uint32_t abase = w2s + static_cast<uint32_t>(slot) * kLayerDecodeW2Rows * Dff * 2 + arow * 128;
            const int bn = lane & 7;
            const uint32_t bbase = hs + static_cast<uint32_t>(r0 + (bn < ne ? bn : 0)) * Dff * 2 + ((lane >> 3) & 1) * 16;
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int ks = k_lo; ks < k_hi; ++ks) {
                const int k0 = ks * 16;
                const int ch = ((k0 & 63) >> 3) + akc;  // 16-byte chunk in the 128-byte row of k-block k0/64
                uint32_t a0, a1, a2, a3, b0, b1;
                ldmatrix_x4(abase + (k0 >> 6) * (kLayerDecodeW2Rows * 128) + ((ch ^ (arow & 7)) << 4), a0, a1, a2, a3);
                ldmatrix_x2(bbase + k0 * 2, b0, b1);
                mma_bf16_16816(d, a0, a1, a2, a3, b0, b1);
            }
            // fragment: d0 (g, 2t), d1 (g, 2t + 1), d2 (g + 8, 2t), d3 (g + 8, 2t + 1) of [W2 row][token row]
            const int g = lane >> 2, t2 = (lane & 3) * 2;
            float* pt = s_tile + it * (kLayerDecodeW2Rows * 8);
            pt[g * 8 + t2] = d[0];
            pt[g * 8 + t2 + 1] = d[1];
            pt[(g + 8) * 8 + t2] = d[2];
            pt[(g + 8) * 8 + t2 + 1] = d[3];
        }
        __syncthreads();
        for (int i = tid; i < T * kLayerDecodeW2Rows * 8; i += kLdThreads) {
            const int slot = i / (kLayerDecodeW2Rows * 8), rem = i - slot * (kLayerDecodeW2Rows * 8);
            const int dd = rem >> 3, n = rem & 7;
            const int e = s_touched[slot], r0 = s_off[e], ne = s_off[e + 1] - r0;
            if (dd < nd && n < ne) {
                const float* pt = s_tile + slot * kparts * (kLayerDecodeW2Rows * 8) + rem;
                float y = pt[0];
                for (int kp = 1; kp < kparts; ++kp) y += pt[kp * (kLayerDecodeW2Rows * 8)];
                const uint16_t yb = bf16_rn_bits(y);
                s_y[(r0 + n) * nd + dd] = yb;
                a.y_perm[static_cast<long long>(r0 + n) * D + d0 + dd] = yb;
            }
        }
    } else {
        // CUDA cores: item = (expert slot, up to kG2Cols consecutive columns of the CTA's)
        const int per_slot = (nd + LdCfg<NR>::G2 - 1) / LdCfg<NR>::G2;
        for (int it = warp; it < T * per_slot; it += kLdWarps) {
            const int slot = it / per_slot, dd0 = (it - slot * per_slot) * LdCfg<NR>::G2;
            const int e = s_touched[slot];
            G2Item g{s_off[e], s_off[e + 1] - s_off[e], dd0, min(LdCfg<NR>::G2, nd - dd0)};
            gemm2_item<NR>(g, reinterpret_cast<const uint4*>(a.w2 + (static_cast<long long>(e) * D + d0 + dd0) * Dff),
                           s_hf, Dff, lane, s_y, nd, a.y_perm, D, d0);
        }
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
static cudaError_t ld_launch(const LayerDecodeArgs& a, const CUtensorMap& tm_w2, int grid, size_t smem,
                             cudaStream_t st) {
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
    return cudaLaunchKernelEx(&cfg, layer_decode_kernel<SWIGLU, NR>, a, tm_w2);
}

template <bool SWIGLU>
static cudaError_t ld_dispatch(const LayerDecodeArgs& a, const CUtensorMap& tm_w2, int grid, size_t smem,
                               cudaStream_t st) {
    if (a.N <= 1) return ld_launch<SWIGLU, 1>(a, tm_w2, grid, smem, st);
    if (a.N <= 2) return ld_launch<SWIGLU, 2>(a, tm_w2, grid, smem, st);
    if (a.N <= 4) return ld_launch<SWIGLU, 4>(a, tm_w2, grid, smem, st);
    return ld_launch<SWIGLU, 8>(a, tm_w2, grid, smem, st);
}

cudaError_t launch_layer_decode(const LayerDecodeArgs& a, const CUtensorMap& tm_w2, int grid, cudaStream_t st) {
    if (a.N < 1 || a.N > kLayerDecodeMaxN || a.N * a.K > kLayerDecodeMaxRows || a.E > kLayerDecodeMaxE ||
        grid < 1 || a.D / 8 > kSmallRouteThreads * kSmallRouteMaxChunks)
        return cudaErrorInvalidValue;
    const size_t smem = layer_decode_smem(a.N, a.D, a.E, a.K, a.Dff, grid, a.w2_smem != 0).total;
    return a.w3 ? ld_dispatch<true>(a, tm_w2, grid, smem, st) : ld_dispatch<false>(a, tm_w2, grid, smem, st);
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
    // W2 staged: every CTA's columns fit one 16-row box, whose k-blocks a box can hold
    const bool w2_fits = 2 * ((D / 2 + nsm - 1) / nsm) <= kLayerDecodeW2Rows && Dff / 64 <= 256;
    // the kernel splits columns and items with 32-bit products
    if (static_cast<long long>(N) * K * Dff * nsm >= (1LL << 31) || static_cast<long long>(D / 2) * nsm >= (1LL << 31))
        return 0;
    *w2_smem = w2_fits && layer_decode_smem(N, D, E, K, Dff, nsm, true).total <= limit ? 1 : 0;
    // 512 threads of at most 128 registers and this shared memory: one CTA per SM
    return nsm;
}

}  // namespace moe
