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
// separated by two grid barriers, for bf16 or e4m3 experts:
//
//   1. router logits: expert e's logits for all N tokens by a group of 256
//      threads (small_logits_expert, the same arithmetic as
//      route_logits_small_kernel), two groups per CTA; e4m3: warp t also
//      quantises token t by the row quantiser's rule (quant.cuh);
//   -- grid barrier 1 --
//   2. routing: every CTA reads the N x E logits and computes the routing
//      itself, spread over its threads (one warp walking the experts serially
//      would take microseconds): topk_token's picks, by ranks counted over
//      four lanes per (token, expert) up to two tokens, by a warp arg-max per
//      token above.  Then, at once on disjoint warps: expert_offsets[e] = the
//      valid picks of experts below e, the row of pick i = that count for its
//      expert + the earlier picks of its expert, each token's weights with
//      topk_token's arithmetic, and the experts that received rows (the work
//      slots).  Same bits as the separate kernels; CTA 0 stores them; CTAs
//      share the x_perm row copy.  Each CTA then asks L2 to prefetch the W2
//      rows its phase 4 will read (or, with w2_smem, starts bulk copies of
//      them into its shared memory), so that the W2 stream runs under GEMM1's;
//   3. GEMM1 + activation on the tensor cores (mma.sync, gemv_steps), the
//      weights as the 16-row operand: a tile is 16 rows f of one expert's W1
//      (and W3), the expert's token rows (<= N, from shared memory) the 8
//      columns of the other operand; each CTA takes a contiguous range of
//      tiles, streams the weights through registers with 32-byte loads and
//      stores h[row][f] = bf16(silu(g) * u) (SwiGLU) or bf16(silu(g)) (SiLU),
//      e4m3: the sums times the token and weight-row scales first;
//   -- grid barrier 2 --
//   4. GEMM2 + combine: CTA b owns output columns [d0, d1) of every row.
//      It stages h (all rows: bf16, e4m3: codes by the row rule) in shared
//      memory, forms y_perm[row][d] = bf16(sum_f h[row][f] W2[e][d][f]) for
//      its columns on the tensor cores (W2 through L2, or from the staged
//      copy), then out[t][d] = bf16(sum_k w[t,k] * y_perm[inv_perm[t,k]][d])
//      in k order (fp32 fused multiply-adds from 0, as combine_kernel).
//
// At these sizes the GEMMs are matrix-vector products (at most N rows per
// expert): the bound is the weight stream, which 16 warps of 32-byte loads
// per SM keep at HBM speed, and mma.sync (fp32 accumulation) takes the
// products off the CUDA cores, where converting every weight to fp32 cost
// more than the stream for e4m3 weights or more than one token.  Routing,
// placement and the combine give the bits of the separate kernels; h and y
// round the same quantities to bf16 but sum in another order than the
// tcgen05 GEMMs.
//
// The grid barriers count arrivals in one 64-bit word of the workspace
// header, which grows by the grid size per barrier and is never reset: each
// CTA reads it once at the start (rounded down to a multiple of the grid
// size, it is the launch's base), then at barrier k adds 1 with release
// semantics and waits (acquire loads) until it reaches base + k * grid, so
// no per-call clearing is needed and a barrier costs one fire-and-forget add
// and the polls.  Every wait is bounded (kWaitLimitNs); on expiry the CTA
// records MOE_DEVERR_TIMEOUT, waits (bounded) for its own bulk copies and
// returns.
#include "quant.cuh"
#include "route_common.cuh"

namespace moe {

constexpr int kLdThreads = 512;
constexpr int kLdWarps = kLdThreads / 32;

// Steps whose weight pieces a warp loads before it multiplies them: 8
// 32-byte loads per lane in flight, with W1 and W3 (kG1Steps) or one weight
// matrix (kG1Steps1).
constexpr int kG1Steps = 2;
constexpr int kG1Steps1 = 4;

// 32-byte streaming load (sm_100 and later; p on a 32-byte boundary): not
// kept in L1, L2 eviction policy `pol`; lo = bytes 0..15, hi = bytes 16..31.
__device__ __forceinline__ void ld_stream_v8(const void* p, uint64_t pol, uint4& lo, uint4& hi) {
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                 : "l"(p), "l"(pol));
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

// d[16 x 8] += a[16 x 32] . b[32 x 8], e4m3 operands, fp32 accumulators (warp-wide)
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9},"
        " {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

// ---------------------------------------------------------------------------
// Matrix-vector products on the tensor cores (mma.sync), the weights as the
// 16-row operand A and up to 8 activation rows as the 8 columns of B.  At
// step s lane (g, t) loads 32-byte piece 4 s + t of weight rows g (ga) and
// g + 8 (ha) -- a warp load covers whole 128-byte lines of 8 rows -- and the
// same piece of activation row g (xr, shared memory; null: a zero column).
// Each 8 bytes of the pieces feed one MMA (a0/a2 from row g, a1/a3 from row
// g + 8, b0/b1 from the activations), so A and B hold the same columns in the
// same k places and every sum runs over its row's terms, in another order.
// acc_a += steps [s_beg, s_end) of (ga, ha); with DUAL also acc_b of (gb, hb)
// (W1 and W3 against the same tokens).
// ---------------------------------------------------------------------------
template <bool FP8, bool DUAL>
__device__ __forceinline__ void gemv_steps(const uint4* ga, const uint4* ha, const uint4* gb, const uint4* hb,
                                           const uint4* xr, int t4, int s_beg, int s_end, uint64_t pol,
                                           float (&acc_a)[4], float (&acc_b)[4]) {
    auto mma_piece = [](float (&acc)[4], const uint4& rg, const uint4& rh, const uint4& xv) {
        if constexpr (FP8) {
            mma_e4m3_16832(acc, rg.x, rh.x, rg.y, rh.y, xv.x, xv.y);
            mma_e4m3_16832(acc, rg.z, rh.z, rg.w, rh.w, xv.z, xv.w);
        } else {
            mma_bf16_16816(acc, rg.x, rh.x, rg.y, rh.y, xv.x, xv.y);
            mma_bf16_16816(acc, rg.z, rh.z, rg.w, rh.w, xv.z, xv.w);
        }
    };
    constexpr int kSteps = DUAL ? kG1Steps : kG1Steps1;
    for (int s0 = s_beg; s0 < s_end; s0 += kSteps) {
        uint4 va[kSteps][2][2], vb[DUAL ? kSteps : 1][2][2];  // [step][row g, row g + 8][bytes 0-15, 16-31]
#pragma unroll
        for (int q = 0; q < kSteps; ++q) {
            if (s0 + q < s_end) {
                const int c = ((s0 + q) * 4 + t4) * 2;
                ld_stream_v8(ga + c, pol, va[q][0][0], va[q][0][1]);
                ld_stream_v8(ha + c, pol, va[q][1][0], va[q][1][1]);
                if constexpr (DUAL) {
                    ld_stream_v8(gb + c, pol, vb[q][0][0], vb[q][0][1]);
                    ld_stream_v8(hb + c, pol, vb[q][1][0], vb[q][1][1]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kSteps; ++q) {
            if (s0 + q < s_end) {
                const int c = ((s0 + q) * 4 + t4) * 2;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const uint4 xv = xr ? xr[c + hf] : make_uint4(0u, 0u, 0u, 0u);
                    mma_piece(acc_a, va[q][0][hf], va[q][1][hf], xv);
                    if constexpr (DUAL) mma_piece(acc_b, vb[q][0][hf], vb[q][1][hf], xv);
                }
            }
        }
    }
}

// The CTA's nt tiles of S steps each over its 16 warps: warp w takes steps
// [w W / 16, (w + 1) W / 16) of the W = nt S steps in tile order, so every
// warp streams the same bytes (to a step).  A tile inside one warp's range is
// finished from its registers; a tile that a warp boundary cuts is summed in
// s_part ([warp][first, last tile of the warp][a, b][16][NR] fp32) by the
// warps that share it, in warp order, after a __syncthreads.
//   run(j, s_beg, s_end, acc_a, acc_b)   accumulates steps of tile j;
//   finish(j, rr, col, a, b)             gets the sums of tile row rr and
//                                        column col < NR (the caller skips
//                                        columns past its rows).
// Called by every thread of the CTA.
template <bool DUAL, int NR, typename Run, typename Finish>
__device__ __forceinline__ void gemv_tiles(int nt, int S, float* s_part, int warp, int lane, int tid, Run run,
                                           Finish finish) {
    constexpr int R = kLayerDecodeW2Rows;
    const int W = nt * S;
    auto first_step = [&](int w) { return w * W / kLdWarps; };
    auto part = [&](int w, int slot, int m, int rr, int col) -> float& {
        return s_part[(((w * 2 + slot) * 2 + m) * R + rr) * NR + col];
    };
    const int g = lane >> 2, t4 = lane & 3;
    const int lo = first_step(warp), hi = first_step(warp + 1);
    if (hi > lo) {
        for (int j = lo / S; j <= (hi - 1) / S; ++j) {
            const int sb = max(lo - j * S, 0), se = min(hi - j * S, S);
            float acc_a[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc_b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            run(j, sb, se, acc_a, acc_b);
            // C fragment: acc[q] is tile row g + 8 (q >> 1), column 2 t4 + (q & 1)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int rr = g + 8 * (q >> 1), col = 2 * t4 + (q & 1);
                if (col < NR) {
                    if (sb == 0 && se == S) {
                        finish(j, rr, col, acc_a[q], acc_b[q]);
                    } else {
                        const int slot = j == lo / S ? 0 : 1;
                        part(warp, slot, 0, rr, col) = acc_a[q];
                        if (DUAL) part(warp, slot, 1, rr, col) = acc_b[q];
                    }
                }
            }
        }
    }
    __syncthreads();
    // the cut tiles: the tile of each warp boundary strictly inside a tile,
    // taken at its first such boundary
    for (int idx = tid; idx < (kLdWarps - 1) * R * NR; idx += kLdThreads) {
        const int wb = 1 + idx / (R * NR), rr = (idx / NR) % R, col = idx % NR;
        const int p = first_step(wb);
        if (p >= W || p % S == 0) continue;
        const int j = p / S;
        if (wb > 1 && first_step(wb - 1) > j * S) continue;  // an earlier boundary cuts this tile too
        // warps owning the tile's first and last steps: owner(q) = (16 (q + 1) - 1) / W
        const int w_a = (kLdWarps * (j * S + 1) - 1) / W, w_b = (kLdWarps * ((j + 1) * S) - 1) / W;
        float sa = 0.0f, sb = 0.0f;
        for (int w = w_a; w <= w_b; ++w) {
            if (first_step(w + 1) == first_step(w)) continue;  // no steps
            const int slot = j == first_step(w) / S ? 0 : 1;
            sa += part(w, slot, 0, rr, col);
            if (DUAL) sb += part(w, slot, 1, rr, col);
        }
        finish(j, rr, col, sa, sb);
    }
}

// The same by groups of warps: with nt <= 16 tile j's steps are split over
// warps [j*16/nt, (j+1)*16/nt), whose partial sums meet in s_part
// ([warp][a, b][16][NR] fp32) and are added in warp order after a
// __syncthreads; with more tiles each warp takes whole tiles j = warp,
// warp + 16, ...  Every warp works on one tile at a time, so its loads are in
// one batch however few its steps, where gemv_tiles cuts ranges across tiles
// into separate batches; the groups are uneven when 16 is not a multiple of
// nt, and with more than 16 tiles some warps take one tile more than others.
// gemv_pick_even chooses between the two per launch.
template <bool DUAL, int NR, typename Run, typename Finish>
__device__ __forceinline__ void gemv_tiles_grouped(int nt, int S, float* s_part, int warp, int lane, int tid, Run run,
                                           Finish finish) {
    constexpr int R = kLayerDecodeW2Rows;
    const int g = lane >> 2, t4 = lane & 3;
    if (nt > 0 && nt <= kLdWarps) {
        int j = 0;
        while ((j + 1) * kLdWarps / nt <= warp) ++j;
        const int w0 = j * kLdWarps / nt, nw = (j + 1) * kLdWarps / nt - w0, i = warp - w0;
        float acc_a[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc_b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        run(j, i * S / nw, (i + 1) * S / nw, acc_a, acc_b);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int rr = g + 8 * (q >> 1), col = 2 * t4 + (q & 1);
            if (col < NR) {
                s_part[((warp * 2 + 0) * R + rr) * NR + col] = acc_a[q];
                if (DUAL) s_part[((warp * 2 + 1) * R + rr) * NR + col] = acc_b[q];
            }
        }
        __syncthreads();
        for (int idx = tid; idx < nt * R * NR; idx += kLdThreads) {
            const int rr = idx % R, col = (idx / R) % NR, jj = idx / (R * NR);
            float sa = 0.0f, sb = 0.0f;
            for (int w = jj * kLdWarps / nt; w < (jj + 1) * kLdWarps / nt; ++w) {
                sa += s_part[((w * 2 + 0) * R + rr) * NR + col];
                if (DUAL) sb += s_part[((w * 2 + 1) * R + rr) * NR + col];
            }
            finish(jj, rr, col, sa, sb);
        }
    } else {
        for (int j = warp; j < nt; j += kLdWarps) {
            float acc_a[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc_b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            run(j, 0, S, acc_a, acc_b);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int rr = g + 8 * (q >> 1), col = 2 * t4 + (q & 1);
                if (col < NR) finish(j, rr, col, acc_a[q], acc_b[q]);
            }
        }
        __syncthreads();
    }
}

// Which of the two schedules to run for nt tiles of S steps with batches of
// kSteps: the one with fewer load batches in its busiest warp, counting a
// batch for every tile a warp's even range touches past its first (a range
// cut across tiles loads each part in its own batches); the groups on a tie.
__device__ __forceinline__ bool gemv_pick_even(int nt, int S, int kSteps) {
    if (nt <= 0) return false;
    auto cdiv = [](int x, int y) { return (x + y - 1) / y; };
    const int grouped = nt <= kLdWarps ? cdiv(cdiv(S, kLdWarps / nt), kSteps) : cdiv(nt, kLdWarps) * cdiv(S, kSteps);
    const int per = cdiv(nt * S, kLdWarps);
    const int even = cdiv(per, kSteps) + cdiv(per, S);
    return even < grouped;
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

template <bool SWIGLU, int NR, bool FP8>
__global__ void __launch_bounds__(kLdThreads, 1)
layer_decode_kernel(const LayerDecodeArgs a, const __grid_constant__ CUtensorMap tmW2) {
    extern __shared__ __align__(16) unsigned char ld_smem[];
    __shared__ float s_part[2][kSmallRouteThreads / 32][kSmallRouteMaxN];
    __shared__ int s_id[kLayerDecodeMaxRows];       // expert of assignment t*K+k (-1: none)
    __shared__ float s_w[kLayerDecodeMaxRows];      // its weight
    __shared__ int s_src[kLayerDecodeMaxRows];      // token of each permuted row
    __shared__ int s_inv[kLayerDecodeMaxRows];      // row of each assignment (-1: none)
    __shared__ int s_touched[kLayerDecodeMaxRows];  // experts with rows, in order of their first pick
    __shared__ int s_T;
    __shared__ volatile int s_abort;
    __shared__ __align__(8) uint64_t s_w2bar;       // W2 bulk copies landed
    __shared__ unsigned long long s_bar_base;       // the barrier count when this launch began
    __shared__ float s_xs[kLayerDecodeMaxN];        // e4m3: token scales
    __shared__ float s_hs[kLayerDecodeMaxRows];     // e4m3: h row scales

    // the GEMVs' schedule is chosen per launch (gemv_pick_even) where carrying
    // both schedules measured faster (bf16 weights from two tokens, e4m3 ones
    // from five); elsewhere the extra code cost more than it saved, and the
    // warp groups run
    constexpr bool kPickSchedule = FP8 ? NR == 8 : NR > 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = a.N, D = a.D, E = a.E, K = a.K, Dff = a.Dff, A = N * K;
    const int G = gridDim.x, b = blockIdx.x;
    const bool writer = b == 0;
    const LayerDecodeSmem L = layer_decode_smem(N, D, E, K, Dff, G, a.w2_smem != 0, FP8);
    unsigned char* sm = ld_smem + ((1024u - (smem_u32(ld_smem) & 1023u)) & 1023u);  // 128-byte swizzle atoms
    float* s_v = reinterpret_cast<float*>(sm + L.logits);   // scores: logit + bias [N][E]
    int* s_off = reinterpret_cast<int*>(sm + L.off);
    uint4* s_x = reinterpret_cast<uint4*>(sm + L.xh);      // x rows, bf16 (phases 1-3), then h rows, bf16
    uint8_t* s_xq = sm + L.xh;                              // e4m3: x codes (phases 1-3)
    uint8_t* s_hq = sm + L.xh;                              // e4m3: h codes (phase 4)
    uint16_t* s_y = reinterpret_cast<uint16_t*>(sm + L.y);
    float* s_tile = reinterpret_cast<float*>(sm + L.part);  // GEMM2 partial tiles (staged)
    float* s_g1 = reinterpret_cast<float*>(sm + L.g1);      // GEMM partial sums [warp][2][16][NR]
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
    const int chunks = D / 8;  // 16-byte chunks of a bf16 x row
    if (!FP8)
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
    if (FP8 && warp < N) {
        // e4m3: token row `warp` -> codes and scale with the row quantiser's
        // rule (quant.cu); the codes are GEMM1's B operand
        const uint4* row = reinterpret_cast<const uint4*>(a.x) + static_cast<size_t>(warp) * chunks;
        uint32_t m = 0;
        for (int c = lane; c < chunks; c += 32) m = max(m, absmax8(__ldg(row + c)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int k = scale_exp_of(m);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);  // 2^-k
        const float sc = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
        if (lane == 0) {
            s_xs[warp] = sc;
            if (writer) a.x_scale[warp] = sc;
        }
        for (int c = lane; c < chunks; c += 32) {
            const uint2 q = to_e4m3x8(__ldg(row + c), inv);
            reinterpret_cast<uint2*>(s_xq + static_cast<size_t>(warp) * D)[c] = q;
            if (writer) reinterpret_cast<uint2*>(a.xq + static_cast<size_t>(warp) * D)[c] = q;
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
    // 2a. the picks of topk_token: the K first experts of each token in the
    //     order (score desc, index asc) among its scores that are not NaN.
    //     Up to two tokens: the rank of (token t, expert e), counted by four
    //     lanes over a quarter of the experts each; rank k < K makes e pick k
    //     (N*E*E comparisons, spread over all threads).  More tokens: a warp
    //     per token runs K rounds of a warp arg-max after the previous pick
    //     (about a microsecond for any N, where the ranks grow with N).
    if (N > 2) {
        for (int t = warp; t < N; t += kLdWarps) {
            float v[kLayerDecodeMaxE / 32];
#pragma unroll
            for (int j = 0; j < kLayerDecodeMaxE / 32; ++j) {
                const int e = lane + 32 * j;
                v[j] = e < E ? s_v[t * E + e] : 0.0f;
            }
            float prev_v = INFINITY;
            int prev_i = -1;
            for (int k = 0; k < K; ++k) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
#pragma unroll
                for (int j = 0; j < kLayerDecodeMaxE / 32; ++j) {
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
                if (lane == 0 && bi >= 0 && bi < E) s_id[t * K + k] = bi;  // none left: stays -1
                prev_v = bv;
                prev_i = bi;
            }
        }
    } else {
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
    const uint32_t w2_bytes = static_cast<uint32_t>(nd) * Dff * (FP8 ? 1 : 2);
    const bool staged = a.w2_smem && nd > 0 && T > 0;
    if (staged) {
        if (tid == kLdThreads - 32) {  // lane 0 of warp 15 issues one 16-row box per expert slot
            const uint32_t box = static_cast<uint32_t>(kLayerDecodeW2Rows) * Dff * (FP8 ? 1 : 2);
            mbar_arrive_expect_tx(&s_w2bar, box * T);
            for (int i = 0; i < T; ++i)
                tma_load_3d(&tmW2, &s_w2bar, reinterpret_cast<char*>(s_w2) + static_cast<size_t>(i) * box, 0,
                            s_touched[i] * D + d0, 0);
        }
    } else if (nd > 0) {
        // not staged: the W2 rows of the first slots, up to the byte budget, into
        // L2; slot i by lane i / 16 of warp i % 16 (a thread issues its bulk
        // prefetches one after another, which held up warp 0's GEMM1 when it
        // issued them all)
        const int i = (tid & 31) * kLdWarps + warp;
        if (i < T && static_cast<long long>(i + 1) * D * Dff * (FP8 ? 1 : 2) <= a.l2_prefetch_max) {
            const long long r = static_cast<long long>(s_touched[i]) * D + d0;
            l2_prefetch_bulk(FP8 ? static_cast<const void*>(a.w2q + r * Dff)
                                 : static_cast<const void*>(a.w2 + r * Dff),
                             w2_bytes);
        }
    }
    for (int r = b; r < rows; r += G) {
        if (FP8) {  // the codes of the token row
            uint4* dst = reinterpret_cast<uint4*>(a.xq_perm + static_cast<long long>(r) * D);
            const uint4* src = reinterpret_cast<const uint4*>(s_xq + static_cast<size_t>(s_src[r]) * D);
            for (int c = tid; c < D / 16; c += kLdThreads) dst[c] = src[c];
        } else {
            uint4* dst = reinterpret_cast<uint4*>(a.x_perm + static_cast<long long>(r) * D);
            for (int c = tid; c < chunks; c += kLdThreads) dst[c] = s_x[s_src[r] * chunks + c];
        }
    }
    // ---- 3. GEMM1 + activation on the tensor cores (gemv_tiles): a tile is
    // 16 consecutive rows f of one expert slot's W1 (and W3) against the
    // slot's token rows; the CTA's tiles are a contiguous range (gemv_tiles).
    {
        const int ft = Dff / kLayerDecodeW2Rows;                 // tiles per expert slot
        const int TT = T * ft;
        const int t_lo = static_cast<int>(static_cast<unsigned>(TT) * b / G);
        const int nt = static_cast<int>(static_cast<unsigned>(TT) * (b + 1) / G) - t_lo;
        const int rstride = FP8 ? D / 16 : D / 8;                // 16-byte chunks per W1 row
        const uint64_t pol = l2_policy_evict_first();
        auto run = [&](int j, int s_beg, int s_end, float (&acc_g)[4], float (&acc_u)[4]) {
            const int tt = t_lo + j, slot = tt / ft;
            const int e = s_touched[slot], r0 = s_off[e], ne = s_off[e + 1] - r0;
            const int g = lane >> 2;
            const long long row = static_cast<long long>(e) * Dff + (tt - slot * ft) * kLayerDecodeW2Rows + g;
            const uint4* p1 = reinterpret_cast<const uint4*>(FP8 ? static_cast<const void*>(a.w1q + row * D)
                                                                 : static_cast<const void*>(a.w1 + row * D));
            const uint4* p3 = reinterpret_cast<const uint4*>(
                SWIGLU ? (FP8 ? static_cast<const void*>(a.w3q + row * D) : static_cast<const void*>(a.w3 + row * D))
                       : static_cast<const void*>(p1));
            const uint4* xr = nullptr;                           // token row of B column g
            if (g < NR && g < ne)
                xr = FP8 ? reinterpret_cast<const uint4*>(s_xq + static_cast<size_t>(s_src[r0 + g]) * D)
                         : s_x + static_cast<size_t>(s_src[r0 + g]) * chunks;
            gemv_steps<FP8, SWIGLU>(p1, p1 + 8 * rstride, p3, p3 + 8 * rstride, xr, lane & 3, s_beg, s_end, pol,
                                    acc_g, acc_u);
        };
        // h[row][f] from the two sums of tile j's row rr and slot row col
        auto finish = [&](int j, int rr, int col, float gs, float us) {
            const int tt = t_lo + j, slot = tt / ft;
            const int f = (tt - slot * ft) * kLayerDecodeW2Rows + rr;
            const int e = s_touched[slot], r0 = s_off[e];
            if (col >= s_off[e + 1] - r0) return;
            float hv;
            if constexpr (FP8) {  // the e4m3 GEMM epilogue: acc * token scale * weight-row scale
                const float rs = s_xs[s_src[r0 + col]];
                const long long wr = static_cast<long long>(e) * Dff + f;
                hv = SWIGLU ? silu_f32(gs * rs * a.s1[wr]) * (us * rs * a.s3[wr]) : silu_f32(gs * rs * a.s1[wr]);
            } else {
                hv = SWIGLU ? silu_f32(gs) * us : silu_f32(gs);
            }
            a.h[static_cast<long long>(r0 + col) * Dff + f] = bf16_rn_bits(hv);
        };
        const int S1 = FP8 ? D / 128 : D / 64;
        if (kPickSchedule && gemv_pick_even(nt, S1, SWIGLU ? kG1Steps : kG1Steps1)) {
            if constexpr (kPickSchedule) gemv_tiles<SWIGLU, NR>(nt, S1, s_g1, warp, lane, tid, run, finish);
        } else {
            gemv_tiles_grouped<SWIGLU, NR>(nt, S1, s_g1, warp, lane, tid, run, finish);
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
    if (FP8) {  // h rows -> e4m3 codes (the MMA's B operand) with the row quantiser's rule, a warp per row
        for (int r = warp; r < rows; r += kLdWarps) {
            const uint4* hrow = reinterpret_cast<const uint4*>(a.h) + static_cast<size_t>(r) * chunks2;
            uint32_t m = 0;
            for (int c = lane; c < chunks2; c += 32) m = max(m, absmax8(ld_cg_v4(hrow + c)));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            const int k = scale_exp_of(m);
            const float inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);  // 2^-k
            const float sc = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
            if (lane == 0) {
                s_hs[r] = sc;
                if (writer) a.h_scale[r] = sc;
            }
            for (int c = lane; c < chunks2; c += 32) {
                const uint2 q = to_e4m3x8(ld_cg_v4(hrow + c), inv);
                reinterpret_cast<uint2*>(s_hq + static_cast<size_t>(r) * Dff)[c] = q;
                if (writer) reinterpret_cast<uint2*>(a.hq + static_cast<size_t>(r) * Dff)[c] = q;
            }
        }
    } else {  // h rows in bf16: the MMA's B operand
        for (int i = tid; i < rows * chunks2; i += kLdThreads)
            s_x[i] = ld_cg_v4(reinterpret_cast<const uint4*>(a.h) + i);
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
        const int row_bytes = Dff * (FP8 ? 1 : 2);
        const int ksteps = row_bytes / 32;  // 32 bytes of K per MMA: 16 bf16 or 32 e4m3
        const uint32_t w2s = smem_u32(s_w2), hs = FP8 ? smem_u32(s_hq) : smem_u32(s_x);
        for (int it = warp; it < T * kparts; it += kLdWarps) {
            const int slot = it / kparts, kp = it - slot * kparts;
            const int e = s_touched[slot], r0 = s_off[e], ne = s_off[e + 1] - r0;
            const int k_lo = ksteps * kp / kparts, k_hi = ksteps * (kp + 1) / kparts;
            // ldmatrix row addresses: A (x4) rows (m & 1) * 8 + lane & 7 at k-chunk m >> 1, m = lane >> 3;
            // B (x2) token row lane & 7 at k-chunk (lane >> 3) & 1
            const int arow = ((lane >> 3) & 1) * 8 + (lane & 7), akc = lane >> 4;
            const uint32_t abase = w2s + static_cast<uint32_t>(slot) * kLayerDecodeW2Rows * row_bytes + arow * 128;
            const int bn = lane & 7;
            const uint32_t bbase =
                hs + static_cast<uint32_t>(r0 + (bn < ne ? bn : 0)) * row_bytes + ((lane >> 3) & 1) * 16;
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int ks = k_lo; ks < k_hi; ++ks) {
                const int kb = ks * 32;  // byte offset of the step's K in a row
                const int ch = ((kb & 127) >> 4) + akc;  // 16-byte chunk in the 128-byte row of its k-block
                uint32_t a0, a1, a2, a3, b0, b1;
                ldmatrix_x4(abase + (kb >> 7) * (kLayerDecodeW2Rows * 128) + ((ch ^ (arow & 7)) << 4), a0, a1, a2, a3);
                ldmatrix_x2(bbase + kb, b0, b1);
                if (FP8)
                    mma_e4m3_16832(d, a0, a1, a2, a3, b0, b1);
                else
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
                if (FP8) y = y * s_hs[r0 + n] * a.s2[static_cast<long long>(e) * D + d0 + dd];  // acc * row * column scale
                const uint16_t yb = bf16_rn_bits(y);
                s_y[(r0 + n) * nd + dd] = yb;
                a.y_perm[static_cast<long long>(r0 + n) * D + d0 + dd] = yb;
            }
        }
    } else {
        // Tensor cores on W2 from global memory (gemv_tiles): a tile is 16 of
        // the CTA's columns d (W2 rows e*D + d0 + d, past nd: the last one
        // again, its sums unused) against the expert's h rows.
        const int tps = (nd + kLayerDecodeW2Rows - 1) / kLayerDecodeW2Rows;  // tiles per expert slot
        const uint64_t pol = l2_policy_evict_first();
        auto run = [&](int j, int s_beg, int s_end, float (&acc)[4], float (&unused)[4]) {
            const int slot = j / tps, dt = j - slot * tps;
            const int e = s_touched[slot], r0 = s_off[e], ne = s_off[e + 1] - r0;
            const int g = lane >> 2;
            const int dg = min(dt * kLayerDecodeW2Rows + g, nd - 1), dh = min(dt * kLayerDecodeW2Rows + g + 8, nd - 1);
            const long long rg = static_cast<long long>(e) * D + d0 + dg, rh = static_cast<long long>(e) * D + d0 + dh;
            const uint4* pg = reinterpret_cast<const uint4*>(FP8 ? static_cast<const void*>(a.w2q + rg * Dff)
                                                                 : static_cast<const void*>(a.w2 + rg * Dff));
            const uint4* ph = reinterpret_cast<const uint4*>(FP8 ? static_cast<const void*>(a.w2q + rh * Dff)
                                                                 : static_cast<const void*>(a.w2 + rh * Dff));
            const uint4* xr = nullptr;                           // h row of B column g
            if (g < NR && g < ne)
                xr = FP8 ? reinterpret_cast<const uint4*>(s_hq + static_cast<size_t>(r0 + g) * Dff)
                         : s_x + static_cast<size_t>(r0 + g) * chunks2;
            gemv_steps<FP8, false>(pg, ph, nullptr, nullptr, xr, lane & 3, s_beg, s_end, pol, acc, unused);
        };
        auto finish = [&](int j, int rr, int n, float y, float) {
            const int slot = j / tps, dd = (j - slot * tps) * kLayerDecodeW2Rows + rr;
            const int e = s_touched[slot], r0 = s_off[e];
            if (dd >= nd || n >= s_off[e + 1] - r0) return;
            if (FP8) y = y * s_hs[r0 + n] * a.s2[static_cast<long long>(e) * D + d0 + dd];  // acc * row * column scale
            const uint16_t yb = bf16_rn_bits(y);
            s_y[(r0 + n) * nd + dd] = yb;
            a.y_perm[static_cast<long long>(r0 + n) * D + d0 + dd] = yb;
        };
        const int nt2 = nd > 0 ? T * tps : 0, S2 = Dff * (FP8 ? 1 : 2) / 128;
        if (kPickSchedule && gemv_pick_even(nt2, S2, kG1Steps1)) {
            if constexpr (kPickSchedule) gemv_tiles<false, NR>(nt2, S2, s_g1, warp, lane, tid, run, finish);
        } else {
            gemv_tiles_grouped<false, NR>(nt2, S2, s_g1, warp, lane, tid, run, finish);
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

template <bool SWIGLU, int NR, bool FP8>
static cudaError_t ld_launch(const LayerDecodeArgs& a, const CUtensorMap& tm_w2, int grid, size_t smem,
                             cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(layer_decode_kernel<SWIGLU, NR, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
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
    return cudaLaunchKernelEx(&cfg, layer_decode_kernel<SWIGLU, NR, FP8>, a, tm_w2);
}

template <bool SWIGLU>
static cudaError_t ld_dispatch(const LayerDecodeArgs& a, const CUtensorMap& tm_w2, int grid, size_t smem,
                               cudaStream_t st) {
    if (a.fp8) {
        if (a.N <= 1) return ld_launch<SWIGLU, 1, true>(a, tm_w2, grid, smem, st);
        if (a.N <= 2) return ld_launch<SWIGLU, 2, true>(a, tm_w2, grid, smem, st);
        if (a.N <= 4) return ld_launch<SWIGLU, 4, true>(a, tm_w2, grid, smem, st);
        return ld_launch<SWIGLU, 8, true>(a, tm_w2, grid, smem, st);
    }
    if (a.N <= 1) return ld_launch<SWIGLU, 1, false>(a, tm_w2, grid, smem, st);
    if (a.N <= 2) return ld_launch<SWIGLU, 2, false>(a, tm_w2, grid, smem, st);
    if (a.N <= 4) return ld_launch<SWIGLU, 4, false>(a, tm_w2, grid, smem, st);
    return ld_launch<SWIGLU, 8, false>(a, tm_w2, grid, smem, st);
}

cudaError_t launch_layer_decode(const LayerDecodeArgs& a, const CUtensorMap& tm_w2, int grid, cudaStream_t st) {
    if (a.N < 1 || a.N > kLayerDecodeMaxN || a.N * a.K > kLayerDecodeMaxRows || a.E > kLayerDecodeMaxE ||
        grid < 1 || a.D / 8 > kSmallRouteThreads * kSmallRouteMaxChunks)
        return cudaErrorInvalidValue;
    if (a.fp8 && (a.D % 128 || a.Dff % 128))
        return cudaErrorInvalidValue;
    const size_t smem = layer_decode_smem(a.N, a.D, a.E, a.K, a.Dff, grid, a.w2_smem != 0, a.fp8 != 0).total;
    const bool swiglu = a.fp8 ? a.w3q != nullptr : a.w3 != nullptr;
    return swiglu ? ld_dispatch<true>(a, tm_w2, grid, smem, st) : ld_dispatch<false>(a, tm_w2, grid, smem, st);
}

int layer_decode_plan(int N, int D, int E, int K, int Dff, bool swiglu, bool fp8, int* w2_smem) {
    int dev = 0, nsm = 0, optin = 0;
    *w2_smem = 0;
    (void)swiglu;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    // the kernel's static shared memory is about 3.7 KB
    const size_t limit = static_cast<size_t>(optin) - 4096;
    // the kernel splits columns and items with 32-bit products
    if (static_cast<long long>(N) * K * Dff * nsm >= (1LL << 31) || static_cast<long long>(D / 2) * nsm >= (1LL << 31))
        return 0;
    // W2 staged: every CTA's columns fit one 16-row box, whose k-blocks a box can hold
    const int esize = fp8 ? 1 : 2;
    const bool w2_fits = 2 * ((D / 2 + nsm - 1) / nsm) <= kLayerDecodeW2Rows && Dff * esize / 128 <= 256;
    *w2_smem = w2_fits && layer_decode_smem(N, D, E, K, Dff, nsm, true, fp8).total <= limit ? 1 : 0;
    if (fp8 && (D % 128 || Dff % 128)) return 0;
    if (!*w2_smem && layer_decode_smem(N, D, E, K, Dff, nsm, false, fp8).total > limit) return 0;
    // 512 threads of at most 128 registers and this shared memory: one CTA per SM
    return nsm;
}

}  // namespace moe
