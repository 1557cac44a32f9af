// grouped_gemm_swap.cuh -- grouped GEMM with the operand roles swapped, for
// calls whose experts own only a few rows each (decode).
//
// The tensor core's M = 128 runs over weight rows and its N = BT (16 or 32)
// over the tokens of one expert: D^T[w, t] = sum_k W[w, k] * X[t, k].  A stage
// then holds 16 KB of weights and BT x 64 bf16 of tokens, instead of a 128-row
// token tile that is mostly past the end of the expert's segment, so ten
// stages of weights stay in flight per SM: decode is a weight-streaming
// problem ("MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im),
// 第二层 "关键 kernel：Grouped GEMM" runs every expert's GEMM in one launch; the
// ragged per-expert row counts are read from expert_offsets on the device).
//
// Tiles: (expert, weight-row tile, token tile, k-split); a SwiGLU weight tile
// is 64 W1 rows over 64 W3 rows, so one accumulator holds gate and up for the
// same 64 output columns.  Epilogue (thread = weight row): the up half goes
// through shared memory to the gate half, which forms silu(gate) * up and
// stores, for every token, 64 consecutive bf16 of h (coalesced).  Split-K
// partials store the raw accumulator (fp32) in the tile-interleaved layout the
// reduction kernels read.
//
// Operand type (template FP8): bf16 or e4m3 as in grouped_gemm.cuh; with e4m3
// each accumulator element is scaled by its weight row's and its token's
// scale before the epilogue uses it.  grouped_gemm_swap.cu instantiates the
// bf16 kernels, grouped_gemm_swap_e4m3.cu the e4m3 ones.
#pragma once

#include <algorithm>
#include <atomic>

#include "gemm_common.cuh"

namespace moe {

template <int EPI, int BT>
struct SwapCfg {
    static constexpr bool DUAL = (EPI == EPI_SWIGLU_BF16 || EPI == EPI_F32_DUAL);
    static constexpr bool F32 = (EPI == EPI_F32 || EPI == EPI_F32_DUAL);
    static constexpr int WROWS = 128;                   // weight rows per tile (MMA M)
    static constexpr int N_OUT_TILE = DUAL ? 64 : 128;  // output columns per tile
    static constexpr int A_BYTES = WROWS * kRowBytes;   // 16 KB of weights
    static constexpr int B_BYTES = BT * kRowBytes;      // the tokens
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 10;
    static constexpr int TMEM_COLS = (2 * BT < 32) ? 32 : 2 * BT;
    static constexpr int U_STRIDE = BT + 1;             // padded row of the up exchange
    static_assert(BT == 16 || BT == 32, "token tile");
};

template <int EPI, int BT, bool FP8, bool GATHER>
__global__ void __launch_bounds__(192, 1)
grouped_gemm_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
                         const __grid_constant__ CUtensorMap tmX, const GemmArgs args) {
    using C = SwapCfg<EPI, BT>;
    using T = OpType<FP8>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* sA = smem;                      // weights
    uint8_t* sB = smem + S * C::A_BYTES;     // tokens
    float* s_u = reinterpret_cast<float*>(sB + S * C::B_BYTES);  // [64][BT+1] up values
    uint64_t* full = reinterpret_cast<uint64_t*>(s_u + 64 * C::U_STRIDE);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_goff = reinterpret_cast<int*>(tmem_slot + 4);
    int* s_tpre = s_goff + (args.G + 1);
    int* s_src = s_tpre + (args.G + 1);  // [BT] gathered tokens: source rows of the token tile

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = args.G;
    uint32_t* err = args.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // gathered tokens: the TMA issuer's expect_tx plus one arrival per producer lane
            mbar_init(&full[s], GATHER ? 33 : 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();  // group offsets and the activations come from earlier kernels
    for (int i = threadIdx.x; i <= G; i += blockDim.x)
        s_goff[i] = args.group_offsets ? args.group_offsets[i] : (i == 0 ? 0 : args.M);
    __syncthreads();
    const int num_kb = args.k_dim / T::KB;
    const int splits = args.splits;
    int bad = 0;
    for (int i = threadIdx.x; i < G; i += blockDim.x) bad |= (s_goff[i] > s_goff[i + 1]);
    if (threadIdx.x == 0) bad |= (s_goff[0] != 0) | (s_goff[G] > args.M) | (splits < 1) | (splits > num_kb);
    const bool args_bad = __syncthreads_or(bad) != 0;
    if (args_bad && blockIdx.x == 0 && threadIdx.x == 0) record_error(err, MOE_DEVERR_BOUNDS);
    if (warp == 0) {  // exclusive prefix of BT-row token tiles per group
        int carry = 0;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int v = (g < G) ? (s_goff[g + 1] - s_goff[g] + BT - 1) / BT : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (g < G) s_tpre[g + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_tpre[0] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int nt = (args.n_out + C::N_OUT_TILE - 1) / C::N_OUT_TILE;
    const int total_tiles = args_bad ? 0 : s_tpre[G] * nt * splits;

    if (GATHER && warp == 0) {
        // ------------------------------------------------------------ producer, gathered tokens
        // lane 0 loads the weight tile by TMA; every lane copies the token
        // rows with cp.async, whose landing arrives on the stage's full barrier
        if (lane == 0) {
            tma_prefetch_desc(&tmW);
            if (C::DUAL) tma_prefetch_desc(&tmW2);
        }
        bool withhold = args.dbg && (*args.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD) && blockIdx.x == 0;
        uint32_t pending = 0, pend_parity = 0;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            const int split = t % splits;
            const TileInfo ti = decode_tile(t / splits, G, nt, s_tpre, s_goff, BT);
            const int wrow = ti.g * args.b_rows_per_group + ti.n_tile * C::N_OUT_TILE;
            const int kb0 = split * num_kb / splits, kb1 = (split + 1) * num_kb / splits;
            gather_rows_fill(s_src, BT, args, ti.row0, ti.rows, lane, err);
            for (int kb = kb0; kb < kb1; ++kb) {
                // every lane waits (each then writes the stage); all go on or all stop
                const bool got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                if (withhold) {
                    withhold = false;  // test hook: this stage never fills
                } else {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[stage], C::A_BYTES);
                        uint8_t* a_dst = sA + stage * C::A_BYTES;
                        if constexpr (C::DUAL) {
                            tma_load_2d(&tmW, &full[stage], a_dst, kb * T::KB, wrow);
                            tma_load_2d(&tmW2, &full[stage], a_dst + 64 * kRowBytes, kb * T::KB, wrow);
                        } else {
                            tma_load_2d(&tmW, &full[stage], a_dst, kb * T::KB, wrow);
                        }
                        pending |= 1u << stage;
                        pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
                    }
                    gather_rows_issue<BT>(smem_u32(sB + stage * C::B_BYTES), s_src, args, kb, lane);
                }
                cp_async_arrive_noinc(&full[stage]);
                if (++stage == S) { stage = 0; phase ^= 1u; }
            }
        }
        cp_async_wait_all();  // no copy may land after this CTA's shared memory is released
        if (lane == 0) {
            for (int s = 0; s < S; ++s)
                if (pending & (1u << s)) drain_wait(&full[s], (pend_parity >> s) & 1u, err);
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmW);
            if (C::DUAL) tma_prefetch_desc(&tmW2);
            tma_prefetch_desc(&tmX);
            bool withhold = args.dbg && (*args.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD) && blockIdx.x == 0;
            uint32_t pending = 0, pend_parity = 0;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const int split = t % splits;
                const TileInfo ti = decode_tile(t / splits, G, nt, s_tpre, s_goff, BT);
                const int wrow = ti.g * args.b_rows_per_group + ti.n_tile * C::N_OUT_TILE;
                const int kb0 = split * num_kb / splits, kb1 = (split + 1) * num_kb / splits;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err)) { ok = false; break; }
                    if (withhold) {
                        withhold = false;  // test hook: this stage never fills
                    } else {
                        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        uint8_t* a_dst = sA + stage * C::A_BYTES;
                        if constexpr (C::DUAL) {
                            tma_load_2d(&tmW, &full[stage], a_dst, kb * T::KB, wrow);
                            tma_load_2d(&tmW2, &full[stage], a_dst + 64 * kRowBytes, kb * T::KB, wrow);
                        } else {
                            tma_load_2d(&tmW, &full[stage], a_dst, kb * T::KB, wrow);
                        }
                        tma_load_2d(&tmX, &full[stage], sB + stage * C::B_BYTES, kb * T::KB, ti.row0);
                        pending |= 1u << stage;
                        pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            for (int s = 0; s < S; ++s)
                if (pending & (1u << s)) drain_wait(&full[s], (pend_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f32acc<FP8>(C::WROWS, BT);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const int split = t % splits;
                const int kb0 = split * num_kb / splits, kb1 = (split + 1) * num_kb / splits;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BT);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, err)) { ok = false; break; }
                    if constexpr (GATHER) fence_proxy_async_smem();  // the gathered tokens, for the tensor core
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::A_BYTES));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                    for (int k = 0; k < T::MMAS; ++k)
                        umma<FP8>(d_tmem, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k),
                                  idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            umma_commit(drain);
            drain_wait(drain, 0, err);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;        // TMEM lanes 32q .. 32q+31
        const int r = q * 32 + lane;   // weight row within the tile
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
            const int split = t % splits;
            const TileInfo ti = decode_tile(t / splits, G, nt, s_tpre, s_goff, BT);
            const int nv = ti.rows;  // valid tokens of this tile
            // e4m3: weight row r's scale (W1 | W3 halves for SwiGLU) and each
            // token's scale, loaded before the accumulator wait: under the
            // weight stream these dependent loads take microseconds, which
            // the wait for the tile's MMAs now hides
            float cs = 1.0f;
            float ts[BT];
            if constexpr (FP8) {
                const long long wbase = static_cast<long long>(ti.g) * args.b_rows_per_group;
                if constexpr (C::DUAL) {
                    cs = (r < 64) ? args.col_scale[wbase + ti.n_tile * 64 + r]
                                  : args.col_scale_up[wbase + ti.n_tile * 64 + (r - 64)];
                } else {
                    cs = args.col_scale[wbase + static_cast<long long>(ti.n_tile) * C::N_OUT_TILE + r];
                }
#pragma unroll
                for (int j = 0; j < BT; ++j) {
                    ts[j] = 0.0f;
                    if (j < nv) {
                        const long long tr = static_cast<long long>(ti.row0) + j;
                        const long long ri = args.row_scale_idx ? static_cast<long long>(args.row_scale_idx[tr]) : tr;
                        ts[j] = args.row_scale[ri];
                    }
                }
            }
            bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, err);
            // all four epilogue warps continue together or stop together
            ok = named_barrier_and(1, 128, ok);
            if (!ok) break;
            tc_fence_after();
            float v[BT];
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BT);
            if constexpr (BT == 16) {
                uint32_t u[16];
                tmem_ld_32x16(t_row, u);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(u[j]);
            } else {
                uint32_t u[32];
                tmem_ld_32x32(t_row, u);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);  // TMEM read: the MMA may reuse it
            if constexpr (FP8) {
#pragma unroll
                for (int j = 0; j < BT; ++j)
                    if (j < nv) v[j] = v[j] * ts[j] * cs;
            }
            if constexpr (C::F32) {
                // raw accumulator: column n*128 + r (DUAL: gate rows then up rows)
                float* out = reinterpret_cast<float*>(args.out) + split * args.split_stride;
                const long long col = static_cast<long long>(ti.n_tile) * C::WROWS + r;
#pragma unroll
                for (int j = 0; j < BT; ++j)
                    if (j < nv) out[(static_cast<long long>(ti.row0) + j) * args.ldo + col] = v[j];
            } else if constexpr (C::DUAL) {
                if (q >= 2) {
#pragma unroll
                    for (int j = 0; j < BT; ++j) s_u[(r - 64) * C::U_STRIDE + j] = v[j];
                }
                named_barrier_sync(1, 128);
                if (q < 2) {
                    uint16_t* out = reinterpret_cast<uint16_t*>(args.out);
                    const long long col = static_cast<long long>(ti.n_tile) * C::N_OUT_TILE + r;
#pragma unroll
                    for (int j = 0; j < BT; ++j) {
                        if (j < nv) {
                            const float h = silu_f32(v[j]) * s_u[r * C::U_STRIDE + j];
                            const __nv_bfloat16 b = __float2bfloat16_rn(h);
                            out[(static_cast<long long>(ti.row0) + j) * args.ldo + col] =
                                *reinterpret_cast<const uint16_t*>(&b);
                        }
                    }
                }
                named_barrier_sync(1, 128);  // s_u free for the next tile
            } else {
                uint16_t* out = reinterpret_cast<uint16_t*>(args.out);
                const long long col = static_cast<long long>(ti.n_tile) * C::N_OUT_TILE + r;
#pragma unroll
                for (int j = 0; j < BT; ++j) {
                    if (j < nv) {
                        const float y = (EPI == EPI_SILU_BF16) ? silu_f32(v[j]) : v[j];
                        const __nv_bfloat16 b = __float2bfloat16_rn(y);
                        out[(static_cast<long long>(ti.row0) + j) * args.ldo + col] =
                            *reinterpret_cast<const uint16_t*>(&b);
                    }
                }
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    __syncwarp();
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------
template <int EPI, int BT>
inline size_t swap_smem_bytes(int G) {
    using C = SwapCfg<EPI, BT>;
    return 1024 + static_cast<size_t>(C::STAGES) * C::STAGE_BYTES + 64 * C::U_STRIDE * sizeof(float) +
           (2 * C::STAGES + 5) * sizeof(uint64_t) + 16 + 2 * static_cast<size_t>(G + 1) * sizeof(int) +
           BT * sizeof(int) /* gathered token rows */;
}

template <int EPI, int BT, bool FP8, bool GATHER = false>
inline cudaError_t swap_launch(const CUtensorMap& tmW, const CUtensorMap& tmW2, const CUtensorMap& tmX,
                               const GemmArgs& a, int grid, cudaStream_t st) {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(grouped_gemm_swap_kernel<EPI, BT, FP8, GATHER>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(swap_smem_bytes<EPI, BT>(1024)));
        if (e != cudaSuccess) return e;
        done.fetch_or(bit, std::memory_order_acq_rel);
    }
    return launch_kernel(grouped_gemm_swap_kernel<EPI, BT, FP8, GATHER>, dim3(grid), dim3(192), swap_smem_bytes<EPI, BT>(a.G),
                         st, tmW, tmW2, tmX, a);
}

}  // namespace moe
