// grouped_gemm.cuh -- persistent grouped GEMM on sm_103a tensor cores
// (tcgen05.mma, accumulators in TMEM, operands staged by TMA).
//
// One launch computes C_g = A_g * B_g^T for every group g (expert), where A_g
// is the ragged row segment group_offsets[g] .. group_offsets[g+1]-1 of one
// row-major [rows, k] bf16 matrix and B_g is a [n, k] slice of a stacked
// weight tensor.  This is the "grouped GEMM" of "MoE 推理完整机制：从 Router 到
// Expert Parallelism 的一切" (zoe.im), 第二层 "关键 kernel：Grouped GEMM": many
// different-size GEMMs in one launch, SMs assigned dynamically to experts.
// Here the assignment is a persistent tile loop: every CTA walks the global
// tile list (group, n-tile, m-tile) with stride gridDim.x, so an expert with
// more rows simply owns more tiles and more SMs (the "hot expert" concern of
// the same section and the persistent idea of 第四层 DeepGEMM / MegaMoE).
//
// CTA layout (192 threads, one CTA per SM):
//   warp 0      TMA producer: A tile [128 x 64] + B tile [BN x 64] per stage
//   warp 1      TMEM allocator and MMA issuer (one thread), 128 x BN x 16 MMAs
//   warps 2..5  epilogue: TMEM -> registers -> activation -> global
// Pipelines: STAGES shared-memory stages (full/empty mbarriers) and two TMEM
// accumulators (tmem_full/tmem_empty) so the epilogue of tile i overlaps the
// main loop of tile i+1.  Every wait is bounded (device.cuh: mbar_wait).
//
// Epilogues:
//   EPI_SWIGLU_BF16  B stage = [W1 rows n..n+BN/2 ; W3 rows n..n+BN/2], so the
//                    accumulator holds gate | up for the same BN/2 columns and
//                    h = silu(gate) * up is formed in registers -> bf16.
//   EPI_SILU_BF16    h = silu(acc) -> bf16
//   EPI_STORE_BF16   y = acc -> bf16
//   EPI_F32          raw fp32 accumulator of one k-split (router logits, or a
//                    split GEMM2); a separate kernel sums the splits in order
//   EPI_F32_DUAL     the same with the W1 | W3 B stage of SwiGLU (split GEMM1)
//
// Split-K: with args.splits = S > 1 every (group, n-tile, m-tile) becomes S
// work items, split s summing k-blocks [s*nkb/S, (s+1)*nkb/S); the splits of
// one tile are consecutive in the work list.  Used when the tile list alone
// would leave SMs idle (router, decode-sized FFN calls).
//
// Operand type (template FP8): bf16 (tcgen05 kind::f16) or e4m3 (kind::f8f6f4,
// one fp32 scale per output row and per weight row applied in the epilogue).
// A stage is one 128-byte swizzle row of K either way (64 bf16 / 128 e4m3),
// so shared-memory layout, descriptors and pipeline depth are the same.
// grouped_gemm.cu instantiates the bf16 kernels, grouped_gemm_e4m3.cu the
// e4m3 ones.
#pragma once

#include <math.h>

#include <atomic>

#include "gemm_common.cuh"

namespace moe {

// ----------------------------------------------------------------------------
template <int EPI, int BN, bool FP8, bool GATHER>
__global__ void __launch_bounds__(192, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, const GemmArgs args) {
    using C = GemmCfg<EPI, BN>;
    using T = OpType<FP8>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + S * C::B_BYTES);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;   // [2]
    uint64_t* tempty = tfull + 2;  // [2]
    uint64_t* drain = tempty + 2;  // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_goff = reinterpret_cast<int*>(tmem_slot + 4);  // [G+1] group row offsets
    int* s_tpre = s_goff + (args.G + 1);                  // [G+1] m-tile prefix
    int* s_src = s_tpre + (args.G + 1);                   // [kBM] gathered A: source rows of the tile

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = args.G;
    uint32_t* err = args.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // gathered A: the TMA issuer's expect_tx plus one arrival per producer lane
            mbar_init(&full[s], GATHER ? 33 : 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 4);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    // Group row ranges.  They must start at 0, never decrease and end within
    // the M rows of A; otherwise nothing is computed and a bounds error is
    // recorded.
    pdl_wait();  // group offsets and A come from earlier kernels
    for (int i = threadIdx.x; i <= G; i += blockDim.x)
        s_goff[i] = args.group_offsets ? args.group_offsets[i] : (i == 0 ? 0 : args.M);
    __syncthreads();
    int bad = 0;
    for (int i = threadIdx.x; i < G; i += blockDim.x) bad |= (s_goff[i] > s_goff[i + 1]);
    if (threadIdx.x == 0) bad |= (s_goff[0] != 0) | (s_goff[G] > args.M);
    const bool offsets_bad = __syncthreads_or(bad) != 0;
    if (offsets_bad && blockIdx.x == 0 && threadIdx.x == 0) record_error(err, MOE_DEVERR_BOUNDS);
    if (warp == 0) {  // exclusive prefix of m-tiles per group
        int carry = 0;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int v = (g < G) ? (s_goff[g + 1] - s_goff[g] + kBM - 1) / kBM : 0;
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
    const int num_kb = args.k_dim / T::KB;
    // every split must own at least one k-block
    const int splits = args.splits;
    const bool split_bad = splits < 1 || splits > num_kb;
    if (split_bad && blockIdx.x == 0 && threadIdx.x == 0) record_error(err, MOE_DEVERR_BOUNDS);
    const int total_tiles = (offsets_bad || split_bad) ? 0 : s_tpre[G] * nt * splits;

    if (GATHER && warp == 0) {
        // ------------------------------------------------------------ producer, gathered A
        // lane 0 loads B by TMA; every lane copies A rows with cp.async, and
        // each lane's copies arrive on the stage's full barrier by themselves
        // when they land (the MMA thread fences them for the async proxy).
        if (lane == 0) {
            tma_prefetch_desc(&tmB);
            if (C::DUAL_B) tma_prefetch_desc(&tmB2);
        }
        bool withhold = args.dbg && (*args.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD) && blockIdx.x == 0;
        uint32_t pending = 0, pend_parity = 0;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            const int split = t % splits;
            const TileInfo ti = decode_tile(t / splits, G, nt, s_tpre, s_goff);
            const int brow = ti.g * args.b_rows_per_group + ti.n_tile * C::N_OUT_TILE;
            const int kb0 = split * num_kb / splits, kb1 = (split + 1) * num_kb / splits;
            gather_rows_fill(s_src, kBM, args, ti.row0, ti.rows, lane, err);
            for (int kb = kb0; kb < kb1; ++kb) {
                // every lane waits (each then writes the stage); all go on or all stop
                const bool got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                if (withhold) {
                    withhold = false;  // test hook: this stage never fills
                } else {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[stage], C::B_BYTES);
                        uint8_t* b_dst = sB + stage * C::B_BYTES;
                        if constexpr (C::DUAL_B) {
                            tma_load_2d(&tmB, &full[stage], b_dst, kb * T::KB, brow);
                            tma_load_2d(&tmB2, &full[stage], b_dst + (BN / 2) * kRowBytes, kb * T::KB, brow);
                        } else {
                            tma_load_2d(&tmB, &full[stage], b_dst, kb * T::KB, brow);
                        }
                        pending |= 1u << stage;
                        pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
                    }
                    gather_rows_issue<kBM>(smem_u32(sA + stage * C::A_BYTES), s_src, args, kb, lane);
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
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            if (C::DUAL_B) tma_prefetch_desc(&tmB2);
            bool withhold = args.dbg && (*args.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD) && blockIdx.x == 0;
            uint32_t pending = 0, pend_parity = 0;  // per-stage: a load issued, its phase parity
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const int split = t % splits;
                const TileInfo ti = decode_tile(t / splits, G, nt, s_tpre, s_goff);
                const int brow = ti.g * args.b_rows_per_group + ti.n_tile * C::N_OUT_TILE;
                const int kb0 = split * num_kb / splits, kb1 = (split + 1) * num_kb / splits;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err)) { ok = false; break; }
                    if (withhold) {
                        withhold = false;  // test hook: this stage never fills
                    } else {
                        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        uint8_t* a_dst = sA + stage * C::A_BYTES;
                        uint8_t* b_dst = sB + stage * C::B_BYTES;
                        tma_load_2d(&tmA, &full[stage], a_dst, kb * T::KB, ti.row0);
                        if constexpr (C::DUAL_B) {
                            tma_load_2d(&tmB, &full[stage], b_dst, kb * T::KB, brow);
                            tma_load_2d(&tmB2, &full[stage], b_dst + (BN / 2) * kRowBytes, kb * T::KB, brow);
                        } else {
                            tma_load_2d(&tmB, &full[stage], b_dst, kb * T::KB, brow);
                        }
                        pending |= 1u << stage;
                        pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            // Every issued copy must land before this CTA's shared memory can
            // be released (immediate unless the pipeline was abandoned).
            for (int s = 0; s < S; ++s)
                if (pending & (1u << s)) drain_wait(&full[s], (pend_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f32acc<FP8>(kBM, BN);
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
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, err)) { ok = false; break; }
                    if constexpr (GATHER) fence_proxy_async_smem();  // the gathered rows, for the tensor core
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::A_BYTES));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                    for (int k = 0; k < T::MMAS; ++k) {
                        // advance 32 bytes along K inside the swizzle atom
                        umma<FP8>(d_tmem, adesc + static_cast<uint64_t>(2 * k),
                                  bdesc + static_cast<uint64_t>(2 * k), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(&empty[stage]);  // stage free once these MMAs finish
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);        // accumulator ready for the epilogue
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // all MMAs of this CTA complete before TMEM is released
            umma_commit(drain);
            drain_wait(drain, 0, err);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // this warp may access TMEM lanes 32q .. 32q+31
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
            const int split = t % splits;
            const TileInfo ti = decode_tile(t / splits, G, nt, s_tpre, s_goff);
            const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int r = q * 32 + lane;
            const bool valid = r < ti.rows;
            const long long grow = static_cast<long long>(ti.row0) + r;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            if constexpr (EPI == EPI_F32 || EPI == EPI_F32_DUAL) {
                epilogue_f32<EPI, BN, FP8>(t_row, valid, grow, ti.g, ti.n_tile, split, args);
            } else {
                epilogue_ffn<EPI, BN, FP8>(t_row, valid, grow, ti.g, ti.n_tile, args);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

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
// host-side dispatch
// ----------------------------------------------------------------------------
template <int EPI, int BN>
inline size_t smem_bytes_for(int G) {
    using C = GemmCfg<EPI, BN>;
    return 1024 /* alignment slack */ + static_cast<size_t>(C::STAGES) * C::STAGE_BYTES +
           (2 * C::STAGES + 5) * sizeof(uint64_t) + 16 + 2 * static_cast<size_t>(G + 1) * sizeof(int) +
           kBM * sizeof(int) /* gathered A: source rows */;
}

// The dynamic shared-memory limit is raised once per (instantiation, device),
// to the size the largest group count (1024) needs.
template <int EPI, int BN, bool FP8, bool GATHER>
inline cudaError_t ensure_smem_attr() {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI, BN, FP8, GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes_for<EPI, BN>(1024)));
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <int EPI, int BN, bool FP8, bool GATHER = false>
inline cudaError_t launch_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                            const GemmArgs& a, int grid, cudaStream_t st) {
    cudaError_t e = ensure_smem_attr<EPI, BN, FP8, GATHER>();
    if (e != cudaSuccess) return e;
    return launch_kernel(grouped_gemm_kernel<EPI, BN, FP8, GATHER>, dim3(grid), dim3(192),
                         smem_bytes_for<EPI, BN>(a.G), st, tmA, tmB, tmB2, a);
}

}  // namespace moe
