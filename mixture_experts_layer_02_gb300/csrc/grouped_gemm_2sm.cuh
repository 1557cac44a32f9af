// grouped_gemm_2sm.cuh -- the grouped GEMM on CTA pairs (tcgen05 cta_group::2).
//
// Same contract as grouped_gemm.cu (ragged expert segments, persistent tile
// loop, SwiGLU or plain bf16 epilogue), for calls whose experts own many rows
// (prefill).  A cluster of two CTAs on two SMs computes a 256 x 256 tile: each
// CTA loads its own 128 rows of A and its own 128 rows of B (the W1 half or the
// W3 half of a SwiGLU tile, or one half of the W2 rows), and the even CTA
// issues `tcgen05.mma.cta_group::2` with M = 256, so every SM reads only half
// of the B operand from L2 and shared memory.  That halves the per-SM operand
// traffic of the one-CTA 128 x 256 tile, which is what limits it.
//
// Tile list: the experts heaviest first, each expert's 256-row m-tiles in
// bands of 8 (band by band, n-tile by n-tile inside a band, the band's m-tiles
// innermost; gemm_common.cuh, decode_tile_banded), so that concurrent pairs
// share weight tiles in L2 and a large expert's token rows are not re-read
// from HBM once per n-tile.
//
// Synchronisation (all waits bounded as in the one-CTA kernel):
//   full[s]    even CTA: the TMA bytes of stage s of BOTH CTAs landed (each
//              CTA's loads count their bytes on the even CTA's barrier)
//   empty[s]   each CTA: the pair MMAs reading stage s finished (multicast commit)
//   tfull[a]   each CTA: accumulator a complete (multicast commit)
//   tempty[a]  even CTA: the 8 epilogue warps of both CTAs drained accumulator a
// Warp roles per CTA: 0 TMA producer, 1 TMEM allocator + (even CTA) MMA
// issuer, 2..5 epilogue.  Before leaving, the even CTA waits for every stage
// it expected (both CTAs' bytes) and a cluster barrier holds the odd CTA until
// then, so no copy can land in a CTA that has exited.
//
// Operand type (template FP8): bf16 or e4m3 as in grouped_gemm.cuh.
// grouped_gemm_2sm.cu instantiates the bf16 kernels, grouped_gemm_2sm_e4m3.cu
// the e4m3 ones.
#pragma once

#include <algorithm>
#include <atomic>

#include "gemm_common.cuh"

namespace moe {

constexpr int kPairRows = 2 * kBM;  // rows of A per pair tile

template <int EPI>
struct PairCfg {
    static constexpr int BN = 256;                         // N of the pair MMA
    static constexpr int A_BYTES = kBM * kRowBytes;        // this CTA's 128 rows of A
    static constexpr int B_BYTES = (BN / 2) * kRowBytes;   // this CTA's 128 rows of B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 6;
    static constexpr bool DUAL_B = (EPI == EPI_SWIGLU_BF16);
    static constexpr int N_OUT_TILE = DUAL_B ? BN / 2 : BN;
    static constexpr int TMEM_COLS = 2 * BN;               // two accumulators
    static_assert(EPI == EPI_SWIGLU_BF16 || EPI == EPI_STORE_BF16, "pair kernel epilogues");
};

template <int EPI, bool FP8, bool GATHER>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmB2, const GemmArgs args) {
    using C = PairCfg<EPI>;
    using T = OpType<FP8>;
    constexpr int S = C::STAGES;
    constexpr int BN = C::BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);  // identical offsets in both CTAs
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + S * C::B_BYTES);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;   // [2]
    uint64_t* tempty = tfull + 2;  // [2]
    uint64_t* drain = tempty + 2;  // [1]
    uint64_t* landed = drain + 1;  // [S] gathered A, odd CTA: its rows of stage s landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(landed + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_goff = reinterpret_cast<int*>(tmem_slot + 4);  // [G+1]
    int* s_tpre = s_goff + (args.G + 1);                  // [G+1] pair m-tiles before list position i
    int* s_ord = s_tpre + (args.G + 1);                   // [G] the groups, heaviest first
    int* s_src = s_ord + args.G;                          // [kBM] gathered A: this CTA's source rows

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = args.G;
    uint32_t* err = args.err;
    const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // gathered A: the even CTA's expect_tx, its 32 producer lanes' copy
            // arrivals and one forwarded arrival for the odd CTA's rows
            mbar_init(&full[s], GATHER ? 34 : 1);
            mbar_init(&empty[s], 1);
            mbar_init(&landed[s], 32);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    pdl_wait();  // group offsets and A come from earlier kernels
    for (int i = threadIdx.x; i <= G; i += blockDim.x)
        s_goff[i] = args.group_offsets ? args.group_offsets[i] : (i == 0 ? 0 : args.M);
    __syncthreads();
    int bad = 0;
    for (int i = threadIdx.x; i < G; i += blockDim.x) bad |= (s_goff[i] > s_goff[i + 1]);
    if (threadIdx.x == 0) bad |= (s_goff[0] != 0) | (s_goff[G] > args.M) | (args.splits != 1);
    const bool offsets_bad = __syncthreads_or(bad) != 0;
    if (offsets_bad && blockIdx.x == 0 && threadIdx.x == 0) record_error(err, MOE_DEVERR_BOUNDS);
    heaviest_first(s_goff, G, s_ord);
    __syncthreads();
    if (warp == 0) {  // exclusive prefix of 256-row m-tiles over the list order
        int carry = 0;
        for (int base = 0; base < G; base += 32) {
            const int i = base + lane;
            const int g = (i < G) ? s_ord[i] : 0;
            int v = (i < G) ? (s_goff[g + 1] - s_goff[g] + kPairRows - 1) / kPairRows : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (i < G) s_tpre[i + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_tpre[0] = 0;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int nt = (args.n_out + C::N_OUT_TILE - 1) / C::N_OUT_TILE;
    const int total_tiles = offsets_bad ? 0 : s_tpre[G] * nt;
    const int band = args.band > 0 ? args.band : kPairBand;
    const int num_kb = args.k_dim / T::KB;
    const int cid = blockIdx.x >> 1;
    const int ncl = gridDim.x >> 1;
    const uint32_t full_lead = mapa_shared(smem_u32(full), 0);
    const uint32_t tempty_lead = mapa_shared(smem_u32(tempty), 0);

    if (GATHER && warp == 0) {
        // ------------------------------------------------------------ producer, gathered A (both CTAs)
        // lane 0 loads this CTA's half of B by TMA (bytes counted on the even
        // CTA's barrier); every lane copies this CTA's 128 A rows with
        // cp.async.  The copies' landing arrives on the even CTA's full barrier
        // directly, or, in the odd CTA, on its local `landed` barrier, which
        // its warp 1 forwards to the even CTA.
        const CUtensorMap* mapB = (C::DUAL_B && rank == 1) ? &tmB2 : &tmB;
        if (lane == 0) tma_prefetch_desc(mapB);
        bool withhold = args.dbg && (*args.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD) && blockIdx.x == 0;
        uint32_t pending = 0, pend_parity = 0;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = cid; t < total_tiles && ok; t += ncl) {
            const TileInfo ti = decode_tile_banded(t, G, nt, s_tpre, s_ord, s_goff, kPairRows, band);
            const int brow = ti.g * args.b_rows_per_group + ti.n_tile * C::N_OUT_TILE +
                             (C::DUAL_B ? 0 : static_cast<int>(rank) * (BN / 2));
            const int my0 = static_cast<int>(rank) * kBM;  // this CTA's rows of the pair tile
            gather_rows_fill(s_src, kBM, args, ti.row0 + my0, max(0, min(kBM, ti.rows - my0)), lane, err);
            for (int kb = 0; kb < num_kb; ++kb) {
                // every lane waits (each then writes the stage); all go on or all stop
                const bool got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                if (withhold) {
                    withhold = false;  // test hook: this stage never fills
                } else {
                    if (lane == 0) {
                        if (leader) {
                            mbar_arrive_expect_tx(&full[stage], 2 * C::B_BYTES);
                            pending |= 1u << stage;
                            pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
                        }
                        tma_load_2d_pair(mapB, full_lead + 8u * stage, sB + stage * C::B_BYTES, kb * T::KB, brow);
                    }
                    gather_rows_issue<kBM>(smem_u32(sA + stage * C::A_BYTES), s_src, args, kb, lane);
                }
                cp_async_arrive_noinc(leader ? &full[stage] : &landed[stage]);
                if (++stage == S) { stage = 0; phase ^= 1u; }
            }
        }
        cp_async_wait_all();  // no copy may land after this CTA's shared memory is released
        if (lane == 0) {
            for (int s = 0; s < S; ++s)
                if (pending & (1u << s)) drain_wait(&full[s], (pend_parity >> s) & 1u, err);
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(C::DUAL_B && rank == 1 ? &tmB2 : &tmB);
            const CUtensorMap* mapB = (C::DUAL_B && rank == 1) ? &tmB2 : &tmB;
            bool withhold = args.dbg && (*args.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD) && blockIdx.x == 0;
            uint32_t pending = 0, pend_parity = 0;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = cid; t < total_tiles && ok; t += ncl) {
                const TileInfo ti = decode_tile_banded(t, G, nt, s_tpre, s_ord, s_goff, kPairRows, band);
                const int arow = ti.row0 + static_cast<int>(rank) * kBM;
                const int brow = ti.g * args.b_rows_per_group + ti.n_tile * C::N_OUT_TILE +
                                 (C::DUAL_B ? 0 : static_cast<int>(rank) * (BN / 2));
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err)) { ok = false; break; }
                    if (withhold) {
                        withhold = false;  // test hook: this stage never fills
                    } else {
                        if (leader) {
                            mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                            pending |= 1u << stage;
                            pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
                        }
                        tma_load_2d_pair(&tmA, full_lead + 8u * stage, sA + stage * C::A_BYTES, kb * T::KB, arow);
                        tma_load_2d_pair(mapB, full_lead + 8u * stage, sB + stage * C::B_BYTES, kb * T::KB, brow);
                    }
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            for (int s = 0; s < S; ++s)
                if (pending & (1u << s)) drain_wait(&full[s], (pend_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if (leader) {
                // ---------------------------------------------------- MMA issuer (even CTA)
                constexpr uint32_t idesc = idesc_f32acc<FP8>(kPairRows, BN);
                int stage = 0;
                uint32_t phase = 0;
                int acc = 0;
                uint32_t acc_phase = 0;
                bool ok = true;
                for (int t = cid; t < total_tiles && ok; t += ncl) {
                    if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err)) break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    for (int kb = 0; kb < num_kb; ++kb) {
                        if (!mbar_wait(&full[stage], phase, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        if constexpr (GATHER) fence_proxy_async_smem();  // the gathered rows, for the tensor core
                        tc_fence_after();
                        const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::A_BYTES));
                        const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                        for (int k = 0; k < T::MMAS; ++k)
                            umma_pair<FP8>(d_tmem, adesc + static_cast<uint64_t>(2 * k),
                                           bdesc + static_cast<uint64_t>(2 * k), idesc,
                                           (kb | k) != 0 ? 1u : 0u);
                        umma_commit_pair_multicast(&empty[stage], 0x3);
                        if (++stage == S) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    umma_commit_pair_multicast(&tfull[acc], 0x3);
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                }
                umma_commit_pair_multicast(drain, 0x3);  // every pair MMA done, in both CTAs
            } else if constexpr (GATHER) {
                // ---------------------------------------------------- forwarder (odd CTA, gathered A)
                // once this CTA's rows of a stage have landed, make them visible
                // to the async proxy and count them on the even CTA's full barrier
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                for (int t = cid; t < total_tiles && ok; t += ncl) {
                    for (int kb = 0; kb < num_kb; ++kb) {
                        if (!mbar_wait(&landed[stage], phase, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_smem();
                        mbar_arrive_cluster(full_lead + 8u * static_cast<uint32_t>(stage));
                        if (++stage == S) { stage = 0; phase ^= 1u; }
                    }
                }
            }
            drain_wait(drain, 0, err);  // the pair MMAs wrote this CTA's TMEM too
        }
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = cid; t < total_tiles; t += ncl) {
            const TileInfo ti = decode_tile_banded(t, G, nt, s_tpre, s_ord, s_goff, kPairRows, band);
            const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int r = static_cast<int>(rank) * kBM + q * 32 + lane;  // row within the pair tile
            const bool valid = r < ti.rows;
            const long long grow = static_cast<long long>(ti.row0) + r;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            epilogue_ffn<EPI, BN, FP8>(t_row, valid, grow, ti.g, ti.n_tile, args);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_lead + 8u * acc);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    __syncwarp();
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while its peer may still signal it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------
template <int EPI>
inline size_t pair_smem_bytes(int G) {
    using C = PairCfg<EPI>;
    return 1024 + static_cast<size_t>(C::STAGES) * C::STAGE_BYTES + (3 * C::STAGES + 5) * sizeof(uint64_t) +
           16 + (2 * static_cast<size_t>(G + 1) + G) * sizeof(int) + kBM * sizeof(int) /* gathered A rows */;
}

template <int EPI, bool FP8, bool GATHER>
inline cudaError_t pair_prepare(int* max_clusters) {
    static std::atomic<unsigned long long> done{0};
    static int clusters[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
        const size_t smem = pair_smem_bytes<EPI>(1024);
        e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<EPI, FP8, GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(192, 1, 1);
        cfg.dynamicSmemBytes = smem;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<EPI, FP8, GATHER>, &cfg);
        if (e != cudaSuccess) return e;
        clusters[dev & 63] = n;
        done.fetch_or(bit, std::memory_order_acq_rel);
    }
    *max_clusters = clusters[dev & 63];
    return cudaSuccess;
}

template <int EPI, bool FP8, bool GATHER = false>
inline cudaError_t pair_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                               const GemmArgs& a, long long tiles_ub, cudaStream_t st) {
    int max_clusters = 0;
    cudaError_t e = pair_prepare<EPI, FP8, GATHER>(&max_clusters);
    if (e != cudaSuccess) return e;
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const long long clusters = std::max<long long>(1, std::min<long long>(tiles_ub, max_clusters));
    return launch_kernel(grouped_gemm_pair_kernel<EPI, FP8, GATHER>, dim3(static_cast<unsigned>(2 * clusters)), dim3(192),
                         pair_smem_bytes<EPI>(a.G), st, tmA, tmB, tmB2, a);
}

}  // namespace moe
