// grouped_gemm_2sm_mixed.cuh -- the CTA-pair grouped GEMM with two kinds of
// tile in one persistent launch, for calls whose experts own very different
// row counts (skewed routing: a few hot experts and a long tail).
//
// "MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im), 第二层
// "关键 kernel：Grouped GEMM": one launch whose SMs are handed out over the
// experts, and a hot expert must not stall the rest.
//
// Hot experts (more than cold_rows rows) run 256 x 256 pair tiles as in
// grouped_gemm_2sm.cuh, heaviest expert first (rows descending, ties by
// index), each expert's m-tiles in bands so that concurrent pairs share a
// weight tile in L2.
//
// Cold experts (1 .. cold_rows rows) run swapped tiles: the pair MMA's M = 256
// runs over weight rows (128 per CTA) and its N = 32 over the expert's tokens
// (16 per CTA), so a cold tile is a stream of its weights.  On GB300 an MMA
// instruction of N <= 64 still takes about 46 cycles (128 at N = 256), so a
// swapped tile consumes its weights about 2.8x faster per byte than a 256-row
// tile; and a TMA copy costs about 0.3 us per SM whatever its size, so the
// weights of a cold stage arrive as one 64 KB box per CTA (128 rows x 4
// k-blocks, a 3-D view of the weight matrix) and its tokens as one 8 KB box.
//
// Work list: the hot tiles and the cold tiles, the cold ones spread evenly
// among the hot ones (position p is cold when floor((p+1)C/T) > floor(pC/T),
// C cold of T tiles), so that the cold experts' weight streaming from HBM
// overlaps the hot experts' tensor-bound tiles instead of forming an
// HBM-bound tail.  Pairs stride over the list as in the other kernels.
//
// SwiGLU (GEMM1) cold tiles: the even CTA holds 128 W1 rows (gate) and the
// odd CTA the 128 W3 rows (up) of the same output columns.  The even CTA
// forms h for the tile's first 16 tokens and the odd CTA for the last 16: each
// CTA's epilogue sends the other half of its accumulator rows to the peer's
// exchange buffer (distributed shared memory) in two rounds of 8 values, with
// one mbarrier for "values landed" and one for "buffer read".
//
// Shared memory: 3 stage slots of 72 KB.  A hot stage holds 2 k-blocks (this
// CTA's 128 token rows, then its 128 weight rows, one 32 KB 3-D box each: 6
// k-blocks in flight, as in grouped_gemm_2sm.cuh); a cold stage holds 4
// k-blocks (64 KB of weights, then 8 KB of tokens).  Up to 256 experts.
// Synchronisation, warp roles, bounded waits and the exit protocol are those
// of grouped_gemm_2sm.cuh.  bf16 operands.
//
// Measured on GB300 this kernel is not faster than grouped_gemm_2sm.cuh on a
// DeepSeek-V3-shaped layer with Zipf-skewed routing: a cold tile is cheaper
// than the 256-row tile it replaces (26-32 against about 40 us), but while
// cold tiles run their single-use weight streams push the hot tiles' working
// set out of L2 and every hot tile slows by about 9%.  The library therefore
// runs it only when MOE_PAIR_COLD_ROWS is set; its results are bitwise those
// of the plain pair kernel.
#pragma once

#include <algorithm>
#include <atomic>

#include "gemm_common.cuh"

namespace moe {

template <int EPI>
struct MixedCfg {
    static constexpr int BN = 256;                              // N of a hot pair MMA
    static constexpr int PAIR_ROWS = 2 * kBM;                   // token rows of a hot pair tile
    static constexpr int KB_BYTES = kBM * kRowBytes;            // 128 rows x one k-block (16 KB)
    static constexpr int HKB = 2;                               // k-blocks per hot stage
    static constexpr int A_BYTES = HKB * KB_BYTES;              // hot: this CTA's 128 token rows
    static constexpr int B_BYTES = HKB * KB_BYTES;              // hot: this CTA's 128 weight rows
    static constexpr int CT = 32;                               // tokens of a cold tile (its N)
    static constexpr int CKB = 4;                               // k-blocks per cold stage
    static constexpr int CW_BYTES = CKB * KB_BYTES;             // cold: 128 weight rows x 4 k-blocks
    static constexpr int CT_KB_BYTES = (CT / 2) * kRowBytes;    // one k-block of this CTA's 16 cold tokens
    static constexpr int CT_BYTES = CKB * CT_KB_BYTES;          // cold: 16 token rows x 4 k-blocks
    static constexpr int SLOT = CW_BYTES + CT_BYTES;            // 72 KB
    static constexpr int STAGES = 3;
    static constexpr bool DUAL_B = (EPI == EPI_SWIGLU_BF16);
    static constexpr int N_OUT_TILE = DUAL_B ? BN / 2 : BN;    // output columns per tile (both kinds)
    static constexpr int TMEM_COLS = 2 * BN;                    // two accumulators
    static constexpr int XR = 8;                                // values per exchange round (2 rounds)
    static constexpr int MAX_G = 256;                           // experts (shared memory bound)
    static constexpr int BAND = kPairBand;                      // hot m-tiles per raster band
    static_assert(EPI == EPI_SWIGLU_BF16 || EPI == EPI_STORE_BF16, "pair kernel epilogues");
    static_assert(A_BYTES + B_BYTES <= SLOT && SLOT % 1024 == 0 && CW_BYTES % 1024 == 0 &&
                      CT_KB_BYTES % 1024 == 0,
                  "stage slots and their operand blocks start on 1024-byte swizzle atoms");
    static_assert(2 * XR == CT / 2, "two exchange rounds cover the half tile");
};

struct MixedTile {
    bool cold;
    int g, row0, rows, n_tile;
};

// Tile p of the mixed list.  H hot tiles (hot list position i owns
// s_hpre[i+1]-s_hpre[i] m-tiles of 256 rows per n-tile) and CC cold tiles
// (cold list position i owns s_cpre[i+1]-s_cpre[i] token tiles of 32 rows per
// n-tile); inside a list, groups in list order.  A cold group's tiles run
// n-tile by n-tile, token tiles innermost.  A hot group's m-tiles run in bands
// of BAND: band by band, inside a band n-tile by n-tile, the band's m-tiles
// innermost.  Concurrent pairs then share a weight tile (the band's m-tiles)
// and re-read only the band's token rows (BAND x 256 rows) from L2 for every
// n-tile: a hot expert's token rows larger than L2 are not re-read from HBM
// once per n-tile, as they would be with every m-tile innermost.
__device__ __forceinline__ bool mixed_is_cold(long long p, long long H, long long CC) {
    if (CC == 0) return false;
    const long long T = H + CC;
    return ((p + 1) * CC) / T > (p * CC) / T;
}

template <int EPI>
__device__ __forceinline__ MixedTile mixed_tile(long long p, long long H, long long CC, int nt, const int* s_goff,
                                                const int* s_hpre, const int* s_hord, int GH, const int* s_cpre,
                                                const int* s_cord, int GC, int band) {
    using C = MixedCfg<EPI>;
    const long long cb = (CC == 0) ? 0 : (p * CC) / (H + CC);
    MixedTile m;
    m.cold = mixed_is_cold(p, H, CC);
    const int* pre = m.cold ? s_cpre : s_hpre;
    const int* ord = m.cold ? s_cord : s_hord;
    const int n = m.cold ? GC : GH;
    const int tile_rows = m.cold ? C::CT : C::PAIR_ROWS;
    const long long t = m.cold ? cb : p - cb;
    int lo = 0, hi = n - 1;
    while (lo < hi) {  // largest i with pre[i] * nt <= t
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<long long>(pre[mid]) * nt <= t) lo = mid; else hi = mid - 1;
    }
    const int mt = pre[lo + 1] - pre[lo];
    const int local = static_cast<int>(t - static_cast<long long>(pre[lo]) * nt);
    int mm;
    if (m.cold) {
        m.n_tile = local / mt;
        mm = local - m.n_tile * mt;
    } else {
        const int full_bands = mt / band;
        const int band_tiles = band * nt;
        if (local < full_bands * band_tiles) {
            const int b = local / band_tiles, r = local - b * band_tiles;
            m.n_tile = r / band;
            mm = b * band + (r - m.n_tile * band);
        } else {  // the last, partial band
            const int ms = mt - full_bands * band, r = local - full_bands * band_tiles;
            m.n_tile = r / ms;
            mm = full_bands * band + (r - m.n_tile * ms);
        }
    }
    m.g = ord[lo];
    m.row0 = s_goff[m.g] + mm * tile_rows;
    m.rows = min(tile_rows, s_goff[m.g + 1] - m.row0);
    return m;
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
grouped_gemm_pair_mixed_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                               const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmT,
                               const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
                               const GemmArgs args) {
    using C = MixedCfg<EPI>;
    constexpr int S = C::STAGES;
    constexpr int BN = C::BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);  // identical offsets in both CTAs
    uint8_t* ring = smem;                 // S slots of C::SLOT bytes
    float* xbuf = reinterpret_cast<float*>(ring + S * C::SLOT);  // [128][XR] values from the peer
    uint64_t* full = reinterpret_cast<uint64_t*>(xbuf + 128 * C::XR);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;   // [2]
    uint64_t* tempty = tfull + 2;  // [2]
    uint64_t* drain = tempty + 2;  // [1]
    uint64_t* xfull = drain + 1;   // [1] the peer's 128 threads wrote their values into xbuf
    uint64_t* xfree = xfull + 1;   // [1] the peer's 128 threads read what this CTA sent
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xfree + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int G = args.G;
    int* s_goff = reinterpret_cast<int*>(tmem_slot + 4);  // [G+1]
    int* s_hpre = s_goff + (G + 1);                       // [G+1] pair m-tiles before hot position i
    int* s_cpre = s_hpre + (G + 1);                       // [G+1] token tiles before cold position i
    int* s_hord = s_cpre + (G + 1);                       // [G] hot groups, heaviest first
    int* s_cord = s_hord + G;                             // [G] cold groups, by index
    int* s_cnt = s_cord + G;                              // [2] hot, cold group counts

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint32_t* err = args.err;
    const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs
    const bool leader = rank == 0;
    const int cold_rows = max(0, args.cold_rows);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);
        }
        mbar_init(drain, 1);
        mbar_init(xfull, 128);
        mbar_init(xfree, 128);
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
    if (threadIdx.x == 0) bad |= (s_goff[0] != 0) | (s_goff[G] > args.M) | (args.splits != 1) | (G > C::MAX_G);
    const bool offsets_bad = __syncthreads_or(bad) != 0;
    if (offsets_bad && blockIdx.x == 0 && threadIdx.x == 0) record_error(err, MOE_DEVERR_BOUNDS);

    // ---- the two lists: hot groups heaviest first, cold groups by index
    if (!offsets_bad) {
        for (int g = threadIdx.x; g < G; g += blockDim.x) {
            const int rg = s_goff[g + 1] - s_goff[g];
            if (rg > cold_rows) {
                int rank_g = 0;
                for (int h = 0; h < G; ++h) {
                    const int rh = s_goff[h + 1] - s_goff[h];
                    rank_g += (rh > cold_rows) & ((rh > rg) | ((rh == rg) & (h < g)));
                }
                s_hord[rank_g] = g;
            }
        }
    }
    if (warp == 0) {
        int nh = 0, nc = 0;
        if (!offsets_bad) {
            for (int base = 0; base < G; base += 32) {
                const int g = base + lane;
                const int rg = (g < G) ? s_goff[g + 1] - s_goff[g] : 0;
                const bool hot = g < G && rg > cold_rows;
                const bool cold = g < G && rg > 0 && rg <= cold_rows;
                const unsigned hm = __ballot_sync(0xffffffffu, hot);
                const unsigned cm = __ballot_sync(0xffffffffu, cold);
                const unsigned lt = (1u << lane) - 1u;
                if (cold) s_cord[nc + __popc(cm & lt)] = g;
                nh += __popc(hm);
                nc += __popc(cm);
            }
        }
        if (lane == 0) {
            s_cnt[0] = nh;
            s_cnt[1] = nc;
        }
    }
    __syncthreads();
    const int GH = s_cnt[0], GC = s_cnt[1];
    if (warp < 2) {  // exclusive prefixes: warp 0 the hot m-tiles, warp 1 the cold token tiles
        const int n = (warp == 0) ? GH : GC;
        const int* ord = (warp == 0) ? s_hord : s_cord;
        int* pre = (warp == 0) ? s_hpre : s_cpre;
        const int tile_rows = (warp == 0) ? C::PAIR_ROWS : C::CT;
        int carry = 0;
        for (int base = 0; base < n; base += 32) {
            const int i = base + lane;
            int v = 0;
            if (i < n) {
                const int g = ord[i];
                v = (s_goff[g + 1] - s_goff[g] + tile_rows - 1) / tile_rows;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (i < n) pre[i + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) pre[0] = 0;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int nt = (args.n_out + C::N_OUT_TILE - 1) / C::N_OUT_TILE;
    const long long H = offsets_bad ? 0 : static_cast<long long>(s_hpre[GH]) * nt;
    const long long CC = offsets_bad ? 0 : static_cast<long long>(s_cpre[GC]) * nt;
    const long long total = H + CC;
    const int band = args.band > 0 ? args.band : C::BAND;
    const int num_kb = args.k_dim / kBK;
    const int num_hs = num_kb / C::HKB;  // hot stages per tile (the host checks num_kb % CKB == 0)
    const int num_cs = num_kb / C::CKB;  // cold stages per tile
    const int cid = blockIdx.x >> 1;
    const int ncl = gridDim.x >> 1;
    const uint32_t full_lead = mapa_shared(smem_u32(full), 0);
    const uint32_t tempty_lead = mapa_shared(smem_u32(tempty), 0);

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            const CUtensorMap* mapB = (C::DUAL_B && rank == 1) ? &tmB2 : &tmB;
            const CUtensorMap* mapW = (C::DUAL_B && rank == 1) ? &tmW2 : &tmW;
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(mapB);
            if (CC > 0) {
                tma_prefetch_desc(&tmT);
                tma_prefetch_desc(mapW);
            }
            bool withhold = args.dbg && (*args.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD) && blockIdx.x == 0;
            uint32_t pending = 0, pend_parity = 0;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (long long p = cid; p < total && ok; p += ncl) {
                const MixedTile ti = mixed_tile<EPI>(p, H, CC, nt, s_goff, s_hpre, s_hord, GH, s_cpre, s_cord, GC, band);
                const int nstages = ti.cold ? num_cs : num_hs;
                // hot: this CTA's 128 token rows and 128 weight rows (W1 | W3 halves or
                // consecutive W2 halves); cold: this CTA's 128 weight rows (W1 | W3 of the
                // same columns, or consecutive halves) and 16 of the 32 tokens
                const int wrow = ti.g * args.b_rows_per_group + ti.n_tile * C::N_OUT_TILE +
                                 (C::DUAL_B ? 0 : static_cast<int>(rank) * kBM);
                const int arow = ti.row0 + static_cast<int>(rank) * (ti.cold ? C::CT / 2 : kBM);
                for (int s = 0; s < nstages; ++s) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err)) { ok = false; break; }
                    if (withhold) {
                        withhold = false;  // test hook: this stage never fills
                    } else {
                        uint8_t* slot = ring + stage * C::SLOT;
                        const uint32_t bar = full_lead + 8u * static_cast<uint32_t>(stage);
                        if (leader) {
                            mbar_arrive_expect_tx(&full[stage], ti.cold ? 2 * C::SLOT : 2 * (C::A_BYTES + C::B_BYTES));
                            pending |= 1u << stage;
                            pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
                        }
                        if (ti.cold) {
                            tma_load_3d_pair(mapW, bar, slot, 0, wrow, s * C::CKB);
                            tma_load_3d_pair(&tmT, bar, slot + C::CW_BYTES, 0, arow, s * C::CKB);
                        } else {
                            tma_load_3d_pair(&tmA, bar, slot, 0, arow, s * C::HKB);
                            tma_load_3d_pair(mapB, bar, slot + C::A_BYTES, 0, wrow, s * C::HKB);
                        }
                    }
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            for (int s = 0; s < S; ++s)
                if (pending & (1u << s)) drain_wait(&full[s], (pend_parity >> s) & 1u, err);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------------------------------------------- MMA issuer (even CTA)
            constexpr uint32_t idesc_hot = idesc_bf16_f32(C::PAIR_ROWS, BN);
            constexpr uint32_t idesc_cold = idesc_bf16_f32(C::PAIR_ROWS, C::CT);
            constexpr int MMAS = OpType<false>::MMAS;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (long long p = cid; p < total && ok; p += ncl) {
                const bool cold = mixed_is_cold(p, H, CC);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const int nstages = cold ? num_cs : num_hs;
                for (int s = 0; s < nstages; ++s) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t slot = smem_u32(ring + stage * C::SLOT);
                    if (cold) {
#pragma unroll
                        for (int j = 0; j < C::CKB; ++j) {
                            const uint64_t wdesc = sw128_kmajor_desc(slot + j * C::KB_BYTES);
                            const uint64_t tdesc = sw128_kmajor_desc(slot + C::CW_BYTES + j * C::CT_KB_BYTES);
#pragma unroll
                            for (int k = 0; k < MMAS; ++k)
                                umma_pair<false>(d_tmem, wdesc + static_cast<uint64_t>(2 * k),
                                                 tdesc + static_cast<uint64_t>(2 * k), idesc_cold,
                                                 (s | j | k) != 0 ? 1u : 0u);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < C::HKB; ++j) {
                            const uint64_t adesc = sw128_kmajor_desc(slot + j * C::KB_BYTES);
                            const uint64_t bdesc = sw128_kmajor_desc(slot + C::A_BYTES + j * C::KB_BYTES);
#pragma unroll
                            for (int k = 0; k < MMAS; ++k)
                                umma_pair<false>(d_tmem, adesc + static_cast<uint64_t>(2 * k),
                                                 bdesc + static_cast<uint64_t>(2 * k), idesc_hot,
                                                 (s | j | k) != 0 ? 1u : 0u);
                        }
                    }
                    umma_commit_pair_multicast(&empty[stage], 0x3);
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair_multicast(&tfull[acc], 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            umma_commit_pair_multicast(drain, 0x3);  // every pair MMA done, in both CTAs
        }
        if (lane == 0) drain_wait(drain, 0, err);  // the pair MMAs wrote this CTA's TMEM too
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int w = q * 32 + lane;  // TMEM lane: token row (hot) or weight row (cold) of this CTA
        const uint32_t peer = rank ^ 1u;
        const uint32_t xrow_peer = mapa_shared(smem_u32(xbuf + w * C::XR), peer);
        const uint32_t xfull_peer = mapa_shared(smem_u32(xfull), peer);
        const uint32_t xfree_peer = mapa_shared(smem_u32(xfree), peer);
        uint16_t* out = reinterpret_cast<uint16_t*>(args.out);
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t xphase = 0;
        for (long long p = cid; p < total; p += ncl) {
            const MixedTile ti = mixed_tile<EPI>(p, H, CC, nt, s_goff, s_hpre, s_hord, GH, s_cpre, s_cord, GC, band);
            const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            if (!ti.cold) {
                const int r = static_cast<int>(rank) * kBM + w;  // row within the pair tile
                const long long grow = static_cast<long long>(ti.row0) + r;
                epilogue_ffn<EPI, BN, false>(t_row, r < ti.rows, grow, ti.g, ti.n_tile, args);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_lead + 8u * acc);
            } else {
                // accumulator row w = weight row; columns = the tile's 32 tokens
                uint32_t v[32];
                tmem_ld_32x32(t_row, v);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_lead + 8u * acc);  // TMEM read: reusable
                const int nv = ti.rows;
                if constexpr (C::DUAL_B) {
                    // even CTA: gate of column w for all 32 tokens, forms tokens 0..15;
                    // odd CTA: up, forms tokens 16..31.  Send the other half to the peer.
                    const long long col = static_cast<long long>(ti.n_tile) * C::N_OUT_TILE + w;
                    float send[C::CT / 2];  // the even CTA sends tokens 16..31, the odd CTA 0..15
#pragma unroll
                    for (int j = 0; j < C::CT / 2; ++j)
                        send[j] = __uint_as_float(rank == 0 ? v[C::CT / 2 + j] : v[j]);
                    float recv[C::CT / 2];
                    bool okx = true;
#pragma unroll
                    for (int round = 0; round < 2; ++round) {  // XR values per round
                        okx = okx && mbar_wait_cluster(xfree, xphase ^ 1u, abort_flag, err);
                        if (okx) {
                            st_cluster_v4(xrow_peer, send[round * C::XR], send[round * C::XR + 1],
                                          send[round * C::XR + 2], send[round * C::XR + 3]);
                            st_cluster_v4(xrow_peer + 16u, send[round * C::XR + 4], send[round * C::XR + 5],
                                          send[round * C::XR + 6], send[round * C::XR + 7]);
                            mbar_arrive_cluster(xfull_peer);
                            okx = mbar_wait_cluster(xfull, xphase, abort_flag, err);
                        }
                        if (okx) {
                            const float4* src = reinterpret_cast<const float4*>(xbuf + w * C::XR);
                            const float4 f0 = src[0], f1 = src[1];
                            recv[round * C::XR] = f0.x;
                            recv[round * C::XR + 1] = f0.y;
                            recv[round * C::XR + 2] = f0.z;
                            recv[round * C::XR + 3] = f0.w;
                            recv[round * C::XR + 4] = f1.x;
                            recv[round * C::XR + 5] = f1.y;
                            recv[round * C::XR + 6] = f1.z;
                            recv[round * C::XR + 7] = f1.w;
                            mbar_arrive_cluster(xfree_peer);  // this CTA's xbuf row may be written again
                        }
                        xphase ^= 1u;
                    }
                    if (!__all_sync(0xffffffffu, okx)) break;
                    const int tok0 = (rank == 0) ? 0 : C::CT / 2;
#pragma unroll
                    for (int j = 0; j < C::CT / 2; ++j) {
                        if (tok0 + j < nv) {
                            const float gate = (rank == 0) ? __uint_as_float(v[j]) : recv[j];
                            const float up = (rank == 0) ? recv[j] : __uint_as_float(v[C::CT / 2 + j]);
                            const __nv_bfloat16 b = __float2bfloat16_rn(silu_f32(gate) * up);
                            out[(static_cast<long long>(ti.row0) + tok0 + j) * args.ldo + col] =
                                *reinterpret_cast<const uint16_t*>(&b);
                        }
                    }
                } else {
                    const long long col = static_cast<long long>(ti.n_tile) * C::N_OUT_TILE +
                                          static_cast<int>(rank) * kBM + w;
#pragma unroll
                    for (int j = 0; j < C::CT; ++j) {
                        if (j < nv) {
                            const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[j]));
                            out[(static_cast<long long>(ti.row0) + j) * args.ldo + col] =
                                *reinterpret_cast<const uint16_t*>(&b);
                        }
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
    cluster_sync_all();  // neither CTA leaves while its peer may still signal it or write its xbuf
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------------------------
template <int EPI>
inline size_t pair_mixed_smem_bytes(int G) {
    using C = MixedCfg<EPI>;
    return 1024 + static_cast<size_t>(C::STAGES) * C::SLOT + 128 * C::XR * sizeof(float) +
           (2 * C::STAGES + 7) * sizeof(uint64_t) + 16 + (3 * static_cast<size_t>(G + 1) + 2 * G + 2) * sizeof(int);
}

template <int EPI>
inline cudaError_t pair_mixed_launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                                     const CUtensorMap& tmT, const CUtensorMap& tmW, const CUtensorMap& tmW2,
                                     const GemmArgs& a, long long tiles_ub, cudaStream_t st) {
    if (a.G > MixedCfg<EPI>::MAX_G) return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> done{0};
    static int clusters[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
        const size_t smem = pair_mixed_smem_bytes<EPI>(MixedCfg<EPI>::MAX_G);
        e = cudaFuncSetAttribute(grouped_gemm_pair_mixed_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(192, 1, 1);
        cfg.dynamicSmemBytes = smem;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_mixed_kernel<EPI>, &cfg);
        if (e != cudaSuccess) return e;
        clusters[dev & 63] = n;
        done.fetch_or(bit, std::memory_order_acq_rel);
    }
    const int max_clusters = clusters[dev & 63];
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const long long ncl = std::max<long long>(1, std::min<long long>(tiles_ub, max_clusters));
    return launch_kernel(grouped_gemm_pair_mixed_kernel<EPI>, dim3(static_cast<unsigned>(2 * ncl)), dim3(192),
                         pair_mixed_smem_bytes<EPI>(a.G), st, tmA, tmB, tmB2, tmT, tmW, tmW2, a);
}

}  // namespace moe
