// ffn_fused_decode.cu -- the grouped SwiGLU FFN of a decode-sized call in ONE
// persistent launch: GEMM1 + SwiGLU and GEMM2 of every expert, with the SMs
// moving from expert to expert inside the kernel.  This is the MegaMoE idea
// of "MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im),
// 第四层 "DeepGEMM & MegaMoE Kernel": one large persistent kernel that assigns
// SMs to experts dynamically and removes the launches between the expert
// GEMMs.  At decode sizes those launches (GEMM1, its split-K reduction, GEMM2,
// its reduction) cost more than the weight stream itself.
//
// Work list (static stride over CTAs, one CTA per SM, all co-resident through
// a cooperative launch):
//   items [0, n1):   GEMM1 work: (expert, token tile, 64-column tile, k-split)
//   items [n1, n2):  GEMM2 work: (expert, token tile, 128-column tile, k-split)
// Each item runs the swapped-operand MMA of grouped_gemm_swap.cuh (weights as
// the 128-row operand, BT tokens as N) and stores its fp32 partial.  The CTA
// that completes the last split of a tile (a per-tile atomic count) sums the
// partials in split order -- deterministic whichever CTA is last -- and writes
// the bf16 result: h = silu(gate) * up for GEMM1, y for GEMM2.  When every
// GEMM1 tile of an expert is written, a per-expert count reaches its total and
// the GEMM2 items of that expert may load h.  A CTA reaches its GEMM2 items
// only after all of its GEMM1 items, and GEMM1 items wait on nothing, so every
// wait ends; each is also bounded (1 s) like every pipeline wait.
#include <algorithm>
#include <atomic>

#include "gemm_common.cuh"

namespace moe {

constexpr int kFusedStages = 10;

template <int BT>
struct FusedCfg {
    static constexpr int A_BYTES = 128 * kRowBytes;     // 128 weight rows
    static constexpr int B_BYTES = BT * kRowBytes;      // BT token rows
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = (2 * BT < 32) ? 32 : 2 * BT;
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

struct FusedItem {
    int phase, tile, split, kb0, kb1;
    TileInfo ti;
};

template <int BT>
__global__ void __launch_bounds__(192, 1)
ffn_fused_decode_kernel(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW3,
                        const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW2,
                        const __grid_constant__ CUtensorMap tmH, const FusedFfnArgs args) {
    using C = FusedCfg<BT>;
    constexpr int S = kFusedStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + S * C::B_BYTES);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* s_last = reinterpret_cast<volatile int*>(tmem_slot + 2);
    int* s_goff = reinterpret_cast<int*>(tmem_slot + 4);
    int* s_tpre = s_goff + (args.G + 1);
    float* s_u = reinterpret_cast<float*>(s_tpre + (args.G + 1));  // [64][BT+1] the up half of a SwiGLU tile

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = args.G;
    uint32_t* err = args.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
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
    pdl_wait();
    for (int i = threadIdx.x; i <= G; i += blockDim.x) s_goff[i] = args.group_offsets[i];
    __syncthreads();
    const int nkb1 = args.D / kBK, nkb2 = args.Dff / kBK;
    const int S1 = args.splits1, S2 = args.splits2;
    int bad = 0;
    for (int i = threadIdx.x; i < G; i += blockDim.x) bad |= (s_goff[i] > s_goff[i + 1]);
    if (threadIdx.x == 0)
        bad |= (s_goff[0] != 0) | (s_goff[G] > args.M) | (S1 < 1) | (S1 > nkb1) | (S2 < 1) | (S2 > nkb2);
    const bool args_bad = __syncthreads_or(bad) != 0;
    if (warp == 0) {  // exclusive prefix of BT-row token tiles per expert
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

    const int nt1 = args.Dff / 64, nt2 = args.D / 128;
    const int tiles1 = s_tpre[G] * nt1, tiles2 = s_tpre[G] * nt2;
    const bool caps_bad = tiles1 > args.tiles1_cap || tiles2 > args.tiles2_cap;
    if ((args_bad || caps_bad) && blockIdx.x == 0 && threadIdx.x == 0) record_error(err, MOE_DEVERR_BOUNDS);
    const int items1 = (args_bad || caps_bad) ? 0 : tiles1 * S1;
    const int total = (args_bad || caps_bad) ? 0 : items1 + tiles2 * S2;

    auto decode = [&](int t) {
        FusedItem it;
        if (t < items1) {
            it.phase = 0;
            it.tile = t / S1;
            it.split = t - it.tile * S1;
            it.ti = decode_tile(it.tile, G, nt1, s_tpre, s_goff, BT);
            it.kb0 = it.split * nkb1 / S1;
            it.kb1 = (it.split + 1) * nkb1 / S1;
        } else {
            const int u = t - items1;
            it.phase = 1;
            it.tile = u / S2;
            it.split = u - it.tile * S2;
            it.ti = decode_tile(it.tile, G, nt2, s_tpre, s_goff, BT);
            it.kb0 = it.split * nkb2 / S2;
            it.kb1 = (it.split + 1) * nkb2 / S2;
        }
        return it;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmW1);
            tma_prefetch_desc(&tmW3);
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmW2);
            tma_prefetch_desc(&tmH);
            bool withhold = args.dbg && (*args.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD) && blockIdx.x == 0;
            uint32_t pending = 0, pend_parity = 0;
            int stage = 0;
            uint32_t phase = 0;
            int ready_g = -1;  // the expert whose h is known complete
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const FusedItem it = decode(t);
                const int g = it.ti.g;
                if (it.phase == 1 && g != ready_g) {
                    // every GEMM1 tile of expert g written: its h rows may be read
                    const int need = ((s_goff[g + 1] - s_goff[g] + BT - 1) / BT) * nt1;
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(args.expert_done + g) < need) {
                        if (*abort_flag) { ok = false; break; }
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            *abort_flag = 1;
                            record_error(err, MOE_DEVERR_TIMEOUT);
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                    fence_proxy_async_global();  // h was written by generic stores; TMA reads it
                    ready_g = g;
                }
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err)) { ok = false; break; }
                    if (withhold) {
                        withhold = false;  // test hook: this stage never fills
                    } else {
                        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        uint8_t* a_dst = sA + stage * C::A_BYTES;
                        uint8_t* b_dst = sB + stage * C::B_BYTES;
                        if (it.phase == 0) {
                            const int wrow = g * args.Dff + it.ti.n_tile * 64;
                            tma_load_2d(&tmW1, &full[stage], a_dst, kb * kBK, wrow);
                            tma_load_2d(&tmW3, &full[stage], a_dst + 64 * kRowBytes, kb * kBK, wrow);
                            tma_load_2d(&tmX, &full[stage], b_dst, kb * kBK, it.ti.row0);
                        } else {
                            const int wrow = g * args.D + it.ti.n_tile * 128;
                            tma_load_2d(&tmW2, &full[stage], a_dst, kb * kBK, wrow);
                            tma_load_2d(&tmH, &full[stage], b_dst, kb * kBK, it.ti.row0);
                        }
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
            constexpr uint32_t idesc = idesc_bf16_f32(128, BT);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const FusedItem it = decode(t);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BT);
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::A_BYTES));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        umma_bf16(d_tmem, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k),
                                  idesc, (kb > it.kb0 || k > 0) ? 1u : 0u);
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
        const int et = threadIdx.x - 64;  // 0..127 among the epilogue threads
        const long long ld1 = 2LL * args.Dff, ld2 = args.D;  // partial row strides
        const long long ss1 = static_cast<long long>(args.M) * ld1, ss2 = static_cast<long long>(args.M) * ld2;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const FusedItem it = decode(t);
            bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, err);
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
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;

            const int nv = it.ti.rows;
            const long long row0 = it.ti.row0;
            const int S_ = (it.phase == 0) ? S1 : S2;
            const long long ld = (it.phase == 0) ? ld1 : ld2;
            const long long ss = (it.phase == 0) ? ss1 : ss2;
            float* part = (it.phase == 0) ? args.part1 : args.part2;
            const long long col = static_cast<long long>(it.ti.n_tile) * 128 + r;  // partial column
            bool last = true;
            if (S_ > 1) {
                // this split's fp32 partial (GEMM1: gate rows, then up rows of the tile)
#pragma unroll
                for (int j = 0; j < BT; ++j)
                    if (j < nv) part[it.split * ss + (row0 + j) * ld + col] = v[j];
                __threadfence();
                named_barrier_sync(1, 128);
                if (et == 0) {
                    int* cnt = (it.phase == 0) ? args.tile_cnt1 + it.tile : args.tile_cnt2 + it.tile;
                    const int prev = atomicAdd(cnt, 1);
                    __threadfence();
                    *s_last = (prev == S_ - 1) ? 1 : 0;
                }
                named_barrier_sync(1, 128);
                last = *s_last != 0;
                if (last) {
                    // sum every split in split order (this one from registers), the
                    // other splits' loads of one split all in flight together
                    float acc[BT];
#pragma unroll
                    for (int j = 0; j < BT; ++j) acc[j] = 0.0f;
                    for (int sp = 0; sp < S_; ++sp) {
                        float t[BT];
                        if (sp == it.split) {
#pragma unroll
                            for (int j = 0; j < BT; ++j) t[j] = v[j];
                        } else {
                            const float* p = part + sp * ss + row0 * ld + col;
#pragma unroll
                            for (int j = 0; j < BT; ++j) t[j] = (j < nv) ? __ldcg(p + j * ld) : 0.0f;
                        }
#pragma unroll
                        for (int j = 0; j < BT; ++j) acc[j] += t[j];
                    }
#pragma unroll
                    for (int j = 0; j < BT; ++j) v[j] = acc[j];
                }
            }
            if (last) {
                if (it.phase == 0) {
                    // h = silu(gate) * up: the up half reaches the gate half through shared memory
                    if (r >= 64) {
#pragma unroll
                        for (int j = 0; j < BT; ++j) s_u[(r - 64) * (BT + 1) + j] = v[j];
                    }
                    named_barrier_sync(1, 128);
                    if (r < 64) {
                        uint16_t* hrow = args.h + row0 * args.Dff + it.ti.n_tile * 64 + r;
#pragma unroll
                        for (int j = 0; j < BT; ++j) {
                            if (j < nv) {
                                const __nv_bfloat16 b = __float2bfloat16_rn(silu_f32(v[j]) * s_u[r * (BT + 1) + j]);
                                hrow[j * args.Dff] = *reinterpret_cast<const uint16_t*>(&b);
                            }
                        }
                        __threadfence();
                    }
                    named_barrier_sync(1, 128);
                    if (et == 0) atomicAdd(args.expert_done + it.ti.g, 1);  // one more GEMM1 tile of h
                } else {
                    uint16_t* yrow = args.y + row0 * args.D + col;
#pragma unroll
                    for (int j = 0; j < BT; ++j) {
                        if (j < nv) {
                            const __nv_bfloat16 b = __float2bfloat16_rn(v[j]);
                            yrow[j * args.D] = *reinterpret_cast<const uint16_t*>(&b);
                        }
                    }
                }
            }
            named_barrier_sync(1, 128);  // s_last and s_u are rewritten by the next item
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
template <int BT>
static size_t fused_smem_bytes(int G) {
    using C = FusedCfg<BT>;
    return 1024 + static_cast<size_t>(kFusedStages) * C::STAGE_BYTES + (2 * kFusedStages + 5) * sizeof(uint64_t) +
           16 + 2 * static_cast<size_t>(G + 1) * sizeof(int) + 64 * (BT + 1) * sizeof(float);
}

template <int BT>
static cudaError_t fused_launch(const CUtensorMap* maps, const FusedFfnArgs& a, int grid, cudaStream_t st) {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(ffn_fused_decode_kernel<BT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(fused_smem_bytes<BT>(1024)));
        if (e != cudaSuccess) return e;
        done.fetch_or(bit, std::memory_order_acq_rel);
    }
    // CTAs wait on each other's results: launch them all at once (cooperative)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = fused_smem_bytes<BT>(a.G);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ffn_fused_decode_kernel<BT>, maps[0], maps[1], maps[2], maps[3], maps[4], a);
}

cudaError_t launch_ffn_fused_decode(int bt, const CUtensorMap* maps, const FusedFfnArgs& a, int grid,
                                    cudaStream_t st) {
    if (bt == 16) return fused_launch<16>(maps, a, grid, st);
    if (bt == 32) return fused_launch<32>(maps, a, grid, st);
    return cudaErrorInvalidValue;
}

int ffn_fused_decode_max_grid(int bt) {
    int dev = 0, nsm = 0, per = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const size_t smem = bt == 16 ? fused_smem_bytes<16>(1024) : fused_smem_bytes<32>(1024);
    cudaError_t e = bt == 16 ? cudaFuncSetAttribute(ffn_fused_decode_kernel<16>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))
                             : cudaFuncSetAttribute(ffn_fused_decode_kernel<32>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return 0;
    e = bt == 16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, ffn_fused_decode_kernel<16>, 192, smem)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, ffn_fused_decode_kernel<32>, 192, smem);
    if (e != cudaSuccess) return 0;
    return nsm * per;
}

}  // namespace moe
