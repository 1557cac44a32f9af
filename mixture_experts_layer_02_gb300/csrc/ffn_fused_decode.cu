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
//   (e4m3 only: quantisation items, below)
//   then:            GEMM2 work: (expert, token tile, 128-column tile, k-split)
// Each item runs the swapped-operand MMA of grouped_gemm_swap.cuh (weights as
// the 128-row operand, BT tokens as N) and stores its fp32 partial.  The CTA
// that completes the last split of a tile (a per-tile atomic count) sums the
// partials in split order -- deterministic whichever CTA is last -- and writes
// the bf16 result: h = silu(gate) * up for GEMM1, y for GEMM2.  When every
// GEMM1 tile of an expert is written, a per-expert count reaches its total and
// the GEMM2 items of that expert may load h.  A GEMM2 item's weight tile does
// not depend on h: while the count is short, the producer streams the weight
// halves of the item's stages into free pipeline slots, and their activation
// halves follow once the count is reached.  A CTA reaches its GEMM2 items only
// after all of its GEMM1 items, and GEMM1 items wait on nothing, so every wait
// ends; each is also bounded (1 s) like every pipeline wait.
//
// e4m3 operands (template FP8): the same, with the scales of
// grouped_gemm.cuh applied to each accumulator, plus a quantisation phase
// between the GEMMs -- items [n1, n1 + nq): one per (expert, token tile).
// GEMM1's last split also folds the magnitude of each bf16 h value into a
// per-row maximum (atomicMax on the bf16 magnitude bits); a quantisation item
// waits for its expert's GEMM1 tiles, then writes the rows' e4m3 codes and
// scales exactly as the row quantiser (quant.cu) does from the same bf16 h,
// and counts the token tile done for its expert; GEMM2 items wait for those
// counts instead.  Phases still only wait on earlier phases.
//
// Publishing a finished tile (making its stores visible GPU-wide before the
// count moves) takes a memory fence whose latency, under the full weight
// stream, was as long as the rest of a GEMM1 epilogue; a seventh warp does
// it.  The epilogue hands each finished tile's count to that warp through a
// small mbarrier ring and goes on with the next tile; the warp fences and
// increments the count in order.
#include <algorithm>
#include <atomic>

#include "gemm_common.cuh"
#include "quant.cuh"

namespace moe {

constexpr int kFusedStages = 10;
constexpr int kFusedThreads = 224;  // producer, MMA, 4 epilogue warps, signaller
constexpr int kSigSlots = 4;        // epilogue -> signaller ring
constexpr int kG2Slots = 4;         // e4m3: producer -> epilogue "GEMM2 input published" ring

template <int BT>
struct FusedCfg {
    static constexpr int A_BYTES = 128 * kRowBytes;     // 128 weight rows
    static constexpr int B_BYTES = BT * kRowBytes;      // BT token rows
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = (2 * BT < 32) ? 32 : 2 * BT;
};

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

struct FusedItem {
    int phase, tile, split, kb0, kb1;
    TileInfo ti;
};

template <int BT, bool FP8>
__global__ void __launch_bounds__(kFusedThreads, 1)
ffn_fused_decode_kernel(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW3,
                        const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW2,
                        const __grid_constant__ CUtensorMap tmH, const FusedFfnArgs args) {
    using C = FusedCfg<BT>;
    using T = OpType<FP8>;
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
    uint64_t* sig_full = drain + 1;
    uint64_t* sig_empty = sig_full + kSigSlots;
    uint64_t* g2ok = sig_empty + kSigSlots;
    uint64_t* g2free = g2ok + kG2Slots;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(g2free + kG2Slots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* s_last = reinterpret_cast<volatile int*>(tmem_slot + 2);
    int* s_sig = reinterpret_cast<int*>(tmem_slot + 4);  // [kSigSlots] counts to publish
    int* s_goff = s_sig + kSigSlots;
    int* s_tpre = s_goff + (args.G + 1);
    float* s_u = reinterpret_cast<float*>(s_tpre + (args.G + 1));  // [64][BT+1] the up half of a SwiGLU tile
    float* s_xs = s_u + 64 * (BT + 1);  // e4m3: [xs_rows] token scale of each permuted row

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
        for (int i = 0; i < kSigSlots; ++i) {
            mbar_init(&sig_full[i], 1);
            mbar_init(&sig_empty[i], 1);
        }
        for (int i = 0; i < kG2Slots; ++i) {
            mbar_init(&g2ok[i], 1);
            mbar_init(&g2free[i], 1);
        }
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
    const int nkb1 = args.D / T::KB, nkb2 = args.Dff / T::KB;
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
    const int itemsq = (args_bad || caps_bad || !FP8) ? 0 : s_tpre[G];  // e4m3: one per token tile
    const int total = (args_bad || caps_bad) ? 0 : items1 + itemsq + tiles2 * S2;
    // GEMM1 tiles of expert g (its h complete) / its token tiles (its hq complete)
    auto need1 = [&](int g) { return ((s_goff[g + 1] - s_goff[g] + BT - 1) / BT) * nt1; };
    auto needq = [&](int g) { return (s_goff[g + 1] - s_goff[g] + BT - 1) / BT; };
    // bounded wait for *p >= need, polled with relaxed loads and a short
    // back-off, then one acquire fence; false on timeout / abort
    auto wait_count = [&](const int* p, int need) {
        if (ld_relaxed_gpu(p) < need) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_relaxed_gpu(p) < need) {
                if (*abort_flag) return false;
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    *abort_flag = 1;
                    record_error(err, MOE_DEVERR_TIMEOUT);
                    return false;
                }
                __nanosleep(64);
            }
        }
        fence_acq_rel_gpu();
        return true;
    };

    auto decode = [&](int t) {
        FusedItem it;
        if (t >= items1 && t < items1 + itemsq) {
            it.phase = 2;  // quantisation of one token tile's h rows
            it.tile = t - items1;
            it.split = 0;
            it.ti = decode_tile(it.tile, G, 1, s_tpre, s_goff, BT);
            it.kb0 = it.kb1 = 0;
        } else if (t < items1) {
            it.phase = 0;
            it.tile = t / S1;
            it.split = t - it.tile * S1;
            it.ti = decode_tile(it.tile, G, nt1, s_tpre, s_goff, BT);
            it.kb0 = it.split * nkb1 / S1;
            it.kb1 = (it.split + 1) * nkb1 / S1;
        } else {
            const int u = t - items1 - itemsq;
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
            int ready_g = -1;  // the expert whose GEMM2 input is known complete
            int gslot = 0;
            uint32_t gphase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const FusedItem it = decode(t);
                if (it.phase == 2) continue;  // quantisation items load nothing
                const int g = it.ti.g;
                int kb_start = it.kb0;  // first k-block still to load in full
                if (it.phase == 1 && g != ready_g) {
                    // GEMM2's input of expert g: h (bf16) or its codes hq (e4m3).  The
                    // W2 tile does not depend on it: while the count is short, stream
                    // the weight half of this item's stages into free slots; their
                    // activation half follows once the count is reached.
                    const int* cnt = FP8 ? args.quant_done + g : args.expert_done + g;
                    const int need = FP8 ? needq(g) : need1(g);
                    const int wrow = g * args.D + it.ti.n_tile * 128;
                    const int st0 = stage;
                    int npre = 0;
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_relaxed_gpu(cnt) < need) {
                        if (kb_start + npre < it.kb1 && npre < S && !withhold &&
                            mbar_test_wait(&empty[stage], phase ^ 1u)) {
                            mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                            tma_load_2d(&tmW2, &full[stage], sA + stage * C::A_BYTES, (kb_start + npre) * T::KB, wrow);
                            pending |= 1u << stage;
                            pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
                            ++npre;
                            if (++stage == S) { stage = 0; phase ^= 1u; }
                            continue;
                        }
                        if (*abort_flag) { ok = false; break; }
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            *abort_flag = 1;
                            record_error(err, MOE_DEVERR_TIMEOUT);
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    if (ok) {
                        fence_acq_rel_gpu();
                        fence_proxy_async_global();  // written by generic stores; TMA reads it
                        ready_g = g;
                    }
                    // the activation half of the prefetched stages (also on the way out,
                    // so that every transaction completes before the CTA drains)
                    for (int i = 0; i < npre; ++i) {
                        const int sti = (st0 + i) % S;
                        tma_load_2d(&tmH, &full[sti], sB + sti * C::B_BYTES, (kb_start + i) * T::KB, it.ti.row0);
                    }
                    kb_start += npre;
                    if (!ok) break;
                }
                if (FP8 && it.phase == 1) {
                    // the epilogue reads this expert's h_scale: pass on what this thread acquired
                    if (!mbar_wait(&g2free[gslot], gphase ^ 1u, abort_flag, err)) break;
                    mbar_arrive(&g2ok[gslot]);
                    if (++gslot == kG2Slots) { gslot = 0; gphase ^= 1u; }
                }
                for (int kb = kb_start; kb < it.kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err)) { ok = false; break; }
                    if (withhold) {
                        withhold = false;  // test hook: this stage never fills
                    } else {
                        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        uint8_t* a_dst = sA + stage * C::A_BYTES;
                        uint8_t* b_dst = sB + stage * C::B_BYTES;
                        if (it.phase == 0) {
                            const int wrow = g * args.Dff + it.ti.n_tile * 64;
                            tma_load_2d(&tmW1, &full[stage], a_dst, kb * T::KB, wrow);
                            tma_load_2d(&tmW3, &full[stage], a_dst + 64 * kRowBytes, kb * T::KB, wrow);
                            tma_load_2d(&tmX, &full[stage], b_dst, kb * T::KB, it.ti.row0);
                        } else {
                            const int wrow = g * args.D + it.ti.n_tile * 128;
                            tma_load_2d(&tmW2, &full[stage], a_dst, kb * T::KB, wrow);
                            tma_load_2d(&tmH, &full[stage], b_dst, kb * T::KB, it.ti.row0);
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
            constexpr uint32_t idesc = idesc_f32acc<FP8>(128, BT);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const FusedItem it = decode(t);
                if (it.phase == 2) continue;  // no MMA for quantisation items
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BT);
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::A_BYTES));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                    for (int k = 0; k < T::MMAS; ++k)
                        umma<FP8>(d_tmem, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k),
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
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;        // TMEM lanes 32q .. 32q+31
        const int r = q * 32 + lane;   // weight row within the tile
        const int et = threadIdx.x - 64;  // 0..127 among the epilogue threads
        const long long ld1 = 2LL * args.Dff, ld2 = args.D;  // partial row strides
        const long long ss1 = static_cast<long long>(args.M) * ld1, ss2 = static_cast<long long>(args.M) * ld2;
        int acc = 0;
        uint32_t acc_phase = 0;
        int sslot = 0;
        uint32_t sphase = 0;
        float cs = 1.0f, rs[BT];  // e4m3 scales of the item in hand
        int gslot = 0;
        uint32_t gphase = 0;
        if (FP8 && args.xs_rows > 0) {
            // every permuted row's token scale, gathered once while the first tiles stream in
            for (int i = et; i < args.xs_rows; i += 128)
                s_xs[i] = args.x_scale[args.x_scale_idx ? static_cast<long long>(args.x_scale_idx[i]) : i];
            named_barrier_sync(1, 128);
        }
        auto load_g1_scales = [&](const FusedItem& it) {
            const long long wi = static_cast<long long>(it.ti.g) * args.Dff + it.ti.n_tile * 64 + (r & 63);
            cs = (r < 64) ? args.s1[wi] : args.s3[wi];
#pragma unroll
            for (int j = 0; j < BT; ++j) {
                rs[j] = 0.0f;
                if (j < it.ti.rows) {
                    const long long tr = static_cast<long long>(it.ti.row0) + j;
                    rs[j] = args.xs_rows > 0 ? s_xs[tr]
                                             : args.x_scale[args.x_scale_idx ? static_cast<long long>(args.x_scale_idx[tr]) : tr];
                }
            }
        };
        // (et == 0) hand a count to the signaller: code g = one more GEMM1 tile
        // of expert g, G + g = one more quantised token tile, -1 = no more.
        // The caller's barrier has ordered every epilogue thread's stores first.
        auto publish = [&](int code) {
            if (!mbar_wait(&sig_empty[sslot], sphase ^ 1u, abort_flag, err)) return;
            s_sig[sslot] = code;
            mbar_arrive(&sig_full[sslot]);
            if (++sslot == kSigSlots) { sslot = 0; sphase ^= 1u; }
        };
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const FusedItem it = decode(t);
            const int nv = it.ti.rows;
            const long long row0 = it.ti.row0;
            if constexpr (FP8) {
                if (it.phase == 2) {
                    // ---- quantisation of h rows row0 .. row0+nv-1 (every GEMM1 tile of the expert written)
                    bool ok = true;
                    if (et == 0) ok = wait_count(args.expert_done + it.ti.g, need1(it.ti.g));
                    ok = named_barrier_and(1, 128, ok);
                    if (!ok) break;
                    if (et < nv) {
                        const int k = scale_exp_of(__ldcg(args.h_amax + row0 + et));
                        s_u[et] = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);  // 2^-k
                        args.h_scale[row0 + et] = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
                    }
                    named_barrier_sync(1, 128);
                    const int chunks = args.Dff / 8;  // 8 values per 16-byte chunk
                    const int n = nv * chunks;
                    for (int base = 0; base < n; base += 8 * 128) {
                        uint4 hv[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int i = base + u * 128 + et;
                            if (i < n) {
                                const int j = i / chunks;
                                hv[u] = __ldcg(reinterpret_cast<const uint4*>(args.h + (row0 + j) * args.Dff) +
                                               (i - j * chunks));
                            }
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int i = base + u * 128 + et;
                            if (i < n) {
                                const int j = i / chunks;
                                reinterpret_cast<uint2*>(args.hq + (row0 + j) * args.Dff)[i - j * chunks] =
                                    to_e4m3x8(hv[u], s_u[j]);
                            }
                        }
                    }
                    named_barrier_sync(1, 128);
                    if (et == 0) publish(G + it.ti.g);  // one more token tile of hq
                    named_barrier_sync(1, 128);  // s_u is rewritten by the next item
                    continue;
                }
            }
            // e4m3: the weight row's scale and each token's, fetched while the MMA
            // runs (GEMM2: once the expert's h codes are published)
            if constexpr (FP8) {
                const int g = it.ti.g;
                if (it.phase == 0) {
                    load_g1_scales(it);
                } else {
                    // h_scale of the expert's rows is written: the producer acquired its
                    // published count before loading this item and hands that on here
                    bool ok = true;
                    if (et == 0) ok = mbar_wait(&g2ok[gslot], gphase, abort_flag, err);
                    ok = named_barrier_and(1, 128, ok);
                    if (!ok) break;
                    if (et == 0) mbar_arrive(&g2free[gslot]);
                    if (++gslot == kG2Slots) { gslot = 0; gphase ^= 1u; }
                    cs = args.s2[static_cast<long long>(g) * args.D + it.ti.n_tile * 128 + r];
#pragma unroll
                    for (int j = 0; j < BT; ++j) rs[j] = (j < nv) ? __ldcg(args.h_scale + row0 + j) : 0.0f;
                }
            }
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
            if constexpr (FP8) {
#pragma unroll
                for (int j = 0; j < BT; ++j)
                    if (j < nv) v[j] = v[j] * rs[j] * cs;
            }

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
                    // other splits' loads of one split all in flight together; the
                    // sum starts from split 0's value, not from +0
                    float acc[BT];
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
                        for (int j = 0; j < BT; ++j) acc[j] = (sp == 0) ? t[j] : acc[j] + t[j];
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
                        uint32_t my_max = 0;  // e4m3: lane j gets token j's magnitude maximum
#pragma unroll
                        for (int j = 0; j < BT; ++j) {
                            if (j < nv) {
                                const __nv_bfloat16 b = __float2bfloat16_rn(silu_f32(v[j]) * s_u[r * (BT + 1) + j]);
                                const uint16_t hb = *reinterpret_cast<const uint16_t*>(&b);
                                hrow[j * args.Dff] = hb;
                                if constexpr (FP8) {
                                    // over this warp's 32 columns of the tile
                                    const uint32_t m = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(hb & 0x7fffu));
                                    if (lane == j) my_max = m;
                                }
                            }
                        }
                        if constexpr (FP8) {
                            if (lane < nv) atomicMax(args.h_amax + row0 + lane, my_max);
                        }
                    }
                    named_barrier_sync(1, 128);
                    if (et == 0) publish(it.ti.g);  // one more GEMM1 tile of h
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
        if (et == 0) publish(-1);
    } else {
        // ------------------------------------------------------------ signaller
        // publishes the epilogue's finished tiles in order: fence (the stores
        // the epilogue ordered before its hand-over become visible GPU-wide),
        // then the count a waiting CTA polls
        if (lane == 0) {
            int slot = 0;
            uint32_t phase = 0;
            while (mbar_wait(&sig_full[slot], phase, abort_flag, err)) {
                const int code = s_sig[slot];
                if (code < 0) break;
                __threadfence();
                atomicAdd(code < G ? args.expert_done + code : args.quant_done + (code - G), 1);
                mbar_arrive(&sig_empty[slot]);
                if (++slot == kSigSlots) { slot = 0; phase ^= 1u; }
            }
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
static size_t fused_smem_bytes(int G, int xs_rows) {
    using C = FusedCfg<BT>;
    return 1024 + static_cast<size_t>(kFusedStages) * C::STAGE_BYTES +
           (2 * kFusedStages + 5 + 2 * kSigSlots + 2 * kG2Slots) * sizeof(uint64_t) + 16 + kSigSlots * sizeof(int) +
           2 * static_cast<size_t>(G + 1) * sizeof(int) + (64 * (BT + 1) + static_cast<size_t>(xs_rows)) * sizeof(float);
}

static int smem_optin_bytes() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    return v;
}

template <int BT, bool FP8>
static cudaError_t set_smem_limit() {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(ffn_fused_decode_kernel<BT, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_optin_bytes());
        if (e != cudaSuccess) return e;
        done.fetch_or(bit, std::memory_order_acq_rel);
    }
    return cudaSuccess;
}

template <int BT, bool FP8>
static cudaError_t fused_launch(const CUtensorMap* maps, const FusedFfnArgs& a, int grid, cudaStream_t st) {
    cudaError_t e = set_smem_limit<BT, FP8>();
    if (e != cudaSuccess) return e;
    // CTAs wait on each other's results: launch them all at once (cooperative)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = fused_smem_bytes<BT>(a.G, a.xs_rows);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ffn_fused_decode_kernel<BT, FP8>, maps[0], maps[1], maps[2], maps[3], maps[4], a);
}

cudaError_t launch_ffn_fused_decode(bool e4m3, int bt, const CUtensorMap* maps, const FusedFfnArgs& a, int grid,
                                    cudaStream_t st) {
    if (bt == 16) return e4m3 ? fused_launch<16, true>(maps, a, grid, st) : fused_launch<16, false>(maps, a, grid, st);
    if (bt == 32) return e4m3 ? fused_launch<32, true>(maps, a, grid, st) : fused_launch<32, false>(maps, a, grid, st);
    return cudaErrorInvalidValue;
}

int ffn_fused_decode_xs_rows(int bt, int G, int rows) {
    const size_t need = bt == 16 ? fused_smem_bytes<16>(G, rows) : fused_smem_bytes<32>(G, rows);
    return need <= static_cast<size_t>(smem_optin_bytes()) ? rows : 0;
}

template <int BT, bool FP8>
static int fused_max_grid(int nsm, size_t smem) {
    int per = 0;
    if (set_smem_limit<BT, FP8>() != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, ffn_fused_decode_kernel<BT, FP8>, kFusedThreads, smem) !=
        cudaSuccess)
        return 0;
    return nsm * per;
}

int ffn_fused_decode_max_grid(bool e4m3, int bt, int G, int xs_rows) {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (bt == 16) {
        const size_t smem = fused_smem_bytes<16>(G, xs_rows);
        return e4m3 ? fused_max_grid<16, true>(nsm, smem) : fused_max_grid<16, false>(nsm, smem);
    }
    if (bt == 32) {
        const size_t smem = fused_smem_bytes<32>(G, xs_rows);
        return e4m3 ? fused_max_grid<32, true>(nsm, smem) : fused_max_grid<32, false>(nsm, smem);
    }
    return 0;
}

}  // namespace moe
