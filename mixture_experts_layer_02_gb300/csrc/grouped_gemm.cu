// grouped_gemm.cu -- persistent grouped GEMM on sm_103a tensor cores
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
//   EPI_ROUTER       acc = router logits of 128 tokens x E experts (E <= BN);
//                    per token: + bias, top-K by (value desc, index asc),
//                    softmax over the K or sigmoid + renormalise ("MoE 推理完整
//                    机制", 第一层 Router 与 Top-K).
#include <math.h>

#include "device.cuh"

namespace moe {

template <int EPI, int BN>
struct GemmCfg {
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BN * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (BN >= 256) ? 4 : (BN >= 128 ? 6 : 8);
    static constexpr int N_OUT_TILE = (EPI == EPI_SWIGLU_BF16) ? BN / 2 : BN;
    static constexpr int TMEM_COLS = 2 * BN;  // two accumulators
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "TMEM allocation must be a power of two in [32, 512]");
};

struct TileInfo {
    int g, row0, rows, n_tile;
};

// Tile t of the global list: groups in order, inside a group n-tiles in
// order, inside an n-tile m-tiles in order (consecutive CTAs share the same
// weight tile, which then comes from L2).
__device__ __forceinline__ TileInfo decode_tile(int t, int G, int nt, const int* s_tpre,
                                                const int* s_goff) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {  // largest g with s_tpre[g] * nt <= t
        const int mid = (lo + hi + 1) >> 1;
        if (s_tpre[mid] * nt <= t) lo = mid; else hi = mid - 1;
    }
    TileInfo ti;
    ti.g = lo;
    const int mt = s_tpre[lo + 1] - s_tpre[lo];
    const int local = t - s_tpre[lo] * nt;
    ti.n_tile = local / mt;
    const int m = local - ti.n_tile * mt;
    ti.row0 = s_goff[lo] + m * kBM;
    ti.rows = min(kBM, s_goff[lo + 1] - ti.row0);
    return ti;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t s = smem_u32(p);
    return p + ((1024u - (s & 1023u)) & 1023u);
}

// Bounded wait that ignores the abort flag (used only to drain in-flight copies
// and MMAs before the CTA exits).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            record_error(err, MOE_DEVERR_TIMEOUT);
            return;
        }
    }
}

// ----------------------------------------------------------------------------
// epilogues: one thread = one accumulator row (TMEM lane), `t_row` addresses
// that warp's lane quarter and the accumulator's first column.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float (&v)[32]) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        d[i] = make_uint4(pack_bf16x2(v[8 * i + 0], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                          pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
    }
}

template <int EPI, int BN>
__device__ __forceinline__ void epilogue_ffn(uint32_t t_row, bool valid, long long grow, int n_tile,
                                             const GemmArgs& a) {
    using C = GemmCfg<EPI, BN>;
    uint16_t* out = reinterpret_cast<uint16_t*>(a.out);
    if constexpr (EPI == EPI_SWIGLU_BF16) {
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
            uint32_t g[32], u[32];
            tmem_ld_32x32(t_row + c * 32, g);
            tmem_ld_32x32(t_row + BN / 2 + c * 32, u);
            tmem_ld_wait();
            const int col = n_tile * C::N_OUT_TILE + c * 32;
            if (valid && col < a.n_out) {
                float h[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    h[j] = silu_f32(__uint_as_float(g[j])) * __uint_as_float(u[j]);
                store_bf16x32(out + grow * a.ldo + col, h);
            }
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32(t_row + c * 32, r);
            tmem_ld_wait();
            const int col = n_tile * C::N_OUT_TILE + c * 32;
            if (valid && col < a.n_out) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float x = __uint_as_float(r[j]);
                    v[j] = (EPI == EPI_SILU_BF16) ? silu_f32(x) : x;
                }
                store_bf16x32(out + grow * a.ldo + col, v);
            }
        }
    }
}

// Router epilogue.  Selection takes K passes over the E logits; pass k keeps
// the first expert, in (value desc, index asc) order, that comes after the one
// pass k-1 chose.  Scanning e upward and replacing only on a strictly larger
// value gives the lower index on ties.
template <int BN>
__device__ __forceinline__ void epilogue_router(uint32_t t_row, bool valid, long long tok,
                                                const GemmArgs& a) {
    const int E = a.E, K = a.K;
    const int nchunks = (E + 31) / 32;
    if (a.logits_out != nullptr) {
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            uint32_t r[32];
            tmem_ld_32x32(t_row + c * 32, r);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int e = c * 32 + j;
                    if (e < E) {
                        const float v = __uint_as_float(r[j]) + (a.bias ? a.bias[e] : 0.0f);
                        a.logits_out[tok * E + e] = v;
                    }
                }
            }
        }
    }
    float sel[32];
    float prev_v = INFINITY;
    int prev_i = -1;
    bool bad = false;
#pragma unroll 1
    for (int k = 0; k < K; ++k) {
        float best_v = -INFINITY;
        int best_i = -1;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            uint32_t r[32];
            tmem_ld_32x32(t_row + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int e = c * 32 + j;
                if (e < E) {
                    const float v = __uint_as_float(r[j]) + (a.bias ? a.bias[e] : 0.0f);
                    const bool after_prev = (v < prev_v) || (v == prev_v && e > prev_i);
                    if (after_prev && (best_i < 0 || v > best_v)) {
                        best_v = v;
                        best_i = e;
                    }
                }
            }
        }
        if (best_i < 0) bad = true;  // only possible with NaN logits
        sel[k] = best_v;
        if (valid) a.topk_ids[tok * K + k] = best_i;
        prev_v = best_v;
        prev_i = best_i;
    }
    if (!valid) return;
    if (bad) record_error(a.err, MOE_DEVERR_BOUNDS);
    float sum = 0.0f;
    if (a.mode == 0) {  // softmax over the K selected logits
        const float top = sel[0];
        for (int k = 0; k < K; ++k) {
            sel[k] = expf(sel[k] - top);
            sum += sel[k];
        }
    } else {            // sigmoid, then renormalise over the K selected
        for (int k = 0; k < K; ++k) {
            sel[k] = 1.0f / (1.0f + expf(-sel[k]));
            sum += sel[k];
        }
    }
    for (int k = 0; k < K; ++k)
        a.topk_w[tok * K + k] = (sum > 0.0f) ? sel[k] / sum : 1.0f / (float)K;
}

// ----------------------------------------------------------------------------
template <int EPI, int BN>
__global__ void __launch_bounds__(192, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, const GemmArgs args) {
    using C = GemmCfg<EPI, BN>;
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
    const int total_tiles = offsets_bad ? 0 : s_tpre[G] * nt;
    const int num_kb = args.k_dim / kBK;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            if (EPI == EPI_SWIGLU_BF16) tma_prefetch_desc(&tmB2);
            bool withhold = args.dbg && (*args.dbg & MOE_DBG_WITHHOLD_FIRST_LOAD) && blockIdx.x == 0;
            uint32_t pending = 0, pend_parity = 0;  // per-stage: a load issued, its phase parity
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(t, G, nt, s_tpre, s_goff);
                const int brow = ti.g * args.b_rows_per_group + ti.n_tile * C::N_OUT_TILE;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err)) { ok = false; break; }
                    if (withhold) {
                        withhold = false;  // test hook: this stage never fills
                    } else {
                        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        uint8_t* a_dst = sA + stage * C::A_BYTES;
                        uint8_t* b_dst = sB + stage * C::B_BYTES;
                        tma_load_2d(&tmA, &full[stage], a_dst, kb * kBK, ti.row0);
                        if constexpr (EPI == EPI_SWIGLU_BF16) {
                            tma_load_2d(&tmB, &full[stage], b_dst, kb * kBK, brow);
                            tma_load_2d(&tmB2, &full[stage], b_dst + (BN / 2) * kBK * 2, kb * kBK, brow);
                        } else {
                            tma_load_2d(&tmB, &full[stage], b_dst, kb * kBK, brow);
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
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::A_BYTES));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        // advance 16 bf16 = 32 bytes along K inside the swizzle atom
                        umma_bf16(d_tmem, adesc + static_cast<uint64_t>(2 * k),
                                  bdesc + static_cast<uint64_t>(2 * k), idesc, (kb | k) != 0 ? 1u : 0u);
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
            const TileInfo ti = decode_tile(t, G, nt, s_tpre, s_goff);
            const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int r = q * 32 + lane;
            const bool valid = r < ti.rows;
            const long long grow = static_cast<long long>(ti.row0) + r;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            if constexpr (EPI == EPI_ROUTER) {
                epilogue_router<BN>(t_row, valid, grow, args);
            } else {
                epilogue_ffn<EPI, BN>(t_row, valid, grow, ti.n_tile, args);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

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
static size_t smem_bytes_for(int G) {
    using C = GemmCfg<EPI, BN>;
    return 1024 /* alignment slack */ + static_cast<size_t>(C::STAGES) * C::STAGE_BYTES +
           (2 * C::STAGES + 5) * sizeof(uint64_t) + 16 + 2 * static_cast<size_t>(G + 1) * sizeof(int);
}

template <int EPI, int BN>
static cudaError_t launch_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB2,
                            const GemmArgs& a, int grid, cudaStream_t st) {
    const size_t smem = smem_bytes_for<EPI, BN>(a.G);
    auto kern = grouped_gemm_kernel<EPI, BN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, 192, smem, st>>>(tmA, tmB, tmB2, a);
    return cudaGetLastError();
}

#define MOE_GEMM_CASE(E_, B_) \
    if (epi == E_ && bn == B_) return launch_t<E_, B_>(tmA, tmB, tmB2, a, grid, st);

cudaError_t launch_grouped_gemm(int epi, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                const CUtensorMap& tmB2, const GemmArgs& a, int grid,
                                cudaStream_t st) {
    MOE_GEMM_CASE(EPI_SWIGLU_BF16, 256)
    MOE_GEMM_CASE(EPI_SWIGLU_BF16, 128)
    MOE_GEMM_CASE(EPI_SWIGLU_BF16, 64)
    MOE_GEMM_CASE(EPI_SILU_BF16, 256)
    MOE_GEMM_CASE(EPI_SILU_BF16, 128)
    MOE_GEMM_CASE(EPI_SILU_BF16, 64)
    MOE_GEMM_CASE(EPI_STORE_BF16, 256)
    MOE_GEMM_CASE(EPI_STORE_BF16, 128)
    MOE_GEMM_CASE(EPI_STORE_BF16, 64)
    MOE_GEMM_CASE(EPI_ROUTER, 256)
    MOE_GEMM_CASE(EPI_ROUTER, 128)
    MOE_GEMM_CASE(EPI_ROUTER, 64)
    MOE_GEMM_CASE(EPI_ROUTER, 32)
    return cudaErrorInvalidValue;
}

#define MOE_SMEM_CASE(E_, B_) \
    if (epi == E_ && bn == B_) return smem_bytes_for<E_, B_>(G);

size_t gemm_smem_bytes(int epi, int bn, int G) {
    MOE_SMEM_CASE(EPI_SWIGLU_BF16, 256)
    MOE_SMEM_CASE(EPI_SWIGLU_BF16, 128)
    MOE_SMEM_CASE(EPI_SWIGLU_BF16, 64)
    MOE_SMEM_CASE(EPI_SILU_BF16, 256)
    MOE_SMEM_CASE(EPI_SILU_BF16, 128)
    MOE_SMEM_CASE(EPI_SILU_BF16, 64)
    MOE_SMEM_CASE(EPI_STORE_BF16, 256)
    MOE_SMEM_CASE(EPI_STORE_BF16, 128)
    MOE_SMEM_CASE(EPI_STORE_BF16, 64)
    MOE_SMEM_CASE(EPI_ROUTER, 256)
    MOE_SMEM_CASE(EPI_ROUTER, 128)
    MOE_SMEM_CASE(EPI_ROUTER, 64)
    MOE_SMEM_CASE(EPI_ROUTER, 32)
    return 0;
}

int gemm_stages(int epi, int bn) {
    (void)epi;
    return bn >= 256 ? 4 : (bn >= 128 ? 6 : 8);
}

}  // namespace moe
