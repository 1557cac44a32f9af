// gemm_common.cuh -- pieces shared by the one-CTA and the CTA-pair grouped
// GEMM kernels: tile configuration, tile-list decoding, bounded drain waits
// and the TMEM -> registers -> global epilogues.
#pragma once

#include "device.cuh"

namespace moe {

template <int EPI, int BN>
struct GemmCfg {
    static constexpr int A_BYTES = kBM * kRowBytes;
    static constexpr int B_BYTES = BN * kRowBytes;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (BN >= 256) ? 4 : (BN >= 128 ? 6 : 8);
    static constexpr bool DUAL_B = (EPI == EPI_SWIGLU_BF16 || EPI == EPI_F32_DUAL);
    static constexpr int N_OUT_TILE = DUAL_B ? BN / 2 : BN;
    static constexpr int TMEM_COLS = 2 * BN;  // two accumulators
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "TMEM allocation must be a power of two in [32, 512]");
};

struct TileInfo {
    int g, row0, rows, n_tile;
};

// Tile t of the global list: groups in order, inside a group n-tiles in
// order, inside an n-tile m-tiles of `tile_rows` rows in order (consecutive
// CTAs share the same weight tile, which then comes from L2).  s_tpre[g] is
// the number of m-tiles before group g.
__device__ __forceinline__ TileInfo decode_tile(int t, int G, int nt, const int* s_tpre,
                                                const int* s_goff, int tile_rows = kBM) {
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
    ti.row0 = s_goff[lo] + m * tile_rows;
    ti.rows = min(tile_rows, s_goff[lo + 1] - ti.row0);
    return ti;
}

// ---- heaviest expert first, in bands (the CTA-pair kernels) ----
// "MoE 推理完整机制" 第二层 "关键 kernel：Grouped GEMM": the SMs of one launch
// are handed out over the experts, and a hot expert must not stall the rest.
// The pair tile list takes the experts heaviest first (rows descending, ties
// by index; index order above kSortMaxGroups experts), so the largest
// experts' many tiles start in the first waves and the small experts fill the
// tail.
constexpr int kSortMaxGroups = 256;
// An expert's m-tiles run in bands of kPairBand: band by band, inside a band
// n-tile by n-tile, the band's m-tiles innermost.  Concurrent pairs then share
// a weight tile, and each n-tile re-reads only the band's token rows (8 x 256
// rows) from L2.  With every m-tile innermost, an expert whose token rows
// exceed L2 re-reads them from HBM once per n-tile; experts of up to 8 m-tiles
// keep exactly that order.  (GemmArgs::band overrides the width, for tuning.)
constexpr int kPairBand = 8;

// s_ord[0 .. G) = the groups heaviest first (every thread of the CTA calls
// this; the caller synchronises before reading s_ord).
__device__ __forceinline__ void heaviest_first(const int* s_goff, int G, int* s_ord) {
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        int r = g;
        if (G <= kSortMaxGroups) {
            const int rg = s_goff[g + 1] - s_goff[g];
            r = 0;
            for (int h = 0; h < G; ++h) {
                const int rh = s_goff[h + 1] - s_goff[h];
                r += (rh > rg) | ((rh == rg) & (h < g));
            }
        }
        s_ord[r] = g;
    }
}

// Tile t of the banded list: groups in s_ord order (s_tpre[i] = m-tiles of
// tile_rows rows before position i), then bands, n-tiles, band m-tiles.
__device__ __forceinline__ TileInfo decode_tile_banded(int t, int G, int nt, const int* s_tpre, const int* s_ord,
                                                       const int* s_goff, int tile_rows, int band = kPairBand) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {  // largest i with s_tpre[i] * nt <= t
        const int mid = (lo + hi + 1) >> 1;
        if (s_tpre[mid] * nt <= t) lo = mid; else hi = mid - 1;
    }
    TileInfo ti;
    ti.g = s_ord[lo];
    const int mt = s_tpre[lo + 1] - s_tpre[lo];
    const int local = t - s_tpre[lo] * nt;
    const int full_bands = mt / band, band_tiles = band * nt;
    int m;
    if (local < full_bands * band_tiles) {
        const int b = local / band_tiles, r = local - b * band_tiles;
        ti.n_tile = r / band;
        m = b * band + (r - ti.n_tile * band);
    } else {  // the last, partial band
        const int ms = mt - full_bands * band, r = local - full_bands * band_tiles;
        ti.n_tile = r / ms;
        m = full_bands * band + (r - ti.n_tile * ms);
    }
    ti.row0 = s_goff[ti.g] + m * tile_rows;
    ti.rows = min(tile_rows, s_goff[ti.g + 1] - ti.row0);
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
// gathered A operand (the permutation fused into GEMM1): the producer warp
// copies each tile row from its source row with 16-byte cp.async into the
// 128-byte-swizzled layout, 8 lanes per row so a warp instruction moves 4
// whole 128-byte rows.  Rows past the segment are not written: they only feed
// accumulator rows the epilogue masks.
// ----------------------------------------------------------------------------
// s_src[i] = source row of tile row i (a_src_rows[row0 + i]) for i < rows,
// -1 otherwise; sources outside 0..a_src_n-1 are flagged and skipped.
__device__ __forceinline__ void gather_rows_fill(int* s_src, int tile_rows, const GemmArgs& a, int row0, int rows,
                                                 int lane, uint32_t* err) {
    for (int i = lane; i < tile_rows; i += 32) {
        int src = -1;
        if (i < rows) {
            src = a.a_src_rows[row0 + i];
            if (src < 0 || src >= a.a_src_n) {
                record_error(err, MOE_DEVERR_BOUNDS);
                src = -1;
            }
        }
        s_src[i] = src;
    }
    __syncwarp();
}

// This lane's copies of k-block kb of an NROWS-row tile at shared address dst.
template <int NROWS>
__device__ __forceinline__ void gather_rows_issue(uint32_t dst, const int* s_src, const GemmArgs& a, int kb,
                                                  int lane) {
    const int c = lane & 7;
    const uint8_t* src = static_cast<const uint8_t*>(a.a_src) + static_cast<long long>(kb) * kRowBytes + c * 16;
#pragma unroll 4
    for (int j = 0; j < NROWS / 4; ++j) {
        const int row = j * 4 + (lane >> 3);
        const int sr = s_src[row];
        if (sr >= 0) cp_async_16(dst + sw128_offset(row, c), src + static_cast<long long>(sr) * a.a_src_ld);
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

// e4m3 scales of one output row (a no-op factor 1 for bf16 operands).
template <bool FP8>
__device__ __forceinline__ float row_scale_of(const GemmArgs& a, bool valid, long long grow) {
    if constexpr (FP8) {
        if (!valid) return 0.0f;
        const long long r = a.row_scale_idx ? static_cast<long long>(a.row_scale_idx[grow]) : grow;
        return a.row_scale[r];
    } else {
        return 1.0f;
    }
}

// 32 consecutive per-column scales (128-byte aligned: col % 32 == 0 and the
// scale arrays are 16-byte aligned with b_rows_per_group % 64 == 0).
__device__ __forceinline__ void load_scales32(const float* p, float (&s)[32]) {
    const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 v = __ldg(q + i);
        s[4 * i] = v.x;
        s[4 * i + 1] = v.y;
        s[4 * i + 2] = v.z;
        s[4 * i + 3] = v.w;
    }
}

template <int EPI, int BN, bool FP8>
__device__ __forceinline__ void epilogue_ffn(uint32_t t_row, bool valid, long long grow, int g, int n_tile,
                                             const GemmArgs& a) {
    using C = GemmCfg<EPI, BN>;
    uint16_t* out = reinterpret_cast<uint16_t*>(a.out);
    const float rs = row_scale_of<FP8>(a, valid, grow);
    const long long wrow0 = static_cast<long long>(g) * a.b_rows_per_group;
    if constexpr (EPI == EPI_SWIGLU_BF16) {
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
            uint32_t gt[32], u[32];
            tmem_ld_32x32(t_row + c * 32, gt);
            tmem_ld_32x32(t_row + BN / 2 + c * 32, u);
            tmem_ld_wait();
            const int col = n_tile * C::N_OUT_TILE + c * 32;
            if (valid && col < a.n_out) {
                float h[32];
                if constexpr (FP8) {
                    float s1[32], s3[32];
                    load_scales32(a.col_scale + wrow0 + col, s1);
                    load_scales32(a.col_scale_up + wrow0 + col, s3);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        h[j] = silu_f32(__uint_as_float(gt[j]) * rs * s1[j]) * (__uint_as_float(u[j]) * rs * s3[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        h[j] = silu_f32(__uint_as_float(gt[j])) * __uint_as_float(u[j]);
                }
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
                if constexpr (FP8) {
                    float sc[32];
                    load_scales32(a.col_scale + wrow0 + col, sc);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * rs * sc[j];
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                }
                if constexpr (EPI == EPI_SILU_BF16) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = silu_f32(v[j]);
                }
                store_bf16x32(out + grow * a.ldo + col, v);
            }
        }
    }
}

// fp32 partial epilogue: the accumulator of one k-split, BN columns per tile
// at column n_tile*BN of slab `split` (for EPI_F32_DUAL the first BN/2 hold
// the gate, the rest the up projection, of output columns n_tile*BN/2 ..).
// With e4m3 operands the row and column scales are applied here (they are
// constant along K), so the reductions only sum.
template <int EPI, int BN, bool FP8>
__device__ __forceinline__ void epilogue_f32(uint32_t t_row, bool valid, long long grow, int g, int n_tile,
                                             int split, const GemmArgs& a) {
    float* out = reinterpret_cast<float*>(a.out) + split * a.split_stride;
    const float rs = row_scale_of<FP8>(a, valid, grow);
    const long long wrow0 = static_cast<long long>(g) * a.b_rows_per_group;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32(t_row + c * 32, r);
        tmem_ld_wait();
        const long long col = static_cast<long long>(n_tile) * BN + c * 32;
        if (valid && col + 32 <= a.ldo) {
            if constexpr (FP8) {
                const bool up = (EPI == EPI_F32_DUAL) && c >= BN / 64;
                const int ocol = (EPI == EPI_F32_DUAL) ? n_tile * (BN / 2) + (up ? c - BN / 64 : c) * 32
                                                       : n_tile * BN + c * 32;
                float sc[32];
                load_scales32((up ? a.col_scale_up : a.col_scale) + wrow0 + ocol, sc);
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * rs * sc[j]);
            }
            uint4* d = reinterpret_cast<uint4*>(out + grow * a.ldo + col);
#pragma unroll
            for (int i = 0; i < 8; ++i) d[i] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
        }
    }
}

}  // namespace moe
