// moe_api.cu -- the C ABI declared in include/moe.h: argument validation,
// workspace carving, TMA descriptor encoding and kernel launches.  No device
// memory is allocated here; every buffer belongs to the caller.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/moe.h"
#include "common.h"

using namespace moe;

namespace {

thread_local std::string g_detail;

}  // namespace

void moe::set_error_detail(const char* msg) { g_detail = msg; }

namespace {

moe_status fail(moe_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_detail = buf;
    return s;
}

moe_status cuda_fail(cudaError_t e, const char* where) {
    return fail(MOE_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---- per-device SM count (the only state the library keeps) ----
int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// ---- TMA descriptor encoding through the driver entry point ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major [rows, cols] matrix of bf16 (or e4m3 bytes), box = [box_rows,
// 128 bytes of columns], 128-byte swizzle (the layout the tcgen05
// shared-memory descriptors expect).
moe_status make_tmap(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows,
                     bool e4m3 = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    const int esize = e4m3 ? 1 : 2;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * esize};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kRowBytes / esize), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) rows=%lld cols=%lld box=%d", (int)r, rows,
                    cols, box_rows);
    return MOE_OK;
}

// The same matrix viewed as {128 bytes of columns, rows, column blocks}
// (strides: the row, then 128 bytes), box = [kbs column blocks][box_rows
// rows][128 bytes]: one copy brings kbs consecutive 128-byte column blocks
// of box_rows rows, each block landing as its own swizzled [box_rows x 128 B]
// tile.
moe_status make_tmap3d(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows, int kbs,
                       bool e4m3 = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    const int esize = e4m3 ? 1 : 2;
    const long long inner = kRowBytes / esize;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(cols / inner)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * esize, static_cast<cuuint64_t>(kRowBytes)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(inner), static_cast<cuuint32_t>(box_rows),
                         static_cast<cuuint32_t>(kbs)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d) rows=%lld cols=%lld box=%dx%d", (int)r,
                    rows, cols, box_rows, kbs);
    return MOE_OK;
}

// ---- shared validation ----
moe_status check_sizes(int N, int D, int E, int K, int Dff, bool need_dff) {
    if (N < 0) return fail(MOE_ERR_INVALID_ARG, "N=%d < 0", N);
    if (E < 1 || E > 1024) return fail(MOE_ERR_INVALID_ARG, "E=%d outside 1..1024", E);
    if (K < 1 || K > E || K > 32) return fail(MOE_ERR_INVALID_ARG, "K=%d outside 1..min(E,32)", K);
    if (D < 64 || D % 64) return fail(MOE_ERR_INVALID_ARG, "D=%d not a positive multiple of 64", D);
    if (need_dff && (Dff < 64 || Dff % 64)) return fail(MOE_ERR_INVALID_ARG, "Dff=%d not a positive multiple of 64", Dff);
    const long long rows = static_cast<long long>(N) * K;
    if (rows >= (1LL << 31)) return fail(MOE_ERR_INVALID_ARG, "N*K=%lld too large", rows);
    if (rows * std::max(D, Dff) >= (1LL << 40)) return fail(MOE_ERR_INVALID_ARG, "rows*width too large");
    // weight rows are addressed with 32-bit tensor-map coordinates
    if (static_cast<long long>(E) * std::max(D, need_dff ? Dff : D) >= (1LL << 31))
        return fail(MOE_ERR_INVALID_ARG, "E*max(D,Dff) too large");
    return MOE_OK;
}

}  // namespace

// The size checks of moe_permute, shared with the allocation-free variant in
// permute.cu so that both reject exactly the same arguments.
int moe::check_permute_sizes(int N, int D, int E, int K) { return check_sizes(N, D, E, K, 64, false); }

namespace {

#define REQUIRE_PTR(p)                                                                   \
    do {                                                                                 \
        if ((p) == nullptr) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", #p);          \
        if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s not 16-byte aligned", #p); \
    } while (0)

#define OPTIONAL_PTR(p)                                                                  \
    do {                                                                                 \
        if ((p) != nullptr && !aligned16(p))                                             \
            return fail(MOE_ERR_INVALID_ARG, "%s not 16-byte aligned", #p);              \
    } while (0)

uint32_t* ws_err(void* ws) { return reinterpret_cast<uint32_t*>(ws); }
const uint32_t* ws_dbg(void* ws) { return reinterpret_cast<uint32_t*>(ws) + 1; }

// ---- split-K planning ----
// The work list of a GEMM has `tiles` (group, n-tile, m-tile) items.  When that
// leaves SMs idle, every item is cut into S k-splits (fp32 partials, summed by
// a follow-up kernel in split order).  Workspaces are sized for at most
// kMaxPlanSms SMs so that their size does not depend on the device.
constexpr int kMaxPlanSms = 256;

// k-splits for `tiles` work items on `nsm` SMs: the S that minimises the
// makespan ceil(tiles*S/nsm)/S (in units of one unsplit tile), plus 0.03 per
// split for the partials and their reduction, plus `split_cost` once for any
// split.  That fixed term is zero for the compute-bound tiles and about a
// third of a tile for the weight-streaming swapped-operand tiles of decode,
// where the partials, the reduction and its ordering add a fixed latency to a
// short tile (measured on GB300: one split beats three for 96 such tiles on
// 152 SMs).
int plan_splits(long long tiles, int max_splits, int nsm, double split_cost = 0.0) {
    nsm = std::min(nsm, kMaxPlanSms);
    if (tiles <= 0 || tiles >= nsm || max_splits <= 1) return 1;
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= max_splits; ++s) {
        const double waves = static_cast<double>((tiles * s + nsm - 1) / nsm);
        const double cost = waves / s + (s > 1 ? split_cost : 0.0) + 0.03 * (s - 1);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// The largest split count plan_splits can return on any device with at most
// kMaxPlanSms SMs: what the workspace sizes for.
int bound_splits(long long tiles, int max_splits) {
    return (tiles > 0 && tiles < kMaxPlanSms) ? std::max(1, max_splits) : 1;
}

// Router: N tile = E rounded up to 32 while E <= 256, else 256 (several n-tiles).
int route_bn(int E) {
    if (E <= 32) return 32;
    if (E <= 64) return 64;
    if (E <= 128) return 128;
    return 256;
}

struct RoutePlan {
    int bn, nt, ldp, splits;
    size_t partial_bytes;
};

RoutePlan plan_route(int N, int D, int E, int nsm, size_t avail = static_cast<size_t>(-1)) {
    RoutePlan p;
    p.bn = route_bn(E);
    p.nt = (E + p.bn - 1) / p.bn;
    p.ldp = p.nt * p.bn;
    const long long tiles = static_cast<long long>((N + kBM - 1) / kBM) * p.nt;
    const int max_s = std::min(16, D / kBK);
    p.splits = plan_splits(tiles, max_s, nsm);
    p.partial_bytes = static_cast<size_t>(bound_splits(tiles, max_s)) * N * p.ldp * sizeof(float);
    // the unsplit partials always fit the sized workspace; a split that would not fit is dropped
    if (static_cast<size_t>(p.splits) * N * p.ldp * sizeof(float) > avail) p.splits = 1;
    return p;
}

// Grouped FFN: N tile = the widest of 256/128/64 whose output columns divide
// the GEMM's width (MOE_FFN_TILE_N=64|128|256 pins it, for tuning and test
// coverage).  The m-tile count is only known on the device; rows/128 +
// min(E, rows) bounds it from above.
int ffn_bn(int n_out, bool swiglu) {
    if (const char* f = getenv("MOE_FFN_TILE_N")) {
        const int bn = atoi(f);
        if ((bn == 64 || bn == 128 || bn == 256) && n_out % (swiglu ? bn / 2 : bn) == 0) return bn;
    }
    const int cands[3] = {256, 128, 64};
    for (int bn : cands)
        if (n_out % (swiglu ? bn / 2 : bn) == 0) return bn;
    return 64;
}

// One GEMM of the grouped FFN: how it runs and where its output goes.
enum GemmMode { MODE_ONE = 0, MODE_PAIR = 1, MODE_SWAP = 2 };

struct GemmPlan {
    int mode;        // MODE_ONE / MODE_PAIR / MODE_SWAP
    int bn;          // N tile (one/pair) or token tile BT (swap)
    int splits;      // k-splits (fp32 partials + reduction when > 1)
    int ldp;         // row stride of the fp32 partials
    long long tiles_ub;
    int cold_rows;   // MODE_PAIR: experts with 1 .. cold_rows rows run weight-streaming tiles (0: none)
};

struct FfnPlan {
    GemmPlan g1, g2;
};

// CTA pairs pay off when experts own many rows: by default when the mean
// rows per touched expert is at least 256; the swapped-operand kernel when it
// is at most 32 (decode).  MOE_PAIR_GEMM=0|1 and MOE_SWAP_GEMM=0|1 force a
// choice wherever the shape allows (tuning and test coverage).
bool env_flag(const char* name, bool dflt) {
    if (const char* f = getenv(name)) return atoi(f) != 0;
    return dflt;
}

// Widest N tile whose output columns divide n_out (no tuning override): the
// fewest tiles any splittable mode can have.
int widest_bn(int n_out, bool swiglu) {
    const int cands[3] = {256, 128, 64};
    for (int bn : cands)
        if (n_out % (swiglu ? bn / 2 : bn) == 0) return bn;
    return 64;
}

// Scratch of the fused decode FFN (one launch for GEMM1 + SwiGLU and GEMM2):
// both GEMMs' fp32 partials plus the per-tile and per-expert counters (and,
// for e4m3 operands, the per-expert quantisation counts and per-row h maxima).
struct FusedDecodeLayout {
    size_t part1, part2, counters, counter_bytes, total;
};

FusedDecodeLayout fused_decode_layout(int rows, int D, int E, int Dff, int s1, int s2, long long tiles1,
                                      long long tiles2) {
    FusedDecodeLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.part1 = take(static_cast<size_t>(s1) * rows * 2 * Dff * sizeof(float));
    L.part2 = take(static_cast<size_t>(s2) * rows * D * sizeof(float));
    L.counter_bytes = static_cast<size_t>(tiles1 + tiles2 + 2LL * E + rows) * sizeof(int);
    L.counters = take(L.counter_bytes);
    L.total = o;
    return L;
}

// The fused decode FFN bound for any call of these sizes (every split count
// the planner may choose), or 0 when decode-sized calls are impossible.
size_t fused_decode_bound(int rows, int D, int E, int Dff) {
    const long long touched_ub = std::min(E, rows);
    if (static_cast<long long>(rows) > 32 * touched_ub) return 0;
    const long long t1 = (rows / 16 + touched_ub) * (Dff / 64), t2 = (rows / 16 + touched_ub) * (D / 128);
    const int s1 = bound_splits(t1, std::min(4, D / kBK / 4)), s2 = bound_splits(t2, std::min(4, Dff / kBK / 4));
    return fused_decode_layout(rows, D, E, Dff, s1, s2, t1, t2).total;
}

// Bytes of fp32 split-K partials any grouped-FFN call of these sizes may
// need, over both activations, every execution mode and every device with at
// most kMaxPlanSms SMs.  Pair tiles never split; swapped tiles are never fewer
// than the widest one-CTA tiles, so the widest one-CTA tiling bounds them.
size_t ffn_partial_bound(int rows, int D, int E, int Dff) {
    const long long touched_ub = std::min(E, rows);
    size_t b = 0;
    for (int sw = 0; sw < 2; ++sw) {
        const bool swiglu = sw == 1;
        const int bn = widest_bn(Dff, swiglu);
        const int per = swiglu ? bn / 2 : bn;
        const long long tiles = (rows / kBM + touched_ub) * ((Dff + per - 1) / per);
        const int sb = bound_splits(tiles, std::min(4, D / kBK / 4));
        const size_t ldp = swiglu ? 2 * static_cast<size_t>(Dff) : Dff;
        if (sb > 1) b = std::max(b, static_cast<size_t>(sb) * rows * ldp * sizeof(float));
    }
    const int bn = widest_bn(D, false);
    const long long tiles = (rows / kBM + touched_ub) * ((D + bn - 1) / bn);
    const int sb = bound_splits(tiles, std::min(4, Dff / kBK / 4));
    if (sb > 1) b = std::max(b, static_cast<size_t>(sb) * rows * D * sizeof(float));
    return std::max(b, fused_decode_bound(rows, D, E, Dff));
}

// MOE_PAIR_COLD_ROWS=n (n > 0) runs pair-mode GEMMs on the mixed pair kernel:
// experts with at most n rows become weight-streaming tiles (weights as the
// MMA's M, 32 tokens as its N), the rest 256-row pair tiles.  Opt-in: on the
// Zipf-skewed DeepSeek-V3 layer (16384 tokens, 256 experts) it measured no
// faster than the plain pair kernel (interleaved medians 8.88 / 9.13 /
// 9.03 ms at n = 16 / 32 / 64 against 8.83 ms), while its hot tiles alone
// match the plain kernel (a single 16384-row expert: 0.786 against
// 0.794 ms).  Results are bitwise identical either way.
int pair_cold_rows(int E, int K, bool swiglu_gemm1, int n_out, int kb_elems) {
    if (kb_elems != kBK) return 0;                                // bf16 operands only
    if (E > 256) return 0;                                        // the kernel's shared memory bound
    if (K % (4 * kBK) != 0) return 0;                            // cold stages of 4 k-blocks
    if (n_out % (swiglu_gemm1 ? 128 : 256) != 0) return 0;       // whole cold tiles
    const char* f = getenv("MOE_PAIR_COLD_ROWS");
    return f ? std::max(0, atoi(f)) : 0;
}

// MOE_PAIR_BAND=n pins the m-tiles per raster band of the pair kernels
// (tuning; a band at least an expert's m-tile count is the unbanded order).
int pair_band() {
    const char* f = getenv("MOE_PAIR_BAND");
    return f ? std::max(0, atoi(f)) : 0;
}

// `avail` = bytes of scratch the caller provided for partials: a split that
// would not fit runs unsplit instead.
FfnPlan plan_ffn(int rows, int D, int E, int Dff, bool swiglu, int nsm, size_t avail, int kb_elems = kBK) {
    FfnPlan p;
    const long long touched_ub = std::min(E, rows);
    const bool swap = env_flag("MOE_SWAP_GEMM", static_cast<long long>(rows) <= 32 * touched_ub);
    const bool pair = !swap && env_flag("MOE_PAIR_GEMM", static_cast<long long>(rows) >= 256 * touched_ub);
    const int bt = (static_cast<long long>(rows) <= 8 * touched_ub) ? 16 : 32;
    const int kb1 = D / kb_elems, kb2 = Dff / kb_elems;

    // ---- GEMM1: rows x D  ->  h (Dff), act fused
    GemmPlan& a = p.g1;
    if (swap && (swiglu || Dff % 128 == 0)) {
        a.mode = MODE_SWAP;
        a.bn = bt;
        const int nt = swiglu ? Dff / 64 : Dff / 128;
        a.tiles_ub = (rows / bt + touched_ub) * nt;
        a.ldp = swiglu ? 2 * Dff : Dff;
    } else {
        a.bn = ffn_bn(Dff, swiglu);
        const int per = swiglu ? a.bn / 2 : a.bn;
        const int nt = (Dff + per - 1) / per;
        a.mode = (pair && swiglu && a.bn == 256) ? MODE_PAIR : MODE_ONE;
        a.tiles_ub = (a.mode == MODE_PAIR ? rows / (2 * kBM) : rows / kBM) * static_cast<long long>(nt) +
                     touched_ub * nt;
        a.ldp = nt * a.bn;
    }
    // splits keep >= 4 k-blocks each and stop at 4
    constexpr double kSwapSplitCost = 0.3;
    const int max_s1 = (a.mode == MODE_PAIR) ? 1 : std::min(4, kb1 / 4);
    a.splits = plan_splits(a.tiles_ub, max_s1, nsm, a.mode == MODE_SWAP ? kSwapSplitCost : 0.0);
    a.cold_rows = (a.mode == MODE_PAIR) ? pair_cold_rows(E, D, swiglu, Dff, kb_elems) : 0;
    if (a.cold_rows > 0) a.tiles_ub += touched_ub * ((a.cold_rows + 31) / 32) * (Dff / 128);

    // ---- GEMM2: rows x Dff  ->  y (D)
    GemmPlan& b = p.g2;
    if (swap && D % 128 == 0) {
        b.mode = MODE_SWAP;
        b.bn = bt;
        b.tiles_ub = (rows / bt + touched_ub) * (D / 128);
    } else {
        b.bn = ffn_bn(D, false);
        const int nt = (D + b.bn - 1) / b.bn;
        b.mode = (pair && b.bn == 256) ? MODE_PAIR : MODE_ONE;
        b.tiles_ub = (b.mode == MODE_PAIR ? rows / (2 * kBM) : rows / kBM) * static_cast<long long>(nt) +
                     touched_ub * nt;
    }
    b.ldp = D;
    const int max_s2 = (b.mode == MODE_PAIR) ? 1 : std::min(4, kb2 / 4);
    b.splits = plan_splits(b.tiles_ub, max_s2, nsm, b.mode == MODE_SWAP ? kSwapSplitCost : 0.0);
    b.cold_rows = (b.mode == MODE_PAIR) ? pair_cold_rows(E, Dff, false, D, kb_elems) : 0;
    if (b.cold_rows > 0) b.tiles_ub += touched_ub * ((b.cold_rows + 31) / 32) * (D / 256);

    // MOE_FFN_SPLITS=s1,s2 pins the k-splits of GEMM1 and GEMM2 (tuning; each
    // clamped to 1 .. its maximum, so the workspace bound still holds)
    if (const char* f = getenv("MOE_FFN_SPLITS")) {
        int s1 = 0, s2 = 0;
        if (sscanf(f, "%d,%d", &s1, &s2) == 2) {
            a.splits = std::max(1, std::min(s1, std::max(1, max_s1)));
            b.splits = std::max(1, std::min(s2, std::max(1, max_s2)));
        }
    }

    if (static_cast<size_t>(a.splits) * rows * a.ldp * sizeof(float) > avail) a.splits = 1;
    if (static_cast<size_t>(b.splits) * rows * b.ldp * sizeof(float) > avail) b.splits = 1;
    return p;
}

size_t route_ws_bytes(int N, int D, int E) {
    return kWsHeaderBytes + align_up(plan_route(N, D, E, kMaxPlanSms).partial_bytes, 256);
}

size_t ffn_ws_bytes(int rows, int D, int E, int Dff) {
    return kWsHeaderBytes + align_up(ffn_partial_bound(rows, D, E, Dff), 256);
}

// ---- layer workspace layout ----
struct LayerLayout {
    size_t ids, w, offsets, perm_src, inv_perm, x_perm, h, y_perm, perm_scratch, gemm_scratch,
        gemm_scratch_bytes, total;
};

LayerLayout layer_layout(int N, int D, int E, int K, int Dff) {
    LayerLayout L;
    const size_t A = static_cast<size_t>(N) * K;
    size_t o = kWsHeaderBytes;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.ids = take(A * 4);
    L.w = take(A * 4);
    L.offsets = take((E + 1) * 4);
    L.perm_src = take(A * 4);
    L.inv_perm = take(A * 4);
    L.perm_scratch = take(permute_scratch_bytes(N, E));
    // fp32 split-K partials: the router's, then (reused) the FFN's
    L.gemm_scratch = take(std::max(plan_route(N, D, E, kMaxPlanSms).partial_bytes,
                                   ffn_partial_bound(N * K, D, E, Dff)));
    L.gemm_scratch_bytes = o - L.gemm_scratch;
    L.x_perm = take(A * D * 2);
    L.h = take(A * Dff * 2);
    L.y_perm = take(A * D * 2);
    L.total = o;
    return L;
}

// ---- paradigm B layer workspace layout ----
struct PaddedLayout {
    size_t ids, w, pad_offsets, kept, slot, x_pad, h, y_pad, perm_scratch, gemm_scratch, gemm_scratch_bytes, total;
};

PaddedLayout padded_layout(int N, int D, int E, int K, int Dff, int C) {
    PaddedLayout L;
    const size_t A = static_cast<size_t>(N) * K;
    const size_t R = static_cast<size_t>(E) * C;  // rows of the padded buffer
    size_t o = kWsHeaderBytes;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.ids = take(A * 4);
    L.w = take(A * 4);
    L.pad_offsets = take((E + 1) * 4);
    L.kept = take(E * 4);
    L.slot = take(A * 4);
    L.perm_scratch = take(permute_scratch_bytes(N, E));
    L.gemm_scratch = take(std::max(plan_route(N, D, E, kMaxPlanSms).partial_bytes,
                                   ffn_partial_bound(static_cast<int>(R), D, E, Dff)));
    L.gemm_scratch_bytes = o - L.gemm_scratch;
    L.x_pad = take(R * D * 2);
    L.h = take(R * Dff * 2);
    L.y_pad = take(R * D * 2);
    L.total = o;
    return L;
}

// ---- e4m3 layer workspace layout ----
struct E4m3Layout {
    size_t ids, w, offsets, perm_src, inv_perm, xq, x_scale, xq_perm, h, hq, h_scale, y_perm, perm_scratch,
        gemm_scratch, gemm_scratch_bytes, total;
};

E4m3Layout e4m3_layout(int N, int D, int E, int K, int Dff) {
    E4m3Layout L;
    const size_t A = static_cast<size_t>(N) * K;
    size_t o = kWsHeaderBytes;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.ids = take(A * 4);
    L.w = take(A * 4);
    L.offsets = take((E + 1) * 4);
    L.perm_src = take(A * 4);
    L.inv_perm = take(A * 4);
    L.perm_scratch = take(permute_scratch_bytes(N, E));
    L.gemm_scratch = take(std::max(plan_route(N, D, E, kMaxPlanSms).partial_bytes,
                                   ffn_partial_bound(N * K, D, E, Dff)));
    L.gemm_scratch_bytes = o - L.gemm_scratch;
    L.xq = take(static_cast<size_t>(N) * D);
    L.x_scale = take(static_cast<size_t>(N) * 4);
    L.xq_perm = take(A * D);
    L.h = take(A * Dff * 2);
    L.hq = take(A * Dff);
    L.h_scale = take(A * 4);
    L.y_perm = take(A * D * 2);
    L.total = o;
    return L;
}

// e4m3 GEMM operands: K of both GEMMs a multiple of 128 (one stage = 128 codes).
moe_status check_e4m3_dims(int D, int Dff) {
    if (D % 128) return fail(MOE_ERR_INVALID_ARG, "e4m3 path: D=%d not a multiple of 128", D);
    if (Dff % 128) return fail(MOE_ERR_INVALID_ARG, "e4m3 path: Dff=%d not a multiple of 128", Dff);
    return MOE_OK;
}

moe_status check_capacity(int E, int C, int D, int Dff) {
    if (C < 0) return fail(MOE_ERR_INVALID_ARG, "capacity=%d < 0", C);
    const long long R = static_cast<long long>(E) * C;
    if (R >= (1LL << 31)) return fail(MOE_ERR_INVALID_ARG, "E*capacity=%lld too large", R);
    if (R * std::max(D, Dff) >= (1LL << 40)) return fail(MOE_ERR_INVALID_ARG, "padded buffer too large");
    return MOE_OK;
}

// ---- stage implementations (no validation: callers validated) ----
// `scratch` (scratch_bytes) holds the fp32 partial logits.
// The permutation a route call may do in the same launch as its top-K.
struct PermuteOut {
    int32_t* offsets;
    int32_t* perm_src;
    int32_t* inv_perm;
    moe_bf16* x_perm;  // null: indices only
};

// Calls of up to 8 tokens (one warp each in every CTA of the fused launch)
// select the top-K and permute in one launch (MOE_FUSED_ROUTE_PERMUTE=0 turns
// it off; same bits either way).  Measured on GB300 (Qwen3-shaped decode
// steps, graph replays): 1 token 39.5 -> 37.5 us, 8 tokens 98.2 -> 96.8 us;
// at 32 tokens the redundant selection in every CTA cost 4 us more than the
// launch it saves.
constexpr int kFusedRoutePermuteTokens = 8;

bool fused_route_permute(int N, int K) {
    return N <= kFusedRoutePermuteTokens && static_cast<long long>(N) * K <= kFusedRoutePermuteMax &&
           env_flag("MOE_FUSED_ROUTE_PERMUTE", true);
}

// The top-K after the logits: with `perm` (and a decode-sized call) the
// fused top-K + permutation, which sets *permuted.
moe_status route_select(const float* partial, int splits, long long split_stride, int ldp, const moe_bf16* x,
                        const float* bias, int N, int D, int E, int K, int mode, int32_t* ids, float* w,
                        float* logits_out, void* ws, const PermuteOut* perm, bool* permuted, cudaStream_t st) {
    cudaError_t e;
    if (perm && fused_route_permute(N, K)) {
        const int grid = std::max(1, std::min(N * K, sm_count()));
        e = launch_route_topk_permute(partial, splits, split_stride, ldp, bias, N, E, K, mode, logits_out, ids, w,
                                      reinterpret_cast<const uint16_t*>(x), D, perm->offsets, perm->perm_src,
                                      perm->inv_perm, reinterpret_cast<uint16_t*>(perm->x_perm), grid, ws_err(ws), st);
        if (e == cudaSuccess && permuted) *permuted = true;
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "router top-K + permute launch");
    }
    e = launch_route_topk(partial, splits, split_stride, ldp, bias, N, E, K, mode, logits_out, ids, w, ws_err(ws),
                          st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "router top-K launch");
}

moe_status do_route(const moe_bf16* x, const moe_bf16* w_gate, const float* bias, int N, int D, int E, int K,
                    int mode, int32_t* ids, float* w, float* logits_out, void* ws, void* scratch,
                    size_t scratch_bytes, cudaStream_t st, const PermuteOut* perm = nullptr,
                    bool* permuted = nullptr) {
    const int nsm = sm_count();
    if (permuted) *permuted = false;
    if (N <= kSmallRouteMaxN && D <= 8192) {
        // decode-sized: logits on the CUDA cores (one warp per expert), then the top-K
        float* logits = static_cast<float*>(scratch);
        cudaError_t e = launch_route_logits_small(reinterpret_cast<const uint16_t*>(x),
                                                  reinterpret_cast<const uint16_t*>(w_gate), N, D, E, logits, st);
        if (e != cudaSuccess) return cuda_fail(e, "router logits launch");
        return route_select(logits, 1, static_cast<long long>(N) * E, E, x, bias, N, D, E, K, mode, ids, w,
                            logits_out, ws, perm, permuted, st);
    }
    const RoutePlan p = plan_route(N, D, E, nsm, scratch_bytes);
    CUtensorMap tA, tB;
    moe_status s = make_tmap(&tA, x, N, D, kBM);
    if (s != MOE_OK) return s;
    s = make_tmap(&tB, w_gate, E, D, p.bn);
    if (s != MOE_OK) return s;
    float* partial = static_cast<float*>(scratch);
    GemmArgs a{};
    a.group_offsets = nullptr;
    a.G = 1;
    a.M = N;
    a.n_out = E;
    a.k_dim = D;
    a.b_rows_per_group = 0;
    a.splits = p.splits;
    a.out = partial;
    a.ldo = p.ldp;
    a.split_stride = static_cast<long long>(N) * p.ldp;
    a.err = ws_err(ws);
    a.dbg = ws_dbg(ws);
    const long long items = static_cast<long long>((N + kBM - 1) / kBM) * p.nt * p.splits;
    const int grid = static_cast<int>(std::min<long long>(items, nsm));
    cudaError_t e = launch_grouped_gemm(EPI_F32, p.bn, tA, tB, tB, a, grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "router GEMM launch");
    return route_select(partial, p.splits, a.split_stride, p.ldp, x, bias, N, D, E, K, mode, ids, w, logits_out, ws,
                        perm, permuted, st);
}

// e4m3 scales of one GEMM (all null for bf16 operands): per output row (with
// an optional index, e.g. token scales read through perm_src) and per weight
// row (W1 / W3 for the SwiGLU GEMM1).
struct GemmScales {
    const float* row;
    const int32_t* row_idx;
    const float* col;
    const float* col_up;
};

// GEMM1's operand rows read through the permutation instead of from a
// permuted copy: row r of A is row rows[r] of src (n rows, ld bytes apart).
struct GatherSrc {
    const void* src;
    const int32_t* rows;
    long long ld;
    int n;
};

// The layer fuses the gather into GEMM1 only when MOE_GATHER=1 (read at each
// call; results are identical either way).  Off by default: with the weights
// streaming from HBM the 16-byte row copies cannot keep enough bytes in
// flight, and the fused GEMM1 runs slower than the separate row copy.
bool gather_enabled() { return env_flag("MOE_GATHER", false); }

// Calls of up to MOE_LAYER_DECODE_MAX_N tokens (default kLayerDecodeTokens
// for bf16 experts, kLayerDecodeTokensE4m3 for e4m3 ones, at most
// kLayerDecodeMaxN) with at most kLayerDecodeMaxRows assignments run the
// whole layer as one cooperative launch (layer_decode.cu);
// MOE_LAYER_DECODE=0 turns it off, and MOE_GATHER=1 selects the gathered
// GEMM1 instead.  Returns the launch's grid, or 0 for the chain of launches.
// The defaults follow measurements on GB300 (Qwen3-shaped layer, graphs of
// 20 calls): the token counts up to which the one launch was faster than
// the chain, whose pipelined TMA weight streams keep more bytes in flight
// once the per-token work outgrows the launch overheads it saves.
constexpr int kLayerDecodeTokens = 4;
constexpr int kLayerDecodeTokensE4m3 = 4;

static bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

int layer_decode_grid(int N, int D, int E, int K, int Dff, int act, bool fp8 = false) {
    if (!env_flag("MOE_LAYER_DECODE", true) || gather_enabled()) return 0;
    int maxn = fp8 ? kLayerDecodeTokensE4m3 : kLayerDecodeTokens;
    if (const char* f = getenv("MOE_LAYER_DECODE_MAX_N")) maxn = atoi(f);
    maxn = std::min(maxn, kLayerDecodeMaxN);
    if (N < 1 || N > maxn || N * K > kLayerDecodeMaxRows || E > kLayerDecodeMaxE || D > 8192) return 0;
    int w2_smem = 0;
    return layer_decode_plan(N, D, E, K, Dff, act == MOE_ACT_SWIGLU, fp8, &w2_smem);
}

// Whether the decode layer stages each CTA's W2 columns in shared memory
// (MOE_LAYER_DECODE_W2_SMEM=1, when they fit).  Off by default: GEMM2
// reading W2 from global memory, prefetched into L2 during GEMM1, measured
// faster on GB300 (Qwen3-shaped layer, bf16 and e4m3).
int layer_decode_w2_smem(int N, int D, int E, int K, int Dff, int act, bool fp8 = false) {
    if (!env_flag("MOE_LAYER_DECODE_W2_SMEM", false)) return 0;
    int w2_smem = 0;
    layer_decode_plan(N, D, E, K, Dff, act == MOE_ACT_SWIGLU, fp8, &w2_smem);
    return w2_smem;
}

// W2 bytes of the chosen experts up to which the decode layer prefetches
// them into L2 while GEMM1 streams (MOE_LAYER_DECODE_L2_MB, default 64 MB of
// the 126 MB L2; 0 turns the prefetch off).
long long layer_decode_prefetch_bytes() {
    long long mb = 64;
    if (const char* f = getenv("MOE_LAYER_DECODE_L2_MB")) mb = atoll(f);
    return std::max(0LL, mb) << 20;
}

// One GEMM of the grouped FFN per its plan.  A = activations [rows, K],
// W = stacked weights [E*n_rows, K] (W3 too for SwiGLU GEMM1), out = bf16
// [rows, n_out]; with splits > 1 the fp32 partials go to `partial` and a
// reduction kernel writes `out` (applying the activation for GEMM1).  With
// e4m3 = true, A and W hold e4m3 codes and `sc` their scales.
moe_status run_ffn_gemm(const GemmPlan& gp, bool gemm1, bool swiglu, bool e4m3, const GemmScales& sc,
                        const void* A, const void* W, const void* W3, const int32_t* offsets, int rows, int E,
                        int K, int n_out, moe_bf16* out, float* partial, void* ws, int nsm, cudaStream_t st,
                        const GatherSrc* gather = nullptr) {
    const bool dual = gemm1 && swiglu;
    const long long wrows = static_cast<long long>(E) * n_out;
    GemmArgs a{};
    if (gather) {
        a.a_src = gather->src;
        a.a_src_rows = gather->rows;
        a.a_src_ld = gather->ld;
        a.a_src_n = gather->n;
    }
    a.row_scale = sc.row;
    a.row_scale_idx = sc.row_idx;
    a.col_scale = sc.col;
    a.col_scale_up = sc.col_up;
    a.group_offsets = offsets;
    a.G = E;
    a.M = rows;
    a.n_out = n_out;
    a.k_dim = K;
    a.b_rows_per_group = n_out;
    a.splits = gp.splits;
    a.band = pair_band();
    a.err = ws_err(ws);
    a.dbg = ws_dbg(ws);
    if (gp.splits == 1) {
        a.out = out;
        a.ldo = n_out;
    } else {
        a.out = partial;
        a.ldo = gp.ldp;
        a.split_stride = static_cast<long long>(rows) * gp.ldp;
    }
    const int bf16_epi = gemm1 ? (swiglu ? EPI_SWIGLU_BF16 : EPI_SILU_BF16) : EPI_STORE_BF16;
    const int epi = (gp.splits == 1) ? bf16_epi : (dual ? EPI_F32_DUAL : EPI_F32);
    CUtensorMap tA, tB, tB2;
    moe_status s = MOE_OK;
    cudaError_t e;
    if (gp.mode == MODE_SWAP) {
        const int wbox = dual ? 64 : 128;
        s = make_tmap(&tB, W, wrows, K, wbox, e4m3);
        if (s == MOE_OK) s = make_tmap(&tB2, dual ? W3 : W, wrows, K, wbox, e4m3);
        if (s == MOE_OK && !gather) s = make_tmap(&tA, A, rows, K, gp.bn, e4m3);
        if (s != MOE_OK) return s;
        const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(gp.tiles_ub * gp.splits, nsm)));
        if (gather)
            e = launch_grouped_gemm_swap_gather(e4m3, epi, gp.bn, tB, tB2, a, grid, st);
        else
            e = e4m3 ? launch_grouped_gemm_swap_e4m3(epi, gp.bn, tB, tB2, tA, a, grid, st)
                     : launch_grouped_gemm_swap(epi, gp.bn, tB, tB2, tA, a, grid, st);
    } else {
        const int box_b = (dual || gp.mode == MODE_PAIR) ? gp.bn / 2 : gp.bn;
        if (!gather) s = make_tmap(&tA, A, rows, K, kBM, e4m3);
        if (s == MOE_OK) s = make_tmap(&tB, W, wrows, K, box_b, e4m3);
        if (s == MOE_OK) s = make_tmap(&tB2, dual ? W3 : W, wrows, K, box_b, e4m3);
        if (s != MOE_OK) return s;
        const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(gp.tiles_ub * gp.splits, nsm)));
        if (gather) {
            e = (gp.mode == MODE_PAIR) ? launch_grouped_gemm_pair_gather(e4m3, bf16_epi, tB, tB2, a, gp.tiles_ub, st)
                                       : launch_grouped_gemm_gather(e4m3, epi, gp.bn, tB, tB2, a, grid, st);
        } else if (gp.mode == MODE_PAIR && !e4m3 && gp.cold_rows > 0) {
            // hot experts on 256-row pair tiles (3-D views: 128 token rows and
            // 128 weight rows by 2 k-blocks), cold ones on weight-streaming
            // tiles (16 token rows and 128 weight rows by 4 k-blocks)
            CUtensorMap hA, hB, hB2, cT, cW, cW2;
            a.cold_rows = gp.cold_rows;
            s = make_tmap3d(&hA, A, rows, K, kBM, 2);
            if (s == MOE_OK) s = make_tmap3d(&hB, W, wrows, K, kBM, 2);
            if (s == MOE_OK) s = make_tmap3d(&hB2, dual ? W3 : W, wrows, K, kBM, 2);
            if (s == MOE_OK) s = make_tmap3d(&cT, A, rows, K, 16, 4);
            if (s == MOE_OK) s = make_tmap3d(&cW, W, wrows, K, kBM, 4);
            if (s == MOE_OK) s = make_tmap3d(&cW2, dual ? W3 : W, wrows, K, kBM, 4);
            if (s != MOE_OK) return s;
            e = launch_grouped_gemm_pair_mixed(bf16_epi, hA, hB, hB2, cT, cW, cW2, a, gp.tiles_ub, st);
        } else if (gp.mode == MODE_PAIR) {
            e = e4m3 ? launch_grouped_gemm_pair_e4m3(bf16_epi, tA, tB, tB2, a, gp.tiles_ub, st)
                     : launch_grouped_gemm_pair(bf16_epi, tA, tB, tB2, a, gp.tiles_ub, st);
        } else {
            e = e4m3 ? launch_grouped_gemm_e4m3(epi, gp.bn, tA, tB, tB2, a, grid, st)
                     : launch_grouped_gemm(epi, gp.bn, tA, tB, tB2, a, grid, st);
        }
    }
    if (e != cudaSuccess) return cuda_fail(e, gemm1 ? "grouped GEMM1 launch" : "grouped GEMM2 launch");
    if (gp.splits > 1) {
        // SwiGLU partials are tile-interleaved: tiles of width gp.ldp / (n_out / half) hold gate | up
        if (dual) {
            const int tile_w = (gp.mode == MODE_SWAP) ? 128 : gp.bn;
            e = launch_ffn_reduce_swiglu(partial, gp.splits, a.split_stride, gp.ldp, rows, n_out, tile_w, out, st);
        } else {
            e = launch_ffn_reduce_store(partial, gp.splits, a.split_stride, gp.ldp, rows, n_out, gemm1, out, st);
        }
        if (e != cudaSuccess) return cuda_fail(e, "split-K reduction launch");
    }
    return MOE_OK;
}

// The decode-sized SwiGLU FFN runs as one persistent launch (both GEMMs with
// swapped operands) from 16 rows up, unless MOE_FUSED_DECODE=0 (or =1 to use
// it at any size).  Below 16 rows (one token with K = 8) the counter reset and
// the cooperative launch, which cannot overlap the previous kernel's tail,
// cost more than the launches they replace (measured on GB300).  With e4m3
// operands it runs only when MOE_FUSED_DECODE=1: there the GEMM1 epilogue
// (scales fetched under the full weight stream, the row maxima for the h
// quantisation) is slower than the halved weight stream per tile, and the
// separate launches measured faster.
constexpr int kFusedDecodeMinRows = 16;

bool use_fused_decode(const FfnPlan& p, bool swiglu, int rows, bool e4m3 = false) {
    if (!swiglu || p.g1.mode != MODE_SWAP || p.g2.mode != MODE_SWAP || p.g1.bn != p.g2.bn) return false;
    if (const char* f = getenv("MOE_FUSED_DECODE")) return atoi(f) != 0;
    return !e4m3 && rows >= kFusedDecodeMinRows;
}

// Operands of the fused decode FFN: bf16 (sc == nullptr) or e4m3 codes with
// their scales (the e4m3 outputs hq, h_scale then written too).
struct FusedOperands {
    const void *x, *w1, *w3, *w2;
    const GemmScales* sc1;  // x_scale, x_scale_idx, s1, s3 (null: bf16)
    const float* s2;
    uint8_t* hq;
    float* h_scale;
};

moe_status run_fused_decode(const FfnPlan& p, const FusedOperands& op, const int32_t* offsets, int rows, int E,
                            int D, int Dff, moe_bf16* h, moe_bf16* y, void* ws, void* scratch,
                            const FusedDecodeLayout& L, int nsm, cudaStream_t st) {
    const int bt = p.g1.bn;
    const bool e4m3 = op.sc1 != nullptr;
    CUtensorMap maps[5];
    moe_status s = make_tmap(&maps[0], op.w1, static_cast<long long>(E) * Dff, D, 64, e4m3);
    if (s == MOE_OK) s = make_tmap(&maps[1], op.w3, static_cast<long long>(E) * Dff, D, 64, e4m3);
    if (s == MOE_OK) s = make_tmap(&maps[2], op.x, rows, D, bt, e4m3);
    if (s == MOE_OK) s = make_tmap(&maps[3], op.w2, static_cast<long long>(E) * D, Dff, 128, e4m3);
    if (s == MOE_OK) s = make_tmap(&maps[4], e4m3 ? static_cast<const void*>(op.hq) : h, rows, Dff, bt, e4m3);
    if (s != MOE_OK) return s;
    char* base = static_cast<char*>(scratch);
    FusedFfnArgs a{};
    a.group_offsets = offsets;
    a.G = E;
    a.M = rows;
    a.D = D;
    a.Dff = Dff;
    a.splits1 = p.g1.splits;
    a.splits2 = p.g2.splits;
    a.part1 = reinterpret_cast<float*>(base + L.part1);
    a.part2 = reinterpret_cast<float*>(base + L.part2);
    a.h = h;
    a.y = y;
    a.tile_cnt1 = reinterpret_cast<int*>(base + L.counters);
    a.tile_cnt2 = a.tile_cnt1 + p.g1.tiles_ub;
    a.expert_done = a.tile_cnt2 + p.g2.tiles_ub;
    a.quant_done = a.expert_done + E;
    a.h_amax = reinterpret_cast<uint32_t*>(a.quant_done + E);
    a.tiles1_cap = static_cast<int>(p.g1.tiles_ub);
    a.tiles2_cap = static_cast<int>(p.g2.tiles_ub);
    a.err = ws_err(ws);
    a.dbg = ws_dbg(ws);
    if (e4m3) {
        a.x_scale = op.sc1->row;
        a.x_scale_idx = op.sc1->row_idx;
        a.s1 = op.sc1->col;
        a.s3 = op.sc1->col_up;
        a.s2 = op.s2;
        a.hq = op.hq;
        a.h_scale = op.h_scale;
        a.xs_rows = ffn_fused_decode_xs_rows(bt, E, rows);
    }
    cudaError_t e = cudaMemsetAsync(base + L.counters, 0, L.counter_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "fused decode counters");
    const long long items = p.g1.tiles_ub * p.g1.splits + p.g2.tiles_ub * p.g2.splits;
    const int grid = static_cast<int>(std::max<long long>(
        1, std::min<long long>({items, static_cast<long long>(nsm),
                                static_cast<long long>(ffn_fused_decode_max_grid(e4m3, bt, E, a.xs_rows))})));
    e = launch_ffn_fused_decode(e4m3, bt, maps, a, grid, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "fused decode FFN launch");
}

// x_perm is ignored when `gather` is given (GEMM1 reads the rows through it).
moe_status do_grouped_ffn(const moe_bf16* x_perm, const int32_t* offsets, int rows, const moe_bf16* w1,
                          const moe_bf16* w3, const moe_bf16* w2, int E, int D, int Dff, int act, moe_bf16* h,
                          moe_bf16* y, void* ws, void* scratch, size_t scratch_bytes, cudaStream_t st,
                          const GatherSrc* gather = nullptr) {
    const bool swiglu = act == MOE_ACT_SWIGLU;
    const int nsm = sm_count();
    const FfnPlan p = plan_ffn(rows, D, E, Dff, swiglu, nsm, scratch_bytes);
    float* partial = static_cast<float*>(scratch);
    if (!gather && use_fused_decode(p, swiglu, rows)) {
        const FusedDecodeLayout L = fused_decode_layout(rows, D, E, Dff, p.g1.splits, p.g2.splits, p.g1.tiles_ub,
                                                        p.g2.tiles_ub);
        if (L.total <= scratch_bytes) {
            const FusedOperands op{x_perm, w1, w3, w2, nullptr, nullptr, nullptr, nullptr};
            return run_fused_decode(p, op, offsets, rows, E, D, Dff, h, y, ws, scratch, L, nsm, st);
        }
    }
    const GemmScales none{};
    moe_status s = run_ffn_gemm(p.g1, true, swiglu, false, none, x_perm, w1, w3, offsets, rows, E, D, Dff, h, partial,
                                ws, nsm, st, gather);
    if (s != MOE_OK) return s;
    return run_ffn_gemm(p.g2, false, swiglu, false, none, h, w2, nullptr, offsets, rows, E, Dff, D, y, partial, ws,
                        nsm, st);
}

// The grouped FFN with e4m3 operands: GEMM1 (+ act) -> h bf16 -> per-row
// e4m3 quantisation (hq, h_scale) -> GEMM2.  x_scale is per row of xq_perm,
// or per token with x_scale_idx = perm_src.
moe_status do_grouped_ffn_e4m3(const uint8_t* xq_perm, const float* x_scale, const int32_t* x_scale_idx,
                               const int32_t* offsets, int rows, const uint8_t* w1q, const float* s1,
                               const uint8_t* w3q, const float* s3, const uint8_t* w2q, const float* s2, int E,
                               int D, int Dff, int act, moe_bf16* h, uint8_t* hq, float* h_scale, moe_bf16* y,
                               void* ws, void* scratch, size_t scratch_bytes, cudaStream_t st,
                               const GatherSrc* gather = nullptr) {
    const bool swiglu = act == MOE_ACT_SWIGLU;
    const int nsm = sm_count();
    const FfnPlan p = plan_ffn(rows, D, E, Dff, swiglu, nsm, scratch_bytes, OpType<true>::KB);
    float* partial = static_cast<float*>(scratch);
    const GemmScales sc1{x_scale, x_scale_idx, s1, swiglu ? s3 : nullptr};
    if (!gather && use_fused_decode(p, swiglu, rows, true)) {
        const FusedDecodeLayout L = fused_decode_layout(rows, D, E, Dff, p.g1.splits, p.g2.splits, p.g1.tiles_ub,
                                                        p.g2.tiles_ub);
        if (L.total <= scratch_bytes) {
            const FusedOperands op{xq_perm, w1q, w3q, w2q, &sc1, s2, hq, h_scale};
            return run_fused_decode(p, op, offsets, rows, E, D, Dff, h, y, ws, scratch, L, nsm, st);
        }
    }
    moe_status s = run_ffn_gemm(p.g1, true, swiglu, true, sc1, xq_perm, w1q, w3q, offsets, rows, E, D, Dff, h,
                                partial, ws, nsm, st, gather);
    if (s != MOE_OK) return s;
    cudaError_t e = launch_quant_rows_e4m3(h, rows, Dff, hq, h_scale, st);
    if (e != cudaSuccess) return cuda_fail(e, "hidden activation quantisation launch");
    const GemmScales sc2{h_scale, nullptr, s2, nullptr};
    return run_ffn_gemm(p.g2, false, swiglu, true, sc2, hq, w2q, nullptr, offsets, rows, E, Dff, D, y, partial, ws,
                        nsm, st);
}

}  // namespace

// ============================================================================
// public ABI
// ============================================================================
extern "C" {

const char* moe_version(void) { return "mixture_experts_layer_02_gb300 0.1 (sm_103a)"; }

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_BOUNDS: return "device-side bounds error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

const char* moe_last_error_detail(void) { return g_detail.c_str(); }

size_t moe_workspace_size(const char* op, int N, int D, int E, int K, int Dff) {
    if (op == nullptr) return 0;
    if (!strcmp(op, "combine")) return kWsHeaderBytes;
    if (!strcmp(op, "route")) {
        if (check_sizes(N, D, E, std::max(K, 1), 64, false) != MOE_OK) return 0;
        return route_ws_bytes(N, D, E);
    }
    if (!strcmp(op, "ffn")) {   // N = total rows of the permuted buffer
        if (check_sizes(N, D, E, 1, Dff, true) != MOE_OK) return 0;
        return ffn_ws_bytes(N, D, E, Dff);
    }
    if (!strcmp(op, "permute")) {
        if (N < 0 || E < 1) return 0;
        return kWsHeaderBytes + align_up(permute_scratch_bytes(N, E), 256);
    }
    if (!strcmp(op, "route_permute")) {  // the router's partials, then the permutation's counts
        if (check_sizes(N, D, E, std::max(K, 1), 64, false) != MOE_OK) return 0;
        return route_ws_bytes(N, D, E) + align_up(permute_scratch_bytes(N, E), 256);
    }
    if (!strcmp(op, "layer")) {
        if (check_sizes(N, D, E, K, Dff, true) != MOE_OK) return 0;
        return layer_layout(N, D, E, K, Dff).total;
    }
    if (!strcmp(op, "layer_e4m3")) {
        if (check_sizes(N, D, E, K, Dff, true) != MOE_OK || D % 128 || Dff % 128) return 0;
        return e4m3_layout(N, D, E, K, Dff).total;
    }
    return 0;
}

int moe_layer_workspace_layout(int N, int D, int E, int K, int Dff, size_t out[8]) {
    if (out == nullptr || check_sizes(N, D, E, K, Dff, true) != MOE_OK) return -1;
    const LayerLayout L = layer_layout(N, D, E, K, Dff);
    out[0] = L.ids;
    out[1] = L.w;
    out[2] = L.offsets;
    out[3] = L.perm_src;
    out[4] = L.inv_perm;
    out[5] = L.x_perm;
    out[6] = L.h;
    out[7] = L.y_perm;
    return 0;
}

moe_status moe_route(const moe_bf16* x, const moe_bf16* w_gate, const float* bias, int N, int D, int E, int K,
                     int mode, int32_t* topk_ids, float* topk_w, float* logits_out, void* ws, size_t ws_bytes,
                     void* stream) {
    moe_status s = check_sizes(N, D, E, K, 64, false);
    if (s != MOE_OK) return s;
    if (mode != MOE_SCORE_SOFTMAX_TOPK && mode != MOE_SCORE_SIGMOID_NORM)
        return fail(MOE_ERR_INVALID_ARG, "mode=%d", mode);
    REQUIRE_PTR(ws);
    if (ws_bytes < moe_workspace_size("route", N, D, E, K, 0)) return fail(MOE_ERR_WORKSPACE, "route workspace");
    if (N == 0) return MOE_OK;
    REQUIRE_PTR(x);
    REQUIRE_PTR(w_gate);
    REQUIRE_PTR(topk_ids);
    REQUIRE_PTR(topk_w);
    OPTIONAL_PTR(bias);
    OPTIONAL_PTR(logits_out);
    return do_route(x, w_gate, bias, N, D, E, K, mode, topk_ids, topk_w, logits_out, ws,
                    static_cast<char*>(ws) + kWsHeaderBytes, ws_bytes - kWsHeaderBytes,
                    static_cast<cudaStream_t>(stream));
}

moe_status moe_permute(const moe_bf16* x, const int32_t* topk_ids, int N, int D, int E, int K,
                       int32_t* expert_offsets, int32_t* perm_src, int32_t* inv_perm, moe_bf16* x_perm, void* ws,
                       size_t ws_bytes, void* stream) {
    moe_status s = check_sizes(N, D, E, K, 64, false);
    if (s != MOE_OK) return s;
    REQUIRE_PTR(ws);
    if (ws_bytes < moe_workspace_size("permute", N, D, E, K, 0)) return fail(MOE_ERR_WORKSPACE, "permute workspace");
    REQUIRE_PTR(expert_offsets);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        cudaError_t e = cudaMemsetAsync(expert_offsets, 0, (E + 1) * sizeof(int32_t), st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "offsets memset");
    }
    REQUIRE_PTR(x);
    REQUIRE_PTR(topk_ids);
    REQUIRE_PTR(perm_src);
    REQUIRE_PTR(inv_perm);
    REQUIRE_PTR(x_perm);
    int32_t* scratch = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kWsHeaderBytes);
    cudaError_t e = launch_permute(x, topk_ids, N, D, E, K, expert_offsets, perm_src, inv_perm, x_perm, scratch,
                                   ws_err(ws), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "permute launch");
}

moe_status moe_route_permute(const moe_bf16* x, const moe_bf16* w_gate, const float* bias, int N, int D, int E,
                             int K, int mode, int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                             int32_t* perm_src, int32_t* inv_perm, moe_bf16* x_perm, void* ws, size_t ws_bytes,
                             void* stream) {
    moe_status s = check_sizes(N, D, E, K, 64, false);
    if (s != MOE_OK) return s;
    if (mode != MOE_SCORE_SOFTMAX_TOPK && mode != MOE_SCORE_SIGMOID_NORM)
        return fail(MOE_ERR_INVALID_ARG, "mode=%d", mode);
    REQUIRE_PTR(ws);
    const size_t rws = route_ws_bytes(N, D, E);
    if (ws_bytes < moe_workspace_size("route_permute", N, D, E, K, 0))
        return fail(MOE_ERR_WORKSPACE, "route_permute workspace");
    REQUIRE_PTR(expert_offsets);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        cudaError_t e = cudaMemsetAsync(expert_offsets, 0, (E + 1) * sizeof(int32_t), st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "offsets memset");
    }
    REQUIRE_PTR(x);
    REQUIRE_PTR(w_gate);
    REQUIRE_PTR(topk_ids);
    REQUIRE_PTR(topk_w);
    REQUIRE_PTR(perm_src);
    REQUIRE_PTR(inv_perm);
    REQUIRE_PTR(x_perm);
    OPTIONAL_PTR(bias);
    char* base = static_cast<char*>(ws);
    const PermuteOut po{expert_offsets, perm_src, inv_perm, x_perm};
    bool permuted = false;
    s = do_route(x, w_gate, bias, N, D, E, K, mode, topk_ids, topk_w, nullptr, ws, base + kWsHeaderBytes,
                 rws - kWsHeaderBytes, st, &po, &permuted);
    if (s != MOE_OK || permuted) return s;
    cudaError_t e = launch_permute(x, topk_ids, N, D, E, K, expert_offsets, perm_src, inv_perm, x_perm,
                                   reinterpret_cast<int32_t*>(base + rws), ws_err(ws), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "permute launch");
}

moe_status moe_grouped_ffn(const moe_bf16* x_perm, const int32_t* expert_offsets, int total_rows,
                           const moe_bf16* w1, const moe_bf16* w3, const moe_bf16* w2, int E, int D, int Dff,
                           int act, moe_bf16* h, moe_bf16* y_perm, void* ws, size_t ws_bytes, void* stream) {
    if (total_rows < 0) return fail(MOE_ERR_INVALID_ARG, "total_rows=%d < 0", total_rows);
    moe_status s = check_sizes(total_rows, D, E, 1, Dff, true);
    if (s != MOE_OK) return s;
    if (act != MOE_ACT_SILU && act != MOE_ACT_SWIGLU) return fail(MOE_ERR_INVALID_ARG, "act=%d", act);
    REQUIRE_PTR(ws);
    if (ws_bytes < moe_workspace_size("ffn", total_rows, D, E, 1, Dff)) return fail(MOE_ERR_WORKSPACE, "ffn workspace");
    if (total_rows == 0) return MOE_OK;
    REQUIRE_PTR(x_perm);
    REQUIRE_PTR(expert_offsets);
    REQUIRE_PTR(w1);
    if (act == MOE_ACT_SWIGLU) REQUIRE_PTR(w3);
    REQUIRE_PTR(w2);
    REQUIRE_PTR(h);
    REQUIRE_PTR(y_perm);
    return do_grouped_ffn(x_perm, expert_offsets, total_rows, w1, w3, w2, E, D, Dff, act, h, y_perm, ws,
                          static_cast<char*>(ws) + kWsHeaderBytes, ws_bytes - kWsHeaderBytes,
                          static_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_bf16* y_perm, const int32_t* inv_perm, const float* topk_w, int N, int D, int K,
                       moe_bf16* out, void* ws, size_t ws_bytes, void* stream) {
    moe_status s = check_sizes(N, D, std::max(K, 1), K, 64, false);
    if (s != MOE_OK) return s;
    REQUIRE_PTR(ws);
    if (ws_bytes < moe_workspace_size("combine", N, D, K, K, 0)) return fail(MOE_ERR_WORKSPACE, "combine workspace");
    if (N == 0) return MOE_OK;
    REQUIRE_PTR(y_perm);
    REQUIRE_PTR(inv_perm);
    REQUIRE_PTR(topk_w);
    REQUIRE_PTR(out);
    cudaError_t e = launch_combine(y_perm, inv_perm, topk_w, N, D, K, out, ws_err(ws),
                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine launch");
}

moe_status moe_layer_forward(const moe_bf16* x, const moe_bf16* w_gate, const float* bias, const moe_bf16* w1,
                             const moe_bf16* w3, const moe_bf16* w2, int N, int D, int E, int K, int Dff, int mode,
                             int act, moe_bf16* out, void* ws, size_t ws_bytes, void* stream) {
    moe_status s = check_sizes(N, D, E, K, Dff, true);
    if (s != MOE_OK) return s;
    if (mode != MOE_SCORE_SOFTMAX_TOPK && mode != MOE_SCORE_SIGMOID_NORM)
        return fail(MOE_ERR_INVALID_ARG, "mode=%d", mode);
    if (act != MOE_ACT_SILU && act != MOE_ACT_SWIGLU) return fail(MOE_ERR_INVALID_ARG, "act=%d", act);
    REQUIRE_PTR(ws);
    const LayerLayout L = layer_layout(N, D, E, K, Dff);
    if (ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "layer workspace needs %zu bytes", L.total);
    if (N == 0) return MOE_OK;
    REQUIRE_PTR(x);
    REQUIRE_PTR(w_gate);
    REQUIRE_PTR(w1);
    if (act == MOE_ACT_SWIGLU) REQUIRE_PTR(w3);
    REQUIRE_PTR(w2);
    REQUIRE_PTR(out);
    OPTIONAL_PTR(bias);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    auto at = [&](size_t off) { return static_cast<void*>(base + off); };
    int32_t* ids = static_cast<int32_t*>(at(L.ids));
    float* w = static_cast<float*>(at(L.w));
    int32_t* offsets = static_cast<int32_t*>(at(L.offsets));
    int32_t* perm_src = static_cast<int32_t*>(at(L.perm_src));
    int32_t* inv_perm = static_cast<int32_t*>(at(L.inv_perm));
    moe_bf16* x_perm = static_cast<moe_bf16*>(at(L.x_perm));
    moe_bf16* h = static_cast<moe_bf16*>(at(L.h));
    moe_bf16* y_perm = static_cast<moe_bf16*>(at(L.y_perm));
    const int rows = N * K;

    // a small decode batch: the whole layer in one launch (its GEMMs read
    // the weights in 32-byte pieces)
    const int ld_grid = layer_decode_grid(N, D, E, K, Dff, act);
    if (ld_grid > 0 && L.gemm_scratch_bytes >= static_cast<size_t>(N) * E * sizeof(float) && aligned32(w1) &&
        aligned32(w2) && (act != MOE_ACT_SWIGLU || aligned32(w3))) {
        LayerDecodeArgs la{};
        la.x = reinterpret_cast<const uint16_t*>(x);
        la.wg = reinterpret_cast<const uint16_t*>(w_gate);
        la.bias = bias;
        la.w1 = reinterpret_cast<const uint16_t*>(w1);
        la.w3 = act == MOE_ACT_SWIGLU ? reinterpret_cast<const uint16_t*>(w3) : nullptr;
        la.w2 = reinterpret_cast<const uint16_t*>(w2);
        la.N = N;
        la.D = D;
        la.E = E;
        la.K = K;
        la.Dff = Dff;
        la.mode = mode;
        la.logits = static_cast<float*>(at(L.gemm_scratch));
        la.ids = ids;
        la.w = w;
        la.offsets = offsets;
        la.perm_src = perm_src;
        la.inv_perm = inv_perm;
        la.x_perm = reinterpret_cast<uint16_t*>(x_perm);
        la.h = reinterpret_cast<uint16_t*>(h);
        la.y_perm = reinterpret_cast<uint16_t*>(y_perm);
        la.out = reinterpret_cast<uint16_t*>(out);
        la.err = ws_err(ws);
        la.dbg = ws_dbg(ws);
        la.bar = reinterpret_cast<unsigned long long*>(base + kWsBarrierCount);
        la.l2_prefetch_max = layer_decode_prefetch_bytes();
        la.w2_smem = layer_decode_w2_smem(N, D, E, K, Dff, act);
        CUtensorMap tm_w2{};
        if (la.w2_smem) {
            s = make_tmap3d(&tm_w2, w2, static_cast<long long>(E) * D, Dff, kLayerDecodeW2Rows, Dff / 64);
            if (s != MOE_OK) return s;
        }
        cudaError_t e = launch_layer_decode(la, tm_w2, ld_grid, st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "decode layer launch");
    }

    // fused: the permutation computes indices only and GEMM1 gathers the rows
    const bool fused = gather_enabled();
    const PermuteOut po{offsets, perm_src, inv_perm, fused ? nullptr : x_perm};
    bool permuted = false;
    s = do_route(x, w_gate, bias, N, D, E, K, mode, ids, w, nullptr, ws, at(L.gemm_scratch), L.gemm_scratch_bytes,
                 st, &po, &permuted);
    if (s != MOE_OK) return s;
    cudaError_t e = cudaSuccess;
    if (!permuted) {
        e = launch_permute(x, ids, N, D, E, K, offsets, perm_src, inv_perm, fused ? nullptr : x_perm,
                           static_cast<int32_t*>(at(L.perm_scratch)), ws_err(ws), st);
        if (e != cudaSuccess) return cuda_fail(e, "permute launch");
    }
    const GatherSrc gs{x, perm_src, static_cast<long long>(D) * 2, N};
    s = do_grouped_ffn(x_perm, offsets, rows, w1, w3, w2, E, D, Dff, act, h, y_perm, ws, at(L.gemm_scratch),
                       L.gemm_scratch_bytes, st, fused ? &gs : nullptr);
    if (s != MOE_OK) return s;
    e = launch_combine(y_perm, inv_perm, w, N, D, K, out, ws_err(ws), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine launch");
}

moe_status moe_permute_indices(const int32_t* topk_ids, int N, int E, int K, int32_t* expert_offsets,
                               int32_t* perm_src, int32_t* inv_perm, void* ws, size_t ws_bytes, void* stream) {
    moe_status s = check_sizes(N, 64, E, K, 64, false);
    if (s != MOE_OK) return s;
    REQUIRE_PTR(ws);
    if (ws_bytes < moe_workspace_size("permute", N, 64, E, K, 0)) return fail(MOE_ERR_WORKSPACE, "permute workspace");
    REQUIRE_PTR(expert_offsets);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        cudaError_t e = cudaMemsetAsync(expert_offsets, 0, (E + 1) * sizeof(int32_t), st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "offsets memset");
    }
    REQUIRE_PTR(topk_ids);
    REQUIRE_PTR(perm_src);
    REQUIRE_PTR(inv_perm);
    int32_t* scratch = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kWsHeaderBytes);
    cudaError_t e = launch_permute(nullptr, topk_ids, N, 64, E, K, expert_offsets, perm_src, inv_perm, nullptr,
                                   scratch, ws_err(ws), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "permute launch");
}

moe_status moe_grouped_ffn_gathered(const moe_bf16* x, int N, const int32_t* perm_src,
                                    const int32_t* expert_offsets, int total_rows, const moe_bf16* w1,
                                    const moe_bf16* w3, const moe_bf16* w2, int E, int D, int Dff, int act,
                                    moe_bf16* h, moe_bf16* y_perm, void* ws, size_t ws_bytes, void* stream) {
    if (total_rows < 0 || N < 0) return fail(MOE_ERR_INVALID_ARG, "total_rows=%d N=%d", total_rows, N);
    moe_status s = check_sizes(total_rows, D, E, 1, Dff, true);
    if (s != MOE_OK) return s;
    if (act != MOE_ACT_SILU && act != MOE_ACT_SWIGLU) return fail(MOE_ERR_INVALID_ARG, "act=%d", act);
    REQUIRE_PTR(ws);
    if (ws_bytes < moe_workspace_size("ffn", total_rows, D, E, 1, Dff)) return fail(MOE_ERR_WORKSPACE, "ffn workspace");
    if (total_rows == 0) return MOE_OK;
    REQUIRE_PTR(x);
    REQUIRE_PTR(perm_src);
    REQUIRE_PTR(expert_offsets);
    REQUIRE_PTR(w1);
    if (act == MOE_ACT_SWIGLU) REQUIRE_PTR(w3);
    REQUIRE_PTR(w2);
    REQUIRE_PTR(h);
    REQUIRE_PTR(y_perm);
    const GatherSrc gs{x, perm_src, static_cast<long long>(D) * 2, N};
    return do_grouped_ffn(nullptr, expert_offsets, total_rows, w1, w3, w2, E, D, Dff, act, h, y_perm, ws,
                          static_cast<char*>(ws) + kWsHeaderBytes, ws_bytes - kWsHeaderBytes,
                          static_cast<cudaStream_t>(stream), &gs);
}

moe_status moe_grouped_ffn_e4m3_gathered(const uint8_t* xq, const float* x_scale, int N, const int32_t* perm_src,
                                         const int32_t* expert_offsets, int total_rows, const uint8_t* w1q,
                                         const float* w1_scale, const uint8_t* w3q, const float* w3_scale,
                                         const uint8_t* w2q, const float* w2_scale, int E, int D, int Dff, int act,
                                         moe_bf16* h, uint8_t* hq, float* h_scale, moe_bf16* y_perm, void* ws,
                                         size_t ws_bytes, void* stream) {
    if (total_rows < 0 || N < 0) return fail(MOE_ERR_INVALID_ARG, "total_rows=%d N=%d", total_rows, N);
    moe_status s = check_sizes(total_rows, D, E, 1, Dff, true);
    if (s != MOE_OK) return s;
    s = check_e4m3_dims(D, Dff);
    if (s != MOE_OK) return s;
    if (act != MOE_ACT_SILU && act != MOE_ACT_SWIGLU) return fail(MOE_ERR_INVALID_ARG, "act=%d", act);
    REQUIRE_PTR(ws);
    if (ws_bytes < moe_workspace_size("ffn", total_rows, D, E, 1, Dff)) return fail(MOE_ERR_WORKSPACE, "ffn workspace");
    if (total_rows == 0) return MOE_OK;
    REQUIRE_PTR(xq);
    REQUIRE_PTR(x_scale);
    REQUIRE_PTR(perm_src);
    REQUIRE_PTR(expert_offsets);
    REQUIRE_PTR(w1q);
    REQUIRE_PTR(w1_scale);
    if (act == MOE_ACT_SWIGLU) {
        REQUIRE_PTR(w3q);
        REQUIRE_PTR(w3_scale);
    }
    REQUIRE_PTR(w2q);
    REQUIRE_PTR(w2_scale);
    REQUIRE_PTR(h);
    REQUIRE_PTR(hq);
    REQUIRE_PTR(h_scale);
    REQUIRE_PTR(y_perm);
    const GatherSrc gs{xq, perm_src, static_cast<long long>(D), N};
    return do_grouped_ffn_e4m3(nullptr, x_scale, perm_src, expert_offsets, total_rows, w1q, w1_scale, w3q, w3_scale,
                               w2q, w2_scale, E, D, Dff, act, h, hq, h_scale, y_perm, ws,
                               static_cast<char*>(ws) + kWsHeaderBytes, ws_bytes - kWsHeaderBytes,
                               static_cast<cudaStream_t>(stream), &gs);
}

moe_status moe_quantize_e4m3(const moe_bf16* src, long long rows, int cols, uint8_t* q, float* scale,
                             void* stream) {
    if (rows < 0) return fail(MOE_ERR_INVALID_ARG, "rows=%lld < 0", rows);
    if (cols < 16 || cols % 16) return fail(MOE_ERR_INVALID_ARG, "cols=%d not a positive multiple of 16", cols);
    if (rows * static_cast<long long>(cols) >= (1LL << 40)) return fail(MOE_ERR_INVALID_ARG, "rows*cols too large");
    if (rows == 0) return MOE_OK;
    REQUIRE_PTR(src);
    REQUIRE_PTR(q);
    REQUIRE_PTR(scale);
    cudaError_t e = launch_quant_rows_e4m3(src, rows, cols, q, scale, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "e4m3 quantisation launch");
}

moe_status moe_permute_e4m3(const uint8_t* xq, const int32_t* topk_ids, int N, int D, int E, int K,
                            int32_t* expert_offsets, int32_t* perm_src, int32_t* inv_perm, uint8_t* xq_perm,
                            void* ws, size_t ws_bytes, void* stream) {
    moe_status s = check_sizes(N, D, E, K, 64, false);
    if (s != MOE_OK) return s;
    if (D % 128) return fail(MOE_ERR_INVALID_ARG, "e4m3 path: D=%d not a multiple of 128", D);
    // an e4m3 row of D codes is moved as D/2 two-byte words by the bf16 row copy
    return moe_permute(reinterpret_cast<const moe_bf16*>(xq), topk_ids, N, D / 2, E, K, expert_offsets, perm_src,
                       inv_perm, reinterpret_cast<moe_bf16*>(xq_perm), ws, ws_bytes, stream);
}

moe_status moe_grouped_ffn_e4m3(const uint8_t* xq_perm, const float* x_scale, const int32_t* x_scale_index,
                                const int32_t* expert_offsets, int total_rows, const uint8_t* w1q,
                                const float* w1_scale, const uint8_t* w3q, const float* w3_scale,
                                const uint8_t* w2q, const float* w2_scale, int E, int D, int Dff, int act,
                                moe_bf16* h, uint8_t* hq, float* h_scale, moe_bf16* y_perm, void* ws,
                                size_t ws_bytes, void* stream) {
    if (total_rows < 0) return fail(MOE_ERR_INVALID_ARG, "total_rows=%d < 0", total_rows);
    moe_status s = check_sizes(total_rows, D, E, 1, Dff, true);
    if (s != MOE_OK) return s;
    s = check_e4m3_dims(D, Dff);
    if (s != MOE_OK) return s;
    if (act != MOE_ACT_SILU && act != MOE_ACT_SWIGLU) return fail(MOE_ERR_INVALID_ARG, "act=%d", act);
    REQUIRE_PTR(ws);
    if (ws_bytes < moe_workspace_size("ffn", total_rows, D, E, 1, Dff)) return fail(MOE_ERR_WORKSPACE, "ffn workspace");
    if (total_rows == 0) return MOE_OK;
    REQUIRE_PTR(xq_perm);
    REQUIRE_PTR(x_scale);
    OPTIONAL_PTR(x_scale_index);
    REQUIRE_PTR(expert_offsets);
    REQUIRE_PTR(w1q);
    REQUIRE_PTR(w1_scale);
    if (act == MOE_ACT_SWIGLU) {
        REQUIRE_PTR(w3q);
        REQUIRE_PTR(w3_scale);
    }
    REQUIRE_PTR(w2q);
    REQUIRE_PTR(w2_scale);
    REQUIRE_PTR(h);
    REQUIRE_PTR(hq);
    REQUIRE_PTR(h_scale);
    REQUIRE_PTR(y_perm);
    return do_grouped_ffn_e4m3(xq_perm, x_scale, x_scale_index, expert_offsets, total_rows, w1q, w1_scale, w3q,
                               w3_scale, w2q, w2_scale, E, D, Dff, act, h, hq, h_scale, y_perm, ws,
                               static_cast<char*>(ws) + kWsHeaderBytes, ws_bytes - kWsHeaderBytes,
                               static_cast<cudaStream_t>(stream));
}

int moe_layer_e4m3_workspace_layout(int N, int D, int E, int K, int Dff, size_t out[12]) {
    if (out == nullptr || check_sizes(N, D, E, K, Dff, true) != MOE_OK || D % 128 || Dff % 128) return -1;
    const E4m3Layout L = e4m3_layout(N, D, E, K, Dff);
    const size_t v[12] = {L.ids, L.w, L.offsets, L.perm_src, L.inv_perm, L.xq,
                          L.x_scale, L.xq_perm, L.h, L.hq, L.h_scale, L.y_perm};
    for (int i = 0; i < 12; ++i) out[i] = v[i];
    return 0;
}

moe_status moe_layer_forward_e4m3(const moe_bf16* x, const moe_bf16* w_gate, const float* bias, const uint8_t* w1q,
                                  const float* w1_scale, const uint8_t* w3q, const float* w3_scale,
                                  const uint8_t* w2q, const float* w2_scale, int N, int D, int E, int K, int Dff,
                                  int mode, int act, moe_bf16* out, void* ws, size_t ws_bytes, void* stream) {
    moe_status s = check_sizes(N, D, E, K, Dff, true);
    if (s != MOE_OK) return s;
    s = check_e4m3_dims(D, Dff);
    if (s != MOE_OK) return s;
    if (mode != MOE_SCORE_SOFTMAX_TOPK && mode != MOE_SCORE_SIGMOID_NORM)
        return fail(MOE_ERR_INVALID_ARG, "mode=%d", mode);
    if (act != MOE_ACT_SILU && act != MOE_ACT_SWIGLU) return fail(MOE_ERR_INVALID_ARG, "act=%d", act);
    REQUIRE_PTR(ws);
    const E4m3Layout L = e4m3_layout(N, D, E, K, Dff);
    if (ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "e4m3 layer workspace needs %zu bytes", L.total);
    if (N == 0) return MOE_OK;
    REQUIRE_PTR(x);
    REQUIRE_PTR(w_gate);
    REQUIRE_PTR(w1q);
    REQUIRE_PTR(w1_scale);
    if (act == MOE_ACT_SWIGLU) {
        REQUIRE_PTR(w3q);
        REQUIRE_PTR(w3_scale);
    }
    REQUIRE_PTR(w2q);
    REQUIRE_PTR(w2_scale);
    REQUIRE_PTR(out);
    OPTIONAL_PTR(bias);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    auto at = [&](size_t off) { return static_cast<void*>(base + off); };
    int32_t* ids = static_cast<int32_t*>(at(L.ids));
    float* w = static_cast<float*>(at(L.w));
    int32_t* offsets = static_cast<int32_t*>(at(L.offsets));
    int32_t* perm_src = static_cast<int32_t*>(at(L.perm_src));
    int32_t* inv_perm = static_cast<int32_t*>(at(L.inv_perm));
    uint8_t* xq = static_cast<uint8_t*>(at(L.xq));
    float* x_scale = static_cast<float*>(at(L.x_scale));
    uint8_t* xq_perm = static_cast<uint8_t*>(at(L.xq_perm));
    moe_bf16* h = static_cast<moe_bf16*>(at(L.h));
    uint8_t* hq = static_cast<uint8_t*>(at(L.hq));
    float* h_scale = static_cast<float*>(at(L.h_scale));
    moe_bf16* y_perm = static_cast<moe_bf16*>(at(L.y_perm));
    const int rows = N * K;

    // a small decode batch: the whole layer in one launch (its GEMMs read
    // the weights in 32-byte pieces)
    const int ld_grid = layer_decode_grid(N, D, E, K, Dff, act, true);
    if (ld_grid > 0 && L.gemm_scratch_bytes >= static_cast<size_t>(N) * E * sizeof(float) && aligned32(w1q) &&
        aligned32(w2q) && (act != MOE_ACT_SWIGLU || aligned32(w3q))) {
        LayerDecodeArgs la{};
        la.x = reinterpret_cast<const uint16_t*>(x);
        la.wg = reinterpret_cast<const uint16_t*>(w_gate);
        la.bias = bias;
        la.N = N;
        la.D = D;
        la.E = E;
        la.K = K;
        la.Dff = Dff;
        la.mode = mode;
        la.logits = static_cast<float*>(at(L.gemm_scratch));
        la.ids = ids;
        la.w = w;
        la.offsets = offsets;
        la.perm_src = perm_src;
        la.inv_perm = inv_perm;
        la.h = reinterpret_cast<uint16_t*>(h);
        la.y_perm = reinterpret_cast<uint16_t*>(y_perm);
        la.out = reinterpret_cast<uint16_t*>(out);
        la.err = ws_err(ws);
        la.dbg = ws_dbg(ws);
        la.bar = reinterpret_cast<unsigned long long*>(base + kWsBarrierCount);
        la.l2_prefetch_max = layer_decode_prefetch_bytes();
        la.w2_smem = layer_decode_w2_smem(N, D, E, K, Dff, act, true);
        la.fp8 = 1;
        la.w1q = w1q;
        la.w3q = act == MOE_ACT_SWIGLU ? w3q : nullptr;
        la.w2q = w2q;
        la.s1 = w1_scale;
        la.s3 = act == MOE_ACT_SWIGLU ? w3_scale : nullptr;
        la.s2 = w2_scale;
        la.xq = xq;
        la.x_scale = x_scale;
        la.xq_perm = xq_perm;
        la.hq = hq;
        la.h_scale = h_scale;
        CUtensorMap tm_w2{};
        if (la.w2_smem) {
            s = make_tmap3d(&tm_w2, w2q, static_cast<long long>(E) * D, Dff, kLayerDecodeW2Rows, Dff / 128, true);
            if (s != MOE_OK) return s;
        }
        cudaError_t e = launch_layer_decode(la, tm_w2, ld_grid, st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "decode layer launch");
    }

    s = do_route(x, w_gate, bias, N, D, E, K, mode, ids, w, nullptr, ws, at(L.gemm_scratch), L.gemm_scratch_bytes,
                 st);
    if (s != MOE_OK) return s;
    // tokens -> e4m3 once (one scale per token), then the permutation moves codes
    cudaError_t e = launch_quant_rows_e4m3(x, N, D, xq, x_scale, st);
    if (e != cudaSuccess) return cuda_fail(e, "token quantisation launch");
    const bool fused = gather_enabled();
    e = launch_permute(reinterpret_cast<const uint16_t*>(xq), ids, N, D / 2, E, K, offsets, perm_src, inv_perm,
                       fused ? nullptr : reinterpret_cast<uint16_t*>(xq_perm),
                       static_cast<int32_t*>(at(L.perm_scratch)), ws_err(ws), st);
    if (e != cudaSuccess) return cuda_fail(e, "permute launch");
    const GatherSrc gs{xq, perm_src, static_cast<long long>(D), N};
    s = do_grouped_ffn_e4m3(xq_perm, x_scale, perm_src, offsets, rows, w1q, w1_scale, w3q, w3_scale, w2q, w2_scale,
                            E, D, Dff, act, h, hq, h_scale, y_perm, ws, at(L.gemm_scratch), L.gemm_scratch_bytes,
                            st, fused ? &gs : nullptr);
    if (s != MOE_OK) return s;
    e = launch_combine(y_perm, inv_perm, w, N, D, K, out, ws_err(ws), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine launch");
}

int moe_layer_launches_e4m3(int N, int D, int E, int K, int Dff, int act) {
    if (check_sizes(N, D, E, K, Dff, true) != MOE_OK || D % 128 || Dff % 128) return -1;
    if (N == 0) return 0;
    if (layer_decode_grid(N, D, E, K, Dff, act, true) > 0 &&
        e4m3_layout(N, D, E, K, Dff).gemm_scratch_bytes >= static_cast<size_t>(N) * E * sizeof(float))
        return 1;  // the whole layer in one launch
    const int rows = N * K;
    int n = 2;                                                  // router GEMM + top-K
    n += 1;                                                     // token quantisation
    n += (static_cast<long long>(rows) <= 4096) ? 1 : 3;        // permute
    const size_t avail = ffn_partial_bound(rows, D, E, Dff);
    const FfnPlan p = plan_ffn(rows, D, E, Dff, act == MOE_ACT_SWIGLU, sm_count(), avail, OpType<true>::KB);
    const bool fused = !gather_enabled() && use_fused_decode(p, act == MOE_ACT_SWIGLU, rows, true) &&
                       fused_decode_layout(rows, D, E, Dff, p.g1.splits, p.g2.splits, p.g1.tiles_ub,
                                           p.g2.tiles_ub).total <= avail;
    n += fused ? 1 : 2 + (p.g1.splits > 1) + (p.g2.splits > 1) + 1;  // GEMMs (+ reductions) + h quantisation
    return n + 1;                                                   // combine
}

moe_status moe_routing_stats(const int32_t* expert_offsets, int E, float decay, float bias_step, float* ema,
                             float* bias, float* kl_out, void* stream) {
    if (E < 1 || E > 1024) return fail(MOE_ERR_INVALID_ARG, "E=%d outside 1..1024", E);
    if (!(decay >= 0.0f && decay <= 1.0f)) return fail(MOE_ERR_INVALID_ARG, "decay outside [0, 1]");
    REQUIRE_PTR(expert_offsets);
    REQUIRE_PTR(ema);
    OPTIONAL_PTR(bias);
    if (kl_out != nullptr && (reinterpret_cast<uintptr_t>(kl_out) & 3u))
        return fail(MOE_ERR_INVALID_ARG, "kl_out not 4-byte aligned");
    cudaError_t e = launch_routing_stats(expert_offsets, E, decay, bias_step, ema, bias, kl_out,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "routing statistics launch");
}

int moe_layer_launches(int N, int D, int E, int K, int Dff, int act, int capacity) {
    if (check_sizes(N, D, E, K, Dff, true) != MOE_OK) return -1;
    if (N == 0) return 0;
    if (capacity < 0 && layer_decode_grid(N, D, E, K, Dff, act) > 0 &&
        layer_layout(N, D, E, K, Dff).gemm_scratch_bytes >= static_cast<size_t>(N) * E * sizeof(float))
        return 1;  // the whole layer in one launch
    const int nsm = sm_count();
    int n = 2;  // router GEMM + top-K
    const bool padded = capacity >= 0;
    if (!padded && fused_route_permute(N, K)) n += 0;                   // permute in the top-K launch
    else n += (!padded && static_cast<long long>(N) * K <= 4096) ? 1 : 3;  // permute
    const int rows = padded ? E * capacity : N * K;
    if (rows > 0) {
        const size_t avail = ffn_partial_bound(rows, D, E, Dff);
        const FfnPlan p = plan_ffn(rows, D, E, Dff, act == MOE_ACT_SWIGLU, nsm, avail);
        const bool fused = (padded || !gather_enabled()) && use_fused_decode(p, act == MOE_ACT_SWIGLU, rows) &&
                           fused_decode_layout(rows, D, E, Dff, p.g1.splits, p.g2.splits, p.g1.tiles_ub,
                                               p.g2.tiles_ub).total <= avail;
        n += fused ? 1 : 2 + (p.g1.splits > 1) + (p.g2.splits > 1);
    }
    return n + 1;  // combine
}

int moe_capacity(int N, int E, int K, float capacity_factor) {
    if (N < 0 || E < 1 || K < 1 || !(capacity_factor >= 0.0f)) return -1;
    const double c = std::ceil(static_cast<double>(capacity_factor) * N * K / E - 1e-9);
    return c > 2147483647.0 ? -1 : static_cast<int>(std::max(0.0, c));
}

size_t moe_workspace_size_padded(const char* op, int N, int D, int E, int K, int Dff, int capacity) {
    if (op == nullptr) return 0;
    if (!strcmp(op, "combine")) return kWsHeaderBytes;
    if (!strcmp(op, "permute")) {
        if (N < 0 || E < 1 || capacity < 0) return 0;
        return kWsHeaderBytes + align_up(permute_scratch_bytes(N, E), 256);
    }
    if (!strcmp(op, "layer")) {
        if (check_sizes(N, D, E, K, Dff, true) != MOE_OK || check_capacity(E, capacity, D, Dff) != MOE_OK) return 0;
        return padded_layout(N, D, E, K, Dff, capacity).total;
    }
    return 0;
}

int moe_layer_padded_workspace_layout(int N, int D, int E, int K, int Dff, int capacity, size_t out[8]) {
    if (out == nullptr || check_sizes(N, D, E, K, Dff, true) != MOE_OK ||
        check_capacity(E, capacity, D, Dff) != MOE_OK)
        return -1;
    const PaddedLayout L = padded_layout(N, D, E, K, Dff, capacity);
    out[0] = L.ids;
    out[1] = L.w;
    out[2] = L.pad_offsets;
    out[3] = L.kept;
    out[4] = L.slot;
    out[5] = L.x_pad;
    out[6] = L.h;
    out[7] = L.y_pad;
    return 0;
}

moe_status moe_permute_padded(const moe_bf16* x, const int32_t* topk_ids, int N, int D, int E, int K, int capacity,
                              int32_t* expert_offsets, int32_t* kept, int32_t* slot, moe_bf16* x_pad, void* ws,
                              size_t ws_bytes, void* stream) {
    moe_status s = check_sizes(N, D, E, K, 64, false);
    if (s != MOE_OK) return s;
    s = check_capacity(E, capacity, D, D);
    if (s != MOE_OK) return s;
    REQUIRE_PTR(ws);
    if (ws_bytes < moe_workspace_size_padded("permute", N, D, E, K, 0, capacity))
        return fail(MOE_ERR_WORKSPACE, "permute workspace");
    REQUIRE_PTR(expert_offsets);
    REQUIRE_PTR(kept);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        // every block is padding: offsets e*C, nothing kept, zero rows
        cudaError_t e = launch_pad_offsets(E, capacity, expert_offsets, kept, st);
        if (e == cudaSuccess && capacity > 0) {
            if (x_pad == nullptr) return fail(MOE_ERR_INVALID_ARG, "x_pad is NULL");
            e = cudaMemsetAsync(x_pad, 0, static_cast<size_t>(E) * capacity * D * 2, st);
        }
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "empty padded permute");
    }
    REQUIRE_PTR(x);
    REQUIRE_PTR(topk_ids);
    REQUIRE_PTR(slot);
    if (capacity > 0) REQUIRE_PTR(x_pad);
    int32_t* scratch = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kWsHeaderBytes);
    cudaError_t e = launch_permute_padded(x, topk_ids, N, D, E, K, capacity, expert_offsets, kept, slot, x_pad,
                                          scratch, ws_err(ws), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "padded permute launch");
}

moe_status moe_combine_padded(const moe_bf16* y_pad, const int32_t* slot, const float* topk_w, int N, int D, int K,
                              int E, int capacity, moe_bf16* out, void* ws, size_t ws_bytes, void* stream) {
    moe_status s = check_sizes(N, D, std::max(E, K), K, 64, false);
    if (s != MOE_OK) return s;
    s = check_capacity(E, capacity, D, D);
    if (s != MOE_OK) return s;
    REQUIRE_PTR(ws);
    if (ws_bytes < kWsHeaderBytes) return fail(MOE_ERR_WORKSPACE, "combine workspace");
    if (N == 0) return MOE_OK;
    if (capacity > 0) REQUIRE_PTR(y_pad);
    REQUIRE_PTR(slot);
    REQUIRE_PTR(topk_w);
    REQUIRE_PTR(out);
    cudaError_t e = launch_combine_rows(y_pad, slot, topk_w, N, D, K, static_cast<long long>(E) * capacity, true, out,
                                        ws_err(ws), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "padded combine launch");
}

moe_status moe_layer_forward_padded(const moe_bf16* x, const moe_bf16* w_gate, const float* bias, const moe_bf16* w1,
                                    const moe_bf16* w3, const moe_bf16* w2, int N, int D, int E, int K, int Dff,
                                    int mode, int act, int capacity, moe_bf16* out, void* ws, size_t ws_bytes,
                                    void* stream) {
    moe_status s = check_sizes(N, D, E, K, Dff, true);
    if (s != MOE_OK) return s;
    s = check_capacity(E, capacity, D, Dff);
    if (s != MOE_OK) return s;
    if (mode != MOE_SCORE_SOFTMAX_TOPK && mode != MOE_SCORE_SIGMOID_NORM)
        return fail(MOE_ERR_INVALID_ARG, "mode=%d", mode);
    if (act != MOE_ACT_SILU && act != MOE_ACT_SWIGLU) return fail(MOE_ERR_INVALID_ARG, "act=%d", act);
    REQUIRE_PTR(ws);
    const PaddedLayout L = padded_layout(N, D, E, K, Dff, capacity);
    if (ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "padded layer workspace needs %zu bytes", L.total);
    if (N == 0) return MOE_OK;
    REQUIRE_PTR(x);
    REQUIRE_PTR(w_gate);
    REQUIRE_PTR(w1);
    if (act == MOE_ACT_SWIGLU) REQUIRE_PTR(w3);
    REQUIRE_PTR(w2);
    REQUIRE_PTR(out);
    OPTIONAL_PTR(bias);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    auto at = [&](size_t off) { return static_cast<void*>(base + off); };
    int32_t* ids = static_cast<int32_t*>(at(L.ids));
    float* w = static_cast<float*>(at(L.w));
    int32_t* pad_off = static_cast<int32_t*>(at(L.pad_offsets));
    int32_t* kept = static_cast<int32_t*>(at(L.kept));
    int32_t* slot = static_cast<int32_t*>(at(L.slot));
    moe_bf16* x_pad = static_cast<moe_bf16*>(at(L.x_pad));
    moe_bf16* h = static_cast<moe_bf16*>(at(L.h));
    moe_bf16* y_pad = static_cast<moe_bf16*>(at(L.y_pad));
    const int rows = E * capacity;

    s = do_route(x, w_gate, bias, N, D, E, K, mode, ids, w, nullptr, ws, at(L.gemm_scratch), L.gemm_scratch_bytes, st);
    if (s != MOE_OK) return s;
    cudaError_t e = launch_permute_padded(x, ids, N, D, E, K, capacity, pad_off, kept, slot, x_pad,
                                          static_cast<int32_t*>(at(L.perm_scratch)), ws_err(ws), st);
    if (e != cudaSuccess) return cuda_fail(e, "padded permute launch");
    if (rows > 0) {
        s = do_grouped_ffn(x_pad, pad_off, rows, w1, w3, w2, E, D, Dff, act, h, y_pad, ws, at(L.gemm_scratch),
                           L.gemm_scratch_bytes, st);
        if (s != MOE_OK) return s;
    }
    e = launch_combine_rows(y_pad, slot, w, N, D, K, rows, true, out, ws_err(ws), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "padded combine launch");
}

moe_status moe_read_device_error(const void* ws, void* stream) {
    if (ws == nullptr) return fail(MOE_ERR_INVALID_ARG, "ws is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof word, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading device error word");
    if (word & MOE_DEVERR_TIMEOUT) return fail(MOE_ERR_DEVICE_TIMEOUT, "device wait timed out (word=0x%x)", word);
    if (word & MOE_DEVERR_BOUNDS) return fail(MOE_ERR_DEVICE_BOUNDS, "device bounds error (word=0x%x)", word);
    return MOE_OK;
}

moe_status moe_clear_device_error(void* ws, void* stream) {
    if (ws == nullptr) return fail(MOE_ERR_INVALID_ARG, "ws is NULL");
    cudaError_t e = cudaMemsetAsync(ws, 0, kWsHeaderBytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "clearing workspace header");
}

moe_status moe_set_debug_flags(void* ws, uint32_t flags, void* stream) {
    if (ws == nullptr) return fail(MOE_ERR_INVALID_ARG, "ws is NULL");
    // one 4-byte word: cudaMemsetAsync writes each byte, so store a flag set
    // whose bytes are all equal or use a memset per byte
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* p = static_cast<char*>(ws) + 4;
    for (int i = 0; i < 4; ++i) {
        cudaError_t e = cudaMemsetAsync(p + i, static_cast<int>((flags >> (8 * i)) & 0xffu), 1, st);
        if (e != cudaSuccess) return cuda_fail(e, "writing debug flags");
    }
    return MOE_OK;
}

}  // extern "C"
