// moe_api.cu -- the C ABI declared in include/moe.h: argument validation,
// workspace carving, TMA descriptor encoding and kernel launches.  No device
// memory is allocated here; every buffer belongs to the caller.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
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

// Row-major [rows, cols] bf16 matrix, box = [box_rows, 64 columns], 128-byte
// swizzle (the layout the tcgen05 shared-memory descriptors expect).
moe_status make_tmap(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) rows=%lld cols=%lld box=%d", (int)r, rows,
                    cols, box_rows);
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
    return MOE_OK;
}

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

// ---- layer workspace layout ----
struct LayerLayout {
    size_t ids, w, offsets, perm_src, inv_perm, x_perm, h, y_perm, perm_scratch, total;
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
    L.x_perm = take(A * D * 2);
    L.h = take(A * Dff * 2);
    L.y_perm = take(A * D * 2);
    L.total = o;
    return L;
}

// ---- stage implementations (no validation: callers validated) ----
int route_bn(int E) {
    if (E <= 32) return 32;
    if (E <= 64) return 64;
    if (E <= 128) return 128;
    return 256;
}

moe_status do_route(const moe_bf16* x, const moe_bf16* w_gate, const float* bias, int N, int D, int E, int K,
                    int mode, int32_t* ids, float* w, float* logits_out, void* ws, cudaStream_t st) {
    const int bn = route_bn(E);
    CUtensorMap tA, tB;
    moe_status s = make_tmap(&tA, x, N, D, kBM);
    if (s != MOE_OK) return s;
    s = make_tmap(&tB, w_gate, E, D, bn);
    if (s != MOE_OK) return s;
    GemmArgs a{};
    a.group_offsets = nullptr;
    a.G = 1;
    a.M = N;
    a.n_out = E;
    a.k_dim = D;
    a.b_rows_per_group = 0;
    a.err = ws_err(ws);
    a.dbg = ws_dbg(ws);
    a.bias = bias;
    a.E = E;
    a.K = K;
    a.mode = mode;
    a.topk_ids = ids;
    a.topk_w = w;
    a.logits_out = logits_out;
    const int tiles = (N + kBM - 1) / kBM;
    const int grid = std::min(tiles, sm_count());
    cudaError_t e = launch_grouped_gemm(EPI_ROUTER, bn, tA, tB, tB, a, grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    return MOE_OK;
}

// Largest N tile (<= 256) whose output-column width divides n_out.
int ffn_bn(int n_out, bool swiglu) {
    const int cands[3] = {256, 128, 64};
    for (int bn : cands) {
        const int per = swiglu ? bn / 2 : bn;
        if (n_out % per == 0) return bn;
    }
    return 64;
}

moe_status do_grouped_ffn(const moe_bf16* x_perm, const int32_t* offsets, int rows, const moe_bf16* w1,
                          const moe_bf16* w3, const moe_bf16* w2, int E, int D, int Dff, int act, moe_bf16* h,
                          moe_bf16* y, void* ws, cudaStream_t st) {
    const bool swiglu = act == MOE_ACT_SWIGLU;
    const int nsm = sm_count();
    // ---- GEMM1 (+ activation): [rows, D] x [E*Dff, D]^T -> h [rows, Dff]
    {
        const int bn = ffn_bn(Dff, swiglu);
        const int box_b = swiglu ? bn / 2 : bn;
        CUtensorMap tA, tB, tB2;
        moe_status s = make_tmap(&tA, x_perm, rows, D, kBM);
        if (s == MOE_OK) s = make_tmap(&tB, w1, static_cast<long long>(E) * Dff, D, box_b);
        if (s == MOE_OK) s = make_tmap(&tB2, swiglu ? w3 : w1, static_cast<long long>(E) * Dff, D, box_b);
        if (s != MOE_OK) return s;
        GemmArgs a{};
        a.group_offsets = offsets;
        a.G = E;
        a.M = rows;
        a.n_out = Dff;
        a.k_dim = D;
        a.b_rows_per_group = Dff;
        a.out = h;
        a.ldo = Dff;
        a.err = ws_err(ws);
        a.dbg = ws_dbg(ws);
        const int per = swiglu ? bn / 2 : bn;
        const long long nt = (Dff + per - 1) / per;
        const long long ub = (static_cast<long long>(rows) / kBM + std::min<long long>(E, rows)) * nt;
        const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(ub, nsm)));
        cudaError_t e = launch_grouped_gemm(swiglu ? EPI_SWIGLU_BF16 : EPI_SILU_BF16, bn, tA, tB, tB2, a, grid, st);
        if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM1 launch");
    }
    // ---- GEMM2: [rows, Dff] x [E*D, Dff]^T -> y [rows, D]
    {
        const int bn = ffn_bn(D, false);
        CUtensorMap tA, tB;
        moe_status s = make_tmap(&tA, h, rows, Dff, kBM);
        if (s == MOE_OK) s = make_tmap(&tB, w2, static_cast<long long>(E) * D, Dff, bn);
        if (s != MOE_OK) return s;
        GemmArgs a{};
        a.group_offsets = offsets;
        a.G = E;
        a.M = rows;
        a.n_out = D;
        a.k_dim = Dff;
        a.b_rows_per_group = D;
        a.out = y;
        a.ldo = D;
        a.err = ws_err(ws);
        a.dbg = ws_dbg(ws);
        const long long nt = (D + bn - 1) / bn;
        const long long ub = (static_cast<long long>(rows) / kBM + std::min<long long>(E, rows)) * nt;
        const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(ub, nsm)));
        cudaError_t e = launch_grouped_gemm(EPI_STORE_BF16, bn, tA, tB, tB, a, grid, st);
        if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM2 launch");
    }
    return MOE_OK;
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
    if (!strcmp(op, "route") || !strcmp(op, "combine") || !strcmp(op, "ffn")) return kWsHeaderBytes;
    if (!strcmp(op, "permute")) {
        if (N < 0 || E < 1) return 0;
        return kWsHeaderBytes + align_up(permute_scratch_bytes(N, E), 256);
    }
    if (!strcmp(op, "layer")) {
        if (check_sizes(N, D, E, K, Dff, true) != MOE_OK) return 0;
        return layer_layout(N, D, E, K, Dff).total;
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
    if (E > 256) return fail(MOE_ERR_UNSUPPORTED, "route supports E <= 256 (got %d)", E);
    return do_route(x, w_gate, bias, N, D, E, K, mode, topk_ids, topk_w, logits_out, ws,
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
    if (E > 256) return fail(MOE_ERR_UNSUPPORTED, "route supports E <= 256 (got %d)", E);
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

    s = do_route(x, w_gate, bias, N, D, E, K, mode, ids, w, nullptr, ws, st);
    if (s != MOE_OK) return s;
    cudaError_t e = launch_permute(x, ids, N, D, E, K, offsets, perm_src, inv_perm, x_perm,
                                   static_cast<int32_t*>(at(L.perm_scratch)), ws_err(ws), st);
    if (e != cudaSuccess) return cuda_fail(e, "permute launch");
    s = do_grouped_ffn(x_perm, offsets, rows, w1, w3, w2, E, D, Dff, act, h, y_perm, ws, st);
    if (s != MOE_OK) return s;
    e = launch_combine(y_perm, inv_perm, w, N, D, K, out, ws_err(ws), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine launch");
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
