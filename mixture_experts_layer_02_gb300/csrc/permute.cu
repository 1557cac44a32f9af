// permute.cu -- contiguous per-expert permutation of token rows.
//
// "MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im), 第二层
// 范式 A Step 1: tokens are regrouped into one contiguous buffer with one
// segment per expert, each segment in token order, plus expert_offsets (the
// prefix sum of per-expert counts); the page's "优化亮点" does the regrouping
// with one scatter/gather pass over HBM.  The count -> prefix sum -> pack order
// is the same one "MoE 大规模分布式推理工程实战" (ybb.press), 2.2 uses to pack
// tokens per destination.
//
// Three launches (one, perm_small_kernel, when N*K <= 4096):
//   1. count    one CTA per block of 16 tokens: per-expert histogram of its
//               assignments, stored as counts[e][block]
//   2. scan     one CTA per expert: exclusive prefix over blocks, in place;
//               total[e] = the expert's row count
//   3. scatter  one CTA per block of tokens: exclusive prefix of totals ->
//               expert base (CTA 0 also stores expert_offsets), stable ranks
//               of the block's assignments in (t, k) order, perm_src /
//               inv_perm, then the bf16 row copy: each token row is read once
//               (16-byte loads) and written to its K destination rows.
// The rank of an assignment only depends on (t, k) order, so the result is
// deterministic and identical to a sequential token-major placement.
#include <algorithm>

#include "device.cuh"

namespace moe {

constexpr int kPermThreads = 256;
constexpr long long kSmallPermAssignments = 4096;  // one-launch path up to this many (t, k)

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// Exclusive scan of one int per thread across a 256-thread block.  Returns the
// exclusive prefix; *total receives the block sum.  `ws8` = 8 ints of shared.
__device__ __forceinline__ int block_excl_scan(int v, int* ws8, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int incl = warp_incl_scan(v, lane);
    if (lane == 31) ws8[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = (lane < kPermThreads / 32) ? ws8[lane] : 0;
        s = warp_incl_scan(s, lane);
        if (lane < kPermThreads / 32) ws8[lane] = s;
    }
    __syncthreads();
    const int before = (warp ? ws8[warp - 1] : 0) + incl - v;
    *total = ws8[kPermThreads / 32 - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kPermThreads)
perm_count_kernel(const int32_t* __restrict__ ids, int N, int E, int K, int nblk,
                  int32_t* __restrict__ counts, uint32_t* err) {
    extern __shared__ int hist[];  // [E]
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    pdl_wait();
    __syncthreads();
    const long long a0 = static_cast<long long>(blockIdx.x) * kPermTokensPerBlock * K;
    const long long a1 = min(static_cast<long long>(N) * K, a0 + kPermTokensPerBlock * K);
    bool bad = false;
    for (long long a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
        const int e = ids[a];
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&hist[e], 1);
        else bad = true;
    }
    if (bad) record_error(err, MOE_DEVERR_BOUNDS);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        counts[static_cast<long long>(e) * nblk + blockIdx.x] = hist[e];
    pdl_trigger();
}

__global__ void __launch_bounds__(kPermThreads)
perm_scan_kernel(int32_t* __restrict__ counts, int nblk, int32_t* __restrict__ totals) {
    __shared__ int ws8[kPermThreads / 32];
    int32_t* row = counts + static_cast<long long>(blockIdx.x) * nblk;
    int carry = 0;
    pdl_wait();
    for (int base = 0; base < nblk; base += kPermThreads) {
        const int i = base + threadIdx.x;
        const int v = (i < nblk) ? row[i] : 0;
        int sum;
        const int before = block_excl_scan(v, ws8, &sum);
        if (i < nblk) row[i] = carry + before;
        carry += sum;
    }
    if (threadIdx.x == 0) totals[blockIdx.x] = carry;
    pdl_trigger();
}

// Steps shared by both scatter kernels, for the block of tokens t0 .. t0+ntok-1
// once s_base[e] holds the first free row of expert e for this block.
// (a) stable ranks of the block's assignments in (t, k) order, 32 at a time
//     by warp 0 -> perm_src, inv_perm, s_dst
__device__ __forceinline__ void place_block(const int32_t* __restrict__ ids, int t0, int ntok, int E, int K,
                                            int* s_base, int* s_dst, int32_t* __restrict__ perm_src,
                                            int32_t* __restrict__ inv_perm, bool write_indices = true) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long a0 = static_cast<long long>(t0) * K;
    const int na = ntok * K;
    if (warp == 0) {
        const unsigned lt = (1u << lane) - 1u;
        for (int base = 0; base < na; base += 32) {
            const int i = base + lane;
            const bool act = i < na;
            const int e = act ? ids[a0 + i] : -1;
            const bool ok = act && static_cast<unsigned>(e) < static_cast<unsigned>(E);
            const int key = ok ? e : -1 - lane;  // invalid lanes never share a key
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            const int rank = __popc(peers & lt);
            const int r = ok ? s_base[e] + rank : -1;
            __syncwarp();
            if (ok && rank == 0) s_base[e] += __popc(peers);
            __syncwarp();
            if (act) {
                s_dst[i] = r;
                if (write_indices) {
                    inv_perm[a0 + i] = r;
                    if (ok) perm_src[r] = t0 + i / K;
                }
            }
        }
    }
}

// (b) row copy: (token, 16-byte chunk) pairs spread over the whole CTA; each
//     token row is read once and written to its K destination rows.  Only
//     chunks [c_lo, c_hi) of each row (a column slice; the whole row by
//     default).  No copy when x_perm is null (index-only permutation: GEMM1
//     gathers the rows).
__device__ __forceinline__ void copy_block(const uint16_t* __restrict__ x, int t0, int ntok, int D, int K,
                                           const int* s_dst, uint16_t* __restrict__ x_perm, int c_lo = 0,
                                           int c_hi = -1) {
    if (x_perm == nullptr) return;
    if (c_hi < 0) c_hi = D / 8;
    const int w = c_hi - c_lo;  // chunks per row in this slice
    const int items = ntok * w;
    constexpr int U = 4;  // chunks in flight per thread
    for (int base = threadIdx.x; base < items; base += U * kPermThreads) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int it = base + u * kPermThreads;
            if (it < items) {
                const int tl = it / w;
                v[u] = __ldg(reinterpret_cast<const uint4*>(x + static_cast<long long>(t0 + tl) * D) + c_lo +
                             (it - tl * w));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int it = base + u * kPermThreads;
            if (it < items) {
                const int tl = it / w;
                const int c = c_lo + (it - tl * w);
                for (int k = 0; k < K; ++k) {
                    const int r = s_dst[tl * K + k];
                    if (r >= 0) reinterpret_cast<uint4*>(x_perm + static_cast<long long>(r) * D)[c] = v[u];
                }
            }
        }
    }
}

// Expert bases: exclusive prefix of totals (each thread a run of experts);
// s_base[e] = offsets[e] + extra[e]; block 0 stores expert_offsets.
__device__ __forceinline__ void expert_bases(const int* totals, const int* extra, long long extra_stride,
                                             int E, int* s_base, int* ws8, int32_t* __restrict__ offsets,
                                             bool store) {
    const int per = (E + kPermThreads - 1) / kPermThreads;
    const int e0 = threadIdx.x * per;
    int run = 0;
    for (int i = 0; i < per; ++i)
        if (e0 + i < E) run += totals[e0 + i];
    int all;
    int before = block_excl_scan(run, ws8, &all);
    for (int i = 0; i < per; ++i) {
        const int e = e0 + i;
        if (e < E) {
            if (store) offsets[e] = before;
            s_base[e] = before + extra[e * extra_stride];
            before += totals[e];
        }
    }
    if (store && threadIdx.x == 0) offsets[E] = all;
    __syncthreads();
}

// Grid (token blocks, column slices): every slice of a block places the
// block's assignments the same way in shared memory, slice 0 alone stores the
// indices, and each slice copies its columns of the rows.  Slices keep enough
// CTAs per SM when there are few token blocks, so the row copies spread
// evenly over the SMs.
__global__ void __launch_bounds__(kPermThreads)
perm_scatter_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ ids, int N, int D,
                    int E, int K, int nblk, const int32_t* __restrict__ counts,
                    const int32_t* __restrict__ totals, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ perm_src, int32_t* __restrict__ inv_perm,
                    uint16_t* __restrict__ x_perm, uint32_t* err) {
    extern __shared__ int sm[];
    int* s_base = sm;                                  // [E] next free row per expert
    int* s_dst = sm + E;                               // [tokens*K] destination rows
    __shared__ int ws8[kPermThreads / 32];
    const int b = blockIdx.x;
    const int slice = blockIdx.y, nslices = gridDim.y;
    pdl_wait();
    expert_bases(totals, counts + b, nblk, E, s_base, ws8, offsets, b == 0 && slice == 0);
    const int t0 = b * kPermTokensPerBlock;
    const int ntok = min(kPermTokensPerBlock, N - t0);
    place_block(ids, t0, ntok, E, K, s_base, s_dst, perm_src, inv_perm, slice == 0);
    __syncthreads();
    const int cpr = D / 8;
    copy_block(x, t0, ntok, D, K, s_dst, x_perm, slice * cpr / nslices, (slice + 1) * cpr / nslices);
    pdl_trigger();
}

// The whole permutation in one launch for small calls (N*K <= kSmallPermAssignments):
// every block counts all assignments itself (the ones before its tokens and
// all of them) instead of reading per-block histograms from scratch.  Blocks
// take `tpb` tokens each (at most kPermTokensPerBlock), few enough that the
// row copies of a decode-sized call spread over the SMs.
__global__ void __launch_bounds__(kPermThreads)
perm_small_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ ids, int N, int D, int E,
                  int K, int tpb, int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
                  int32_t* __restrict__ inv_perm, uint16_t* __restrict__ x_perm, uint32_t* err) {
    extern __shared__ int sm[];
    int* s_before = sm;            // [E] assignments to e before this block's tokens
    int* s_total = sm + E;         // [E] all assignments to e
    int* s_base = sm + 2 * E;      // [E]
    int* s_dst = sm + 3 * E;       // [tokens*K]
    __shared__ int ws8[kPermThreads / 32];
    for (int e = threadIdx.x; e < E; e += kPermThreads) {
        s_before[e] = 0;
        s_total[e] = 0;
    }
    pdl_wait();
    __syncthreads();
    const int t0 = blockIdx.x * tpb;
    const long long a0 = static_cast<long long>(t0) * K;
    const long long na = static_cast<long long>(N) * K;
    bool bad = false;
    for (long long a = threadIdx.x; a < na; a += kPermThreads) {
        const int e = ids[a];
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
            atomicAdd(&s_total[e], 1);
            if (a < a0) atomicAdd(&s_before[e], 1);
        } else {
            bad = true;
        }
    }
    if (bad && blockIdx.x == 0) record_error(err, MOE_DEVERR_BOUNDS);
    __syncthreads();
    expert_bases(s_total, s_before, 1, E, s_base, ws8, offsets, blockIdx.x == 0);
    const int ntok = min(tpb, N - t0);
    place_block(ids, t0, ntok, E, K, s_base, s_dst, perm_src, inv_perm);
    __syncthreads();
    copy_block(x, t0, ntok, D, K, s_dst, x_perm);
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Paradigm B ("MoE 推理完整机制", 第二层 范式 B): every expert owns a fixed
// block of C rows, e*C .. e*C+C-1, filled in token order; assignments past
// the block are dropped (slot -1); unused rows of a block are zero.  Uses the
// same count and scan launches as the contiguous permutation.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPermThreads)
perm_padded_scatter_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ ids, int N, int D, int E,
                           int K, int C, int nblk, const int32_t* __restrict__ counts,
                           const int32_t* __restrict__ totals, int32_t* __restrict__ pad_offsets,
                           int32_t* __restrict__ kept, int32_t* __restrict__ slot, uint16_t* __restrict__ x_pad) {
    extern __shared__ int sm[];
    int* s_base = sm;           // [E] next row of expert e's block for this block of tokens
    int* s_dst = sm + E;        // [tokens*K]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = blockIdx.x;
    pdl_wait();
    for (int e = threadIdx.x; e < E; e += kPermThreads) {
        s_base[e] = e * C + counts[static_cast<long long>(e) * nblk + b];
        if (b == 0) kept[e] = min(totals[e], C);
    }
    if (b == 0)
        for (int e = threadIdx.x; e <= E; e += kPermThreads) pad_offsets[e] = e * C;
    __syncthreads();
    const int t0 = b * kPermTokensPerBlock;
    const int ntok = min(kPermTokensPerBlock, N - t0);
    const long long a0 = static_cast<long long>(t0) * K;
    const int na = ntok * K;
    if (warp == 0) {  // stable ranks in (t, k) order; past the block -> dropped
        const unsigned lt = (1u << lane) - 1u;
        for (int base = 0; base < na; base += 32) {
            const int i = base + lane;
            const bool act = i < na;
            const int e = act ? ids[a0 + i] : -1;
            const bool ok = act && static_cast<unsigned>(e) < static_cast<unsigned>(E);
            const int key = ok ? e : -1 - lane;
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            const int rank = __popc(peers & lt);
            int r = -1;
            if (ok) {
                r = s_base[e] + rank;
                if (r >= (e + 1) * C) r = -1;
            }
            __syncwarp();
            if (ok && rank == 0) s_base[e] += __popc(peers);
            __syncwarp();
            if (act) {
                s_dst[i] = r;
                slot[a0 + i] = r;
            }
        }
    }
    __syncthreads();
    copy_block(x, t0, ntok, D, K, s_dst, x_pad);
    // zero the unused rows: this CTA takes an even share of all E*C rows, one
    // warp per row; a row past its block's kept count is cleared
    const int cpr = D / 8;
    const long long R = static_cast<long long>(E) * C;
    const long long q0 = R * b / nblk, q1 = R * (b + 1) / nblk;
    for (long long row = q0 + warp; row < q1; row += kPermThreads / 32) {
        const int e = static_cast<int>(row / C);
        if (row - static_cast<long long>(e) * C < min(totals[e], C)) continue;
        uint4* dst = reinterpret_cast<uint4*>(x_pad + row * D);
        for (int c = lane; c < cpr; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
    }
    pdl_trigger();
}

// The padded buffer of an empty batch: offsets e*C, nothing kept.
__global__ void pad_offsets_kernel(int E, int C, int32_t* __restrict__ pad_offsets, int32_t* __restrict__ kept) {
    pdl_wait();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        pad_offsets[e] = e * C;
        if (e < E) kept[e] = 0;
    }
    pdl_trigger();
}

cudaError_t launch_pad_offsets(int E, int C, int32_t* pad_offsets, int32_t* kept, cudaStream_t st) {
    return launch_kernel(pad_offsets_kernel, dim3(1), dim3(256), 0, st, E, C, pad_offsets, kept);
}

cudaError_t launch_permute_padded(const uint16_t* x, const int32_t* ids, int N, int D, int E, int K, int C,
                                  int32_t* pad_offsets, int32_t* kept, int32_t* slot, uint16_t* x_pad,
                                  int32_t* scratch, uint32_t* err, cudaStream_t st) {
    const int nblk = (N + kPermTokensPerBlock - 1) / kPermTokensPerBlock;
    int32_t* counts = scratch;
    int32_t* totals = scratch + static_cast<long long>(nblk) * E;
    cudaError_t e = launch_kernel(perm_count_kernel, dim3(nblk), dim3(kPermThreads), E * sizeof(int), st, ids, N, E,
                                  K, nblk, counts, err);
    if (e == cudaSuccess)
        e = launch_kernel(perm_scan_kernel, dim3(E), dim3(kPermThreads), 0, st, counts, nblk, totals);
    const size_t smem = (E + kPermTokensPerBlock * K) * sizeof(int);
    if (e == cudaSuccess)
        e = launch_kernel(perm_padded_scatter_kernel, dim3(nblk), dim3(kPermThreads), smem, st, x, ids, N, D, E, K,
                          C, nblk, counts, totals, pad_offsets, kept, slot, x_pad);
    return e;
}

size_t permute_scratch_bytes(int N, int E) {
    const long long nblk = (static_cast<long long>(N) + kPermTokensPerBlock - 1) / kPermTokensPerBlock;
    return static_cast<size_t>((nblk * E + E) * sizeof(int32_t));
}

static int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

cudaError_t launch_permute(const uint16_t* x, const int32_t* ids, int N, int D, int E, int K,
                           int32_t* offsets, int32_t* perm_src, int32_t* inv_perm,
                           uint16_t* x_perm, int32_t* scratch, uint32_t* err, cudaStream_t st) {
    const int nblk = (N + kPermTokensPerBlock - 1) / kPermTokensPerBlock;
    if (static_cast<long long>(N) * K <= kSmallPermAssignments) {
        // one token per block up to one block per SM, then just enough tokens per block
        const int nsm = std::max(1, device_sm_count());
        const int tpb = std::min(kPermTokensPerBlock, std::max(1, (N + nsm - 1) / nsm));
        const int grid = std::max(1, (N + tpb - 1) / tpb);
        const size_t smem = (3 * E + tpb * K) * sizeof(int);
        return launch_kernel(perm_small_kernel, dim3(grid), dim3(kPermThreads), smem, st, x, ids, N, D, E, K, tpb,
                             offsets, perm_src, inv_perm, x_perm, err);
    }
    int32_t* counts = scratch;                                   // [E][nblk]
    int32_t* totals = scratch + static_cast<long long>(nblk) * E;  // [E]
    cudaError_t e = launch_kernel(perm_count_kernel, dim3(nblk), dim3(kPermThreads), E * sizeof(int), st, ids, N, E,
                                  K, nblk, counts, err);
    if (e == cudaSuccess)
        e = launch_kernel(perm_scan_kernel, dim3(E), dim3(kPermThreads), 0, st, counts, nblk, totals);
    const size_t smem = (E + kPermTokensPerBlock * K) * sizeof(int);
    // column slices: about four CTAs per SM at least, each slice >= 64 chunks (1 KB) of a row
    const int nsm = std::max(1, device_sm_count());
    const int max_slices = std::max(1, D / 8 / 64);
    const int nslices = (x_perm == nullptr) ? 1 : std::min(max_slices, std::max(1, (4 * nsm + nblk - 1) / nblk));
    if (e == cudaSuccess)
        e = launch_kernel(perm_scatter_kernel, dim3(nblk, nslices), dim3(kPermThreads), smem, st, x, ids, N, D, E, K,
                          nblk, counts, totals, offsets, perm_src, inv_perm, x_perm, err);
    return e;
}

}  // namespace moe

// ============================================================================
// moe_permute_static_scratch -- the permutation without a caller workspace.
//
// moe_permute needs a few bytes of scratch per (expert, block of 16 tokens)
// for its per-block histograms.  Some callers cannot hand it a workspace:
// runtimes that plan every device buffer ahead of time and forbid allocation
// while the model runs (a plugin's enqueue step in a pre-built inference
// engine, a serving loop on a fixed memory budget), or code paths where a
// cudaMalloc would stall on an implicit device synchronisation.  This entry
// point keeps that scratch in a fixed array of device global memory owned by
// the library instead: kStaticPermuteScratchInts int32 values (4 MiB), which
// every GPU that loads the library holds until the process exits.
// ============================================================================
#include <cstdio>
#include <mutex>

#include "../../include/moe.h"

namespace moe {

constexpr long long kStaticPermuteScratchInts = 1LL << 20;  // 4 MiB

// Shared by every call on a device; the histogram kernel rewrites every entry
// a call reads, so nothing needs clearing between calls.
static __device__ __align__(256) int32_t g_static_permute_scratch[kStaticPermuteScratchInts];

namespace {
std::mutex g_static_mu;
int32_t* g_static_ptr[64];  // device address of the array, per device ordinal

// The array's device address on the current device.  Host code only sees a
// host-side stand-in under the array's name, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.  The
// address is cached for the life of the process: after cudaDeviceReset the
// module may be reloaded elsewhere, so calls after a reset are not supported.
cudaError_t static_scratch_on_current_device(int32_t** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_permute_scratch);
        if (e != cudaSuccess) return e;
        g_static_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_static_ptr[dev];
    return cudaSuccess;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

}  // namespace moe

extern "C" moe_status moe_permute_static_scratch(const moe_bf16* x, const int32_t* topk_ids, int N, int D,
                                                 int E, int K, int32_t* expert_offsets, int32_t* perm_src,
                                                 int32_t* inv_perm, moe_bf16* x_perm, void* stream) {
    using namespace moe;
    char msg[256];
    const int sizes = check_permute_sizes(N, D, E, K);  // exactly moe_permute's checks
    if (sizes != MOE_OK) return static_cast<moe_status>(sizes);
    const void* ptrs[5] = {expert_offsets, x, topk_ids, perm_src, inv_perm};
    const int nreq = (N == 0) ? 1 : 5;
    for (int i = 0; i < nreq; ++i) {
        if (ptrs[i] == nullptr || !al16(ptrs[i])) {
            set_error_detail("moe_permute_static_scratch: a required pointer is NULL or not 16-byte aligned");
            return MOE_ERR_INVALID_ARG;
        }
    }
    if (N > 0 && (x_perm == nullptr || !al16(x_perm))) {
        set_error_detail("moe_permute_static_scratch: x_perm is NULL or not 16-byte aligned");
        return MOE_ERR_INVALID_ARG;
    }
    const long long need = static_cast<long long>(permute_scratch_bytes(N, E) / sizeof(int32_t));
    if (need > kStaticPermuteScratchInts) {
        snprintf(msg, sizeof msg,
                 "moe_permute_static_scratch: N=%d, E=%d needs %lld int32 of scratch; the static maximum "
                 "is %lld (E * ceil(N/16) + E <= 1048576); use moe_permute with a workspace",
                 N, E, need, kStaticPermuteScratchInts);
        set_error_detail(msg);
        return MOE_ERR_UNSUPPORTED;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (N == 0) {
        e = cudaMemsetAsync(expert_offsets, 0, (E + 1) * sizeof(int32_t), st);
    } else {
        int32_t* scratch = nullptr;
        e = static_scratch_on_current_device(&scratch);
        if (e == cudaSuccess)
            e = launch_permute(x, topk_ids, N, D, E, K, expert_offsets, perm_src, inv_perm, x_perm, scratch,
                               nullptr, st);
    }
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "moe_permute_static_scratch: %s", cudaGetErrorString(e));
        set_error_detail(msg);
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
