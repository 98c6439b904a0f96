// permute.cu -- MoE routing permute into a contiguous, padded per-expert layout.
//
// Counting sort over the flattened (token, slot) pairs, stable in (token, slot)
// order, with all metadata left on the device ("miniTE report", section
// "Transformer Engine path optimisation": contiguous layouts and device-side
// metadata feed the grouped GEMM without a host round trip).
//   1. count:   one block per chunk of kChunk pairs -> per-chunk expert histogram,
//               and the per-expert totals (atomic adds of the block histograms)
//   2. scan:    one block per expert: the padded sizes of the experts before it
//               -> its segment start (offsets), then an exclusive scan of its
//               column of chunk counts -> each chunk's first row in the segment
//               (up to 64 chunks: one block over the whole histogram instead)
//   3. scatter: one block per chunk, in order: rank inside the chunk from
//               warp match + per-warp histograms -> gather_rows / dst_rows
#include <mutex>

#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int kChunk = 1024;
constexpr int kPermThreads = 256;
constexpr int kMaxExperts = 1024;

__global__ void __launch_bounds__(kPermThreads) perm_count_kernel(const int32_t* ids, int64_t n,
                                                                  int E, int32_t* counts, int32_t* totals,
                                                                  unsigned* status) {
    extern __shared__ int32_t s_hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int64_t c1 = min(c0 + kChunk, n);
    for (int64_t i = c0 + threadIdx.x; i < c1; i += blockDim.x) {
        const int32_t e = ids[i];
        if (e >= 0 && e < E) atomicAdd(&s_hist[e], 1);
        else record_error(status, NVFP4_ERR_DEVICE_INPUT, DETAIL_EXPERT_ID);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t h = s_hist[e];
        counts[static_cast<int64_t>(blockIdx.x) * E + e] = h;
        if (totals != nullptr && h != 0) atomicAdd(totals + e, h);
    }
}

// Small histograms (up to kScanOneMaxChunks chunks): one block of
// kScanOneThreads threads: Ew = round_up(E, 32) experts across and
// G = kScanOneThreads / Ew groups of chunks down; thread (g, e) sums expert e's
// counts over its group's chunks (loads batched so that many are in flight),
// the first Ew threads scan the padded totals, then every thread rewrites its
// chunks' counts as their first rows in the expert segment.
constexpr int kScanOneThreads = 1024;
constexpr int kScanOneMaxChunks = 64;
constexpr int kScanBatch = 8;

__global__ void __launch_bounds__(kScanOneThreads) perm_scan_one_block_kernel(int32_t* counts, int nchunks, int E, int align,
                                                                 int32_t* offsets) {
    __shared__ int32_t s_part[kScanOneThreads];   // [G][Ew] per-group sums, then per-group bases
    __shared__ int32_t s_warp[32];
    const int Ew = (E + 31) & ~31;
    const int G = kScanOneThreads / Ew;
    const int e = threadIdx.x % Ew;
    const int g = threadIdx.x / Ew;
    const bool mine = g < G && e < E;
    const int per = (nchunks + G - 1) / G;
    const int c0 = g * per;
    const int c1 = min(c0 + per, nchunks);
    int32_t sum = 0;
    if (mine) {
        for (int c = c0; c < c1; c += kScanBatch) {
            int32_t v[kScanBatch];
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j)
                v[j] = (c + j < c1) ? counts[static_cast<int64_t>(c + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j) sum += v[j];
        }
    }
    if (g < G) s_part[g * Ew + e] = sum;
    __syncthreads();
    // the first Ew threads (whole warps): expert totals, padded, block-wide exclusive scan
    int32_t padded = 0, incl = 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < Ew) {
        int64_t total = 0;
        for (int gg = 0; gg < G; ++gg) total += s_part[gg * Ew + e];
        padded = (e < E) ? static_cast<int32_t>((total + align - 1) / align * align) : 0;
        incl = padded;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) s_warp[warp] = incl;
    }
    __syncthreads();
    if (warp == 0) {
        const int nw = Ew >> 5;
        int32_t w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o) w += t;
        }
        if (lane < nw) s_warp[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    if (threadIdx.x < Ew && e < E) {
        const int32_t excl = incl - padded + (warp > 0 ? s_warp[warp - 1] : 0);
        offsets[e] = excl;
        if (e == E - 1) offsets[E] = excl + padded;
        // group gg of expert e starts after the segment start and the earlier groups
        int32_t base = excl;
        for (int gg = 0; gg < G; ++gg) {
            const int32_t part = s_part[gg * Ew + e];
            s_part[gg * Ew + e] = base;
            base += part;
        }
    }
    __syncthreads();
    if (mine) {
        int32_t base = s_part[g * Ew + e];
        for (int c = c0; c < c1; c += kScanBatch) {
            int32_t v[kScanBatch];
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j)
                v[j] = (c + j < c1) ? counts[static_cast<int64_t>(c + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j) {
                if (c + j < c1) counts[static_cast<int64_t>(c + j) * E + e] = base;
                base += v[j];
            }
        }
    }
}

// Exclusive scan of one value per thread over the block (blockDim.x a multiple
// of 32, at most 1024); returns the thread's exclusive prefix and the block sum.
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* total, int64_t* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int64_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t t = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o) w += t;
        }
        if (lane < nw) s_warp[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const int64_t excl = incl - v + (warp > 0 ? s_warp[warp - 1] : 0);
    *total = s_warp[nw - 1];
    __syncthreads();   // s_warp is reused by the next call
    return excl;
}

// Larger histograms: one block per expert e.  Its segment starts after the padded sizes of experts
// 0 .. e-1 (from the count pass's totals); chunk c's first row in the segment
// is the start plus the counts of expert e in chunks 0 .. c-1, written over
// counts[c][e] (only this block reads or writes column e).
constexpr int kScanThreads = 512;

__global__ void __launch_bounds__(kScanThreads) perm_scan_kernel(int32_t* counts, const int32_t* totals, int nchunks,
                                                                 int E, int align, int32_t* offsets) {
    __shared__ int64_t s_warp[kScanThreads / 32];
    const int e = blockIdx.x;
    auto padded = [align](int32_t t) { return (static_cast<int64_t>(t) + align - 1) / align * align; };
    int64_t part = 0;
    for (int j = threadIdx.x; j < e; j += blockDim.x) part += padded(totals[j]);
    int64_t start = 0;
    (void)block_exclusive_scan(part, &start, s_warp);
    if (threadIdx.x == 0) {
        offsets[e] = static_cast<int32_t>(start);
        if (e == E - 1) offsets[E] = static_cast<int32_t>(start + padded(totals[e]));
    }
    int64_t carry = start;
    for (int c0 = 0; c0 < nchunks; c0 += blockDim.x) {
        const int c = c0 + threadIdx.x;
        const int64_t v = c < nchunks ? counts[static_cast<int64_t>(c) * E + e] : 0;
        int64_t sum = 0;
        const int64_t excl = block_exclusive_scan(v, &sum, s_warp);
        if (c < nchunks) counts[static_cast<int64_t>(c) * E + e] = static_cast<int32_t>(carry + excl);
        carry += sum;
    }
}

__global__ void __launch_bounds__(kPermThreads) perm_scatter_kernel(const int32_t* ids, int64_t n,
                                                                    int topk, int E,
                                                                    const int32_t* chunk_base,
                                                                    int32_t* gather,
                                                                    int32_t* dst_rows) {
    extern __shared__ int32_t smem[];
    int32_t* s_next = smem;                 // [E] next free row of each expert for this chunk
    int32_t* s_wcnt = smem + E;             // [kPermThreads/32][E] pairs per warp this round
    constexpr int kWarps = kPermThreads / 32;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        s_next[e] = chunk_base[static_cast<int64_t>(blockIdx.x) * E + e];
        for (int w = 0; w < kWarps; ++w) s_wcnt[w * E + e] = 0;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int64_t c1 = min(c0 + kChunk, n);
    int32_t e_next = (c0 + threadIdx.x < c1) ? ids[c0 + threadIdx.x] : -1;   // read a round ahead
    for (int64_t base = c0; base < c1; base += kPermThreads) {
        const int64_t i = base + threadIdx.x;
        int32_t e = e_next;
        e_next = (i + kPermThreads < c1) ? ids[i + kPermThreads] : -1;
        if (e >= E) e = -1;
        if (i < c1 && e < 0) dst_rows[i] = -1;   // dropped id (already reported by the count pass)
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        const unsigned lower = peers & ((1u << lane) - 1u);
        if (e >= 0 && lower == 0u) s_wcnt[warp * E + e] = __popc(peers);
        __syncthreads();
        if (e >= 0) {
            int32_t row = s_next[e] + __popc(lower);
            for (int w = 0; w < warp; ++w) row += s_wcnt[w * E + e];
            gather[row] = static_cast<int32_t>(i / topk);
            dst_rows[i] = row;
        }
        __syncthreads();
        for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
            int32_t add = 0;
            for (int w = 0; w < kWarps; ++w) {
                add += s_wcnt[w * E + ee];
                s_wcnt[w * E + ee] = 0;
            }
            s_next[ee] += add;
        }
        __syncthreads();
    }
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

int64_t nvfp4_moe_capacity(int64_t tokens, int32_t topk, int32_t num_experts, int32_t row_align) {
    if (tokens < 0 || topk <= 0 || num_experts <= 0 || row_align <= 0) return 0;
    return round_up(tokens * topk + static_cast<int64_t>(num_experts) * (row_align - 1), row_align);
}

size_t nvfp4_moe_permute_workspace_bytes(int64_t tokens, int32_t topk, int32_t num_experts) {
    if (tokens < 0 || topk <= 0 || num_experts <= 0) return 0;
    const int64_t chunks = ceil_div(tokens * topk, kChunk);
    // per-expert totals (padded to 256 bytes), then the per-chunk histograms
    return static_cast<size_t>(round_up(static_cast<int64_t>(num_experts), 64) * 4 + chunks * num_experts * 4);
}

nvfp4_status nvfp4_moe_permute(const int32_t* topk_ids, int64_t tokens, int32_t topk,
                               int32_t num_experts, int32_t row_align, int32_t* expert_offsets,
                               int32_t* gather_rows, int64_t capacity, int32_t* dst_rows,
                               void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (tokens < 0 || topk < 1 || topk > 64 || num_experts < 1 || num_experts > kMaxExperts ||
        row_align < 1)
        return NVFP4_ERR_SHAPE;
    const int64_t n = tokens * topk;
    if (n > (int64_t(1) << 30)) return NVFP4_ERR_SHAPE;
    if (capacity < nvfp4_moe_capacity(tokens, topk, num_experts, row_align)) return NVFP4_ERR_SHAPE;
    if (capacity > (int64_t(1) << 31) - 1) return NVFP4_ERR_SHAPE;
    if (expert_offsets == nullptr || gather_rows == nullptr || (n > 0 && (topk_ids == nullptr || dst_rows == nullptr)))
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(topk_ids, 4) || !aligned(expert_offsets, 4) || !aligned(gather_rows, 4) ||
        !aligned(dst_rows, 4) || !aligned(workspace, 4))
        return NVFP4_ERR_ALIGNMENT;
    if (workspace == nullptr ||
        workspace_bytes < nvfp4_moe_permute_workspace_bytes(tokens, topk, num_experts))
        return NVFP4_ERR_WORKSPACE;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int nchunks = static_cast<int>(ceil_div(n, kChunk));
    const int E = num_experts;
    int32_t* totals = static_cast<int32_t*>(workspace);
    int32_t* counts = totals + round_up(static_cast<int64_t>(E), 64);
    // a few chunks: one scan block reads the whole histogram (no totals);
    // more: the count pass also sums per-expert totals and one block per
    // expert scans its column
    const bool one_block = nchunks <= kScanOneMaxChunks;
    if (cudaMemsetAsync(gather_rows, 0xFF, static_cast<size_t>(capacity) * 4, s) != cudaSuccess ||
        (!one_block && cudaMemsetAsync(totals, 0, static_cast<size_t>(E) * 4, s) != cudaSuccess))
        return NVFP4_ERR_CUDA;
    if (nchunks > 0) {
        perm_count_kernel<<<nchunks, kPermThreads, E * sizeof(int32_t), s>>>(
            topk_ids, n, E, counts, one_block ? nullptr : totals, ctx.status);
        NVFP4_CHECK_LAUNCH();
    }
    if (one_block)
        perm_scan_one_block_kernel<<<1, kScanOneThreads, 0, s>>>(counts, nchunks, E, row_align, expert_offsets);
    else
        perm_scan_kernel<<<E, kScanThreads, 0, s>>>(counts, totals, nchunks, E, row_align, expert_offsets);
    NVFP4_CHECK_LAUNCH();
    if (nchunks > 0) {
        const size_t smem = static_cast<size_t>(E) * (1 + kPermThreads / 32) * sizeof(int32_t);
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        perm_scatter_kernel<<<nchunks, kPermThreads, smem, s>>>(topk_ids, n, topk, E, counts,
                                                                gather_rows, dst_rows);
        NVFP4_CHECK_LAUNCH();
    }
    return NVFP4_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Permute for callers that cannot allocate device memory
// ---------------------------------------------------------------------------
// Some callers of this library cannot call cudaMalloc at the point where they
// route tokens: host runtimes whose device memory is owned by a different
// allocator (a framework's caching allocator, a serving engine's pre-reserved
// pool), or decode loops that forbid allocation on the hot path (cudaMalloc
// synchronises the device).  For them the routing permute's scratch (per-chunk
// expert histograms) lives in the fixed file-scope array below, which every
// device that loads this library keeps until the process exits.
// nvfp4_moe_permute itself is unchanged; this entry point only supplies that
// array as its workspace.
namespace nvfp4 {
namespace {

constexpr int64_t kNoAllocScratchBytes = int64_t(1) << 20;   // 1 MiB
static __device__ __align__(256) int32_t g_noalloc_permute_scratch[kNoAllocScratchBytes / 4];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];
unsigned long long g_noalloc_ctx[64];

// Device address of the scratch array in the current device's current CUDA
// context.  Looked up (with that device current) on the first call in each
// context -- a cudaDeviceReset or another context made current gives the array
// another address -- and cached; the host-side name of a __device__ array is
// not a device address, so it is never passed to a kernel directly.
nvfp4_status noalloc_scratch(const DeviceCtx& ctx, void** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    const int dev = ctx.device & 63;
    if (!ctx_cached(g_noalloc_ctx, ctx) || g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_permute_scratch) != cudaSuccess || p == nullptr)
            return NVFP4_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
        ctx_cache_set(g_noalloc_ctx, ctx);
    }
    *out = g_noalloc_ptr[dev];
    return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_moe_permute_noalloc(const int32_t* topk_ids, int64_t tokens,
                                                  int32_t topk, int32_t num_experts,
                                                  int32_t row_align, int32_t* expert_offsets,
                                                  int32_t* gather_rows, int64_t capacity,
                                                  int32_t* dst_rows, nvfp4_stream_t stream) {
    // the same device checks, in the same order, as the allocating permute
    nvfp4::DeviceCtx ctx;
    nvfp4_status st = nvfp4::device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    const size_t need = nvfp4_moe_permute_workspace_bytes(tokens, topk, num_experts);
    if (need == 0) return NVFP4_ERR_SHAPE;
    if (need > static_cast<size_t>(nvfp4::kNoAllocScratchBytes)) return NVFP4_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = nvfp4::noalloc_scratch(ctx, &scratch);
    if (st != NVFP4_OK) return st;
    return nvfp4_moe_permute(topk_ids, tokens, topk, num_experts, row_align, expert_offsets,
                             gather_rows, capacity, dst_rows, scratch,
                             static_cast<size_t>(nvfp4::kNoAllocScratchBytes), stream);
}
