// gather.cu -- per-token quantized rows scattered into the expert layout.
//
// Per-token quantization of a row depends on that row alone (its own amax,
// S = amax / 2688, its own block scales and codes: "Towards Blackwell-Native
// 8-bit and 4-bit RL", "Online computation of the per-token scale"), so
// quantizing the tokens once and copying row gather[r] of the result to row r
// of the routed layout gives, bit for bit, what quantizing the gathered rows
// gives -- with top-k routing, at 1/k of the quantization work.  A row with no
// source (layout padding) becomes a zero row (zero codes, zero scales, S = 0:
// the quantization of a zero row); the scale rows past rows_out up to a
// multiple of 128 are zeroed, as the quantizer does.
#include <type_traits>

#include "common.cuh"
#include "rowquant.cuh"

namespace nvfp4 {
namespace {

constexpr int kGqThreads = 256;
constexpr int kGqWarps = kGqThreads / 32;
constexpr int kRowsPerBatch = 4;
constexpr int kGqMaxExperts = 256;

// Order in which a CTA visits the layout's 128-row tiles.  Expert e owns tiles
// [ts[e], ts[e+1]) (ts[e] = ceil(offset[e] / 128)); every expert owns at least
// m of them.  Visit k maps to: tile j = k / E of expert e = k % E while
// k < E m (the j-th tiles of all experts, j = 0, 1, ...), then the experts'
// tiles past their first m, expert by expert (q[e] counts those before e),
// then the tiles outside [ts[0], ts[E]).  A bijection on [0, tiles) for any
// non-decreasing ts; E = 0 is the identity.
struct TileOrder {
    int32_t ts[kGqMaxExperts + 1];
    int32_t q[kGqMaxExperts + 1];
    int32_t m;
    int32_t E;
};

__device__ __forceinline__ int64_t tile_of(const TileOrder& o, int64_t k) {
    if (o.E == 0) return k;
    const int64_t a = static_cast<int64_t>(o.E) * o.m;
    if (k < a) return o.ts[k % o.E] + k / o.E;
    k -= a;
    if (k < o.q[o.E]) {
        int lo = 0, hi = o.E - 1;   // the last expert e with q[e] <= k
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (o.q[mid] <= k) lo = mid;
            else hi = mid - 1;
        }
        return o.ts[lo] + o.m + (k - o.q[lo]);
    }
    k -= o.q[o.E];
    return k < o.ts[0] ? k : o.ts[o.E] + (k - o.ts[0]);
}

// Fills *o from the expert offsets (all threads of the CTA call it; E = 0 when
// there are none or they are unusable: the identity order).
__device__ void build_tile_order(TileOrder* o, const int32_t* __restrict__ offsets, int num_experts, int64_t tiles) {
    const int E = (offsets != nullptr && num_experts >= 1 && num_experts <= kGqMaxExperts && tiles <= 0x7FFFFFFF)
                      ? num_experts : 0;
    bool good = true;
    for (int e = threadIdx.x; e <= E && E > 0; e += blockDim.x) {
        const int32_t off = __ldg(offsets + e);
        const int64_t t = (static_cast<int64_t>(off) + 127) / 128;
        good = good && off >= 0;
        o->ts[e] = static_cast<int32_t>(off < 0 ? 0 : (t < tiles ? t : tiles));
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) good = good && o->ts[e + 1] >= o->ts[e];
    const bool ok = __syncthreads_and(good) != 0 && E > 0;
    if (threadIdx.x == 0) {
        o->E = ok ? E : 0;
        o->m = 0x7FFFFFFF;
    }
    __syncthreads();
    if (!ok) return;
    for (int e = threadIdx.x; e < E; e += blockDim.x) atomicMin(&o->m, o->ts[e + 1] - o->ts[e]);
    __syncthreads();
    if (threadIdx.x < 32) {
        // exclusive prefix of the tiles past m: lane l sums experts 8l .. 8l + 7
        const int lane = threadIdx.x;
        int32_t part = 0;
        for (int e = 8 * lane; e < 8 * lane + 8 && e < E; ++e) part += o->ts[e + 1] - o->ts[e] - o->m;
        int32_t incl = part;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += v;
        }
        int32_t run = incl - part;
        for (int e = 8 * lane; e < 8 * lane + 8 && e < E; ++e) {
            o->q[e] = run;
            run += o->ts[e + 1] - o->ts[e] - o->m;
        }
        if (lane == 31) o->q[E] = incl;
    }
    __syncthreads();
}

// One CTA per 128-row tile of the output (a tile of the swizzled scale layout),
// tiles visited in TileOrder: the tile's 128 source row indices are read once
// into shared memory; the codes are copied in 16- (or 8-) byte pieces, the
// lanes of a warp on consecutive pieces of a row, four rows' loads in flight
// before their stores; each 512-byte scale atom (128 rows x one word) is
// written as 32 16-byte lines, lane l gathering the words of rows l, l+32,
// l+64, l+96.
template <bool kVec16>
__global__ void __launch_bounds__(kGqThreads) gather_quantized_kernel(
    const uint8_t* __restrict__ q_src, const uint8_t* __restrict__ sf_src, const float* __restrict__ s_src,
    int64_t rows_src, const int32_t* __restrict__ gather, int64_t rows_out, int64_t tiles, int row_bytes,
    int kgroups, const int32_t* __restrict__ offsets, int num_experts, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sf, float* __restrict__ s, unsigned* status) {
    pdl_launch_dependents();    // a dependent waits for this grid's completion itself
    __shared__ int64_t src_of[128];
    __shared__ TileOrder order;
    build_tile_order(&order, offsets, num_experts, tiles);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    constexpr int kPiece = kVec16 ? 16 : 8;
    const int pieces = row_bytes / kPiece;
    using Piece = typename std::conditional<kVec16, uint4, uint2>::type;
    auto zero_piece = []() -> Piece {
        Piece z;
        memset(&z, 0, sizeof(z));
        return z;
    };
    auto load_piece = [](const uint8_t* row, int pc) -> Piece { return __ldg(reinterpret_cast<const Piece*>(row) + pc); };
    auto store_piece = [](uint8_t* row, int pc, const Piece& v) { reinterpret_cast<Piece*>(row)[pc] = v; };
    for (int64_t visit = blockIdx.x; visit < tiles; visit += gridDim.x) {
        const int64_t tile = tile_of(order, visit);
        const int64_t r0 = tile * 128;
        __syncthreads();                    // the previous tile's src_of is no longer read
        if (threadIdx.x < 128) {
            const int64_t r = r0 + threadIdx.x;
            int64_t src = -1;
            if (r < rows_out) {
                src = __ldg(gather + r);
                if (src >= rows_src) {
                    record_error(status, NVFP4_ERR_DEVICE_INPUT, DETAIL_GATHER_INDEX);
                    src = -1;
                }
                s[r] = src >= 0 ? __ldg(s_src + src) : 0.0f;
            }
            src_of[threadIdx.x] = src;
        }
        __syncthreads();
        // codes of the tile's rows (rows past rows_out have none): warp w copies
        // rows w, w + 8, ..., kRowsPerBatch rows at a time with every load of
        // the batch issued before its stores (lane l on pieces l, l + 32)
        const int rows_here = static_cast<int>(rows_out - r0 < 128 ? rows_out - r0 : 128);
        for (int rb = warp; rb < rows_here; rb += kGqWarps * kRowsPerBatch) {
            for (int pb = 0; pb < pieces; pb += 64) {
                Piece v[kRowsPerBatch][2];
#pragma unroll
                for (int j = 0; j < kRowsPerBatch; ++j) {
                    const int rr = rb + j * kGqWarps;
                    const int64_t src = rr < rows_here ? src_of[rr] : -1;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int pc = pb + lane + 32 * h;
                        v[j][h] = (src >= 0 && pc < pieces) ? load_piece(q_src + src * row_bytes, pc) : zero_piece();
                    }
                }
#pragma unroll
                for (int j = 0; j < kRowsPerBatch; ++j) {
                    const int rr = rb + j * kGqWarps;
                    if (rr >= rows_here) continue;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int pc = pb + lane + 32 * h;
                        if (pc < pieces) store_piece(q + (r0 + rr) * row_bytes, pc, v[j][h]);
                    }
                }
            }
        }
        // scale atoms: warp w builds atoms g = w, w + 8, ...; lane l writes line l
        for (int g = warp; g < kgroups; g += kGqThreads / 32) {
            uint32_t w4[4];
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                const int64_t src = src_of[lane + 32 * qd];
                w4[qd] = src >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(sf_src + sf_word_offset(src, g, kgroups)))
                                  : 0u;
            }
            reinterpret_cast<uint4*>(sf + (tile * kgroups + g) * 512)[lane] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
    }
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_moe_gather_quantized(const void* q_src, const void* sf_src, const float* s_src,
                                                   int64_t rows_src, int64_t cols, const int32_t* gather_rows,
                                                   int64_t rows_out, const int32_t* expert_offsets,
                                                   int32_t num_experts, void* q, void* sf, float* s,
                                                   nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (rows_src < 0 || rows_out < 0 || cols <= 0 || cols % 16 != 0 || cols > (int64_t(1) << 24))
        return NVFP4_ERR_SHAPE;
    if (rows_out == 0) return NVFP4_OK;
    if (gather_rows == nullptr || q == nullptr || sf == nullptr || s == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (rows_src > 0 && (q_src == nullptr || sf_src == nullptr || s_src == nullptr)) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(q_src, 16) || !aligned(sf_src, 16) || !aligned(s_src, 4) || !aligned(gather_rows, 4) ||
        !aligned(q, 16) || !aligned(sf, 16) || !aligned(s, 4) || !aligned(expert_offsets, 4))
        return NVFP4_ERR_ALIGNMENT;
    const int row_bytes = static_cast<int>(cols / 2);
    const int kgroups = static_cast<int>(ceil_div(cols, 64));
    const int64_t tiles = ceil_div(rows_out, 128);
    const int64_t cap = static_cast<int64_t>(ctx.sm_count) * 8;
    const int grid = static_cast<int>(tiles < cap ? tiles : cap);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t* qs = static_cast<const uint8_t*>(q_src);
    const uint8_t* ss = static_cast<const uint8_t*>(sf_src);
    if (row_bytes % 16 == 0)
        gather_quantized_kernel<true><<<grid, kGqThreads, 0, cs>>>(qs, ss, s_src, rows_src, gather_rows, rows_out,
                                                                   tiles, row_bytes, kgroups, expert_offsets,
                                                                   num_experts, static_cast<uint8_t*>(q),
                                                                   static_cast<uint8_t*>(sf),
                                                                   s, ctx.status);
    else
        gather_quantized_kernel<false><<<grid, kGqThreads, 0, cs>>>(qs, ss, s_src, rows_src, gather_rows, rows_out,
                                                                    tiles, row_bytes, kgroups, expert_offsets,
                                                                    num_experts, static_cast<uint8_t*>(q),
                                                                    static_cast<uint8_t*>(sf),
                                                                    s, ctx.status);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}
