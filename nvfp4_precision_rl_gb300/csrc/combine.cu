// combine.cu -- unpermute + weighted combine of the routed experts' outputs.
//
//   out[t, h] = bf16_rn( sum_{j < topk} w[t, j] * y2[dst[t * topk + j], h] )
//
// ("Towards Blackwell-Native 8-bit and 4-bit RL", shared-expert section: the
// routed experts' outputs pass through a high-precision weighted reduction.)
// The reduction is binary32 in slot order, multiply then add, each one IEEE
// operation (__fmul_rn / __fadd_rn: never contracted into an FMA), so the
// result is bit-exact.  Memory-bound gather: one thread per (token, 8 columns)
// -- with topk fixed at compile time (an even number of 8-column chunks, and
// enough of them), per (token, chunks c and c + chunks / 2) -- the topk 16-byte row loads
// issued before any arithmetic; in the fixed-topk kernel the next item's rows
// and weights are read while the current item's rows load, so each item waits
// on one memory latency instead of two.
#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int kCbThreads = 256;
constexpr int kCbMaxTopk = 32;

template <int kTopk, int kPer>   // kTopk 0: runtime topk; kPer: 8-column chunks per item (1 or 2)
__global__ void __launch_bounds__(kCbThreads) combine_kernel(const uint16_t* __restrict__ y2, int64_t rows,
                                                             int64_t ld_y2, const int32_t* __restrict__ dst,
                                                             const float* __restrict__ w, int64_t tokens,
                                                             int topk_rt, int chunks, uint16_t* __restrict__ out,
                                                             int64_t ld_out, unsigned* status) {
    const int topk = kTopk > 0 ? kTopk : topk_rt;
    const int64_t total = tokens * chunks;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if constexpr (kTopk > 0) {
        // kPer chunks per item (c, and c + chunks / 2 when kPer is 2, of one
        // token): the next item's rows and weights are read while the current
        // one's rows load
        const int half = chunks / kPer;
        const int64_t items = tokens * half;
        int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        int32_t rn[kTopk];
        float wn[kTopk];
        auto fetch = [&](int64_t it) {
            const int64_t t = it / half;
#pragma unroll
            for (int u = 0; u < kTopk; ++u) {
                rn[u] = it < items ? __ldg(dst + t * kTopk + u) : -1;
                wn[u] = it < items ? __ldg(w + t * kTopk + u) : 0.0f;
            }
        };
        fetch(i);
        for (; i < items; i += stride) {
            const int64_t t = i / half;
            const int c = static_cast<int>(i - t * half);
            int32_t r[kTopk];
            float wj[kTopk];
#pragma unroll
            for (int u = 0; u < kTopk; ++u) {
                r[u] = rn[u];
                wj[u] = wn[u];
            }
            uint4 v[kTopk][kPer];
#pragma unroll
            for (int u = 0; u < kTopk; ++u) {
#pragma unroll
                for (int hh = 0; hh < kPer; ++hh) v[u][hh] = make_uint4(0u, 0u, 0u, 0u);
                if (r[u] >= 0 && r[u] < rows) {
                    const uint4* row = reinterpret_cast<const uint4*>(y2 + r[u] * ld_y2);
#pragma unroll
                    for (int hh = 0; hh < kPer; ++hh) v[u][hh] = __ldg(row + c + hh * half);
                } else if (c == 0) {
                    record_error(status, NVFP4_ERR_DEVICE_INPUT, DETAIL_GATHER_INDEX);
                }
            }
            fetch(i + stride);
#pragma unroll
            for (int hh = 0; hh < kPer; ++hh) {
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
                for (int u = 0; u < kTopk; ++u) {
                    if (r[u] < 0 || r[u] >= rows) continue;   // contributes nothing
                    const uint32_t words[4] = {v[u][hh].x, v[u][hh].y, v[u][hh].z, v[u][hh].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[2 * e] = __fadd_rn(acc[2 * e], __fmul_rn(wj[u], bf16lo(words[e])));
                        acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __fmul_rn(wj[u], bf16hi(words[e])));
                    }
                }
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
                    o[e] = *reinterpret_cast<const uint32_t*>(&h);
                }
                reinterpret_cast<uint4*>(out + t * ld_out)[c + hh * half] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        return;
    }
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / chunks;
        const int c = static_cast<int>(i - t * chunks);
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
        constexpr int kUnroll = kTopk > 0 ? kTopk : 8;
        for (int j0 = 0; j0 < topk; j0 += kUnroll) {
            uint4 v[kUnroll];
            float wj[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                wj[u] = 0.0f;
                if (j < topk) {
                    const int64_t r = __ldg(dst + t * topk + j);
                    if (r >= 0 && r < rows) {
                        v[u] = __ldg(reinterpret_cast<const uint4*>(y2 + r * ld_y2) + c);
                        wj[u] = __ldg(w + t * topk + j);
                    } else if (c == 0) {
                        record_error(status, NVFP4_ERR_DEVICE_INPUT, DETAIL_GATHER_INDEX);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (j0 + u >= topk) break;
                const int64_t r = __ldg(dst + t * topk + j0 + u);
                if (r < 0 || r >= rows) continue;   // contributes nothing
                const uint32_t words[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[2 * e] = __fadd_rn(acc[2 * e], __fmul_rn(wj[u], bf16lo(words[e])));
                    acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __fmul_rn(wj[u], bf16hi(words[e])));
                }
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
            o[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        reinterpret_cast<uint4*>(out + t * ld_out)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_moe_combine(const void* y2, int64_t rows, int64_t ld_y2, const int32_t* dst_rows,
                                          const float* weights, int64_t tokens, int32_t topk, int64_t hidden,
                                          void* out, int64_t ld_out, nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (rows < 0 || tokens < 0 || topk < 1 || topk > kCbMaxTopk || hidden <= 0 || hidden % 8 != 0 ||
        ld_y2 < hidden || ld_y2 % 8 != 0 || ld_out < hidden || ld_out % 8 != 0)
        return NVFP4_ERR_SHAPE;
    if (hidden > (int64_t(1) << 24) || tokens > (int64_t(1) << 31) / topk) return NVFP4_ERR_SHAPE;
    if (tokens == 0) return NVFP4_OK;
    if (!y2 || !dst_rows || !weights || !out) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(y2, 16) || !aligned(out, 16) || !aligned(dst_rows, 4) || !aligned(weights, 4))
        return NVFP4_ERR_ALIGNMENT;
    const int chunks = static_cast<int>(hidden / 8);
    const int64_t total = tokens * chunks;
    const int64_t want = ceil_div(total, kCbThreads);
    const int64_t cap = static_cast<int64_t>(ctx.sm_count) * 16;
    const int grid = static_cast<int>(want < cap ? want : cap);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t* src = static_cast<const uint16_t*>(y2);
    uint16_t* dst = static_cast<uint16_t*>(out);
    // the two-chunk kernel holds 2 CTAs per SM; with fewer than ~8 of its items
    // per resident thread the one-chunk kernel, with twice the CTAs, is faster
    const bool two_chunks = chunks % 2 == 0 && total / 2 >= static_cast<int64_t>(ctx.sm_count) * 2 * kCbThreads * 8;
    if (topk == 8 && two_chunks)
        combine_kernel<8, 2><<<grid, kCbThreads, 0, s>>>(src, rows, ld_y2, dst_rows, weights, tokens, topk, chunks,
                                                         dst, ld_out, ctx.status);
    else if (topk == 8)
        combine_kernel<8, 1><<<grid, kCbThreads, 0, s>>>(src, rows, ld_y2, dst_rows, weights, tokens, topk, chunks,
                                                         dst, ld_out, ctx.status);
    else
        combine_kernel<0, 1><<<grid, kCbThreads, 0, s>>>(src, rows, ld_y2, dst_rows, weights, tokens, topk, chunks,
                                                      dst, ld_out, ctx.status);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}
