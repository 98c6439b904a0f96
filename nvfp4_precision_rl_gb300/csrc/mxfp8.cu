// mxfp8.cu -- MXFP8 quantization and dequantization.
//
// MXFP8 ("Towards Blackwell-Native 8-bit and 4-bit RL", "MXFP8 format
// background"): 32 consecutive values share one E8M0 scale, a power of two
// rounded up so that the block maximum is not clipped; the values are E4M3.
// Scale 2^e with e the smallest integer >= -127 such that 448 * 2^e >= amax
// (E8M0 code e + 127); element E4M3_RNE_sat(x * 2^-e), the product exact.
// The 1x32 row-wise copy and the 32x1 column-wise copy are quantized
// independently from the bf16 data ("Backward activation representation
// trade-off").  Scale bytes use the same 128 x 4 swizzled tiles as NVFP4
// (one 32-bit word = four consecutive blocks = 128 values).  Bit-exact.
#include <cuda_fp16.h>

#include "common.cuh"
#include "rowquant.cuh"

namespace nvfp4 {
namespace {

constexpr int kMxThreads = 256;

// smallest e >= -127 with 448 * 2^e >= amax (amax >= 0, finite): amax = m 2^E,
// 448 = 1.75 2^8, so e = E - 8 when m <= 1.75, else E - 7.
__device__ __forceinline__ int mx_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int ef = static_cast<int>(b >> 23);
    if (ef == 0) return -127;   // zero or subnormal: 448 * 2^-127 covers it
    const int e = ef - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return e < -127 ? -127 : e;
}

__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t m, uint32_t v) {
    uint32_t out;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(out) : "r"(m), "r"(v & 0x7FFF7FFFu));
    return out;
}

// two floats -> two E4M3 codes, `lo` in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
    return h;
}

// 32 bf16 values (16 words) scaled by 2^-e -> 32 E4M3 codes (8 words)
__device__ __forceinline__ void mx_encode32(const uint32_t (&w)[16], int e, uint32_t (&c)[8]) {
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);   // 2^-e, normal
    const float2 i2 = make_float2(inv, inv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 a = __fmul2_rn(make_float2(bf16lo(w[2 * j]), bf16hi(w[2 * j])), i2);
        const float2 b = __fmul2_rn(make_float2(bf16lo(w[2 * j + 1]), bf16hi(w[2 * j + 1])), i2);
        c[j] = e4m3x2(a.x, a.y) | (e4m3x2(b.x, b.y) << 16);
    }
}

// Rows: one thread per 1x32 block.
__global__ void __launch_bounds__(kMxThreads) mx_rows_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                             int nb, int64_t ld, uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ sf, int kgroups) {
    const int64_t total = rows * nb;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t r = i / nb;
        const int b = static_cast<int>(i - r * nb);
        const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + static_cast<int64_t>(b) * 32);
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 v = __ldg(src + j);
            w[4 * j] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
        }
        uint32_t m = 0u;
#pragma unroll
        for (int j = 0; j < 16; ++j) m = absmax_bf16x2(m, w[j]);
        const int e = mx_exponent(fmaxf(bf16lo(m), bf16hi(m)));
        uint32_t c[8];
        mx_encode32(w, e, c);
        uint4* dst = reinterpret_cast<uint4*>(q + r * (static_cast<int64_t>(nb) * 32) + static_cast<int64_t>(b) * 32);
        dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
        dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
        sf[sf_word_offset(r, b >> 2, kgroups) + (b & 3)] = static_cast<uint8_t>(e + 127);
    }
}

// Columns (X^T, 32x1 blocks): one thread per two adjacent columns x 32 rows.
__global__ void __launch_bounds__(kMxThreads) mx_cols_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                             int cols, int64_t ld, uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ sf, int kgroups) {
    const int pairs = cols >> 1;
    const int64_t total = static_cast<int64_t>(pairs) * (rows >> 5);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t g = i / pairs;                        // 32-row group
        const int k0 = static_cast<int>(i - g * pairs) * 2;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(x + (g * 32) * ld + k0);
        const int64_t step = ld >> 1;
        uint32_t v[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] = __ldg(src + t * step);
        uint32_t m = 0u;
#pragma unroll
        for (int t = 0; t < 32; ++t) m = absmax_bf16x2(m, v[t]);
        const int e0 = mx_exponent(bf16lo(m));
        const int e1 = mx_exponent(bf16hi(m));
        uint32_t w0[16], w1[16];   // column k0 / k0 + 1 values as bf16 pairs along the rows
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            w0[t] = (v[2 * t] & 0xFFFFu) | (v[2 * t + 1] << 16);
            w1[t] = (v[2 * t] >> 16) | (v[2 * t + 1] & 0xFFFF0000u);
        }
        uint32_t c0[8], c1[8];
        mx_encode32(w0, e0, c0);
        mx_encode32(w1, e1, c1);
        uint4* d0 = reinterpret_cast<uint4*>(q + static_cast<int64_t>(k0) * rows + g * 32);
        uint4* d1 = reinterpret_cast<uint4*>(q + static_cast<int64_t>(k0 + 1) * rows + g * 32);
        d0[0] = make_uint4(c0[0], c0[1], c0[2], c0[3]);
        d0[1] = make_uint4(c0[4], c0[5], c0[6], c0[7]);
        d1[0] = make_uint4(c1[0], c1[1], c1[2], c1[3]);
        d1[1] = make_uint4(c1[4], c1[5], c1[6], c1[7]);
        const int blk = static_cast<int>(g);
        sf[sf_word_offset(k0, blk >> 2, kgroups) + (blk & 3)] = static_cast<uint8_t>(e0 + 127);
        sf[sf_word_offset(k0 + 1, blk >> 2, kgroups) + (blk & 3)] = static_cast<uint8_t>(e1 + 127);
    }
}

// Dequantization: one thread per block; dec(q) * 2^(code - 127) is exact in
// binary32 and rounded once to bf16.
// One thread per quarter block (8 values, 16 bytes of output): a warp's store
// covers 512 contiguous bytes of a row.
__global__ void __launch_bounds__(kMxThreads) mx_dequant_kernel(const uint8_t* __restrict__ q,
                                                                const uint8_t* __restrict__ sf, int64_t rows,
                                                                int nb, int kgroups, uint16_t* __restrict__ y,
                                                                int64_t ld_y) {
    const int parts = 4 * nb;                            // 8-value parts per row
    const int64_t total = rows * parts;
    const bool narrow = total <= 0xFFFFFFFFll;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t r = narrow ? static_cast<int64_t>(static_cast<uint32_t>(i) / static_cast<uint32_t>(parts))
                                 : i / parts;
        const int pq = static_cast<int>(i - r * parts);
        const int b = pq >> 2;
        const uint2 c = __ldg(reinterpret_cast<const uint2*>(q + r * (static_cast<int64_t>(nb) * 32)) + pq);
        const uint32_t code = __ldg(sf + sf_word_offset(r, b >> 2, kgroups) + (b & 3));
        const float f = code ? __uint_as_float(code << 23) : __uint_as_float(0x00400000u);   // 2^(code-127)
        const float2 f2 = make_float2(f, f);
        const uint32_t words[2] = {c.x, c.y};
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t hv;
                const uint16_t pair = static_cast<uint16_t>(words[j] >> (16 * h));
                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hv) : "h"(pair));
                const float2 v = __fmul2_rn(__half22float2(*reinterpret_cast<const __half2*>(&hv)), f2);
                const __nv_bfloat162 o = __floats2bfloat162_rn(v.x, v.y);
                out[2 * j + h] = *reinterpret_cast<const uint32_t*>(&o);
            }
        }
        *reinterpret_cast<uint4*>(y + r * ld_y + static_cast<int64_t>(pq) * 8) = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

int grid_for(int64_t work, const DeviceCtx& ctx) {
    const int64_t want = ceil_div(work, kMxThreads);
    const int64_t cap = static_cast<int64_t>(ctx.sm_count) * 16;
    return static_cast<int>(want < cap ? want : cap);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

size_t nvfp4_mxfp8_sf_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return static_cast<size_t>(round_up(rows, 128) * round_up(ceil_div(cols, 32), 4));
}

nvfp4_status nvfp4_mxfp8_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x, void* q, void* sf,
                                  void* q_col, void* sf_col, nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (rows < 0 || cols <= 0 || cols % 32 != 0 || cols > (int64_t(1) << 24) || ld_x < cols || ld_x % 8 != 0)
        return NVFP4_ERR_SHAPE;
    const bool want_col = q_col != nullptr || sf_col != nullptr;
    if (want_col && (q_col == nullptr || sf_col == nullptr)) return NVFP4_ERR_INVALID_ARG;
    if (want_col && rows % 32 != 0) return NVFP4_ERR_SHAPE;
    if (rows == 0) return NVFP4_OK;
    if (!x || !q || !sf) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(q_col, 16)) return NVFP4_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    const int nb = static_cast<int>(cols / 32);
    // the padding of the swizzled scales reads as zero (the kernels write every
    // real block; there is padding only for ragged row or block counts)
    if ((rows % 128 != 0 || nb % 4 != 0) &&
        cudaMemsetAsync(sf, 0, nvfp4_mxfp8_sf_bytes(rows, cols), s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    mx_rows_kernel<<<grid_for(rows * nb, ctx), kMxThreads, 0, s>>>(xb, rows, nb, ld_x, static_cast<uint8_t*>(q),
                                                                    static_cast<uint8_t*>(sf), (nb + 3) / 4);
    NVFP4_CHECK_LAUNCH();
    if (want_col) {
        const int nbc = static_cast<int>(rows / 32);
        if ((cols % 128 != 0 || nbc % 4 != 0) &&
            cudaMemsetAsync(sf_col, 0, nvfp4_mxfp8_sf_bytes(cols, rows), s) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        mx_cols_kernel<<<grid_for((cols / 2) * nbc, ctx), kMxThreads, 0, s>>>(
            xb, rows, static_cast<int>(cols), ld_x, static_cast<uint8_t*>(q_col), static_cast<uint8_t*>(sf_col),
            (nbc + 3) / 4);
        NVFP4_CHECK_LAUNCH();
    }
    return NVFP4_OK;
}

nvfp4_status nvfp4_mxfp8_dequantize(const void* q, const void* sf, int64_t rows, int64_t cols, void* y,
                                    int64_t ld_y, nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (rows < 0 || cols <= 0 || cols % 32 != 0 || cols > (int64_t(1) << 24) || ld_y < cols || ld_y % 8 != 0)
        return NVFP4_ERR_SHAPE;
    if (rows == 0) return NVFP4_OK;
    if (!q || !sf || !y) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(y, 16)) return NVFP4_ERR_ALIGNMENT;
    const int nb = static_cast<int>(cols / 32);
    mx_dequant_kernel<<<grid_for(rows * nb * 4, ctx), kMxThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(q), static_cast<const uint8_t*>(sf), rows, nb, (nb + 3) / 4,
        static_cast<uint16_t*>(y), ld_y);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}

}  // extern "C"
