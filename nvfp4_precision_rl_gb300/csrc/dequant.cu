// dequant.cu -- NVFP4 -> BF16 dequantization.
//
//   y[r, k] = bf16_rn( fl32( S_r * fl32( dec(q[r, k]) * dec(s_b) ) ) )
//
// ("TRIAGE", section "NVFP4 quantization format and W4A4 execution": the
// NVFP4 value is the outer FP32 scale times the E4M3 block scale times the E2M1
// code.)  HBM-bound: 0.5625 bytes read and 2 bytes written per element.  One
// thread per 16-element block: 8 code bytes, one scale byte (swizzled layout)
// and the row's outer scale in; 32 bf16 bytes out.  The E2M1 x E4M3 product is
// exact in fp16 (at most 5 significant bits, |x| <= 6 * 448, >= 2^-10), so the
// decode runs on packed halves; the multiply by S is one binary32 rounding and
// cvt.rn.bf16x2.f32 the final one.
#include <cuda_fp16.h>

#include "common.cuh"
#include "rowquant.cuh"

namespace nvfp4 {
namespace {

constexpr int kDqThreads = 256;

// byte of two E2M1 codes -> f16x2 (low nibble in the low half)
__device__ __forceinline__ __half2 e2m1x2_to_half2(uint32_t byte) {
    uint32_t h;
    const uint16_t in = static_cast<uint16_t>(byte & 0xFFu);
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u16 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(h) : "h"(in));
    return *reinterpret_cast<__half2*>(&h);
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t out;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
    return out;
}

__global__ void __launch_bounds__(kDqThreads) dequant_kernel(const uint8_t* __restrict__ q,
                                                            const uint8_t* __restrict__ sf,
                                                            const float* __restrict__ s, int s_per_row,
                                                            int64_t rows, int nblocks, int kgroups,
                                                            uint16_t* __restrict__ y, int64_t ld_y) {
    const int64_t total = rows * nblocks;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t r = i / nblocks;
        const int b = static_cast<int>(i - r * nblocks);
        const uint2 codes = __ldg(reinterpret_cast<const uint2*>(q + r * (static_cast<int64_t>(nblocks) * 8)) + b);
        const uint32_t sb = __ldg(sf + sf_word_offset(r, b >> 2, kgroups) + (b & 3));
        const float S = __ldg(s + (s_per_row ? r : 0));
        uint32_t h2;
        const uint16_t sb2 = static_cast<uint16_t>(sb | (sb << 8));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(sb2));
        const __half2 scale = *reinterpret_cast<__half2*>(&h2);
        const float2 S2 = make_float2(S, S);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t word = j < 4 ? codes.x : codes.y;
            const __half2 v = __hmul2(e2m1x2_to_half2(word >> (8 * (j & 3))), scale);   // exact
            const float2 f = __fmul2_rn(__half22float2(v), S2);
            w[j] = bf16x2_rn(f.x, f.y);
        }
        uint4* dst = reinterpret_cast<uint4*>(y + r * ld_y + static_cast<int64_t>(b) * 16);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_dequantize(const void* q, const void* sf, const float* s, int32_t s_per_row,
                                         int64_t rows, int64_t cols, void* y, int64_t ld_y,
                                         nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (rows < 0 || cols <= 0 || cols % 16 != 0 || ld_y < cols || ld_y % 8 != 0) return NVFP4_ERR_SHAPE;
    if (cols > (int64_t(1) << 24) || rows > (int64_t(1) << 31)) return NVFP4_ERR_SHAPE;
    if (rows == 0) return NVFP4_OK;
    if (!q || !sf || !s || !y) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(q, 8) || !aligned(y, 16) || !aligned(s, 4)) return NVFP4_ERR_ALIGNMENT;
    const int nblocks = static_cast<int>(cols / 16);
    const int kgroups = static_cast<int>(ceil_div(cols, 64));
    const int64_t total = rows * nblocks;
    const int64_t want = ceil_div(total, kDqThreads);
    const int64_t cap = static_cast<int64_t>(ctx.sm_count) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    dequant_kernel<<<grid, kDqThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(q), static_cast<const uint8_t*>(sf), s, s_per_row, rows, nblocks,
        kgroups, static_cast<uint16_t*>(y), ld_y);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}
