// swiglu.cu -- fused SwiGLU + per-token NVFP4 quantize: the input of the MoE fc2
// GEMM built straight from the fc1 output, h = bf16(silu(gate) * up), without
// writing h to HBM unless asked ("Towards Blackwell-Native 8-bit and 4-bit RL",
// "Parallelism and tensor-conversion contract": gate and up projections are one
// fused GEMM in a SwiGLU MoE layer).  The quantize step is the row quantizer's
// own code (rowquant.cuh), so it is bit-exact given h; h itself is within one
// bf16 ulp of bf16(silu(g) u) evaluated exactly.
#include "rowquant.cuh"
#include "swiglu.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

struct SwiParams {
    const uint16_t* y1;
    int64_t rows;
    int64_t rows_pad;
    int64_t ld;
    const int32_t* row_count;
    uint32_t* q;
    uint8_t* sf;
    float* s;
    uint16_t* h;
    int ffn;
    int kgroups;
};

template <int NCH>
__global__ void __launch_bounds__(kThreads) swiglu_quant_kernel(SwiParams p) {
    pdl_launch_dependents();    // a dependent waits for this grid's completion itself
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    const int nchunks = p.ffn >> 3;
    int64_t limit = p.rows;
    if (p.row_count != nullptr) {
        const int64_t rc = *p.row_count;
        limit = rc < 0 ? 0 : (rc < p.rows ? rc : p.rows);
    }
    for (int64_t r = warp0; r < p.rows_pad; r += nwarps) {
        if (r >= p.rows) {
            zero_sf_row(p.sf, p.kgroups, r, lane);
            continue;
        }
        uint4 g[NCH], u[NCH];
        const uint4* gr = reinterpret_cast<const uint4*>(p.y1 + r * p.ld);
        const uint4* ur = reinterpret_cast<const uint4*>(p.y1 + r * p.ld + p.ffn);
        uint32_t bits = 0u;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int c = i * 32 + lane;
            g[i] = make_uint4(0u, 0u, 0u, 0u);
            u[i] = g[i];
            if (r < limit && c < nchunks) {
                g[i] = ldg_stream(gr + c);
                u[i] = ldg_stream(ur + c);
            }
            bits |= g[i].x | g[i].y | g[i].z | g[i].w | u[i].x | u[i].y | u[i].z | u[i].w;
        }
        // A row whose inputs are all +0 (an expert layout's padding, or a row
        // past row_count) gives h = +0 and quantizes to zero codes, zero
        // scales and S = 0: written directly.
        if (!__any_sync(0xFFFFFFFFu, bits != 0u)) {
            for (int c = lane; c < nchunks; c += 32) {
                p.q[r * nchunks + c] = 0u;
                if (p.h != nullptr) reinterpret_cast<uint4*>(p.h + r * p.ffn)[c] = make_uint4(0u, 0u, 0u, 0u);
            }
            zero_sf_row(p.sf, p.kgroups, r, lane);
            if (lane == 0) p.s[r] = 0.0f;
            continue;
        }
        uint4 v[NCH];
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int c = i * 32 + lane;
            uint4 hv;
            hv.x = swiglu_pair(g[i].x, u[i].x);
            hv.y = swiglu_pair(g[i].y, u[i].y);
            hv.z = swiglu_pair(g[i].z, u[i].z);
            hv.w = swiglu_pair(g[i].w, u[i].w);
            if (p.h != nullptr && c < nchunks)
                reinterpret_cast<uint4*>(p.h + r * p.ffn)[c] = hv;
            v[i] = hv;
        }
        float bmax[NCH];
        const float amax = row_block_max<NCH>(v, bmax);
        encode_row<NCH>(v, bmax, amax, nchunks, p.kgroups, p.q, p.sf, p.s, r, lane);
    }
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_swiglu_quantize(const void* y1, int64_t rows, int64_t ffn,
                                              int64_t ld_y1, const int32_t* row_count, void* q,
                                              void* sf, float* s, void* h, nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (rows < 0 || ffn <= 0 || ffn % 16 != 0 || ffn > 16 * 256 || ld_y1 < 2 * ffn || ld_y1 % 8 != 0)
        return NVFP4_ERR_SHAPE;
    if (rows > 0 && (y1 == nullptr || q == nullptr || sf == nullptr || s == nullptr))
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(y1, 16) || !aligned(q, 16) || !aligned(sf, 16) || !aligned(s, 4) ||
        !aligned(row_count, 4) || !aligned(h, 16))
        return NVFP4_ERR_ALIGNMENT;
    if (rows == 0) return NVFP4_OK;
    SwiParams p;
    p.y1 = static_cast<const uint16_t*>(y1);
    p.rows = rows;
    p.rows_pad = round_up(rows, 128);
    p.ld = ld_y1;
    p.row_count = row_count;
    p.q = static_cast<uint32_t*>(q);
    p.sf = static_cast<uint8_t*>(sf);
    p.s = s;
    p.h = static_cast<uint16_t*>(h);
    p.ffn = static_cast<int>(ffn);
    p.kgroups = static_cast<int>(round_up(ffn / 16, 4) / 4);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const int blocks = static_cast<int>(ceil_div(p.rows_pad, kThreads / 32));
    const int need = static_cast<int>((ffn / 8 + 31) / 32);
    if (need <= 1) swiglu_quant_kernel<1><<<blocks, kThreads, 0, cs>>>(p);
    else if (need <= 2) swiglu_quant_kernel<2><<<blocks, kThreads, 0, cs>>>(p);
    else if (need <= 3) swiglu_quant_kernel<3><<<blocks, kThreads, 0, cs>>>(p);
    else if (need <= 4) swiglu_quant_kernel<4><<<blocks, kThreads, 0, cs>>>(p);
    else if (need <= 8) swiglu_quant_kernel<8><<<blocks, kThreads, 0, cs>>>(p);
    else swiglu_quant_kernel<16><<<blocks, kThreads, 0, cs>>>(p);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}
