// rowquant.cuh -- the per-row NVFP4 encode shared by the row quantizer and the
// fused SwiGLU + quantize kernel (one warp per row; lane l holds 8-element
// chunks l, l+32, ...; a 16-element block is the chunk pair held by lanes 2j
// and 2j+1).
#pragma once

#include "common.cuh"

namespace nvfp4 {

constexpr uint32_t kAbsMask2 = 0x7FFF7FFFu;  // clears both bf16 sign bits

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a),
                               *reinterpret_cast<__nv_bfloat162*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

// max |x| over 8 bf16 values, as float
__device__ __forceinline__ float chunk_absmax(const uint4& v) {
    uint32_t m = bmax2(bmax2(v.x & kAbsMask2, v.y & kAbsMask2), bmax2(v.z & kAbsMask2, v.w & kAbsMask2));
    return fmaxf(bf16lo(m), bf16hi(m));
}

__device__ __forceinline__ uint32_t encode_chunk(const uint4& v, float r) {
    return cvt_e2m1x8(__fmul_rn(bf16lo(v.x), r), __fmul_rn(bf16hi(v.x), r),
                      __fmul_rn(bf16lo(v.y), r), __fmul_rn(bf16hi(v.y), r),
                      __fmul_rn(bf16lo(v.z), r), __fmul_rn(bf16hi(v.z), r),
                      __fmul_rn(bf16lo(v.w), r), __fmul_rn(bf16hi(v.w), r));
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ int64_t sf_word_offset(int64_t r, int g, int kgroups) {
    return ((r >> 7) * kgroups + g) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4;
}


// Scale words of one row: lanes 8g..8g+7 hold blocks 4g'..4g'+3 of a chunk
// round (each block twice); lane 8g writes the four codes as one word.
__device__ __forceinline__ void store_sf_word(uint8_t* sf, int kgroups, int64_t r, int round,
                                              int lane, uint32_t sb) {
    const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
    const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sb, 4);
    const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sb, 6);
    if ((lane & 7) == 0) {
        const int g = round * 4 + (lane >> 3);
        if (g < kgroups)
            *reinterpret_cast<uint32_t*>(sf + sf_word_offset(r, g, kgroups)) =
                sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
    }
}

__device__ __forceinline__ void zero_sf_row(uint8_t* sf, int kgroups, int64_t r, int lane) {
    for (int g = lane; g < kgroups; g += 32)
        *reinterpret_cast<uint32_t*>(sf + sf_word_offset(r, g, kgroups)) = 0u;
}

// Block maxima (per lane chunk pair) and the row amax of a row held in registers.
template <int NCH>
__device__ __forceinline__ float row_block_max(const uint4 (&v)[NCH], float (&bmax)[NCH]) {
    float row_amax = 0.0f;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const float m8 = chunk_absmax(v[i]);
        bmax[i] = fmaxf(m8, __shfl_xor_sync(0xFFFFFFFFu, m8, 1));
        row_amax = fmaxf(row_amax, m8);
    }
    return warp_max(row_amax);
}

// Encode a register-resident row with outer-scale amax `amax`: codes, scale
// words and the FP32 outer scale of row r.
template <int NCH>
__device__ __forceinline__ void encode_row(const uint4 (&v)[NCH], const float (&bmax)[NCH],
                                           float amax, int nchunks, int kgroups, uint32_t* q,
                                           uint8_t* sf, float* s, int64_t r, int lane) {
    const ScaleRecipe rec(amax);
    uint32_t* qrow = q + r * nchunks;
    auto encode = [&](auto form) {
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int c = i * 32 + lane;
            float rb;
            const uint32_t sb = rec.template block_as<decltype(form)::value>(bmax[i], &rb);
            const uint32_t w = encode_chunk(v[i], rb);
            if (c < nchunks) qrow[c] = w;
            store_sf_word(sf, kgroups, r, i, lane, sb);
        }
    };
    if (rec.fast) encode(std::true_type{});
    else encode(std::false_type{});
    if (lane == 0) s[r] = rec.S;
}

// ---------------------------------------------------------------------------
// Block-per-lane variant: lane l owns 16-element blocks l, l+32, ... of a row
// (32 contiguous bytes each, read from shared memory), so the block scale is
// computed once per block and the 16 multiplies run as 8 packed FP32x2 ops.
// ---------------------------------------------------------------------------
struct Block16 {
    uint4 lo, hi;   // elements 0..7 and 8..15 of the block (bf16 pairs)
};

// max(|a|, |b|) per bf16 half, with the sign of a XOR b (max.xorsign.abs): the
// magnitudes of a max tree need no masking until its root
__device__ __forceinline__ uint32_t amax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float block_absmax(const Block16& b) {
    const uint32_t m = amax2(amax2(amax2(b.lo.x, b.lo.y), amax2(b.lo.z, b.lo.w)),
                             amax2(amax2(b.hi.x, b.hi.y), amax2(b.hi.z, b.hi.w))) & kAbsMask2;
    return fmaxf(bf16lo(m), bf16hi(m));
}

// x * r for the two bf16 values of a word (correctly rounded, like __fmul_rn).
__device__ __forceinline__ float2 scale_pair(uint32_t w, float2 r2) {
    return __fmul2_rn(make_float2(bf16lo(w), bf16hi(w)), r2);
}

__device__ __forceinline__ uint32_t encode8(const uint4& v, float2 r2) {
    const float2 a = scale_pair(v.x, r2), b = scale_pair(v.y, r2);
    const float2 c = scale_pair(v.z, r2), d = scale_pair(v.w, r2);
    return cvt_e2m1x8(a.x, a.y, b.x, b.y, c.x, c.y, d.x, d.y);
}

// Encode a row whose blocks sit in registers (NB blocks per lane, block
// b = i * 32 + lane): codes, scale words and the outer scale of row r.
template <int NB>
__device__ __forceinline__ void encode_row_blocks(const Block16 (&v)[NB], const float (&bmax)[NB],
                                                  float amax, int nblocks, int kgroups, uint2* q,
                                                  uint8_t* sf, float* s, int64_t r, int lane) {
    const ScaleRecipe rec(amax);
    uint2* qrow = q + r * nblocks;
    uint8_t* const sfrow = sf + sf_word_offset(r, 0, kgroups);   // group g is 512 g bytes further
    auto encode = [&](auto form) {
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int b = i * 32 + lane;
            float rb;
            const uint32_t sb = rec.template block_as<decltype(form)::value>(bmax[i], &rb);
            const float2 r2 = make_float2(rb, rb);
            const uint2 w = make_uint2(encode8(v[i].lo, r2), encode8(v[i].hi, r2));
            if (b < nblocks) qrow[b] = w;
            // each lane writes its block's scale byte: four consecutive lanes
            // fill one swizzled word (blocks past the row's end write zero bytes)
            if ((b >> 2) < kgroups) sfrow[(static_cast<uint32_t>(b >> 2) << 9) + (b & 3)] = static_cast<uint8_t>(sb);
        }
    };
    if (rec.fast) encode(std::true_type{});
    else encode(std::false_type{});
    if (lane == 0) s[r] = rec.S;
}

}  // namespace nvfp4
