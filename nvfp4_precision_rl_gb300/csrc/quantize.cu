// quantize.cu -- per-token two-level NVFP4 quantization (rows), the per-tensor
// variant, and the column-wise copy for the backward pass.
//
// Row kernel: one warp per row, 16-byte coalesced loads, the whole row held in
// registers so the amax (found with bf16x2 max and warp shuffles) is reused for
// the outer scale, the block scales and the encode without re-reading HBM
// ("Towards Blackwell-Native 8-bit and 4-bit RL", "Online per-token scale": the
// per-token FP32 scale is computed inside the quantize kernel and returned by the
// same call; "miniTE report", "Transformer Engine path optimisation": amax reuse).
// Lane l holds 8-element chunks l, l+32, ...; a 16-element block is the chunk
// pair (2j, 2j+1) held by lanes 2j and 2j+1, so block maxima need one shuffle.
#include "rowquant.cuh"

namespace nvfp4 {

namespace {

constexpr int kRowThreads = 256;            // 8 warps = 8 rows per block iteration

enum RowMode { kPerToken = 0, kPerTensor = 1, kAmaxOnly = 2 };

struct RowParams {
    const uint16_t* x;
    int64_t rows_in;
    int64_t ld_x;
    const int32_t* gather;
    int64_t rows_out;
    int64_t rows_pad;   // rows_out rounded up to 128 (rows of the swizzled scales)
    uint32_t* q;        // packed codes viewed as 32-bit words (8 codes each)
    uint8_t* sf;
    float* s;
    unsigned* amax_ws;  // global amax as float bits (non-negative floats order as unsigned)
    unsigned* status;
    int cols;
    int kgroups;        // 4-block groups per row = scale words per row
};

__device__ __forceinline__ int64_t source_row(const RowParams& p, int64_t r) {
    int64_t src = p.gather ? static_cast<int64_t>(p.gather[r]) : r;
    if (src >= p.rows_in) {
        record_error(p.status, NVFP4_ERR_DEVICE_INPUT, DETAIL_GATHER_INDEX);
        src = -1;
    }
    return src;
}

// Row kernel with the row held in registers: NCH chunks of 8 per lane (cols <= 256 * NCH).
template <int NCH, int MODE>
__global__ void __launch_bounds__(kRowThreads) quant_rows_kernel(RowParams p) {
    pdl_launch_dependents();    // a dependent waits for this grid's completion itself
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * (kRowThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kRowThreads / 32);
    const int nchunks = p.cols >> 3;
    const float tensor_amax = (MODE == kPerTensor) ? __uint_as_float(*p.amax_ws) : 0.0f;
    const int64_t row_end = (MODE == kAmaxOnly) ? p.rows_out : p.rows_pad;
    float seen_amax = 0.0f;

    for (int64_t r = warp0; r < row_end; r += nwarps) {
        if (r >= p.rows_out) {
            zero_sf_row(p.sf, p.kgroups, r, lane);
            continue;
        }
        const int64_t src = source_row(p, r);
        const uint4* xr = reinterpret_cast<const uint4*>(p.x + (src < 0 ? 0 : src) * p.ld_x);
        uint4 v[NCH];
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int c = i * 32 + lane;
            v[i] = (src >= 0 && c < nchunks) ? ldg_stream(xr + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        float bmax[NCH];
        const float row_amax = row_block_max<NCH>(v, bmax);
        seen_amax = fmaxf(seen_amax, row_amax);
        if (MODE == kAmaxOnly) continue;
        encode_row<NCH>(v, bmax, MODE == kPerTensor ? tensor_amax : row_amax, nchunks, p.kgroups,
                        p.q, p.sf, p.s, r, lane);
    }
    if (MODE != kPerTensor && p.amax_ws != nullptr && lane == 0 && seen_amax > 0.0f)
        atomicMax(p.amax_ws, __float_as_uint(seen_amax));
}

// Rows staged through shared memory by bulk TMA copies: persistent CTAs, each
// warp owns `depth` row buffers and keeps up to `depth` rows of its grid-stride
// sequence in flight (one cp.async.bulk per row, completion on a per-buffer
// mbarrier), so memory-level parallelism no longer depends on how many rows fit
// in registers.  The per-row arithmetic is the register kernel's (rowquant.cuh).
struct StageCfg {
    int depth;          // row buffers per warp
    uint32_t row_pad;   // bytes per row buffer (row bytes rounded up to 128)
};

__device__ __forceinline__ void bulk_row_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Rows of up to two tensors with the same number of columns: row slots
// [0, split) are tensor 0's rows and padding rows (rows_out .. rows_pad, whose
// swizzled scale words are zeroed), [split, total) tensor 1's.  One launch
// then quantizes, e.g., a linear layer's activation and its weight.
struct RowJob {
    RowParams t0, t1;
    int64_t split;      // row slots of tensor 0
    int64_t total;      // row slots of both
};

// Rows of up to 96 blocks (1536 columns) fit 64 registers per thread, so two
// CTAs share an SM when their row buffers fit: a warp's rows are a chain of
// dependent steps (wait, amax, the exact scale divides, encode), and more warps
// per SM keep more rows in flight.
template <int NB>
constexpr int staged_ctas_per_sm() { return NB <= 3 ? 2 : 1; }

template <int NB, int MODE>
__global__ void __launch_bounds__(512, staged_ctas_per_sm<NB>()) quant_rows_staged_kernel(RowJob job, StageCfg cfg) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();    // a dependent waits for this grid's completion itself
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    uint8_t* bufs = smem + static_cast<size_t>(warp) * cfg.depth * cfg.row_pad;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nwarps) * cfg.depth * cfg.row_pad) +
                     warp * cfg.depth;
    const int nblocks = job.t0.cols >> 4;
    const int kgroups = job.t0.kgroups;
    const uint32_t row_bytes = static_cast<uint32_t>(job.t0.cols) * 2u;
    const float tensor_amax = (MODE == kPerTensor) ? __uint_as_float(*job.t0.amax_ws) : 0.0f;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * nwarps;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * nwarps + warp;

    if (lane == 0) {
        for (int d = 0; d < cfg.depth; ++d) mbar_init(&bars[d], 1);
        fence_barrier_init();
    }
    __syncwarp();

    // source row of slot r (-1: a zero row or a padding row; no copy is issued)
    auto source = [&](int64_t r) -> int64_t {
        const bool sec = r >= job.split;
        const int64_t lr = sec ? r - job.split : r;
        const int64_t rows_out = sec ? job.t1.rows_out : job.t0.rows_out;
        if (lr >= rows_out) return -1;
        const int32_t* gather = sec ? job.t1.gather : job.t0.gather;
        int64_t src = gather ? static_cast<int64_t>(gather[lr]) : lr;
        if (src >= (sec ? job.t1.rows_in : job.t0.rows_in)) {
            record_error(job.t0.status, NVFP4_ERR_DEVICE_INPUT, DETAIL_GATHER_INDEX);
            src = -1;
        }
        return src;
    };
    // Start the copy of slot r into buffer d (a zero row only completes the phase).
    auto issue = [&](int64_t r, int d) {
        if (r >= job.total || lane != 0) return;
        const int64_t src = source(r);
        if (src >= 0) {
            const bool sec = r >= job.split;
            const uint16_t* x = sec ? job.t1.x : job.t0.x;
            const int64_t ld = sec ? job.t1.ld_x : job.t0.ld_x;
            mbar_arrive_expect_tx(&bars[d], row_bytes);
            bulk_row_load(bufs + static_cast<size_t>(d) * cfg.row_pad, x + src * ld, row_bytes, &bars[d]);
        } else {
            mbar_arrive(&bars[d]);
        }
    };
    for (int d = 0; d < cfg.depth; ++d) issue(first + d * stride, d);

    float seen0 = 0.0f, seen1 = 0.0f;
    uint32_t parity = 0;   // bit d = phase parity expected next on buffer d
    int d = 0;
    for (int64_t r = first; r < job.total; r += stride) {
        const bool sec = r >= job.split;
        const int64_t lr = sec ? r - job.split : r;
        const int64_t rows_out = sec ? job.t1.rows_out : job.t0.rows_out;
        const bool pad_row = lr >= rows_out;
        bool zero_row = pad_row;
        if (!pad_row) {
            const int32_t* gather = sec ? job.t1.gather : job.t0.gather;
            const int64_t src = gather ? static_cast<int64_t>(gather[lr]) : lr;
            zero_row = src < 0 || src >= (sec ? job.t1.rows_in : job.t0.rows_in);   // no copy was issued
        }
        bool ok = mbar_wait_bounded(&bars[d], (parity >> d) & 1u, 2000000000ull, nullptr);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
            if (lane == 0) {
                record_error(job.t0.status, NVFP4_ERR_TIMEOUT, DETAIL_NONE);
                // let the copies this warp still has in flight land before it exits
                for (int k = 0; k < cfg.depth; ++k) {
                    const int bb = (d + k) % cfg.depth;
                    if (r + k * stride < job.total)
                        mbar_wait_bounded(&bars[bb], (parity >> bb) & 1u, 200000000ull, nullptr);
                }
            }
            break;
        }
        parity ^= 1u << d;
        // A padding row gets zero scale words; a zero row of the output (no
        // source row) quantizes, per token, to zero codes, zero scales and S = 0,
        // written directly.
        if (pad_row || (MODE == kPerToken && zero_row)) {
            __syncwarp();
            issue(r + cfg.depth * stride, d);
            d = (d + 1 == cfg.depth) ? 0 : d + 1;
            zero_sf_row(sec ? job.t1.sf : job.t0.sf, kgroups, lr, lane);
            if (!pad_row) {
                uint2* qrow = reinterpret_cast<uint2*>(sec ? job.t1.q : job.t0.q) + lr * nblocks;
                for (int b = lane; b < nblocks; b += 32) qrow[b] = make_uint2(0u, 0u);
                if (lane == 0) (sec ? job.t1.s : job.t0.s)[lr] = 0.0f;
            }
            continue;
        }
        const uint4* row = reinterpret_cast<const uint4*>(bufs + static_cast<size_t>(d) * cfg.row_pad);
        Block16 v[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int b = i * 32 + lane;
            const bool in = !zero_row && b < nblocks;
            v[i].lo = in ? row[2 * b] : make_uint4(0u, 0u, 0u, 0u);
            v[i].hi = in ? row[2 * b + 1] : make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();                       // every lane has read the buffer
        issue(r + cfg.depth * stride, d);   // refill it with the row `depth` steps ahead
        d = (d + 1 == cfg.depth) ? 0 : d + 1;
        float bmax[NB];
        float row_amax = 0.0f;
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            bmax[i] = block_absmax(v[i]);
            row_amax = fmaxf(row_amax, bmax[i]);
        }
        row_amax = warp_max(row_amax);
        if (sec) seen1 = fmaxf(seen1, row_amax);
        else seen0 = fmaxf(seen0, row_amax);
        if (MODE == kAmaxOnly) continue;
        encode_row_blocks<NB>(v, bmax, MODE == kPerTensor ? tensor_amax : row_amax, nblocks, kgroups,
                              reinterpret_cast<uint2*>(sec ? job.t1.q : job.t0.q), sec ? job.t1.sf : job.t0.sf,
                              sec ? job.t1.s : job.t0.s, lr, lane);
    }
    if (MODE != kPerTensor && lane == 0) {
        if (job.t0.amax_ws != nullptr && seen0 > 0.0f) atomicMax(job.t0.amax_ws, __float_as_uint(seen0));
        if (job.t1.amax_ws != nullptr && seen1 > 0.0f) atomicMax(job.t1.amax_ws, __float_as_uint(seen1));
    }
}

// Rows longer than 256 * 16 elements: two passes over the row (the second from L1/L2).
// Narrow rows (up to 64 blocks = 1024 columns): each warp quantizes TWO rows
// per step, so a step's 2 x nblocks blocks fill whole lane rounds (768
// columns: 96 blocks = three rounds of 32 instead of 1.5 rounds per row with
// a quarter of the lanes idle) and the per-row work (the wait, the copy issue,
// the amax reduction, the outer scale) is shared by two rows.  Row pairs
// (2k, 2k+1) of the job's row slots are walked grid-stride per warp; a pair
// sits in one staging slot (both rows copied by bulk TMA, one mbarrier).  The
// per-block arithmetic is the one-row kernel's (rowquant.cuh): same bytes.
template <int NU, int MODE>
__global__ void __launch_bounds__(512, 2) quant_row_pairs_kernel(RowJob job, StageCfg cfg) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();    // a dependent waits for this grid's completion itself
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t slot_bytes = 2 * cfg.row_pad;
    uint8_t* bufs = smem + static_cast<size_t>(warp) * cfg.depth * slot_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nwarps) * cfg.depth * slot_bytes) +
                     warp * cfg.depth;
    const int nblocks = job.t0.cols >> 4;
    const int kgroups = job.t0.kgroups;
    const uint32_t row_bytes = static_cast<uint32_t>(job.t0.cols) * 2u;
    const float tensor_amax = (MODE == kPerTensor) ? __uint_as_float(*job.t0.amax_ws) : 0.0f;
    const int64_t pairs = (job.total + 1) >> 1;   // a last odd slot (amax-only pass) pairs with a pad row
    const int64_t stride = static_cast<int64_t>(gridDim.x) * nwarps;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * nwarps + warp;

    if (lane == 0) {
        for (int d = 0; d < cfg.depth; ++d) mbar_init(&bars[d], 1);
        fence_barrier_init();
    }
    __syncwarp();

    // source row of row slot r (-1: a pad row past rows_out, or a dropped gather index)
    auto source = [&](int64_t r) -> int64_t {
        const bool sec = r >= job.split;
        const RowParams& t = sec ? job.t1 : job.t0;
        const int64_t lr = sec ? r - job.split : r;
        if (lr >= t.rows_out) return -1;
        int64_t src = t.gather ? static_cast<int64_t>(t.gather[lr]) : lr;
        if (src >= t.rows_in) {
            record_error(job.t0.status, NVFP4_ERR_DEVICE_INPUT, DETAIL_GATHER_INDEX);
            src = -1;
        }
        return src;
    };
    // lane 0: copy pair k's rows with a source into slot d (one arrival; bytes as copied)
    auto issue = [&](int64_t k, int d) {
        if (k >= pairs || lane != 0) return;
        const int64_t s0 = source(2 * k), s1 = source(2 * k + 1);
        const bool sec = 2 * k >= job.split;
        const uint16_t* x = sec ? job.t1.x : job.t0.x;
        const int64_t ld = sec ? job.t1.ld_x : job.t0.ld_x;
        mbar_arrive_expect_tx(&bars[d], (s0 >= 0 ? row_bytes : 0u) + (s1 >= 0 ? row_bytes : 0u));
        uint8_t* dst = bufs + static_cast<size_t>(d) * slot_bytes;
        if (s0 >= 0) bulk_row_load(dst, x + s0 * ld, row_bytes, &bars[d]);
        if (s1 >= 0) bulk_row_load(dst + cfg.row_pad, x + s1 * ld, row_bytes, &bars[d]);
    };
    for (int d = 0; d < cfg.depth; ++d) issue(first + d * stride, d);

    float seen0 = 0.0f, seen1 = 0.0f;
    uint32_t parity = 0;
    int d = 0;
    for (int64_t k = first; k < pairs; k += stride) {
        const int64_t r0 = 2 * k;
        const bool sec = r0 >= job.split;
        const RowParams& t = sec ? job.t1 : job.t0;
        const int64_t lr0 = sec ? r0 - job.split : r0;
        // per row of the pair: pad (past rows_out: only its scale words are
        // written, as zeros) or zero (no source: encodes as a zero row)
        auto no_source = [&](int64_t lr) {
            if (lr >= t.rows_out) return true;
            const int64_t src = t.gather ? static_cast<int64_t>(t.gather[lr]) : lr;
            return src < 0 || src >= t.rows_in;
        };
        const bool pad0 = lr0 >= t.rows_out, pad1 = lr0 + 1 >= t.rows_out;
        const bool zero0 = no_source(lr0), zero1 = no_source(lr0 + 1);
        bool ok = mbar_wait_bounded(&bars[d], (parity >> d) & 1u, 2000000000ull, nullptr);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
            if (lane == 0) {
                record_error(job.t0.status, NVFP4_ERR_TIMEOUT, DETAIL_NONE);
                for (int j = 0; j < cfg.depth; ++j) {
                    const int bb = (d + j) % cfg.depth;
                    if (k + j * stride < pairs) mbar_wait_bounded(&bars[bb], (parity >> bb) & 1u, 200000000ull, nullptr);
                }
            }
            break;
        }
        parity ^= 1u << d;
        const uint8_t* slot = bufs + static_cast<size_t>(d) * slot_bytes;
        // unit u = i * 32 + lane: row u / nblocks, block u % nblocks
        Block16 v[NU];
        int hrow[NU], blk[NU];
#pragma unroll
        for (int i = 0; i < NU; ++i) {
            const int u = i * 32 + lane;
            hrow[i] = u >= nblocks ? 1 : 0;
            blk[i] = u - hrow[i] * nblocks;
            const bool in = u < 2 * nblocks && !(hrow[i] ? zero1 : zero0);
            const uint4* row = reinterpret_cast<const uint4*>(slot + hrow[i] * cfg.row_pad);
            v[i].lo = in ? row[2 * blk[i]] : make_uint4(0u, 0u, 0u, 0u);
            v[i].hi = in ? row[2 * blk[i] + 1] : make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();                       // every lane has read the slot
        issue(k + cfg.depth * stride, d);   // refill it with the pair `depth` steps ahead
        d = (d + 1 == cfg.depth) ? 0 : d + 1;
        float bmax[NU];
        float am0 = 0.0f, am1 = 0.0f;
#pragma unroll
        for (int i = 0; i < NU; ++i) {
            bmax[i] = block_absmax(v[i]);
            if (hrow[i]) am1 = fmaxf(am1, bmax[i]);
            else am0 = fmaxf(am0, bmax[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            am0 = fmaxf(am0, __shfl_xor_sync(0xFFFFFFFFu, am0, o));
            am1 = fmaxf(am1, __shfl_xor_sync(0xFFFFFFFFu, am1, o));
        }
        if (sec) seen1 = fmaxf(seen1, fmaxf(am0, am1));
        else seen0 = fmaxf(seen0, fmaxf(am0, am1));
        if (MODE == kAmaxOnly) continue;
        const ScaleRecipe rec0(MODE == kPerTensor ? tensor_amax : am0);
        const ScaleRecipe rec1(MODE == kPerTensor ? tensor_amax : am1);
        // the pair's two code rows are consecutive: unit u is block u of the pair
        uint2* const qpair = reinterpret_cast<uint2*>(t.q) + lr0 * nblocks;
        // the pair's scale bytes: both rows lie in one 32-row group of a 128-row
        // scale tile (lr0 even), row lr0 + 1 16 bytes after row lr0, group g of a
        // row 512 g bytes after its group 0
        uint8_t* const sfpair = t.sf + sf_word_offset(lr0, 0, kgroups);
        // the FMA form of the scale arithmetic when both rows allow it
        auto encode = [&](auto form) {
#pragma unroll
            for (int i = 0; i < NU; ++i) {
                const int u = i * 32 + lane;
                const int h = hrow[i];
                const int b = blk[i];
                if (u >= 2 * nblocks) continue;
                const uint32_t sfo = (static_cast<uint32_t>(h) << 4) + (static_cast<uint32_t>(b >> 2) << 9) + (b & 3);
                if (h ? pad1 : pad0) {
                    // a pad row's scale words are zero (blocks 4g.. of its row, one byte each)
                    if ((b >> 2) < kgroups) sfpair[sfo] = 0;
                    continue;
                }
                float rb;
                const uint32_t sb = (h ? rec1 : rec0).template block_as<decltype(form)::value>(bmax[i], &rb);
                const float2 r2 = make_float2(rb, rb);
                qpair[u] = make_uint2(encode8(v[i].lo, r2), encode8(v[i].hi, r2));
                sfpair[sfo] = static_cast<uint8_t>(sb);
            }
        };
        if (rec0.fast && rec1.fast) encode(std::true_type{});
        else encode(std::false_type{});
        // the padding of a row's last scale word (blocks nblocks .. 4 kgroups) is zero
        if (lane < 2 && (nblocks & 3) != 0) {
            const int64_t lr = lr0 + lane;
            for (int b = nblocks; b < 4 * kgroups; ++b) t.sf[sf_word_offset(lr, b >> 2, kgroups) + (b & 3)] = 0;
        }
        if (lane < 2 && !(lane ? pad1 : pad0)) t.s[lr0 + lane] = (lane ? rec1 : rec0).S;
    }
    if (MODE != kPerTensor && lane == 0) {
        if (job.t0.amax_ws != nullptr && seen0 > 0.0f) atomicMax(job.t0.amax_ws, __float_as_uint(seen0));
        if (job.t1.amax_ws != nullptr && seen1 > 0.0f) atomicMax(job.t1.amax_ws, __float_as_uint(seen1));
    }
}

template <int MODE>
__global__ void __launch_bounds__(kRowThreads) quant_rows_long_kernel(RowParams p) {
    pdl_launch_dependents();    // a dependent waits for this grid's completion itself
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * (kRowThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kRowThreads / 32);
    const int nchunks = p.cols >> 3;
    const int rounds = (nchunks + 31) / 32;
    const float tensor_amax = (MODE == kPerTensor) ? __uint_as_float(*p.amax_ws) : 0.0f;
    const int64_t row_end = (MODE == kAmaxOnly) ? p.rows_out : p.rows_pad;
    float seen_amax = 0.0f;

    for (int64_t r = warp0; r < row_end; r += nwarps) {
        if (r >= p.rows_out) {
            zero_sf_row(p.sf, p.kgroups, r, lane);
            continue;
        }
        const int64_t src = source_row(p, r);
        const uint4* xr = reinterpret_cast<const uint4*>(p.x + (src < 0 ? 0 : src) * p.ld_x);
        float row_amax = 0.0f;
        for (int i = 0; i < rounds; ++i) {
            const int c = i * 32 + lane;
            if (src >= 0 && c < nchunks) row_amax = fmaxf(row_amax, chunk_absmax(__ldg(xr + c)));
        }
        row_amax = warp_max(row_amax);
        seen_amax = fmaxf(seen_amax, row_amax);
        if (MODE == kAmaxOnly) continue;
        const ScaleRecipe rec(MODE == kPerTensor ? tensor_amax : row_amax);
        uint32_t* qrow = p.q + r * nchunks;
        for (int i = 0; i < rounds; ++i) {
            const int c = i * 32 + lane;
            const uint4 v = (src >= 0 && c < nchunks) ? __ldg(xr + c) : make_uint4(0u, 0u, 0u, 0u);
            const float m8 = chunk_absmax(v);
            const float bm = fmaxf(m8, __shfl_xor_sync(0xFFFFFFFFu, m8, 1));
            float rb;
            const uint32_t sb = rec.block(bm, &rb);
            const uint32_t w = encode_chunk(v, rb);
            if (c < nchunks) qrow[c] = w;
            store_sf_word(p.sf, p.kgroups, r, i, lane, sb);
        }
        if (lane == 0) p.s[r] = rec.S;
    }
    if (MODE != kPerTensor && p.amax_ws != nullptr && lane == 0 && seen_amax > 0.0f)
        atomicMax(p.amax_ws, __float_as_uint(seen_amax));
}

// ---------------------------------------------------------------------------
// Column-wise copy: X^T quantized along tokens with the per-tensor scale.
// A warp owns 64 columns (2 per lane, read as bf16x2 so each token row is one
// 128-byte load) and 64 tokens = 4 blocks of 16 = one scale word per column.
// ---------------------------------------------------------------------------
struct ColParams {
    const uint16_t* x;
    int64_t rows_in;
    int64_t ld_x;
    const int32_t* gather;
    int64_t rows_out;   // tokens, % 16 == 0
    uint8_t* q;         // [cols, rows_out / 2]
    uint8_t* sf;        // swizzled [round_up(cols, 128), round_up(rows_out / 16, 4)]
    float* s;
    const unsigned* amax_ws;
    unsigned* status;
    int cols;
    int kgroups;        // scale words per column row = ceil(rows_out / 64)
};

constexpr int kColThreads = 128;

// |a| max |b| on bf16 pairs (exact: max of bf16 values).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t m, uint32_t v) {
    uint32_t out;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(out) : "r"(m), "r"(v & 0x7FFF7FFFu));
    return out;
}

// Codes of one column's 16-token block: tokens t (low nibble) and t + 1 (high).
// `sel` picks the column's half of each 32-bit pair of columns.
template <bool kHi>
__device__ __forceinline__ uint2 encode_col_block(const uint32_t* v, float r) {
    const float2 rr = make_float2(r, r);
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float x0 = kHi ? bf16hi(v[2 * i]) : bf16lo(v[2 * i]);
        const float x1 = kHi ? bf16hi(v[2 * i + 1]) : bf16lo(v[2 * i + 1]);
        const float2 y = __fmul2_rn(make_float2(x0, x1), rr);
        b[i] = cvt_e2m1x2(y.x, y.y);
    }
    return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                      b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// Column-wise copy: thread = 2 adjacent columns (one 32-bit load per token) x
// 64 tokens (4 blocks of 16 = one swizzled scale word per column); all 64 loads
// are in flight before any arithmetic.  Amax uses packed bf16 max, the
// multiply packed FP32x2; each column's 32 code bytes of the group are written
// as two 16-byte stores when the row pitch allows it.
template <bool kGather>
__global__ void __launch_bounds__(kColThreads) quant_cols_kernel(ColParams p) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int k0 = blockIdx.x * 64 + lane * 2;
    const int g = blockIdx.y * (kColThreads / 32) + warp;   // token group of 64
    if (g >= p.kgroups) return;
    const int64_t m0 = static_cast<int64_t>(g) * 64;
    const bool col_ok = k0 < p.cols;

    // x and the gather rows are complete before this kernel starts: the row
    // pass it follows is launched without programmatic serialization, so it
    // began only after their producers had finished, and this kernel begins
    // after the row pass has.  The loads therefore run ahead of the wait;
    // only the tensor amax comes from the row pass.
    uint32_t v[64];
    if (!kGather && col_ok && m0 + 64 <= p.rows_out) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.x + m0 * p.ld_x + k0);
        const int64_t step = p.ld_x >> 1;   // 32-bit words per row
#pragma unroll
        for (int t = 0; t < 64; ++t) v[t] = __ldg(src + t * step);
    } else {
#pragma unroll
        for (int t = 0; t < 64; ++t) {
            const int64_t m = m0 + t;
            int64_t src = -1;
            if (m < p.rows_out) {
                src = kGather ? static_cast<int64_t>(p.gather[m]) : m;
                if (src >= p.rows_in) src = -1;   // reported by the row pass
            }
            v[t] = (col_ok && src >= 0)
                       ? __ldg(reinterpret_cast<const uint32_t*>(p.x + src * p.ld_x + k0))
                       : 0u;
        }
    }
    pdl_wait();                 // the row pass's tensor amax
    const ScaleRecipe rec(__uint_as_float(*p.amax_ws));
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) p.s[0] = rec.S;
    uint32_t word0 = 0u, word1 = 0u;
    uint2 c0[4], c1[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t m = 0u;
#pragma unroll
        for (int t = 0; t < 16; ++t) m = bf16x2_absmax(m, v[16 * b + t]);
        float r0, r1;
        const uint32_t s0 = rec.block(bf16lo(m), &r0);
        const uint32_t s1 = rec.block(bf16hi(m), &r1);
        word0 |= s0 << (8 * b);
        word1 |= s1 << (8 * b);
        c0[b] = encode_col_block<false>(v + 16 * b, r0);
        c1[b] = encode_col_block<true>(v + 16 * b, r1);
    }
    if (col_ok) {
        const int64_t qstride = p.rows_out >> 1;
        uint8_t* q0 = p.q + k0 * qstride + (m0 >> 1);
        uint8_t* q1 = q0 + qstride;
        if (m0 + 64 <= p.rows_out && (qstride & 15) == 0) {
            reinterpret_cast<uint4*>(q0)[0] = make_uint4(c0[0].x, c0[0].y, c0[1].x, c0[1].y);
            reinterpret_cast<uint4*>(q0)[1] = make_uint4(c0[2].x, c0[2].y, c0[3].x, c0[3].y);
            reinterpret_cast<uint4*>(q1)[0] = make_uint4(c1[0].x, c1[0].y, c1[1].x, c1[1].y);
            reinterpret_cast<uint4*>(q1)[1] = make_uint4(c1[2].x, c1[2].y, c1[3].x, c1[3].y);
        } else {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                if (m0 + 16 * b < p.rows_out) {
                    reinterpret_cast<uint2*>(q0)[b] = c0[b];
                    reinterpret_cast<uint2*>(q1)[b] = c1[b];
                }
            }
        }
    }
    // scale words (padding columns k >= cols get zero words)
    *reinterpret_cast<uint32_t*>(p.sf + sf_word_offset(k0, g, p.kgroups)) = col_ok ? word0 : 0u;
    *reinterpret_cast<uint32_t*>(p.sf + sf_word_offset(k0 + 1, g, p.kgroups)) = col_ok ? word1 : 0u;
}

// Staged-kernel geometry: as many warps x row buffers as fit in ~200 KB.
bool staged_config(int cols, int* warps, StageCfg* cfg) {
    const uint32_t pad = static_cast<uint32_t>(round_up(static_cast<int64_t>(cols) * 2, 128));
    const size_t budget = 200 * 1024;
    const int choices[5][2] = {{16, 3}, {16, 2}, {12, 2}, {8, 3}, {8, 2}};
    for (const auto& c : choices) {
        if (static_cast<size_t>(c[0]) * c[1] * (pad + 8) <= budget) {
            *warps = c[0];
            cfg->depth = c[1];
            cfg->row_pad = pad;
            return true;
        }
    }
    return false;
}

template <int NB, int MODE>
nvfp4_status launch_staged(const RowJob& job, int warps, StageCfg cfg, const DeviceCtx& ctx, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(warps) * cfg.depth * (cfg.row_pad + 8);
    static unsigned long long attr[64] = {};   // per context: see ctx_cached
    if (!ctx_cached(attr, ctx)) {
        if (cudaFuncSetAttribute(quant_rows_staged_kernel<NB, MODE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 210 * 1024) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        ctx_cache_set(attr, ctx);
    }
    const int64_t want = ceil_div(job.total, warps);
    const int per_sm = (staged_ctas_per_sm<NB>() == 2 && 2 * smem <= 220 * 1024) ? 2 : 1;
    const int64_t cap = static_cast<int64_t>(ctx.sm_count) * per_sm;
    const int grid = static_cast<int>(want < cap ? want : cap);
    quant_rows_staged_kernel<NB, MODE><<<grid, warps * 32, smem, s>>>(job, cfg);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}

template <int NU, int MODE>
nvfp4_status launch_row_pairs(const RowJob& job, const DeviceCtx& ctx, cudaStream_t s) {
    constexpr int kWarps = 16;
    StageCfg cfg;
    cfg.depth = 2;
    cfg.row_pad = static_cast<uint32_t>(round_up(static_cast<int64_t>(job.t0.cols) * 2, 128));
    const size_t smem = static_cast<size_t>(kWarps) * cfg.depth * (2 * cfg.row_pad + 8);
    static unsigned long long attr[64] = {};   // per context: see ctx_cached
    if (!ctx_cached(attr, ctx)) {
        if (cudaFuncSetAttribute(quant_row_pairs_kernel<NU, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 210 * 1024) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        ctx_cache_set(attr, ctx);
    }
    const int64_t want = ceil_div((job.total + 1) / 2, kWarps);
    const int64_t cap = static_cast<int64_t>(ctx.sm_count) * (2 * smem <= 220 * 1024 ? 2 : 1);
    const int grid = static_cast<int>(want < cap ? want : cap);
    quant_row_pairs_kernel<NU, MODE><<<grid, kWarps * 32, smem, s>>>(job, cfg);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}

// Staged path for a job (one or two tensors with the same columns); false if
// the row does not fit the staged geometry (the caller falls back).  Rows of
// up to 64 blocks go two per warp step.
template <int MODE>
bool try_launch_staged(const RowJob& job, const DeviceCtx& ctx, cudaStream_t s, nvfp4_status* st) {
    const int nblocks = job.t0.cols / 16;
    if (nblocks <= 64) {
        const int nu = (2 * nblocks + 31) / 32;    // units (blocks of the row pair) per lane
        if (nu <= 1) *st = launch_row_pairs<1, MODE>(job, ctx, s);
        else if (nu <= 2) *st = launch_row_pairs<2, MODE>(job, ctx, s);
        else if (nu <= 3) *st = launch_row_pairs<3, MODE>(job, ctx, s);
        else *st = launch_row_pairs<4, MODE>(job, ctx, s);
        return true;
    }
    int warps = 0;
    StageCfg cfg{0, 0};
    const int nb = (job.t0.cols / 16 + 31) / 32;   // 16-element blocks per lane
    if (nb > 8 || !staged_config(job.t0.cols, &warps, &cfg)) return false;
    if (nb <= 1) *st = launch_staged<1, MODE>(job, warps, cfg, ctx, s);
    else if (nb <= 2) *st = launch_staged<2, MODE>(job, warps, cfg, ctx, s);
    else if (nb <= 3) *st = launch_staged<3, MODE>(job, warps, cfg, ctx, s);
    else if (nb <= 4) *st = launch_staged<4, MODE>(job, warps, cfg, ctx, s);
    else if (nb <= 5) *st = launch_staged<5, MODE>(job, warps, cfg, ctx, s);
    else if (nb <= 6) *st = launch_staged<6, MODE>(job, warps, cfg, ctx, s);
    else *st = launch_staged<8, MODE>(job, warps, cfg, ctx, s);
    return true;
}

template <int MODE>
nvfp4_status launch_rows(const RowParams& p, int blocks, const DeviceCtx& ctx, cudaStream_t s) {
    RowJob job;
    job.t0 = p;
    job.t1 = p;
    job.t1.rows_out = 0;
    job.t1.rows_pad = 0;
    job.t1.amax_ws = nullptr;
    job.split = (MODE == kAmaxOnly) ? p.rows_out : p.rows_pad;
    job.total = job.split;
    nvfp4_status st = NVFP4_OK;
    if (try_launch_staged<MODE>(job, ctx, s, &st)) return st;
    const int need = (p.cols / 8 + 31) / 32;
    if (need <= 1) quant_rows_kernel<1, MODE><<<blocks, kRowThreads, 0, s>>>(p);
    else if (need <= 2) quant_rows_kernel<2, MODE><<<blocks, kRowThreads, 0, s>>>(p);
    else if (need <= 4) quant_rows_kernel<4, MODE><<<blocks, kRowThreads, 0, s>>>(p);
    else if (need <= 8) quant_rows_kernel<8, MODE><<<blocks, kRowThreads, 0, s>>>(p);
    else if (need <= 12) quant_rows_kernel<12, MODE><<<blocks, kRowThreads, 0, s>>>(p);
    else if (need <= 16) quant_rows_kernel<16, MODE><<<blocks, kRowThreads, 0, s>>>(p);
    else quant_rows_long_kernel<MODE><<<blocks, kRowThreads, 0, s>>>(p);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}

}  // namespace

// Per-token rows of two tensors with the same columns in one launch (row
// kernel's staged path; two launches when the row is too long for it).
nvfp4_status quantize_rows_pair_launch(const RowParams& a, const RowParams& b, const DeviceCtx& ctx,
                                       cudaStream_t s) {
    RowJob job;
    job.t0 = a;
    job.t1 = b;
    job.split = a.rows_pad;
    job.total = a.rows_pad + b.rows_pad;
    if (job.total == 0) return NVFP4_OK;
    nvfp4_status st = NVFP4_OK;
    if (try_launch_staged<kPerToken>(job, ctx, s, &st)) return st;
    if (a.rows_pad > 0) {
        const int64_t want = ceil_div(a.rows_pad, kRowThreads / 32);
        st = launch_rows<kPerToken>(a, static_cast<int>(want < 1048576 ? want : 1048576), ctx, s);
        if (st != NVFP4_OK) return st;
    }
    if (b.rows_pad > 0) {
        const int64_t want = ceil_div(b.rows_pad, kRowThreads / 32);
        st = launch_rows<kPerToken>(b, static_cast<int>(want < 1048576 ? want : 1048576), ctx, s);
    }
    return st;
}

RowParams row_params(const void* x, int64_t rows, int64_t cols, int64_t ld, void* q, void* sf, float* s,
                     unsigned* amax_ws, unsigned* status) {
    RowParams p;
    p.x = static_cast<const uint16_t*>(x);
    p.rows_in = rows;
    p.ld_x = ld;
    p.gather = nullptr;
    p.rows_out = rows;
    p.rows_pad = round_up(rows, 128);
    p.q = static_cast<uint32_t*>(q);
    p.sf = static_cast<uint8_t*>(sf);
    p.s = s;
    p.amax_ws = amax_ws;
    p.status = status;
    p.cols = static_cast<int>(cols);
    p.kgroups = static_cast<int>(round_up(cols / 16, 4) / 4);
    return p;
}

// Shared by the ABI entry and by the SwiGLU file's requantize check.
nvfp4_status quantize_rows_launch(const uint16_t* x, int64_t rows_in, int64_t cols, int64_t ld_x,
                                  const int32_t* gather, int64_t rows_out, int mode, void* q,
                                  void* sf, float* s, unsigned* amax_ws, bool publish_amax,
                                  const DeviceCtx& ctx, cudaStream_t stream) {
    RowParams p;
    p.x = x;
    p.rows_in = rows_in;
    p.ld_x = ld_x;
    p.gather = gather;
    p.rows_out = rows_out;
    p.rows_pad = round_up(rows_out, 128);
    p.q = static_cast<uint32_t*>(q);
    p.sf = static_cast<uint8_t*>(sf);
    p.s = s;
    p.amax_ws = (mode == kPerTensor || publish_amax) ? amax_ws : nullptr;
    p.status = ctx.status;
    p.cols = static_cast<int>(cols);
    p.kgroups = static_cast<int>(round_up(cols / 16, 4) / 4);
    const int64_t rows_launch = (mode == kAmaxOnly) ? rows_out : p.rows_pad;
    if (rows_launch == 0) return NVFP4_OK;
    const int64_t want = ceil_div(rows_launch, kRowThreads / 32);
    const int blocks = static_cast<int>(want < 1048576 ? want : 1048576);
    if (mode == kPerToken) return launch_rows<kPerToken>(p, blocks, ctx, stream);
    if (mode == kPerTensor) return launch_rows<kPerTensor>(p, blocks, ctx, stream);
    return launch_rows<kAmaxOnly>(p, blocks, ctx, stream);
}

nvfp4_status quantize_cols_launch(const uint16_t* x, int64_t rows_in, int64_t cols, int64_t ld_x,
                                  const int32_t* gather, int64_t rows_out, void* q, void* sf,
                                  float* s, const unsigned* amax_ws, const DeviceCtx& ctx,
                                  cudaStream_t stream) {
    ColParams p;
    p.x = x;
    p.rows_in = rows_in;
    p.ld_x = ld_x;
    p.gather = gather;
    p.rows_out = rows_out;
    p.q = static_cast<uint8_t*>(q);
    p.sf = static_cast<uint8_t*>(sf);
    p.s = s;
    p.amax_ws = amax_ws;
    p.status = ctx.status;
    p.cols = static_cast<int>(cols);
    p.kgroups = static_cast<int>(ceil_div(rows_out, 64));
    if (p.kgroups == 0) {
        return cudaMemsetAsync(s, 0, sizeof(float), stream) == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
    }
    dim3 grid(static_cast<unsigned>(round_up(cols, 128) / 64),
              static_cast<unsigned>(ceil_div(p.kgroups, kColThreads / 32)));
    // programmatic serialization: the kernel may start while the row pass
    // finishes; it loads x at once and waits (griddepcontrol.wait) before
    // reading the row pass's amax.  The row pass must therefore be launched
    // without that attribute (it starts after x's producers have finished).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kColThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = (gather != nullptr) ? cudaLaunchKernelEx(&cfg, quant_cols_kernel<true>, p)
                                              : cudaLaunchKernelEx(&cfg, quant_cols_kernel<false>, p);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

size_t nvfp4_quantize_workspace_bytes(void) { return 256; }

nvfp4_status nvfp4_quantize_per_token(const void* x, int64_t rows_in, int64_t cols, int64_t ld_x,
                                      const int32_t* gather_rows, int64_t rows_out,
                                      nvfp4_scale_mode mode, void* q_row, void* sf_row,
                                      float* s_row, void* q_col, void* sf_col, float* s_col,
                                      void* workspace, size_t workspace_bytes,
                                      nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (mode != NVFP4_SCALE_PER_TOKEN && mode != NVFP4_SCALE_PER_TENSOR) return NVFP4_ERR_INVALID_ARG;
    if (rows_in < 0 || rows_out < 0 || cols <= 0) return NVFP4_ERR_SHAPE;
    if (cols % 16 != 0 || cols > (int64_t(1) << 24) || ld_x < cols || ld_x % 8 != 0) return NVFP4_ERR_SHAPE;
    if (gather_rows == nullptr && rows_out > rows_in) return NVFP4_ERR_SHAPE;
    const bool want_col = (q_col != nullptr) || (sf_col != nullptr) || (s_col != nullptr);
    if (want_col && (q_col == nullptr || sf_col == nullptr || s_col == nullptr)) return NVFP4_ERR_INVALID_ARG;
    if (want_col && rows_out % 16 != 0) return NVFP4_ERR_SHAPE;
    if (rows_out > 0 && (q_row == nullptr || sf_row == nullptr || s_row == nullptr)) return NVFP4_ERR_INVALID_ARG;
    if (rows_out > 0 && rows_in > 0 && x == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q_row, 16) || !aligned(sf_row, 16) || !aligned(s_row, 4) ||
        !aligned(gather_rows, 4) || !aligned(q_col, 16) || !aligned(sf_col, 16) || !aligned(s_col, 4))
        return NVFP4_ERR_ALIGNMENT;
    const bool need_ws = want_col || mode == NVFP4_SCALE_PER_TENSOR;
    if (need_ws && (workspace == nullptr || workspace_bytes < nvfp4_quantize_workspace_bytes()))
        return NVFP4_ERR_WORKSPACE;
    if (need_ws && !aligned(workspace, 4)) return NVFP4_ERR_ALIGNMENT;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    unsigned* amax_ws = static_cast<unsigned*>(workspace);
    if (need_ws && cudaMemsetAsync(amax_ws, 0, sizeof(unsigned), s) != cudaSuccess) return NVFP4_ERR_CUDA;

    if (mode == NVFP4_SCALE_PER_TENSOR) {
        st = quantize_rows_launch(xb, rows_in, cols, ld_x, gather_rows, rows_out, kAmaxOnly, nullptr,
                                  nullptr, nullptr, amax_ws, true, ctx, s);
        if (st != NVFP4_OK) return st;
    }
    st = quantize_rows_launch(xb, rows_in, cols, ld_x, gather_rows, rows_out, mode, q_row, sf_row,
                              s_row, amax_ws, want_col && mode == NVFP4_SCALE_PER_TOKEN, ctx, s);
    if (st != NVFP4_OK) return st;
    if (want_col)
        st = quantize_cols_launch(xb, rows_in, cols, ld_x, gather_rows, rows_out, q_col, sf_col,
                                  s_col, amax_ws, ctx, s);
    return st;
}

nvfp4_status nvfp4_quantize_per_token_pair(const void* x, int64_t rows_x, int64_t ld_x, void* q_x,
                                           void* sf_x, float* s_x, void* q_col, void* sf_col,
                                           float* s_col, const void* w, int64_t rows_w, int64_t ld_w,
                                           void* q_w, void* sf_w, float* s_w, int64_t cols,
                                           void* workspace, size_t workspace_bytes,
                                           nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (rows_x < 0 || rows_w < 0 || cols <= 0 || cols % 16 != 0 || cols > (int64_t(1) << 24))
        return NVFP4_ERR_SHAPE;
    if (ld_x < cols || ld_x % 8 != 0 || ld_w < cols || ld_w % 8 != 0) return NVFP4_ERR_SHAPE;
    const bool want_col = (q_col != nullptr) || (sf_col != nullptr) || (s_col != nullptr);
    if (want_col && (q_col == nullptr || sf_col == nullptr || s_col == nullptr)) return NVFP4_ERR_INVALID_ARG;
    if (want_col && rows_x % 16 != 0) return NVFP4_ERR_SHAPE;
    if (rows_x > 0 && (x == nullptr || q_x == nullptr || sf_x == nullptr || s_x == nullptr))
        return NVFP4_ERR_INVALID_ARG;
    if (rows_w > 0 && (w == nullptr || q_w == nullptr || sf_w == nullptr || s_w == nullptr))
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q_x, 16) || !aligned(sf_x, 16) || !aligned(s_x, 4) ||
        !aligned(w, 16) || !aligned(q_w, 16) || !aligned(sf_w, 16) || !aligned(s_w, 4) ||
        !aligned(q_col, 16) || !aligned(sf_col, 16) || !aligned(s_col, 4))
        return NVFP4_ERR_ALIGNMENT;
    if (want_col && (workspace == nullptr || workspace_bytes < nvfp4_quantize_workspace_bytes()))
        return NVFP4_ERR_WORKSPACE;
    if (want_col && !aligned(workspace, 4)) return NVFP4_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned* amax_ws = want_col ? static_cast<unsigned*>(workspace) : nullptr;
    if (want_col && cudaMemsetAsync(amax_ws, 0, sizeof(unsigned), s) != cudaSuccess) return NVFP4_ERR_CUDA;
    const RowParams a = row_params(x, rows_x, cols, ld_x, q_x, sf_x, s_x, amax_ws, ctx.status);
    const RowParams b = row_params(w, rows_w, cols, ld_w, q_w, sf_w, s_w, nullptr, ctx.status);
    // the weight's rows first, the activation's last: its column-wise copy (the
    // next kernel) then re-reads it from L2 rather than HBM
    st = quantize_rows_pair_launch(b, a, ctx, s);
    if (st != NVFP4_OK) return st;
    if (want_col)
        st = quantize_cols_launch(static_cast<const uint16_t*>(x), rows_x, cols, ld_x, nullptr, rows_x, q_col,
                                  sf_col, s_col, amax_ws, ctx, s);
    return st;
}

}  // extern "C"
