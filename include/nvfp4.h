/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) per-token NVFP4 W4A4 linear-layer path.
 *
 * The computation is the two-level NVFP4 contract
 *     X ~ s_token * s_block * X_FP4
 * ("Towards Blackwell-Native 8-bit and 4-bit RL: End-to-End MXFP8 and NVFP4 RL
 * in Miles", section "How it works": X_FP4 are 16 E2M1 values, s_block their E4M3
 * block scale, s_token an FP32 per-token scale computed online inside the
 * quantizer; "TRIAGE: Direction-Aware Mismatch Stabilization of Native NVFP4 RL",
 * section "NVFP4 quantization format and W4A4 execution":
 * x^_j = S * s_b * Q_E2M1(x_j / (S * s_b))), followed by block-scaled FP4 GEMMs
 * with the per-token scale applied in the GEMM epilogue ("Towards Blackwell-Native
 * 8-bit and 4-bit RL", results item 10).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All data pointers are DEVICE pointers unless a parameter says "host".  The
 *    caller allocates every buffer; the library never allocates.  Sizes of the
 *    derived buffers come from the *_bytes helpers below.
 *  - Every call is asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *    NULL is the legacy default stream).  Nothing synchronises the host except
 *    nvfp4_get_device_status().
 *  - Errors are returned as nvfp4_status; nothing is thrown across the ABI.  A
 *    call that returns an error has launched nothing.  Errors detected on the
 *    device (a bounded wait that ran out, an out-of-range device-side index) are
 *    recorded in a per-device status word and reported by
 *    nvfp4_get_device_status().
 *  - Calls work in the CUDA context current on the calling thread.  The device
 *    addresses the library caches (its status word, the no-alloc permute's
 *    scratch array) and its per-kernel attributes belong to one context: they
 *    are looked up or set again whenever the current context differs from the
 *    one they were taken in (another context made current, or a new primary
 *    context after cudaDeviceReset).
 *  - The device must be compute capability 10.3 (GB300, sm_103a).
 *  - Matrix layouts are row-major with the contraction axis K contiguous
 *    (nn.Linear layout: X [M, K], W [N, K]).  bf16 data are 2-byte bfloat16.
 *
 * Quantized tensor format (produced by nvfp4_quantize_per_token, consumed by the
 * GEMMs) for a [rows, cols] matrix, cols % 16 == 0:
 *  - packed codes  uint8 [rows, cols/2]: byte j holds element 2j in its low
 *                  nibble and element 2j+1 in its high nibble; an E2M1 code is
 *                  sign(bit 3) | exponent(bits 2..1) | mantissa(bit 0).
 *  - block scales  E4M3 (bias 7, max 448) codes, one per 16 contiguous elements
 *                  of a row, stored SWIZZLED: rows padded to a multiple of 128,
 *                  blocks per row padded to a multiple of 4, cut into 128 x 4
 *                  tiles of 512 bytes in row-tile-major order; inside a tile row
 *                  r sits at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + block % 4.
 *                  Padding bytes are written as 0.  (The pages ask that such
 *                  backend layouts be explicit and verifiable: "Towards
 *                  Blackwell-Native 8-bit and 4-bit RL", future work item 3.)
 *  - outer scales  float32 [rows]: S_t = amax_t / 2688 (2688 = 6 * 448).
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* nvfp4_stream_t;

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,        /* NULL where a buffer is required, bad enum, negative size */
    NVFP4_ERR_ALIGNMENT = 2,          /* a pointer or leading dimension breaks its alignment rule */
    NVFP4_ERR_SHAPE = 3,              /* a size breaks its divisibility / range rule */
    NVFP4_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
    NVFP4_ERR_CUDA = 5,               /* a CUDA runtime call failed (launch, memset, ...) */
    NVFP4_ERR_TIMEOUT = 6,            /* device side: a bounded wait ran out; the kernel exited early */
    NVFP4_ERR_DEVICE_INPUT = 7,       /* device side: an input value was out of range (e.g. expert id) */
    NVFP4_ERR_WORKSPACE = 8           /* workspace missing or smaller than the *_workspace_bytes() size */
} nvfp4_status;

typedef enum {
    NVFP4_SCALE_PER_TOKEN = 0,   /* one FP32 outer scale per row (the recipe's choice) */
    NVFP4_SCALE_PER_TENSOR = 1   /* one FP32 outer scale for the whole matrix (comparison mode) */
} nvfp4_scale_mode;

/* ------------------------------------------------------------------------- */
/* Sizes                                                                     */
/* ------------------------------------------------------------------------- */

/* Bytes of the packed codes of a [rows, cols] matrix: rows * cols / 2. */
NVFP4_API size_t nvfp4_packed_bytes(int64_t rows, int64_t cols);

/* Bytes of the swizzled block scales of a [rows, cols] matrix:
 * round_up(rows, 128) * round_up(cols / 16, 4). */
NVFP4_API size_t nvfp4_sf_bytes(int64_t rows, int64_t cols);

/* ------------------------------------------------------------------------- */
/* Per-token two-level quantization                                          */
/* ------------------------------------------------------------------------- */

/* Scratch bytes nvfp4_quantize_per_token needs when mode is
 * NVFP4_SCALE_PER_TENSOR or a column-wise copy is requested (one global amax
 * word, padded); 0 is never returned. */
NVFP4_API size_t nvfp4_quantize_workspace_bytes(void);

/*
 * Quantize the rows of X (per-token amax, FP32 outer scale, E4M3 16-block
 * scales, E2M1 codes, round-to-nearest-even, saturating), in one pass that
 * keeps each row in registers and reuses its amax for the scale and the encode
 * ("Towards Blackwell-Native 8-bit and 4-bit RL", "Online per-token scale": one
 * call returns the packed FP4 values, the E4M3 block scales and the per-token
 * FP32 scale; "miniTE report", "Transformer Engine path optimisation": amax
 * reuse).  Exact IEEE arithmetic, no fast math (same page, "Bit-exact quantizer
 * contract"); the operation order is:
 *   S = amax / 2688, T = 6 * S, per block: d = amax_b / T (0 if T == 0),
 *   s_b = E4M3(d), D = S * s_b, r = 1 / D (0 if D == 0, clamped to FLT_MAX),
 *   q = E2M1(x * r).
 *
 *  x            bf16 [rows_in, ld_x]; row i starts at x + i * ld_x elements.
 *               16-byte aligned, ld_x % 8 == 0, ld_x >= cols.
 *  rows_in      rows of x (>= 0).
 *  cols         K, > 0, % 16 == 0.  (The GEMMs additionally need K % 64 == 0.)
 *  gather_rows  NULL: output row r reads x row r (rows_out <= rows_in).
 *               Otherwise int32 [rows_out]: output row r reads x row
 *               gather_rows[r], or is a zero row when gather_rows[r] < 0 (MoE
 *               padding).  An index >= rows_in makes a zero row and records
 *               NVFP4_ERR_DEVICE_INPUT.
 *  rows_out     rows produced (>= 0).
 *  mode         NVFP4_SCALE_PER_TOKEN or NVFP4_SCALE_PER_TENSOR (amax over all
 *               output rows; every s_row entry is then equal).
 *  q_row        uint8 [rows_out, cols/2], 16-byte aligned.
 *  sf_row       nvfp4_sf_bytes(rows_out, cols) bytes, 16-byte aligned; padding
 *               rows and blocks are written as 0.
 *  s_row        float [rows_out].
 *  q_col, sf_col, s_col
 *               all NULL: no column-wise copy.  Otherwise the column-wise copy
 *               for the backward pass ("Towards Blackwell-Native 8-bit and 4-bit
 *               RL", "Backward activation representation": row- and column-wise
 *               copies quantized independently from full precision): X^T
 *               [cols, rows_out] quantized with 16-blocks along the token axis
 *               and ONE per-tensor outer scale S_col = (max over rows of
 *               amax_t) / 2688.  q_col uint8 [cols, rows_out/2], sf_col
 *               nvfp4_sf_bytes(cols, rows_out) bytes, s_col float [1].
 *               Requires rows_out % 16 == 0.
 *  workspace    device scratch of workspace_bytes >= nvfp4_quantize_workspace_bytes(),
 *               4-byte aligned; required for per-tensor mode or a column copy,
 *               ignored (may be NULL) otherwise.  Its contents need not be
 *               initialised; it must not be shared with a call in flight on
 *               another stream.
 * Returns NVFP4_OK or an error code (nothing launched on error).
 */
NVFP4_API nvfp4_status nvfp4_quantize_per_token(
    const void* x, int64_t rows_in, int64_t cols, int64_t ld_x,
    const int32_t* gather_rows, int64_t rows_out, nvfp4_scale_mode mode,
    void* q_row, void* sf_row, float* s_row,
    void* q_col, void* sf_col, float* s_col,
    void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * Per-token quantization of a linear layer's two GEMM operands with the same
 * K in one launch: x (an activation, optionally with its column-wise copy) and
 * w (a weight, per output row).  Each tensor's bytes are exactly those of
 * nvfp4_quantize_per_token on it alone (per-token scales make every row
 * independent: "Towards Blackwell-Native 8-bit and 4-bit RL", "Online
 * computation of the per-token scale").  One kernel walks the rows of both,
 * so the two small quantizations share one ramp-up.
 *
 *  x, w           bf16 [rows_x, ld_x], [rows_w, ld_w]; 16-byte aligned, ld % 8 == 0.
 *  q_x, sf_x, s_x and q_w, sf_w, s_w   as nvfp4_quantize_per_token's row outputs.
 *  q_col, sf_col, s_col   all NULL, or x's column-wise copy (rows_x % 16 == 0;
 *                 needs the workspace, nvfp4_quantize_workspace_bytes()).
 *  cols           > 0, % 16 == 0.
 */
NVFP4_API nvfp4_status nvfp4_quantize_per_token_pair(
    const void* x, int64_t rows_x, int64_t ld_x, void* q_x, void* sf_x, float* s_x,
    void* q_col, void* sf_col, float* s_col,
    const void* w, int64_t rows_w, int64_t ld_w, void* q_w, void* sf_w, float* s_w,
    int64_t cols, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------- */
/* MoE routing permute                                                       */
/* ------------------------------------------------------------------------- */

/* Rows a padded per-expert layout can need: tokens * topk + num_experts *
 * (row_align - 1), rounded up to row_align. */
NVFP4_API int64_t nvfp4_moe_capacity(int64_t tokens, int32_t topk, int32_t num_experts, int32_t row_align);

/* Scratch bytes of nvfp4_moe_permute (per-expert totals and per-chunk expert histograms). */
NVFP4_API size_t nvfp4_moe_permute_workspace_bytes(int64_t tokens, int32_t topk, int32_t num_experts);

/*
 * Build the contiguous per-expert row layout the grouped GEMM consumes, with
 * all metadata left on the device ("miniTE report", "Transformer Engine path
 * optimisation": contiguous layouts and device-side metadata).  Expert e owns
 * rows [expert_offsets[e], expert_offsets[e+1]), its routed (token, slot) pairs
 * first in ascending (token, slot) order, then padding rows up to a multiple of
 * row_align.
 *
 *  topk_ids        int32 [tokens, topk], values in [0, num_experts).  An id out
 *                  of range is dropped (dst_rows = -1) and NVFP4_ERR_DEVICE_INPUT
 *                  is recorded.
 *  tokens, topk    >= 0 and 1..64.
 *  num_experts     1..1024.
 *  row_align       >= 1; the grouped GEMM needs a multiple of 128 (256
 *                  balances its tiles best).
 *  expert_offsets  int32 [num_experts + 1] (output).
 *  gather_rows     int32 [capacity] (output): source token of each row, -1 for
 *                  padding and for rows past expert_offsets[num_experts].
 *  capacity        rows of gather_rows, >= nvfp4_moe_capacity(...).
 *  dst_rows        int32 [tokens, topk] (output): row of each (token, slot).
 *  workspace       >= nvfp4_moe_permute_workspace_bytes(...) bytes, 4-byte aligned.
 */
NVFP4_API nvfp4_status nvfp4_moe_permute(
    const int32_t* topk_ids, int64_t tokens, int32_t topk, int32_t num_experts,
    int32_t row_align, int32_t* expert_offsets, int32_t* gather_rows, int64_t capacity,
    int32_t* dst_rows, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_moe_permute for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers that
 * cannot call cudaMalloc (or any allocating routine) where they route tokens:
 * runtimes whose device memory is owned by another allocator (a framework's
 * caching allocator, a serving engine's pre-reserved pool) that nothing else
 * may grow, and decode loops that forbid allocation on the hot path, where a
 * cudaMalloc would synchronise the device.  It computes exactly what
 * nvfp4_moe_permute computes, with the same arguments minus the workspace: the
 * per-chunk histogram scratch lives in a fixed 1 MiB __device__ array inside
 * this library, which every device that loads the library holds until the
 * process exits.
 *
 *  Limit: nvfp4_moe_permute_workspace_bytes(tokens, topk, num_experts) must be
 *  <= 1 MiB (for 128 experts: up to 2,096,128 routed (token, slot) pairs);
 *  larger sizes return NVFP4_ERR_WORKSPACE and launch nothing.
 *  The first call on a device (and the first in each further CUDA context on
 *  it) looks up the array's device address, with that device current, and so
 *  should come before any stream capture.
 *  Nothing in the array needs to start at zero (every histogram entry read is
 *  first written by the same call), but every call shares it: calls that
 *  overlap on the GPU (other streams, other host threads) race and must be
 *  serialised by the caller.  Nothing is allocated or freed by this call.
 */
NVFP4_API nvfp4_status nvfp4_moe_permute_noalloc(
    const int32_t* topk_ids, int64_t tokens, int32_t topk, int32_t num_experts,
    int32_t row_align, int32_t* expert_offsets, int32_t* gather_rows, int64_t capacity,
    int32_t* dst_rows, nvfp4_stream_t stream);

/*
 * Scatter per-token quantized rows into the routed (expert) layout: output row
 * r is row gather_rows[r] of the source quantization -- its packed codes, its
 * swizzled block-scale words and its FP32 outer scale -- or a zero row (zero
 * codes, zero scales, S = 0) when gather_rows[r] < 0.  Per-token quantization
 * of a row depends on that row alone ("Towards Blackwell-Native 8-bit and
 * 4-bit RL", "Online computation of the per-token scale"), so
 * nvfp4_quantize_per_token(X) followed by this call produces, bit for bit,
 * what nvfp4_quantize_per_token(X, gather_rows) produces, with 1/topk of the
 * quantization work.
 *
 *  q_src, sf_src, s_src  a per-token quantization of X [rows_src, cols]
 *               (nvfp4_quantize_per_token without gather): uint8 [rows_src,
 *               cols/2], nvfp4_sf_bytes(rows_src, cols) bytes, float [rows_src].
 *  cols         > 0, % 16 == 0.
 *  gather_rows  int32 [rows_out] (device); an index >= rows_src makes a zero row
 *               and records NVFP4_ERR_DEVICE_INPUT.
 *  expert_offsets  int32 [num_experts + 1] (device) or NULL: the layout's
 *               expert offsets (nvfp4_moe_permute's output for these
 *               gather_rows).  They set only the ORDER in which the 128-row
 *               tiles are written, never the result: tile j of every expert,
 *               then tile j + 1, so that the k copies of a token (whose rows sit
 *               at about the same relative place in each expert, the permute
 *               being stable in token order) are read while the token's row is
 *               still in L2.  NULL, num_experts outside [1, 256] or offsets
 *               that are negative or decreasing give the layout's own order.
 *  num_experts  number of experts of expert_offsets (ignored when it is NULL).
 *  q, sf, s     uint8 [rows_out, cols/2], nvfp4_sf_bytes(rows_out, cols) bytes
 *               (scale rows past rows_out written as 0), float [rows_out].
 *  Pointers 16-byte aligned (s, s_src, gather_rows, expert_offsets: 4).
 *  rows_out == 0 is a no-op.
 */
NVFP4_API nvfp4_status nvfp4_moe_gather_quantized(
    const void* q_src, const void* sf_src, const float* s_src, int64_t rows_src, int64_t cols,
    const int32_t* gather_rows, int64_t rows_out, const int32_t* expert_offsets, int32_t num_experts,
    void* q, void* sf, float* s, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Block-scaled W4A4 GEMMs                                                   */
/* ------------------------------------------------------------------------- */

/*
 * Y[m, n] = bf16_rn( S_a[m] * S_b[n] * sum_k dec(a)[m,k] * dec(b)[n,k] ), with
 * dec(.) = E4M3 block scale * E2M1 value, accumulated in FP32 by the tcgen05
 * block-scaled tensor-core MMA; the per-token scale is applied in the epilogue
 * (not as a separate pass: "Towards Blackwell-Native 8-bit and 4-bit RL",
 * results item 10).
 *
 *  a_q, a_sf, a_s  quantized A (activations) [M, K] as produced by
 *                  nvfp4_quantize_per_token: packed codes, swizzled scales
 *                  (nvfp4_sf_bytes(M, K) bytes), float [M].
 *  b_q, b_sf, b_s  quantized B (weights) [N, K], same format.
 *  M >= 0, N > 0 with N % 16 == 0, K > 0 with K % 64 == 0.
 *  y               bf16 [M, ld_y], ld_y >= N, ld_y % 8 == 0, 16-byte aligned.
 *  a_q, b_q, a_sf, b_sf: 16-byte aligned.
 */
NVFP4_API nvfp4_status nvfp4_gemm(
    const void* a_q, const void* a_sf, const float* a_s, int64_t M,
    const void* b_q, const void* b_sf, const float* b_s, int64_t N, int64_t K,
    void* y, int64_t ld_y, nvfp4_stream_t stream);

/*
 * nvfp4_gemm with a choice of outer-scale granularity per operand:
 * a_s_per_row / b_s_per_row != 0 read S_a[m] / S_b[n] from arrays as above;
 * == 0 read one scale a_s[0] / b_s[0] for every row -- the column-wise copies'
 * single per-tensor scale.  This makes the NVFP4 backward GEMMs ("Towards
 * Blackwell-Native 8-bit and 4-bit RL", "Backward activation representation
 * trade-off" and the backward modes; the pages' recipe itself runs these in
 * BF16):
 *   dgrad  dX[M, K]  = dY[M, N] W[N, K]:   A = dY (rows, per token),
 *                      B = W's column-wise copy [K, N] (one scale);
 *   wgrad  dW[N, K]  = dY^T X:             A = dY's column-wise copy [N, M],
 *                      B = X's column-wise copy [K, M] (one scale each).
 * Shapes and alignment as nvfp4_gemm (the contraction length K % 64 == 0).
 */
NVFP4_API nvfp4_status nvfp4_gemm_ex(
    const void* a_q, const void* a_sf, const float* a_s, int32_t a_s_per_row, int64_t M,
    const void* b_q, const void* b_sf, const float* b_s, int32_t b_s_per_row, int64_t N, int64_t K,
    void* y, int64_t ld_y, nvfp4_stream_t stream);

/*
 * Grouped (MoE) W4A4 GEMM: for every expert e, rows m in
 * [expert_offsets[e], expert_offsets[e+1]) of A are multiplied by expert e's
 * weights:  Y[m, n] = bf16_rn( S_a[m] * S_b[e, n] * sum_k dec(a)[m,k] dec(b_e)[n,k] ).
 * The offsets are read on the device; no host synchronisation is needed after
 * nvfp4_moe_permute ("miniTE report", "Transformer Engine path optimisation":
 * grouped GEMM with device-side metadata).
 *
 *  a_q, a_sf, a_s   quantized A with rows_capacity rows (the padded per-expert
 *                   layout; sf: nvfp4_sf_bytes(rows_capacity, K) bytes).
 *  rows_capacity    rows of A and Y; expert_offsets[E] must be <= rows_capacity
 *                   and every expert_offsets[e] % 128 == 0 (else
 *                   NVFP4_ERR_DEVICE_INPUT is recorded and the tile is skipped).
 *                   When every offset is a multiple of 256 (nvfp4_moe_permute
 *                   with row_align 256) the kernel walks 256-row slots, each a
 *                   full two-SM tile, which spreads the tiles evenly over the
 *                   SM pairs; with 128-row alignment an expert with an odd
 *                   number of 128-row tiles computes (and drops) 128 rows
 *                   past its segment.
 *  expert_offsets   int32 [E + 1] (device), nondecreasing.
 *  E                1..1024.
 *  b_q              uint8 [E, N, K/2]: expert e's packed weights at b_q + e*N*K/2.
 *  b_sf             E blocks of nvfp4_sf_bytes(N, K) bytes, expert e's at
 *                   b_sf + e * nvfp4_sf_bytes(N, K).
 *  b_s              float [E, N].
 *  N % 16 == 0, K % 64 == 0.
 *  y                bf16 [rows_capacity, N]; rows >= expert_offsets[E] are not written.
 */
NVFP4_API nvfp4_status nvfp4_grouped_gemm(
    const void* a_q, const void* a_sf, const float* a_s, int64_t rows_capacity,
    const int32_t* expert_offsets, int32_t E,
    const void* b_q, const void* b_sf, const float* b_s, int64_t N, int64_t K,
    void* y, nvfp4_stream_t stream);

/*
 * Grouped W4A4 GEMM of a SwiGLU expert's fused gate + up projection with the
 * SwiGLU in its epilogue: for every expert e and row m of its segment,
 *     g[m, j] = Y[m, j],  u[m, j] = Y[m, F + j]    (Y as nvfp4_grouped_gemm
 *                                                   computes it, rounded to bf16)
 *     h[m, j] = bf16(silu(g) * u)                  (j < F)
 * -- the same bits as nvfp4_grouped_gemm with N = 2F followed by
 * nvfp4_swiglu_quantize's h, without writing or re-reading Y ("Towards
 * Blackwell-Native 8-bit and 4-bit RL", "Parallelism and tensor-conversion
 * consistency contract": gate and up are one fused GEMM in a SwiGLU MoE layer;
 * the gate is the first half).  A pair tile multiplies gate rows n0 .. n0+127
 * and the matching up rows F+n0 .. of B, so no weight reordering is needed.
 *
 *  a_*, rows_capacity, expert_offsets, E   as for nvfp4_grouped_gemm.
 *  b_q, b_sf, b_s   expert weights with 2F rows each (gate rows 0..F-1, up rows
 *                   F..2F-1), laid out as for nvfp4_grouped_gemm with N = 2F.
 *  ffn              F; F % 128 == 0, K % 64 == 0.
 *  h                bf16 [rows_capacity, F]; rows >= expert_offsets[E] are
 *                   written as zeros (so a per-token quantization of all
 *                   rows_capacity rows gives zero rows there).
 */
NVFP4_API nvfp4_status nvfp4_grouped_gemm_swiglu(
    const void* a_q, const void* a_sf, const float* a_s, int64_t rows_capacity,
    const int32_t* expert_offsets, int32_t E,
    const void* b_q, const void* b_sf, const float* b_s, int64_t ffn, int64_t K,
    void* h, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Unpermute + weighted combine (after the MoE fc2)                          */
/* ------------------------------------------------------------------------- */

/*
 * out[t, h] = bf16_rn( sum_{j < topk} w[t, j] * y2[dst_rows[t*topk + j], h] ),
 * the routed experts' outputs brought back to token order and reduced with the
 * router weights in high precision ("Towards Blackwell-Native 8-bit and 4-bit
 * RL", shared-expert section): binary32, slot order j = 0..topk-1, each step
 * one rounded multiply and one rounded add.  Bit-exact.
 *
 *  y2        bf16 [rows, ld_y2] (the fc2 output in the padded expert layout),
 *            ld_y2 >= hidden, ld_y2 % 8 == 0, 16-byte aligned.
 *  dst_rows  int32 [tokens * topk] on the device (nvfp4_moe_permute's dst_rows).
 *            A row outside [0, rows) contributes nothing and sets the device
 *            status to NVFP4_ERR_DEVICE_INPUT.
 *  weights   float [tokens, topk] on the device.
 *  topk      1..32.  hidden > 0, % 8 == 0.
 *  out       bf16 [tokens, ld_out], ld_out >= hidden, ld_out % 8 == 0, 16-byte aligned.
 */
NVFP4_API nvfp4_status nvfp4_moe_combine(
    const void* y2, int64_t rows, int64_t ld_y2, const int32_t* dst_rows, const float* weights,
    int64_t tokens, int32_t topk, int64_t hidden, void* out, int64_t ld_out, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Dequantize (NVFP4 -> BF16)                                                */
/* ------------------------------------------------------------------------- */

/*
 * y[r, k] = bf16_rn( fl32( S_r * fl32( dec(q[r, k]) * dec(s_b[r, k / 16]) ) ) ):
 * the NVFP4 value x^ = S * dec(s_b) * dec(q) ("TRIAGE", section "NVFP4
 * quantization format and W4A4 execution") evaluated in binary32 -- the
 * code-times-block-scale product is exact, the multiply by the FP32 outer
 * scale rounds once to binary32 -- then rounded to bf16, nearest-even.  Serves
 * the dequantized-BF16 backward ("Towards Blackwell-Native 8-bit and 4-bit RL",
 * NVFP4 backward modes).  Bit-exact.
 *
 *  q          packed E2M1 [rows, cols/2], low nibble = even k; 8-byte aligned.
 *  sf         swizzled E4M3 block scales, nvfp4_sf_bytes(rows, cols) bytes.
 *  s          float outer scales: s[r] when s_per_row != 0, else s[0] for every
 *             row (the column-wise copy's single per-tensor scale).
 *  cols       > 0, % 16 == 0.
 *  y          bf16 [rows, ld_y], ld_y >= cols, ld_y % 8 == 0, 16-byte aligned.
 *  Errors: NVFP4_ERR_SHAPE / _ALIGNMENT / _INVALID_ARG; rows == 0 is a no-op.
 */
NVFP4_API nvfp4_status nvfp4_dequantize(
    const void* q, const void* sf, const float* s, int32_t s_per_row, int64_t rows, int64_t cols,
    void* y, int64_t ld_y, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------- */
/* MXFP8 (E4M3 values, E8M0 scale per 32 values)                             */
/* ------------------------------------------------------------------------- */

/* Bytes of a swizzled E8M0 scale array for [rows, cols]: the 128 x 4 tile
 * layout of nvfp4_sf_bytes with one byte per 32 values,
 * round_up(rows, 128) * round_up(ceil(cols / 32), 4); 0 when either is <= 0. */
NVFP4_API size_t nvfp4_mxfp8_sf_bytes(int64_t rows, int64_t cols);

/*
 * MXFP8 quantization ("Towards Blackwell-Native 8-bit and 4-bit RL", MXFP8
 * format background; "Backward activation representation trade-off"): each
 * 1x32 block of a row shares the scale 2^e, e the smallest integer >= -127
 * with 448 * 2^e >= the block's amax (stored as the E8M0 code e + 127); each
 * value is E4M3_RNE_satfinite(x * 2^-e), the product exact.  With q_col/sf_col
 * the same is done for the 32x1 blocks of each column, stored as X^T.
 * Bit-exact.
 *
 *  x       bf16 [rows, ld_x], ld_x >= cols, ld_x % 8 == 0, 16-byte aligned.
 *  cols    > 0, % 32 == 0.
 *  q       E4M3 codes [rows, cols] (device, 16-byte aligned).
 *  sf      swizzled E8M0 codes, nvfp4_mxfp8_sf_bytes(rows, cols) bytes; the
 *          padding is zeroed.
 *  q_col   NULL, or E4M3 codes of X^T [cols, rows] (16-byte aligned); needs
 *          rows % 32 == 0.
 *  sf_col  swizzled E8M0 codes of X^T, nvfp4_mxfp8_sf_bytes(cols, rows) bytes;
 *          NULL exactly when q_col is.
 *  Errors: NVFP4_ERR_SHAPE / _ALIGNMENT / _INVALID_ARG; rows == 0 is a no-op.
 */
NVFP4_API nvfp4_status nvfp4_mxfp8_quantize(
    const void* x, int64_t rows, int64_t cols, int64_t ld_x, void* q, void* sf, void* q_col, void* sf_col,
    nvfp4_stream_t stream);

/*
 * y[r, k] = bf16_rn( dec(q[r, k]) * 2^(code - 127) ), the product exact in
 * binary32 (E8M0 code 0 is 2^-127).  Bit-exact.
 *
 *  q       E4M3 codes [rows, cols], 16-byte aligned;  sf  swizzled E8M0 codes.
 *  cols    > 0, % 32 == 0.
 *  y       bf16 [rows, ld_y], ld_y >= cols, ld_y % 8 == 0, 16-byte aligned.
 *  Errors: NVFP4_ERR_SHAPE / _ALIGNMENT / _INVALID_ARG; rows == 0 is a no-op.
 */
NVFP4_API nvfp4_status nvfp4_mxfp8_dequantize(
    const void* q, const void* sf, int64_t rows, int64_t cols, void* y, int64_t ld_y, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------- */
/* SwiGLU + requantize (the MoE fc2 input)                                   */
/* ------------------------------------------------------------------------- */

/*
 * h[r, f] = bf16_rn( silu(g) * u ), g = y1[r, f], u = y1[r, ffn + f] (the fused
 * gate/up projection: "Towards Blackwell-Native 8-bit and 4-bit RL",
 * "Parallelism and tensor-conversion contract", SwiGLU MoE), then h quantized
 * per token exactly as nvfp4_quantize_per_token does, in the same kernel.
 * silu is evaluated in binary32 with the hardware approximations ex2.approx
 * and rcp.approx on exp(-|g|) (which never overflows: sigma(g) = 1/(1+e) for
 * g >= 0, e/(1+e) for g < 0), ~2^-17 relative error at most, so h may differ
 * from an exact evaluation by one bf16 ulp (for gates g >= -96; below that
 * |silu(g)| < 1e-39 and the bound can fail when |u| is very large);
 * the quantization of h is bit-exact.
 *
 *  y1        bf16 [rows, ld_y1], ld_y1 >= 2*ffn, ld_y1 % 8 == 0, 16-byte aligned.
 *  ffn       > 0, % 16 == 0.
 *  row_count NULL, or an int32 on the device: rows >= *row_count are written as
 *            zero rows (e.g. expert_offsets + E, the used part of the layout).
 *  q, sf, s  quantized h: [rows, ffn/2], nvfp4_sf_bytes(rows, ffn), float [rows].
 *  h         NULL, or bf16 [rows, ffn] to also receive h itself.
 */
NVFP4_API nvfp4_status nvfp4_swiglu_quantize(
    const void* y1, int64_t rows, int64_t ffn, int64_t ld_y1, const int32_t* row_count,
    void* q, void* sf, float* s, void* h, nvfp4_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Status and diagnostics                                                    */
/* ------------------------------------------------------------------------- */

/* Synchronise `stream`, then return and clear the current device's status word
 * (the first device-side error recorded since the last call), or NVFP4_ERR_CUDA
 * if the synchronisation itself failed. */
NVFP4_API nvfp4_status nvfp4_get_device_status(nvfp4_stream_t stream);

/* Static, human-readable name of a status code. */
NVFP4_API const char* nvfp4_status_string(nvfp4_status status);

/*
 * Exhaustive check of the device's E2M1 and E4M3 conversions, the ones the
 * quantizer uses.  Over every non-negative float32 bit pattern p (0 ..
 * 0x7F800000, i.e. +0 to +inf) it records, for each E2M1 code c (0..7) and
 * each E4M3 code c (0..127), the first and last p that encode to c:
 * first[c] / last[c] at index c for E2M1 and 16 + c for E4M3 (0xFFFFFFFF / 0
 * when a code never occurs).  counters[0] counts patterns whose E2M1 code is
 * below that of p - 1 (non-monotone), counters[1] the same for E4M3,
 * counters[2] the p whose negation -p does not encode to (code of p) | 8 in
 * E2M1, counters[3] the E4M3 NaN codes produced.
 *  first, last  uint32 [144] each (device); counters uint32 [4] (device).
 */
NVFP4_API nvfp4_status nvfp4_debug_cvt_probe(uint32_t* first, uint32_t* last, uint32_t* counters,
                                   nvfp4_stream_t stream);

/*
 * Self-check of the quantizers' scale arithmetic (outer scale, block scale code
 * and element multiplier, "Towards Blackwell-Native 8-bit and 4-bit RL",
 * "Bit-exact quantizer contract"): rows whose outer scale lies in [2^-90, 2^90]
 * compute the correctly rounded quotients amax / 2688 and amax_b / T and the
 * reciprocals 1 / T and 1 / D with fused multiply-adds instead of IEEE
 * division.  This compares the two forms for every bf16 row amax and over every
 * pair of bf16 values the quantizers can meet (row amax, block amax <= row
 * amax; about 5e8 pairs).
 *  counters  uint64 [2] (device, 8-byte aligned): [0] pairs compared, [1]
 *            pairs whose code or multiplier differ, plus rows whose S, T, 1/T or
 *            range decision differ (0 when the forms agree).
 *  mismatch  uint32 [17] (device): [0] mismatches recorded, then up to 8 pairs
 *            (row amax bits >> 16, block amax bits >> 16; 0xFFFFFFFF when the
 *            row's own S, T, 1/T or range decision differ).
 * Both are cleared on the stream first; results are ready when it completes.
 */
NVFP4_API nvfp4_status nvfp4_debug_scale_recipe_check(unsigned long long* counters, uint32_t* mismatch,
                                                      nvfp4_stream_t stream);

/*
 * Failure-detection check: launch one block that waits, with the library's
 * bounded wait, on an mbarrier nothing will ever arrive at.  After timeout_ns
 * (1 ms .. 10 s) the wait gives up, the kernel records NVFP4_ERR_TIMEOUT in the
 * status word and returns normally, leaving the context usable.
 */
NVFP4_API nvfp4_status nvfp4_debug_wait_timeout(int64_t timeout_ns, nvfp4_stream_t stream);

/*
 * Failure-detection check of the GEMMs' abort path: every wait of the GEMM
 * pipelines launched after this call (until it is called again) gives up after
 * limit_ns instead of the default 2 s; 0 restores the default (0 .. 10 s).
 * Limits are enforced at the resolution of the GPU's global timer (so a limit
 * of a few microseconds may outlast every wait); with 1 ns, every wait that is
 * not complete at its first attempt gives up: the role that gave up records
 * NVFP4_ERR_TIMEOUT and raises the CTA's abort flag, every
 * role of both CTAs of a pair leaves its loop, copies and tensor-core work in
 * flight complete, TMEM is freed and the kernel returns, leaving the context
 * usable (the output is then incomplete).  Process-wide; not for use while
 * other threads launch GEMMs.  The GEMMs run a separate build of their kernels
 * while a limit other than the default is set (the default build keeps the
 * default limit as a constant); nvfp4_grouped_gemm_swiglu then returns
 * NVFP4_ERR_INVALID_ARG.
 */
NVFP4_API nvfp4_status nvfp4_debug_set_gemm_wait_limit(int64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H_ */
