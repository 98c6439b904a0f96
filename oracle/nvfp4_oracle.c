/*
 * nvfp4_oracle.c -- CPU oracle for the per-token NVFP4 W4A4 linear-layer path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
 * reference arm do.  It shares no code, header, table or constant generator with
 * the CUDA library (nvfp4_precision_rl_gb300/csrc).
 *
 * Plain, slow, obviously correct.  Every float operation of the quantizer is one
 * IEEE-754 binary32 operation with round-to-nearest-even (compile with
 * -ffp-contract=off so that no multiply-add is fused); the GEMM is an exact
 * integer sum scaled in binary64.
 *
 * Sources (web pages; cited by title and section):
 *  [Miles]  "Towards Blackwell-Native 8-bit and 4-bit RL: End-to-End MXFP8 and
 *           NVFP4 RL in Miles" (LMSYS blog, summarised on papercache.org).
 *  [TRIAGE] "TRIAGE: Direction-Aware Mismatch Stabilization of Native NVFP4
 *           Reinforcement Learning", section "NVFP4 quantization format and W4A4
 *           execution" (the decode formula x^ = S * s_b * Q_E2M1(x / (S * s_b))).
 *  [miniTE] "miniTE report: why native NVFP4 RL destabilises late in training"
 *           (aitest123.com), section "NVFP4 format, two-level scaling and
 *           conversion error".
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  R1  outer scale S = fl(amax / 2688), 2688 = 6 * 448: the token's largest
 *      block lands on the E4M3 maximum ([Miles] "NVFP4 format background": the
 *      FP32 scale maps the token into the representable range).
 *  R2  operation order: S, T = fl(6*S), d_b = fl(amax_b / T), s_b = E4M3(d_b),
 *      D_b = fl(S * dec(s_b)), r_b = fl(1 / D_b) (0 if D_b == 0, clamped to
 *      FLT_MAX), q = E2M1(fl(x * r_b)).
 *  R3  both encoders round to the nearest table entry, ties to the even code
 *      (code LSB 0), and saturate to the largest finite entry; the E2M1 sign
 *      bit is kept even when the magnitude rounds to zero.
 *  R6  packed byte j of a row holds element 2j in its low nibble.
 *  R7  the column-wise copy quantizes X^T (16-blocks along tokens) with one
 *      per-tensor scale from the global amax.
 *  R9  swizzled scale-factor layout: 128 x 4 tiles of 512 bytes, row-tile major.
 *  R11 dequantization to bf16 evaluates S * dec(s_b) * dec(q) in binary32 (the
 *      product of the two codes is exact) and rounds the binary32 result to bf16.
 *  R12 the routed-expert combine accumulates in binary32 in slot order.
 *  R13 MXFP8 scale: the smallest power of two 2^e (e >= -127) with
 *      448 * 2^e >= amax_b; elements E4M3(x / 2^e), ties to even, sign kept.
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Element formats ([miniTE] "NVFP4 format"; [Miles] "NVFP4 format background") */
/* ------------------------------------------------------------------------ */

/* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf / NaN. */
static double e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (the "FN" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * S.1111.111 is NaN, no inf, so the largest finite value is 448. */
static double e4m3_value(int code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

static double g_e2m1[16];
static double g_e4m3[256];
static pthread_once_t g_tables_once = PTHREAD_ONCE_INIT;

static void build_tables(void) {
    for (int c = 0; c < 16; ++c) g_e2m1[c] = e2m1_value(c);
    for (int c = 0; c < 256; ++c) g_e4m3[c] = e4m3_value(c);
}
static void tables(void) { pthread_once(&g_tables_once, build_tables); }

/* Nearest entry of an ascending list of non-negative values (codes 0..n-1 of
 * the format), ties to the even code, values past the end saturate. */
static int nearest_code(double v, const double* vals, int n) {
    if (!(v < vals[n - 1])) return n - 1;          /* >= max, or +inf */
    for (int i = 0; i + 1 < n; ++i) {
        if (v <= vals[i + 1]) {
            double mid = 0.5 * (vals[i] + vals[i + 1]);  /* exact in binary64 */
            if (v < mid) return i;
            if (v > mid) return i + 1;
            return (i & 1) ? i + 1 : i;                  /* tie: even code */
        }
    }
    return n - 1;
}

static int enc_e2m1(float x) {
    int sign = signbit(x) ? 8 : 0;
    return sign | nearest_code(fabs((double)x), g_e2m1, 8);
}

/* Block scales are non-negative; codes 0x00..0x7E are the non-negative finite
 * E4M3 values in ascending order. */
static int enc_e4m3(float d) {
    return nearest_code(fabs((double)d), g_e4m3, 127);
}

ORC_API void orc_e2m1_table(double* out16) { tables(); memcpy(out16, g_e2m1, sizeof g_e2m1); }
ORC_API void orc_e4m3_table(double* out256) { tables(); memcpy(out256, g_e4m3, sizeof g_e4m3); }

ORC_API void orc_e2m1_encode(const float* x, int64_t n, uint8_t* codes) {
    tables();
    for (int64_t i = 0; i < n; ++i) codes[i] = (uint8_t)enc_e2m1(x[i]);
}

ORC_API void orc_e4m3_encode(const float* x, int64_t n, uint8_t* codes) {
    tables();
    for (int64_t i = 0; i < n; ++i) codes[i] = (uint8_t)enc_e4m3(x[i]);
}

static float bf16_to_float(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, 4);
    return f;
}

/* ------------------------------------------------------------------------ */
/* Two-level quantization of one vector ([TRIAGE] NVFP4 section formula;     */
/* [Miles] "NVFP4 format background" and "online per-token scale").          */
/* ------------------------------------------------------------------------ */

/* Quantize n values (n % 16 == 0) with a given amax (the token's own amax in
 * per-token mode, the tensor's amax in per-tensor mode).
 * q: n/2 packed bytes (low nibble = even element), sf: n/16 E4M3 codes. */
static float quantize_vector(const float* x, int64_t n, float amax, uint8_t* q, uint8_t* sf) {
    const float S = amax / 2688.0f;   /* R1: 2688 = 6 * 448 */
    const float T = 6.0f * S;
    for (int64_t b = 0; b < n / 16; ++b) {
        const float* xb = x + 16 * b;
        float amax_b = 0.0f;
        for (int k = 0; k < 16; ++k) amax_b = fmaxf(amax_b, fabsf(xb[k]));
        float d = (T == 0.0f) ? 0.0f : amax_b / T;
        int s_b = enc_e4m3(d);
        float D = S * (float)g_e4m3[s_b];
        float r = (D == 0.0f) ? 0.0f : 1.0f / D;
        if (r > FLT_MAX) r = FLT_MAX;
        sf[b] = (uint8_t)s_b;
        for (int k = 0; k < 16; k += 2) {
            int lo = enc_e2m1(xb[k] * r);
            int hi = enc_e2m1(xb[k + 1] * r);
            q[8 * b + k / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
    return S;
}

static float vector_amax(const float* x, int64_t n) {
    float a = 0.0f;
    for (int64_t k = 0; k < n; ++k) a = fmaxf(a, fabsf(x[k]));
    return a;
}

/* Source row of output row r (gather index, -1 = zero row). */
static void load_row(const uint16_t* x, int64_t cols, int64_t ld, const int32_t* gather,
                     int64_t r, float* dst) {
    int64_t src = gather ? (int64_t)gather[r] : r;
    if (src < 0) {
        for (int64_t k = 0; k < cols; ++k) dst[k] = 0.0f;
        return;
    }
    for (int64_t k = 0; k < cols; ++k) dst[k] = bf16_to_float(x[src * ld + k]);
}

typedef struct {
    const uint16_t* x; int64_t cols, ld; const int32_t* gather;
    int64_t r0, r1;
    int per_tensor; float amax_tensor;
    uint8_t* q; uint8_t* sf; float* s;
    float amax_out;
} row_job;

static void* row_amax_worker(void* p) {
    row_job* j = (row_job*)p;
    float* buf = (float*)malloc(sizeof(float) * (size_t)j->cols);
    float a = 0.0f;
    for (int64_t r = j->r0; r < j->r1; ++r) {
        load_row(j->x, j->cols, j->ld, j->gather, r, buf);
        a = fmaxf(a, vector_amax(buf, j->cols));
    }
    free(buf);
    j->amax_out = a;
    return NULL;
}

static void* row_quant_worker(void* p) {
    row_job* j = (row_job*)p;
    float* buf = (float*)malloc(sizeof(float) * (size_t)j->cols);
    for (int64_t r = j->r0; r < j->r1; ++r) {
        load_row(j->x, j->cols, j->ld, j->gather, r, buf);
        float amax = j->per_tensor ? j->amax_tensor : vector_amax(buf, j->cols);
        j->s[r] = quantize_vector(buf, j->cols, amax, j->q + r * (j->cols / 2),
                                  j->sf + r * (j->cols / 16));
    }
    free(buf);
    return NULL;
}

static void run_rows(void* (*fn)(void*), row_job* proto, int64_t rows, int nthreads, float* amax_max) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    row_job jobs[256];
    int64_t per = (rows + nthreads - 1) / nthreads;
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].r0 = t * per;
        jobs[t].r1 = (t + 1) * per < rows ? (t + 1) * per : rows;
        jobs[t].amax_out = 0.0f;
        if (jobs[t].r0 >= jobs[t].r1) break;
        pthread_create(&th[t], NULL, fn, &jobs[t]);
        ++used;
    }
    float a = 0.0f;
    for (int t = 0; t < used; ++t) {
        pthread_join(th[t], NULL);
        a = fmaxf(a, jobs[t].amax_out);
    }
    if (amax_max) *amax_max = a;
}

/* Row-wise quantization of X (bf16 [rows_in, cols], leading dimension ld) into
 * rows_out rows; output row r reads source row gather[r] (gather == NULL:
 * identity; -1: a zero row).  mode 0 = per-token outer scale, 1 = per-tensor.
 * Outputs: q [rows_out, cols/2], sf row-major [rows_out, cols/16], s [rows_out].
 * Returns the amax over all output rows (the per-tensor amax). */
ORC_API float orc_quantize_rows(const uint16_t* x, int64_t cols, int64_t ld, const int32_t* gather,
                                int64_t rows_out, int mode, uint8_t* q, uint8_t* sf, float* s,
                                int nthreads) {
    tables();
    row_job proto = {x, cols, ld, gather, 0, 0, mode == 1, 0.0f, q, sf, s, 0.0f};
    float amax = 0.0f;
    run_rows(row_amax_worker, &proto, rows_out, nthreads, &amax);
    proto.amax_tensor = amax;
    run_rows(row_quant_worker, &proto, rows_out, nthreads, NULL);
    return amax;
}

typedef struct {
    const uint16_t* x; int64_t cols, ld; const int32_t* gather; int64_t rows;
    int64_t k0, k1; float amax;
    uint8_t* q; uint8_t* sf; float S;
} col_job;

static void* col_quant_worker(void* p) {
    col_job* j = (col_job*)p;
    float* buf = (float*)malloc(sizeof(float) * (size_t)j->rows);
    /* column k of the gathered X is row k of X^T */
    for (int64_t k = j->k0; k < j->k1; ++k) {
        for (int64_t r = 0; r < j->rows; ++r) {
            int64_t src = j->gather ? (int64_t)j->gather[r] : r;
            buf[r] = src < 0 ? 0.0f : bf16_to_float(j->x[src * j->ld + k]);
        }
        j->S = quantize_vector(buf, j->rows, j->amax, j->q + k * (j->rows / 2),
                               j->sf + k * (j->rows / 16));
    }
    free(buf);
    return NULL;
}

/* Column-wise copy (R7): X^T [cols, rows] quantized with 16-blocks along the
 * token axis and one per-tensor outer scale from amax (the global amax that the
 * row pass already found).  q [cols, rows/2], sf row-major [cols, rows/16]. */
ORC_API float orc_quantize_cols(const uint16_t* x, int64_t cols, int64_t ld, const int32_t* gather,
                                int64_t rows, float amax, uint8_t* q, uint8_t* sf, int nthreads) {
    tables();
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    col_job jobs[256];
    int64_t per = (cols + nthreads - 1) / nthreads;
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        col_job j = {x, cols, ld, gather, rows, t * per, (t + 1) * per < cols ? (t + 1) * per : cols,
                     amax, q, sf, 0.0f};
        jobs[t] = j;
        if (j.k0 >= j.k1) break;
        pthread_create(&th[t], NULL, col_quant_worker, &jobs[t]);
        ++used;
    }
    for (int t = 0; t < used; ++t) pthread_join(th[t], NULL);
    return amax / 2688.0f;
}

/* ------------------------------------------------------------------------ */
/* Swizzled scale-factor layout (R9)                                          */
/* ------------------------------------------------------------------------ */

static int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

ORC_API int64_t orc_sf_swizzled_bytes(int64_t rows, int64_t kb) {
    return round_up(rows, 128) * round_up(kb, 4);
}

/* Byte offset of scale factor (row r, block c) in the swizzled buffer: the
 * matrix is cut into 128-row x 4-block tiles of 512 bytes, tiles ordered with
 * the block index fastest; inside a tile, row r sits in 16-byte line r % 32,
 * at 4-byte slot (r % 128) / 32, byte c % 4. */
static int64_t swz_offset(int64_t r, int64_t c, int64_t kb) {
    int64_t tiles_per_row = round_up(kb, 4) / 4;
    int64_t tile = (r / 128) * tiles_per_row + c / 4;
    return tile * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

ORC_API void orc_sf_swizzle(const uint8_t* sf_rm, int64_t rows, int64_t kb, uint8_t* out) {
    memset(out, 0, (size_t)orc_sf_swizzled_bytes(rows, kb));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < kb; ++c) out[swz_offset(r, c, kb)] = sf_rm[r * kb + c];
}

ORC_API void orc_sf_unswizzle(const uint8_t* swz, int64_t rows, int64_t kb, uint8_t* sf_rm) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < kb; ++c) sf_rm[r * kb + c] = swz[swz_offset(r, c, kb)];
}

/* ------------------------------------------------------------------------ */
/* Dequantization: x^ = S * dec(s_b) * dec(q)  ([TRIAGE] NVFP4 formula)        */
/* ------------------------------------------------------------------------ */

ORC_API void orc_dequantize(const uint8_t* q, const uint8_t* sf_rm, const float* s, int64_t rows,
                            int64_t cols, double* out) {
    tables();
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < cols; ++k) {
            uint8_t byte = q[r * (cols / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            out[r * cols + k] = (double)s[r] * g_e4m3[sf_rm[r * (cols / 16) + k / 16]] * g_e2m1[code];
        }
}

/* bf16 from binary32, round to nearest, ties to even (finite inputs; NaN kept). */
static uint16_t bf16_from_float_rne(float f) {
    uint32_t bits;
    memcpy(&bits, &f, 4);
    if ((bits & 0x7F800000u) == 0x7F800000u && (bits & 0x007FFFFFu) != 0) return 0x7FC0;
    uint32_t lower = bits & 0xFFFFu;
    uint32_t upper = bits >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;   /* carries into the exponent */
    return (uint16_t)upper;
}

/* Dequantization to bf16 (R11), the input of the dequantized backward:
 * c = dec(q) * dec(s_b) (exact in binary32), p = fl32(S * c), y = bf16_rn(p).
 * s_per_row == 0: s[0] for every row. */
ORC_API void orc_dequantize_bf16(const uint8_t* q, const uint8_t* sf_rm, const float* s, int s_per_row,
                                 int64_t rows, int64_t cols, uint16_t* out) {
    tables();
    for (int64_t r = 0; r < rows; ++r) {
        float S = s[s_per_row ? r : 0];
        for (int64_t k = 0; k < cols; ++k) {
            uint8_t byte = q[r * (cols / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            float c = (float)g_e2m1[code] * (float)g_e4m3[sf_rm[r * (cols / 16) + k / 16]];
            float p = S * c;
            out[r * cols + k] = bf16_from_float_rne(p);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* W4A4 GEMM:  Y[m,n] = S_a[m] * S_b[n] * sum_k x^_mk w^_nk / (S_a S_b)       */
/* ------------------------------------------------------------------------ */

/* Every 2*E2M1 value is an integer in [-12, 12] and every 512*E4M3 value an
 * integer in [0, 229376], so sum_k dec(qa)dec(sa)dec(qb)dec(sb) * 2^20 is an
 * integer, summed here exactly in int64 (|sum| < 3.1e16 for K <= 4096). */
typedef struct {
    int8_t* q2;     /* rows x K, 2 * E2M1 value */
    int64_t* s9;    /* rows x K/16, 512 * E4M3 value */
} int_operand;

static void make_int_operand(const uint8_t* q, const uint8_t* sf_rm, int64_t rows, int64_t K,
                             int_operand* o) {
    o->q2 = (int8_t*)malloc((size_t)(rows * K));
    o->s9 = (int64_t*)malloc(sizeof(int64_t) * (size_t)(rows * (K / 16)));
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = q[r * (K / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            o->q2[r * K + k] = (int8_t)(2.0 * g_e2m1[code]);
        }
        for (int64_t b = 0; b < K / 16; ++b)
            o->s9[r * (K / 16) + b] = (int64_t)(512.0 * g_e4m3[sf_rm[r * (K / 16) + b]]);
    }
}

static void free_int_operand(int_operand* o) { free(o->q2); free(o->s9); }

/* One output element: exact value and sum of |products| (both scaled). */
static void exact_dot(const int_operand* a, int64_t m, const int_operand* b, int64_t n, int64_t K,
                      float sa, float sb, double* y, double* absy) {
    int64_t acc = 0, abs_acc = 0;
    const int8_t* qa = a->q2 + m * K;
    const int8_t* qb = b->q2 + n * K;
    for (int64_t blk = 0; blk < K / 16; ++blk) {
        int64_t dot = 0, adot = 0;
        for (int k = 0; k < 16; ++k) {
            int64_t p = (int64_t)qa[16 * blk + k] * (int64_t)qb[16 * blk + k];
            dot += p;
            adot += p < 0 ? -p : p;
        }
        int64_t ss = a->s9[m * (K / 16) + blk] * b->s9[n * (K / 16) + blk];
        acc += ss * dot;
        abs_acc += ss * adot;
    }
    double scale = ldexp(1.0, -20) * (double)sa * (double)sb;
    *y = (double)acc * scale;
    if (absy) *absy = (double)abs_acc * scale;
}

typedef struct {
    const int_operand *a, *b; const float *sa, *sb; int64_t N, K;
    const int64_t *mi, *ni; int64_t i0, i1;   /* sampled list, or ... */
    int64_t m0, m1;                           /* ... a row range of the full product */
    double *y, *absy;
} gemm_job;

static void* gemm_full_worker(void* p) {
    gemm_job* j = (gemm_job*)p;
    for (int64_t m = j->m0; m < j->m1; ++m)
        for (int64_t n = 0; n < j->N; ++n)
            exact_dot(j->a, m, j->b, n, j->K, j->sa[m], j->sb[n], &j->y[m * j->N + n],
                      j->absy ? &j->absy[m * j->N + n] : NULL);
    return NULL;
}

static void* gemm_sampled_worker(void* p) {
    gemm_job* j = (gemm_job*)p;
    for (int64_t i = j->i0; i < j->i1; ++i)
        exact_dot(j->a, j->mi[i], j->b, j->ni[i], j->K, j->sa[j->mi[i]], j->sb[j->ni[i]], &j->y[i],
                  j->absy ? &j->absy[i] : NULL);
    return NULL;
}

static void run_gemm(void* (*fn)(void*), gemm_job* proto, int64_t count, int nthreads, int rows_mode) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    gemm_job jobs[256];
    int64_t per = (count + nthreads - 1) / nthreads;
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        int64_t lo = t * per, hi = (t + 1) * per < count ? (t + 1) * per : count;
        if (lo >= hi) break;
        if (rows_mode) { jobs[t].m0 = lo; jobs[t].m1 = hi; }
        else { jobs[t].i0 = lo; jobs[t].i1 = hi; }
        pthread_create(&th[t], NULL, fn, &jobs[t]);
        ++used;
    }
    for (int t = 0; t < used; ++t) pthread_join(th[t], NULL);
}

/* Full product: y, absy (optional) are [M, N] row-major binary64. */
ORC_API void orc_gemm_exact(const uint8_t* qa, const uint8_t* sfa_rm, const float* sa, int64_t M,
                            const uint8_t* qb, const uint8_t* sfb_rm, const float* sb, int64_t N,
                            int64_t K, double* y, double* absy, int nthreads) {
    tables();
    int_operand a, b;
    make_int_operand(qa, sfa_rm, M, K, &a);
    make_int_operand(qb, sfb_rm, N, K, &b);
    gemm_job proto = {&a, &b, sa, sb, N, K, NULL, NULL, 0, 0, 0, 0, y, absy};
    run_gemm(gemm_full_worker, &proto, M, nthreads, 1);
    free_int_operand(&a);
    free_int_operand(&b);
}

/* Sampled outputs (mi[i], ni[i]), i < count. */
ORC_API void orc_gemm_exact_sampled(const uint8_t* qa, const uint8_t* sfa_rm, const float* sa,
                                    int64_t M, const uint8_t* qb, const uint8_t* sfb_rm,
                                    const float* sb, int64_t N, int64_t K, const int64_t* mi,
                                    const int64_t* ni, int64_t count, double* y, double* absy,
                                    int nthreads) {
    tables();
    int_operand a, b;
    make_int_operand(qa, sfa_rm, M, K, &a);
    make_int_operand(qb, sfb_rm, N, K, &b);
    gemm_job proto = {&a, &b, sa, sb, N, K, mi, ni, 0, 0, 0, 0, y, absy};
    run_gemm(gemm_sampled_worker, &proto, count, nthreads, 0);
    free_int_operand(&a);
    free_int_operand(&b);
}

/* The same product as a plain binary64 loop over the decoded operands (the
 * oracle's self-check: it must agree with the exact sum to ~1e-12). */
ORC_API void orc_gemm_fp64(const uint8_t* qa, const uint8_t* sfa_rm, const float* sa, int64_t M,
                           const uint8_t* qb, const uint8_t* sfb_rm, const float* sb, int64_t N,
                           int64_t K, double* y) {
    tables();
    double* xa = (double*)malloc(sizeof(double) * (size_t)(M * K));
    double* xb = (double*)malloc(sizeof(double) * (size_t)(N * K));
    orc_dequantize(qa, sfa_rm, sa, M, K, xa);
    orc_dequantize(qb, sfb_rm, sb, N, K, xb);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += xa[m * K + k] * xb[n * K + k];
            y[m * N + n] = acc;
        }
    free(xa);
    free(xb);
}

/* ------------------------------------------------------------------------ */
/* MoE routing permute: per-expert contiguous rows, segments padded to align  */
/* ------------------------------------------------------------------------ */

/* topk [T, k] expert ids.  offsets [E+1]: segment e is rows
 * [offsets[e], offsets[e+1]), its length the expert's count rounded up to
 * align.  Inside a segment, routed pairs (t, j) keep ascending (t, j) order.
 * gather [capacity]: source token of each row, -1 for padding.  dst [T*k]: row
 * of pair (t, j).  Returns 0, or -1 if an id is out of range or the rows do
 * not fit in capacity. */
ORC_API int orc_moe_permute(const int32_t* topk, int64_t T, int32_t k, int32_t E, int32_t align,
                            int32_t* offsets, int32_t* gather, int64_t capacity, int32_t* dst) {
    int64_t* count = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int64_t* cursor = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int rc = 0;
    for (int64_t i = 0; i < T * k; ++i) {
        if (topk[i] < 0 || topk[i] >= E) { rc = -1; goto done; }
        count[topk[i]]++;
    }
    int64_t off = 0;
    for (int32_t e = 0; e < E; ++e) {
        offsets[e] = (int32_t)off;
        cursor[e] = off;
        off += round_up(count[e], align);
    }
    offsets[E] = (int32_t)off;
    if (off > capacity) { rc = -1; goto done; }
    for (int64_t r = 0; r < capacity; ++r) gather[r] = -1;
    for (int64_t i = 0; i < T * k; ++i) {
        int64_t row = cursor[topk[i]]++;
        gather[row] = (int32_t)(i / k);
        dst[i] = (int32_t)row;
    }
done:
    free(count);
    free(cursor);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* SwiGLU between fc1 and fc2 ([Miles] "SwiGLU MoE" gate/up contract)         */
/* ------------------------------------------------------------------------ */

/* Round a binary64 value to bfloat16, nearest-even, in one step. */
static uint16_t bf16_from_double(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);                      /* a = f * 2^ex, f in [0.5, 1) */
    int lsb = ex - 8;                   /* 8 significant bits */
    if (lsb < -133) lsb = -133;         /* subnormal spacing 2^-133 */
    double r = nearbyint(ldexp(a, -lsb));   /* default rounding: nearest-even */
    double mag = ldexp(r, lsb);
    if (mag > 3.3895313892515355e38) return sign | 0x7F80;   /* past the largest bf16 */
    float f = (float)mag;               /* exact */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return sign | (uint16_t)(bits >> 16);
}

/* h[r, f] = bf16(silu(g) * u), g = y1[r, f], u = y1[r, F + f], in binary64. */
ORC_API void orc_swiglu(const uint16_t* y1, int64_t rows, int64_t F, int64_t ld, uint16_t* h) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t f = 0; f < F; ++f) {
            double g = bf16_to_float(y1[r * ld + f]);
            double u = bf16_to_float(y1[r * ld + F + f]);
            double silu = g / (1.0 + exp(-g));
            h[r * F + f] = bf16_from_double(silu * u);
        }
}

/* Unpermute + weighted combine after the expert GEMMs ([Miles], section on
 * keeping shared experts in high precision: the sparsely selected routed
 * experts' outputs pass through a high-precision weighted reduction).
 * Reading R12: the reduction is binary32, in slot order, multiply then add:
 * out[t, h] = bf16_rn(acc), acc = 0, then for j = 0 .. topk-1
 * acc = fl32(acc + fl32(w[t, j] * y2[dst[t*topk + j], h])).  A dst row outside
 * [0, rows) contributes nothing. */
ORC_API void orc_moe_combine(const uint16_t* y2, int64_t rows, int64_t ld, const int32_t* dst,
                             const float* w, int64_t tokens, int topk, int64_t hidden, uint16_t* out) {
    for (int64_t t = 0; t < tokens; ++t)
        for (int64_t h = 0; h < hidden; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < topk; ++j) {
                int64_t r = dst[t * topk + j];
                if (r < 0 || r >= rows) continue;
                float prod = w[t * topk + j] * bf16_to_float(y2[r * ld + h]);
                acc = acc + prod;
            }
            out[t * hidden + h] = bf16_from_float_rne(acc);
        }
}

/* ------------------------------------------------------------------------ */
/* MXFP8 ([Miles] "MXFP8 format background": 1x32 blocks of E4M3 values      */
/* sharing one E8M0 power-of-two scale, rounded up so that the block maximum */
/* is not clipped; row-wise 1x32 and column-wise 32x1 copies are quantized   */
/* independently from the full-precision data, "Backward activation         */
/* representation trade-off").                                              */
/* ------------------------------------------------------------------------ */

/* Reading R13: the scale is 2^e with e the smallest integer >= -127 such that
 * 448 * 2^e >= amax_b (amax_b = 0 gives -127); E8M0 code = e + 127. */
static int mx_exponent(float amax) {
    int e = -127;
    while (ldexp(448.0, e) < (double)amax) ++e;
    return e;
}

/* E4M3 of x / 2^e, nearest with ties to the even code, saturating, sign kept. */
static uint8_t mx_element(float x, int e) {
    double v = ldexp((double)x, -e);                 /* exact */
    int sign = signbit(x) ? 0x80 : 0;
    return (uint8_t)(sign | nearest_code(fabs(v), g_e4m3, 127));
}

/* Rows: q [rows, cols] E4M3 codes, sf_rm [rows, cols/32] E8M0 codes. */
ORC_API void orc_mxfp8_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q,
                                     uint8_t* sf_rm) {
    tables();
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < cols / 32; ++b) {
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(bf16_to_float(x[r * ld + b * 32 + i]));
                if (a > amax) amax = a;
            }
            int e = mx_exponent(amax);
            sf_rm[r * (cols / 32) + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i)
                q[r * cols + b * 32 + i] = mx_element(bf16_to_float(x[r * ld + b * 32 + i]), e);
        }
}

/* Columns (X^T, 32x1 blocks along the rows): q [cols, rows], sf_rm [cols, rows/32]. */
ORC_API void orc_mxfp8_quantize_cols(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q,
                                     uint8_t* sf_rm) {
    tables();
    for (int64_t k = 0; k < cols; ++k)
        for (int64_t b = 0; b < rows / 32; ++b) {
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(bf16_to_float(x[(b * 32 + i) * ld + k]));
                if (a > amax) amax = a;
            }
            int e = mx_exponent(amax);
            sf_rm[k * (rows / 32) + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i)
                q[k * rows + b * 32 + i] = mx_element(bf16_to_float(x[(b * 32 + i) * ld + k]), e);
        }
}

/* bf16 of dec(q) * 2^(code - 127), one rounding of the exact product. */
ORC_API void orc_mxfp8_dequantize_bf16(const uint8_t* q, const uint8_t* sf_rm, int64_t rows, int64_t cols,
                                       uint16_t* out) {
    tables();
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < cols; ++k) {
            double v = g_e4m3[q[r * cols + k]] * ldexp(1.0, (int)sf_rm[r * (cols / 32) + k / 32] - 127);
            out[r * cols + k] = bf16_from_double(v);
        }
}

ORC_API void orc_bf16_from_double(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_from_double(v[i]);
}
