/*
 * q8_oracle.c -- the ORACLE for the Q8_0 block-quantized decode product.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously correct CPU
 * restatement of what the GPU library computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or helper with the CUDA library and includes nothing
 * from it; the CUDA library never loads it.
 *
 * Sources (web pages, cited by title and section):
 *   [Ferro]  "Ferro" README (github paragontasx/ferro), section "How the iGPU
 *            path is fast", item 1: Q8_0 weights, activations quantized per
 *            32-wide block following llama.cpp, int8 DP4A dot products.
 *   [Ember]  "Ember: packed Q8 decode" post (voidwest.dev/ember/
 *            packed-q8-decode), the row-contiguous source figure (each row's
 *            block is a scale, then quants q0..q31) and the packed 16-row
 *            tile figure (eight 64-byte groups of four coordinates for 16
 *            rows, then 16 fp16 scales; one record = 544 bytes = 16 blocks).
 *
 * Readings taken where the pages are silent:
 *   - scale rule: d = amax / 127 in fp32, q = roundf(x * (1/d)) (ties away
 *     from zero), 1/d taken from the fp32 d (not from the stored fp16), d
 *     stored as IEEE binary16 rounded to nearest-even, subnormals kept.
 *   - amax == 0: d = 0, all q = 0.
 *   - d below 2^-128 (amax subnormal or nearly): 1/d overflows to inf, nonzero
 *     values clamp to +-127, and a zero value (0 * inf = NaN) stays 0.
 *   - block byte order: fp16 d little-endian at bytes 0..1, q[0..31] at
 *     bytes 2..33 (34 bytes per block).
 *   - output: y[m][n] = sum_b isum_b * d_w * d_a, accumulated here in fp64;
 *     every term is exact in fp64 (20 + 11 + 11 significant bits).
 *   - fused producers (the norm and SwiGLU before quantization): see the
 *     section at the end of this file.
 *
 * Build: any C99 compiler, -O2 -ffp-contract=off, no fast-math.  Portable C:
 * no intrinsics, no inline assembly, no reliance on the signedness of char.
 *
 * Every function here is pinned by the CPU tests (tests/test_oracle_pins.py)
 * against closed forms, library routines (numpy float16), brute force and the
 * pages' byte accounting.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 32               /* values per block  [Ferro, item 1; Ember figure] */
#define BLOCK_BYTES 34      /* 2-byte scale + 32 int8                [Ember]   */
#define EMBER_ROWS 16       /* rows per packed tile                  [Ember]   */
#define EMBER_TILE_BYTES 544

int q8o_qk(void) { return QK; }
int q8o_block_bytes(void) { return BLOCK_BYTES; }
int q8o_ember_tile_bytes(void) { return EMBER_TILE_BYTES; }

/* ---------------------------------------------------------------------------
 * IEEE-754 binary32 -> binary16, round to nearest, ties to even.
 * Written from the definition of the two formats: take the 24-bit significand,
 * shift it to the binary16 grid (13 bits for normal results, more for
 * subnormal ones), round on the discarded bits, and let a carry out of the
 * significand bump the exponent (which also produces infinity on overflow).
 * ------------------------------------------------------------------------- */
uint16_t q8o_f32_to_f16(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint32_t sign = (bits >> 31) << 15;
    uint32_t exp = (bits >> 23) & 0xffu;
    uint32_t mant = bits & 0x7fffffu;

    if (exp == 0xffu)                       /* inf or NaN */
        return (uint16_t)(sign | 0x7c00u | (mant ? 0x200u : 0u));
    if (exp == 0u)                          /* zero or fp32 subnormal (< 2^-126) */
        return (uint16_t)sign;

    int e = (int)exp - 127;                 /* value = sig * 2^(e-23) */
    uint32_t sig = mant | 0x800000u;        /* 24 significant bits    */
    int shift;                              /* bits dropped from sig  */
    if (e >= -14)
        shift = 13;                         /* binary16 normal: 11-bit significand */
    else
        shift = 13 + (-14 - e);             /* binary16 subnormal: grid 2^-24      */
    if (shift > 24)                         /* below half the smallest subnormal  */
        return (uint16_t)sign;

    uint32_t r = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (r & 1u)))
        r += 1u;

    uint32_t h;
    if (e >= -14) {
        if (e > 15)
            return (uint16_t)(sign | 0x7c00u);
        /* r in [1024, 2048]; a carry to 2048 moves into the exponent field */
        h = ((uint32_t)(e + 15) << 10) + (r - 1024u);
        if (h >= 0x7c00u)
            h = 0x7c00u;
    } else {
        h = r;                              /* r <= 1024; 1024 is the smallest normal */
    }
    return (uint16_t)(sign | h);
}

/* binary16 -> binary32, exact (every binary16 value is a binary32 value). */
float q8o_f16_to_f32(uint16_t h)
{
    uint32_t sign = h >> 15;
    uint32_t exp = (h >> 10) & 0x1fu;
    uint32_t mant = h & 0x3ffu;
    float v;
    if (exp == 0u)
        v = ldexpf((float)mant, -24);
    else if (exp == 31u)
        v = mant ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024u + mant), (int)exp - 25);
    return sign ? -v : v;
}

/* ---------------------------------------------------------------------------
 * Quantize one block of 32 fp32 values to one 34-byte Q8_0 block.
 * [Ferro, item 1] names the per-32-block activation scheme; the rounding rule
 * is the reading stated in the header.  All arithmetic is single precision,
 * one operation at a time, in this order:
 *   amax = max_i |x_i|;  d = amax / 127;  id = d != 0 ? 1/d : 0;
 *   q_i = roundf(x_i * id)  (clamped to [-127, 127], which never binds);
 *   stored scale = binary16(d).
 * ------------------------------------------------------------------------- */
void q8o_quantize_block(const float *x, uint8_t *out)
{
    float amax = 0.0f;
    for (int i = 0; i < QK; ++i) {
        float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    uint16_t d16 = q8o_f32_to_f16(d);
    out[0] = (uint8_t)(d16 & 0xffu);
    out[1] = (uint8_t)(d16 >> 8);
    for (int i = 0; i < QK; ++i) {
        float v = x[i] * id;
        float r = roundf(v);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        /* x * (1/d) is NaN only for x = 0 with 1/d = inf (d below 2^-128):
         * a zero value quantizes to zero */
        if (r != r) r = 0.0f;
        int qi = (int)r;
        out[2 + i] = (uint8_t)(qi & 0xff);   /* two's-complement int8 byte */
    }
}

/* Quantize a row-major [rows][K] fp32 matrix to [rows][K/32] blocks. */
void q8o_quantize_rows(const float *x, int64_t rows, int64_t K, uint8_t *out)
{
    int64_t nb = K / QK;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            q8o_quantize_block(x + r * K + b * QK, out + (r * nb + b) * BLOCK_BYTES);
}

static int8_t q_at(const uint8_t *block, int i)
{
    int v = block[2 + i];
    return (int8_t)(v >= 128 ? v - 256 : v);
}

static float scale_of(const uint8_t *block)
{
    uint16_t h = (uint16_t)(block[0] | ((uint16_t)block[1] << 8));
    return q8o_f16_to_f32(h);
}

/* ---------------------------------------------------------------------------
 * Per-block integer dot products (exact, int32):
 *   isum[m][n][b] = sum_{i<32} q_w[n][b][i] * q_a[m][b][i]
 * [Ferro, item 1] (int8 DP4A dot products over per-32-block activations).
 * W: [N][K/32] blocks, A: [M][K/32] blocks, isum: [M][N][K/32].
 * ------------------------------------------------------------------------- */
void q8o_block_dots(const uint8_t *W, int64_t N, int64_t K,
                    const uint8_t *A, int64_t M, int32_t *isum)
{
    int64_t nb = K / QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *wb = W + (n * nb + b) * BLOCK_BYTES;
                const uint8_t *ab = A + (m * nb + b) * BLOCK_BYTES;
                int32_t s = 0;
                for (int i = 0; i < QK; ++i)
                    s += (int32_t)q_at(wb, i) * (int32_t)q_at(ab, i);
                isum[(m * N + n) * nb + b] = s;
            }
}

/* ---------------------------------------------------------------------------
 * The product: y[m][n] = sum_b isum_b * d_w[n][b] * d_a[m][b], in fp64, with
 * the stored (binary16) scales.  Also returns S[m][n] = sum_b |term_b|, the
 * magnitude the parity tolerance is scaled by.  Either output may be NULL.
 * ------------------------------------------------------------------------- */
void q8o_gemm(const uint8_t *W, int64_t N, int64_t K,
              const uint8_t *A, int64_t M, double *y, double *S)
{
    int64_t nb = K / QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *wb = W + (n * nb + b) * BLOCK_BYTES;
                const uint8_t *ab = A + (m * nb + b) * BLOCK_BYTES;
                int32_t s = 0;
                for (int i = 0; i < QK; ++i)
                    s += (int32_t)q_at(wb, i) * (int32_t)q_at(ab, i);
                double term = (double)s * (double)scale_of(wb) * (double)scale_of(ab);
                acc += term;
                mag += fabs(term);
            }
            if (y) y[m * N + n] = acc;
            if (S) S[m * N + n] = mag;
        }
}

/* ---------------------------------------------------------------------------
 * The prefill product's single-precision summation order.  [Ferro],
 * "Exactness contract": prefill rows take the tile GEMM, and a row's result
 * depends neither on how many rows share the launch nor on how the prompt
 * is sliced.  The page fixes no order; the reading taken is a plain one a
 * tile GEMM can keep per row and split along K into two halves: for each
 * output, the blocks in order, cut into nseg segments of `seg` consecutive
 * blocks (the last may be shorter), the first h = ceil(nseg / 2) segments
 * forming the low half and the rest the high half;
 *   s_b   = d_w * d_a in fp32 (exact: two 11-bit significands),
 *   sigma = fma(isum_b, s_b, sigma) through a segment, from +0,
 *   Y_lo  = Y_lo + sigma through the low half's segments, from +0,
 *   Y_hi  = Y_hi + sigma through the high half's segments, from +0,
 *   y     = Y_lo + Y_hi.
 * Every step is one IEEE single-precision operation rounded to nearest
 * even; fmaf rounds once.
 * ------------------------------------------------------------------------- */
void q8o_gemm_prefill_order(const uint8_t *W, int64_t N, int64_t K,
                            const uint8_t *A, int64_t M, int64_t seg, float *y)
{
    int64_t nb = K / QK;
    int64_t nseg = (nb + seg - 1) / seg;
    int64_t h = (nseg + 1) / 2;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            float Y_lo = 0.0f, Y_hi = 0.0f, sigma = 0.0f;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *wb = W + (n * nb + b) * BLOCK_BYTES;
                const uint8_t *ab = A + (m * nb + b) * BLOCK_BYTES;
                int32_t isum = 0;
                for (int i = 0; i < QK; ++i)
                    isum += (int32_t)q_at(wb, i) * (int32_t)q_at(ab, i);
                float s_b = scale_of(wb) * scale_of(ab);
                sigma = fmaf((float)isum, s_b, sigma);
                if ((b + 1) % seg == 0 || b == nb - 1) {
                    if (b / seg < h)
                        Y_lo = Y_lo + sigma;
                    else
                        Y_hi = Y_hi + sigma;
                    sigma = 0.0f;
                }
            }
            y[m * N + n] = Y_lo + Y_hi;
        }
}

/* Quantize fp32 activations, then the product: the fused operation. */
void q8o_quant_gemm(const uint8_t *W, int64_t N, int64_t K,
                    const float *x, int64_t M, uint8_t *A_scratch,
                    double *y, double *S)
{
    q8o_quantize_rows(x, M, K, A_scratch);
    q8o_gemm(W, N, K, A_scratch, M, y, S);
}

/* ---------------------------------------------------------------------------
 * [Ember] packed 16-row tile, used only to pin the byte accounting: 16
 * row-contiguous blocks of one block column become one 544-byte record.
 * Group g (g = 0..7) holds, for rows 0..15 in order, the four quants
 * q[4g..4g+3] of that row (64 bytes); then the 16 fp16 scales follow in row
 * order (32 bytes).  src: 16 blocks (row r at src + 34*r).
 * ------------------------------------------------------------------------- */
void q8o_ember_tile_pack(const uint8_t *src, uint8_t *out)
{
    uint8_t *p = out;
    for (int g = 0; g < QK / 4; ++g)
        for (int r = 0; r < EMBER_ROWS; ++r)
            for (int k = 0; k < 4; ++k)
                *p++ = src[r * BLOCK_BYTES + 2 + 4 * g + k];
    for (int r = 0; r < EMBER_ROWS; ++r) {
        *p++ = src[r * BLOCK_BYTES + 0];
        *p++ = src[r * BLOCK_BYTES + 1];
    }
}

void q8o_ember_tile_unpack(const uint8_t *tile, uint8_t *dst)
{
    const uint8_t *p = tile;
    for (int g = 0; g < QK / 4; ++g)
        for (int r = 0; r < EMBER_ROWS; ++r)
            for (int k = 0; k < 4; ++k)
                dst[r * BLOCK_BYTES + 2 + 4 * g + k] = *p++;
    for (int r = 0; r < EMBER_ROWS; ++r) {
        dst[r * BLOCK_BYTES + 0] = *p++;
        dst[r * BLOCK_BYTES + 1] = *p++;
    }
}

/* ---------------------------------------------------------------------------
 * Fused producers [Ferro, "How the iGPU path is fast", item 3: the residual
 * add, the norm and the int8 quantization in one pass; SwiGLU emits the next
 * GEMM's int8 input].  The pages name these fusions, not their arithmetic.
 * Readings, all in single precision, every
 * operation one IEEE rounding (sqrt and division correctly rounded):
 *   - RMSNorm as in the Llama family: h = x + delta (or x); s = sum_k h_k^2
 *     summed as the pairwise tree over k padded with zeros to a power of
 *     two; ms = s / K; r = 1 / sqrt(ms + eps); y_k = (h_k * r) * gamma_k.
 *   - SwiGLU: h = silu(g) * u with silu(g) = g / (1 + e^-g), e^x being the
 *     fixed procedure q8o_exp below (fused multiply-adds, each one
 *     rounding); gate g and up u are the first and the second half of each
 *     row of the gate/up product.
 *   - then every 32-block of y (or h) is quantized by q8o_quantize_block.
 * ------------------------------------------------------------------------- */

/* Pairwise sum: the n values padded with zeros to p = 2^ceil(log2 n) leaves,
 * then level by level each adjacent pair is added (a complete binary tree). */
float q8o_pairwise_sum(const float *v, int64_t n)
{
    if (n <= 0)
        return 0.0f;
    int64_t p = 1;
    while (p < n)
        p <<= 1;
    float *buf = (float *)malloc((size_t)p * sizeof(float));
    if (buf == NULL)
        return NAN;
    for (int64_t i = 0; i < p; ++i)
        buf[i] = i < n ? v[i] : 0.0f;
    for (int64_t w = p; w > 1; w >>= 1)
        for (int64_t i = 0; i < w / 2; ++i)
            buf[i] = buf[2 * i] + buf[2 * i + 1];
    float s = buf[0];
    free(buf);
    return s;
}

/* e^x by a fixed single-precision procedure: Cody and Waite's reduction
 * x = n ln2 + r with ln2 split into 355/512 (9 significant bits, so n * 355/512
 * is exact for |n| <= 128) plus the rest of ln2 rounded to single precision,
 * each step one fused multiply-add (fmaf, one rounding); then the Taylor
 * polynomial of degree 7 of e^r in Horner form, each step one fmaf (|r| <=
 * 0.35, truncation below 6e-9 relative); then the exact scaling by 2^n.
 * Outside [-87, 88] the result is 0 or +infinity. */
#define Q8O_LOG2E 0x1.715476p+0f      /* 1/ln 2 rounded            */
#define Q8O_LN2_HI 0x1.63p-1f         /* 355/512                   */
#define Q8O_LN2_LO -0x1.bd0106p-13f   /* ln 2 - 355/512 rounded    */
#define Q8O_C3 0x1.555556p-3f         /* 1/3! rounded              */
#define Q8O_C4 0x1.555556p-5f         /* 1/4!                      */
#define Q8O_C5 0x1.111112p-7f         /* 1/5!                      */
#define Q8O_C6 0x1.6c16c2p-10f        /* 1/6!                      */
#define Q8O_C7 0x1.a01a02p-13f        /* 1/7!                      */
float q8o_exp(float x)
{
    if (x > 88.0f)
        return INFINITY;
    if (x < -87.0f)
        return 0.0f;
    float n = rintf(x * Q8O_LOG2E);
    float r = fmaf(-n, Q8O_LN2_HI, x);
    r = fmaf(-n, Q8O_LN2_LO, r);
    float p = Q8O_C7;
    p = fmaf(p, r, Q8O_C6);
    p = fmaf(p, r, Q8O_C5);
    p = fmaf(p, r, Q8O_C4);
    p = fmaf(p, r, Q8O_C3);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return p * ldexpf(1.0f, (int)n);
}

float q8o_silu(float g)
{
    return g / (1.0f + q8o_exp(-g));
}

void q8o_exp_array(const float *x, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = q8o_exp(x[i]);
}

void q8o_silu_array(const float *x, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = q8o_silu(x[i]);
}

/* Residual add + RMSNorm + quantization of M rows of K values.
 * x, delta (may be NULL): [M][K]; gamma: [K]; h_out (may be NULL): [M][K]
 * receives h = x + delta; out: [M][K/32] blocks. */
void q8o_residual_rmsnorm_quantize(const float *x, const float *delta, const float *gamma,
                                   float eps, int64_t M, int64_t K, float *h_out, uint8_t *out)
{
    float *h = (float *)malloc((size_t)K * sizeof(float));
    float *sq = (float *)malloc((size_t)K * sizeof(float));
    float *y = (float *)malloc((size_t)K * sizeof(float));
    if (h == NULL || sq == NULL || y == NULL) {
        free(h); free(sq); free(y);
        return;
    }
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) {
            h[k] = delta != NULL ? x[m * K + k] + delta[m * K + k] : x[m * K + k];
            sq[k] = h[k] * h[k];
        }
        if (h_out != NULL)
            memcpy(h_out + m * K, h, (size_t)K * sizeof(float));
        float s = q8o_pairwise_sum(sq, K);
        float ms = s / (float)K;
        float r = 1.0f / sqrtf(ms + eps);
        for (int64_t k = 0; k < K; ++k)
            y[k] = (h[k] * r) * gamma[k];
        q8o_quantize_rows(y, 1, K, out + m * (K / QK) * BLOCK_BYTES);
    }
    free(h); free(sq); free(y);
}

/* SwiGLU + quantization: gu is [M][2F] (gate = gu[m][0..F), up =
 * gu[m][F..2F)), out is [M][F/32] blocks of h = silu(gate) * up. */
void q8o_swiglu_quantize(const float *gu, int64_t M, int64_t F, uint8_t *out)
{
    float h[QK];
    int64_t nb = F / QK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < QK; ++i) {
                float g = gu[m * 2 * F + b * QK + i];
                float u = gu[m * 2 * F + F + b * QK + i];
                h[i] = q8o_silu(g) * u;
            }
            q8o_quantize_block(h, out + (m * nb + b) * BLOCK_BYTES);
        }
}

/* ---------------------------------------------------------------------------
 * Int8 KV cache codec ("Ferro" README, "Exactness, scheduling and operations
 * (LM serving)", item "KV cache": K/V rows stored as int8 with one fp32
 * scale per 32 values, llama.cpp's q8_0 scheme for the cache, written by the
 * cache-write kernel and dequantized where attention reads it).
 *
 * Readings: the 32-value codebook is the one of q8o_quantize_block (d =
 * amax / 127, q = roundf(x * (1/d)), 1/d from the fp32 d); the stored scale
 * is that fp32 d itself, not rounded to binary16; a cache entry is D int8
 * quants in the quant plane [slot][D] plus D/32 fp32 scales in the scale
 * plane [slot][D/32] (36 bytes per 32 values); row r of the input goes to
 * cache slot slots[r] (slot r when slots is NULL); a slot outside [0,
 * capacity) is not written.  Dequantization is one single-precision
 * multiply per value: x' = (float)q * d.
 * ------------------------------------------------------------------------- */
#define KV_BLOCK_BYTES 36   /* 32 int8 + one fp32 scale */

int q8o_kv_block_bytes(void) { return KV_BLOCK_BYTES; }

void q8o_kv_quantize(const float *x, int64_t rows, int64_t D, const int32_t *slots,
                     int64_t capacity, int8_t *cache_q, float *cache_d)
{
    int64_t nb = D / QK;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t s = slots != NULL ? (int64_t)slots[r] : r;
        if (s < 0 || s >= capacity)
            continue;
        for (int64_t b = 0; b < nb; ++b) {
            const float *v = x + r * D + b * QK;
            float amax = 0.0f;
            for (int i = 0; i < QK; ++i) {
                float a = fabsf(v[i]);
                if (a > amax)
                    amax = a;
            }
            float d = amax / 127.0f;
            float id = (d != 0.0f) ? 1.0f / d : 0.0f;
            cache_d[s * nb + b] = d;
            for (int i = 0; i < QK; ++i) {
                float t = roundf(v[i] * id);
                if (t > 127.0f) t = 127.0f;
                if (t < -127.0f) t = -127.0f;
                if (t != t) t = 0.0f;       /* 0 * inf: a zero value stays zero */
                cache_q[s * D + b * QK + i] = (int8_t)(int)t;
            }
        }
    }
}

void q8o_kv_dequantize(const int8_t *cache_q, const float *cache_d, int64_t capacity, int64_t D,
                       const int32_t *slots, int64_t rows, float *out)
{
    int64_t nb = D / QK;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t s = slots != NULL ? (int64_t)slots[r] : r;
        if (s < 0 || s >= capacity)
            continue;
        for (int64_t k = 0; k < D; ++k)
            out[r * D + k] = (float)cache_q[s * D + k] * cache_d[s * nb + k / QK];
    }
}
