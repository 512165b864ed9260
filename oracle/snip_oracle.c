/*
 * snip_oracle.c -- plain, slow, single-threaded CPU oracle for the quantized
 * linear layer of sub-byte mixed-precision training (SNIP with NVFP4 / FP8).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant generator
 * with the CUDA library.
 *
 * Sources (page title, section):
 *  - "FP4 all the way" (Chmiel, Fishman, Banner, Soudry), summary page,
 *    Outline: NVFP4 = blocks of 16 E2M1 values sharing one scale stored in
 *    E4M3; round-to-nearest in the forward pass, stochastic rounding in the
 *    backpropagation and update passes; quantized learning loses efficiency
 *    once the gradient norm falls below about sqrt(3) times the quantization
 *    noise.
 *  - "Research on Mixed-Precision Training for LLMs" (newline.co), paragraph
 *    on stochastic rounding: round up or down with a probability set by the
 *    distance to the two neighbouring representable values, so that the
 *    expected value is preserved.
 *  - "SNIP: An Adaptive Mixed Precision Framework for Subbyte LLM Training",
 *    Abstract and Figure 2: per-layer FP8/FP4 choice, periodic statistics on
 *    activations, weights and gradients; Figure 5: each linear layer's
 *    forward and backward GEMMs run in the chosen low precision.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  R1  two-level scale: an fp32 tensor scale g = amax / (6 * 448) above the
 *      E4M3 block scales (g = 1 when amax == 0).
 *  R2  block scale = E4M3(amax_block / (6 g)), round-to-nearest-even, saturated
 *      at 448; elements whose scaled magnitude exceeds 6 saturate to 6.
 *  R3  element ties go to the even code.
 *  R4  the sign of the input is kept, including for results of magnitude 0.
 *  R5  elements are scaled as x * (1 / p), p = decode(s_b) * g, in fp32.
 *  R6  stochastic rounding draws 16 random bits per element from
 *      Philox4x32-10; round up iff u16 < floor(frac * 65536).
 *  R15 an element equal to zero encodes to magnitude 0 (sign kept) whatever
 *      its block's scale is; a block whose p is 0 encodes to all zeros.
 *
 * Floating point: every fp32 step below is one IEEE-754 binary32 operation
 * with round-to-nearest-even (build with -ffp-contract=off, no fast-math);
 * accumulations and dequantized values are fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 input                                                               */
/* ------------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32: widening is exact. */
static float bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static int bf16_is_finite(uint16_t h) { return (h & 0x7f80u) != 0x7f80u; }

/* ------------------------------------------------------------------------ */
/* E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.              */
/* ------------------------------------------------------------------------ */

/* Value of a 4-bit E2M1 code, from the bit fields (exponent 0 = subnormal). */
double oracle_e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* Magnitude code (0..7) nearest to y >= 0; ties go to the even code;
 * anything above the largest value (6) saturates to it. */
int oracle_e2m1_rtn(float y) {
    if (y >= 6.0f) return 7;
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 7; ++c) {
        double d = fabs((double)y - oracle_e2m1_value(c));
        if (d < bestd || (d == bestd && (c & 1) == 0)) { best = c; bestd = d; }
    }
    return best;
}

/* Stochastic rounding of y >= 0 onto the E2M1 grid with 16 random bits u16.
 * lo = largest grid value <= y, hi = the next one; go up iff
 * u16 < floor(frac * 2^16), frac = (y - lo) / (hi - lo).  y >= 6 gives 6. */
int oracle_e2m1_sr(float y, uint32_t u16) {
    if (y >= 6.0f) return 7;
    int lo = 0;
    for (int c = 0; c <= 7; ++c)
        if (oracle_e2m1_value(c) <= (double)y) lo = c;
    double vlo = oracle_e2m1_value(lo), vhi = oracle_e2m1_value(lo + 1);
    double frac = ((double)y - vlo) / (vhi - vlo);
    uint32_t thr = (uint32_t)floor(frac * 65536.0);
    return (u16 < thr) ? lo + 1 : lo;
}

/* ------------------------------------------------------------------------ */
/* E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;        */
/* S.1111.111 is NaN, the largest finite magnitude is 448.                   */
/* ------------------------------------------------------------------------ */

double oracle_e4m3_value(int code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* The 127 finite non-negative E4M3 values in code order, which is also
 * ascending order (codes 0x00..0x7e). */
static double e4m3_table[0x7f];
static int e4m3_table_ready = 0;
static void e4m3_table_init(void) {
    if (e4m3_table_ready) return;
    for (int c = 0; c <= 0x7e; ++c) e4m3_table[c] = oracle_e4m3_value(c);
    e4m3_table_ready = 1;
}

/* Largest code c with value(c) <= y, for 0 <= y (binary search on the
 * ascending table). */
static int e4m3_floor_code(double y) {
    e4m3_table_init();
    int lo = 0, hi = 0x7e;
    if (y >= e4m3_table[hi]) return hi;
    while (hi - lo > 1) {          /* invariant: value(lo) <= y < value(hi) */
        int mid = (lo + hi) / 2;
        if (e4m3_table[mid] <= y) lo = mid; else hi = mid;
    }
    return lo;
}

/* Magnitude code (0..0x7e) of the finite E4M3 value nearest to t >= 0;
 * ties go to the even code; values beyond 448 saturate to 448. */
int oracle_e4m3_rtn(float t) {
    int c = e4m3_floor_code((double)t);
    if (c == 0x7e) return c;
    double dlo = (double)t - e4m3_table[c], dhi = e4m3_table[c + 1] - (double)t;
    if (dlo < dhi) return c;
    if (dhi < dlo) return c + 1;
    return (c & 1) == 0 ? c : c + 1;
}

/* Stochastic rounding of y >= 0 onto the finite E4M3 grid (same rule as
 * oracle_e2m1_sr); y >= 448 gives 448. */
int oracle_e4m3_sr(float y, uint32_t u16) {
    if (y >= 448.0f) return 0x7e;
    int lo = e4m3_floor_code((double)y);
    double vlo = e4m3_table[lo], vhi = e4m3_table[lo + 1];
    double frac = ((double)y - vlo) / (vhi - vlo);
    uint32_t thr = (uint32_t)floor(frac * 65536.0);
    return (u16 < thr) ? lo + 1 : lo;
}

/* ------------------------------------------------------------------------ */
/* E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits; exponent 31 holds    */
/* infinities and NaNs, the largest finite magnitude is 57344 (code 0x7b).   */
/* The gradient format of FP8 training recipes; here the NEXT-2 variant for  */
/* dY and dY^T.                                                              */
/* ------------------------------------------------------------------------ */

double oracle_e5m2_value(int code) {
    int s = (code >> 7) & 1, e = (code >> 2) & 31, m = code & 3;
    if (e == 31) return m == 0 ? (s ? -INFINITY : INFINITY) : NAN;
    double mag = (e == 0) ? ldexp((double)m, -16) : ldexp(1.0 + m / 4.0, e - 15);
    return s ? -mag : mag;
}

/* The 124 finite non-negative E5M2 values in code order (0x00..0x7b), which
 * is also ascending order. */
static double e5m2_table[0x7c];
static int e5m2_table_ready = 0;
static void e5m2_table_init(void) {
    if (e5m2_table_ready) return;
    for (int c = 0; c <= 0x7b; ++c) e5m2_table[c] = oracle_e5m2_value(c);
    e5m2_table_ready = 1;
}

static int e5m2_floor_code(double y) {
    e5m2_table_init();
    int lo = 0, hi = 0x7b;
    if (y >= e5m2_table[hi]) return hi;
    while (hi - lo > 1) {          /* invariant: value(lo) <= y < value(hi) */
        int mid = (lo + hi) / 2;
        if (e5m2_table[mid] <= y) lo = mid; else hi = mid;
    }
    return lo;
}

/* Nearest finite E5M2 magnitude code to t >= 0, ties to even, saturating at 57344. */
int oracle_e5m2_rtn(float t) {
    int c = e5m2_floor_code((double)t);
    if (c == 0x7b) return c;
    double dlo = (double)t - e5m2_table[c], dhi = e5m2_table[c + 1] - (double)t;
    if (dlo < dhi) return c;
    if (dhi < dlo) return c + 1;
    return (c & 1) == 0 ? c : c + 1;
}

/* Stochastic rounding of y >= 0 onto the finite E5M2 grid (the rule of
 * oracle_e2m1_sr); y >= 57344 gives 57344. */
int oracle_e5m2_sr(float y, uint32_t u16) {
    if (y >= 57344.0f) return 0x7b;
    int lo = e5m2_floor_code((double)y);
    double vlo = e5m2_table[lo], vhi = e5m2_table[lo + 1];
    double frac = ((double)y - vlo) / (vhi - vlo);
    uint32_t thr = (uint32_t)floor(frac * 65536.0);
    return (u16 < thr) ? lo + 1 : lo;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As   */
/* Easy as 1, 2, 3", SC'11): a 4x32-bit counter, 2x32-bit key, ten rounds of */
/* two 32x32->64 multiplies, with a Weyl-sequence key schedule.              */
/* ------------------------------------------------------------------------ */

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;   /* round multipliers */
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;   /* key increments    */
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 16 random bits of source element e (row-major index into the tensor
 * being quantized, whatever the output orientation).  One Philox call serves
 * 8 consecutive elements: counter = (e/8 low word, e/8 high word, stream id
 * low, stream id high), key = (seed low, seed high); element e takes 32-bit
 * word (e/2) mod 4, low half for even e and high half for odd e. */
uint32_t oracle_sr_bits(uint64_t seed, uint64_t stream_id, uint64_t e) {
    uint64_t group = e >> 3;
    uint32_t ctr[4] = {(uint32_t)group, (uint32_t)(group >> 32),
                       (uint32_t)stream_id, (uint32_t)(stream_id >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    uint32_t w = out[(e >> 1) & 3];
    return (e & 1) ? (w >> 16) : (w & 0xffffu);
}

/* ------------------------------------------------------------------------ */
/* amax                                                                     */
/* ------------------------------------------------------------------------ */

/* Largest magnitude of a bf16 tensor; returns 1 (and m = NaN) if any element
 * is infinite or NaN, else 0. */
int oracle_amax_bf16(const uint16_t* x, int64_t n, float* m_out) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        if (!bf16_is_finite(x[i])) { *m_out = NAN; return 1; }
        float a = fabsf(bf16_to_float(x[i]));
        if (a > m) m = a;
    }
    *m_out = m;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Orientation helpers.                                                      */
/* orient 0: blocks run along the columns; output has rows x cols.          */
/* orient 1: blocks run along the rows (the transposed operand); output has */
/*           cols x rows, output row i is input column i.                    */
/* ------------------------------------------------------------------------ */

/* Source row-major index of element k of output row i. */
static int64_t src_index(int orient, int64_t rows, int64_t cols, int64_t i, int64_t k) {
    (void)rows;
    return orient == 0 ? i * cols + k : k * cols + i;
}

/* ------------------------------------------------------------------------ */
/* NVFP4                                                                     */
/* ------------------------------------------------------------------------ */

/* Tensor scale from the tensor's amax (R1). */
float oracle_nvfp4_global_scale(float amax) {
    if (amax == 0.0f) return 1.0f;
    return amax / 2688.0f; /* 2688 = 6 * 448: largest E2M1 x largest E4M3 */
}

/* Quantize a bf16 rows x cols tensor to NVFP4.
 *   orient   0 = blocks of 16 along cols (needs cols % 16 == 0),
 *            1 = blocks of 16 along rows (needs rows % 16 == 0), output is
 *                the transpose.
 *   rnd      0 = round to nearest, 1 = stochastic (seed, stream_id).
 *   g_in     if non-NULL, use *g_in as the tensor scale instead of amax/2688.
 * Outputs (output shape OR x OC: OR = rows, OC = cols for orient 0, swapped
 * for orient 1):
 *   codes        OR x OC/2 bytes, element 2j in bits 0..3 of byte j,
 *                element 2j+1 in bits 4..7; bit 3 of a code is the sign.
 *   scales       OR x OC/16 E4M3 bytes, row-major.
 *   g_out        the tensor scale used.
 *   block_sqerr  (nullable) OR x OC/16 sums of squared dequantization error.
 *   sel, n_sel   (nullable) compute only output rows sel[0..n_sel) (the tensor
 *                scale still comes from the whole tensor, the random bits from
 *                each element's index in it); outputs then have n_sel rows.
 * Returns 0, or 1 if the input holds a non-finite value (outputs untouched),
 * or 2 on a shape error. */
int oracle_quantize_nvfp4_at(const uint16_t* x, int64_t rows, int64_t cols, int orient, int rnd,
                             uint64_t seed, uint64_t stream_id, const float* g_in, uint64_t index_base,
                             uint8_t* codes, uint8_t* scales, float* g_out, double* block_sqerr,
                             const int64_t* sel, int64_t n_sel);
int oracle_quantize_nvfp4(const uint16_t* x, int64_t rows, int64_t cols, int orient, int rnd,
                          uint64_t seed, uint64_t stream_id, const float* g_in,
                          uint8_t* codes, uint8_t* scales, float* g_out, double* block_sqerr,
                          const int64_t* sel, int64_t n_sel) {
    return oracle_quantize_nvfp4_at(x, rows, cols, orient, rnd, seed, stream_id, g_in, 0, codes, scales, g_out,
                                    block_sqerr, sel, n_sel);
}

/* The same, for x holding a part of a larger row-major tensor that starts at
 * element index_base of it (a shard of whole rows, index_base = first row *
 * cols): every element draws the random bits of its index in the whole tensor
 * (R6), so the shards of a tensor quantize exactly as the tensor does when
 * they share its tensor scale (g_in). */
int oracle_quantize_nvfp4_at(const uint16_t* x, int64_t rows, int64_t cols, int orient, int rnd,
                             uint64_t seed, uint64_t stream_id, const float* g_in, uint64_t index_base,
                             uint8_t* codes, uint8_t* scales, float* g_out, double* block_sqerr,
                             const int64_t* sel, int64_t n_sel) {
    int64_t OR = orient == 0 ? rows : cols, OC = orient == 0 ? cols : rows;
    if (OC % 16 != 0) return 2;
    float amax;
    if (oracle_amax_bf16(x, rows * cols, &amax)) return 1;
    float g = g_in ? *g_in : oracle_nvfp4_global_scale(amax);
    *g_out = g;
    int64_t nb = OC / 16;
    int64_t nout = sel ? n_sel : OR;
    for (int64_t ii = 0; ii < nout; ++ii) {
        int64_t i = sel ? sel[ii] : ii;   /* output row computed; results go to row ii */
        for (int64_t b = 0; b < nb; ++b) {
            float xs[16];
            uint64_t es[16];
            float ab = 0.0f;
            for (int k = 0; k < 16; ++k) {
                es[k] = (uint64_t)src_index(orient, rows, cols, i, b * 16 + k);
                xs[k] = bf16_to_float(x[es[k]]);
                if (fabsf(xs[k]) > ab) ab = fabsf(xs[k]);
            }
            /* block scale: E4M3 of amax_block / (6 g), the product 6 g first */
            float six_g = 6.0f * g;
            float t = ab / six_g;
            int sb = oracle_e4m3_rtn(t);
            scales[ii * nb + b] = (uint8_t)sb;
            float p = (float)oracle_e4m3_value(sb) * g;
            double q = oracle_e4m3_value(sb) * (double)g; /* exact step of one grid unit */
            double err = 0.0;
            for (int k = 0; k < 16; ++k) {
                int sign = signbit(xs[k]) ? 8 : 0;
                int mag = 0;
                if (p != 0.0f && xs[k] != 0.0f) {
                    float inv = 1.0f / p;
                    float y = fabsf(xs[k]) * inv;
                    mag = rnd == 0 ? oracle_e2m1_rtn(y)
                                   : oracle_e2m1_sr(y, oracle_sr_bits(seed, stream_id, index_base + es[k]));
                }
                int code = sign | mag;
                int64_t col = b * 16 + k;
                uint8_t* byte = &codes[ii * (OC / 2) + col / 2];
                if ((col & 1) == 0) *byte = (uint8_t)((*byte & 0xf0) | code);
                else *byte = (uint8_t)((*byte & 0x0f) | (code << 4));
                double xhat = oracle_e2m1_value(code) * q;
                err += (xhat - (double)xs[k]) * (xhat - (double)xs[k]);
            }
            if (block_sqerr) block_sqerr[ii * nb + b] = err;
        }
    }
    return 0;
}

/* Dequantize NVFP4 (OR x OC) into fp64: value(code) * decode(scale) * g. */
void oracle_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales, float g,
                          int64_t OR, int64_t OC, double* out) {
    for (int64_t i = 0; i < OR; ++i)
        for (int64_t k = 0; k < OC; ++k) {
            uint8_t byte = codes[i * (OC / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            double s = oracle_e4m3_value(scales[i * (OC / 16) + k / 16]);
            out[i * OC + k] = oracle_e2m1_value(code) * s * (double)g;
        }
}

/* ------------------------------------------------------------------------ */
/* NVFP4 element and scale formats with longer blocks (the block-size axis   */
/* of the FP4 study in "FP4 all the way", summary page, Outline): B = 16,    */
/* 32, 64 or 128 E2M1 values share one E4M3 scale under the same tensor     */
/* scale g.  B = 16 is NVFP4 itself.                                          */
/* ------------------------------------------------------------------------ */

/* Quantize a bf16 rows x cols tensor with one E4M3 scale per `block`
 * consecutive elements along the blocked dim (orient as for NVFP4; the
 * blocked dim must be a multiple of block).  Every step is NVFP4's (R1, R2,
 * R5, R6, R15) with the block maximum taken over `block` elements.
 * Outputs: codes OR x OC/2 bytes as for NVFP4; scales OR x OC/block E4M3
 * bytes (one per block, row-major); g_out; sel / n_sel as for NVFP4.
 * Returns 0, 1 (non-finite input) or 2 (shape). */
int oracle_quantize_nvfp4_block(const uint16_t* x, int64_t rows, int64_t cols, int orient, int rnd,
                                uint64_t seed, uint64_t stream_id, const float* g_in, int block,
                                uint8_t* codes, uint8_t* scales, float* g_out,
                                const int64_t* sel, int64_t n_sel) {
    int64_t OR = orient == 0 ? rows : cols, OC = orient == 0 ? cols : rows;
    if (block < 16 || block > 128 || (block & (block - 1)) != 0 || OC % block != 0) return 2;
    float amax;
    if (oracle_amax_bf16(x, rows * cols, &amax)) return 1;
    float g = g_in ? *g_in : oracle_nvfp4_global_scale(amax);
    *g_out = g;
    int64_t nb = OC / block;
    int64_t nout = sel ? n_sel : OR;
    for (int64_t ii = 0; ii < nout; ++ii) {
        int64_t i = sel ? sel[ii] : ii;
        for (int64_t b = 0; b < nb; ++b) {
            /* the block's largest magnitude over all of its elements */
            float ab = 0.0f;
            for (int k = 0; k < block; ++k) {
                float v = fabsf(bf16_to_float(x[src_index(orient, rows, cols, i, b * block + k)]));
                if (v > ab) ab = v;
            }
            float six_g = 6.0f * g;
            int sb = oracle_e4m3_rtn(ab / six_g);
            scales[ii * nb + b] = (uint8_t)sb;
            float p = (float)oracle_e4m3_value(sb) * g;
            for (int k = 0; k < block; ++k) {
                uint64_t e = (uint64_t)src_index(orient, rows, cols, i, b * block + k);
                float xv = bf16_to_float(x[e]);
                int sign = signbit(xv) ? 8 : 0;
                int mag = 0;
                if (p != 0.0f && xv != 0.0f) {
                    float inv = 1.0f / p;
                    float y = fabsf(xv) * inv;
                    mag = rnd == 0 ? oracle_e2m1_rtn(y) : oracle_e2m1_sr(y, oracle_sr_bits(seed, stream_id, e));
                }
                int code = sign | mag;
                int64_t col = b * block + k;
                uint8_t* byte = &codes[ii * (OC / 2) + col / 2];
                if ((col & 1) == 0) *byte = (uint8_t)((*byte & 0xf0) | code);
                else *byte = (uint8_t)((*byte & 0x0f) | (code << 4));
            }
        }
    }
    return 0;
}

/* Dequantize (OR x OC, one scale per `block` elements) into fp64. */
void oracle_dequant_nvfp4_block(const uint8_t* codes, const uint8_t* scales, float g, int block,
                                int64_t OR, int64_t OC, double* out) {
    for (int64_t i = 0; i < OR; ++i)
        for (int64_t k = 0; k < OC; ++k) {
            uint8_t byte = codes[i * (OC / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            double s = oracle_e4m3_value(scales[i * (OC / block) + k / block]);
            out[i * OC + k] = oracle_e2m1_value(code) * s * (double)g;
        }
}

/* ------------------------------------------------------------------------ */
/* MXFP4 (OCP Microscaling Formats specification v1.0, the format the FP4    */
/* study of "FP4 all the way" weighs against NVFP4 on block size and scale  */
/* format): 32 E2M1 elements share one E8M0 scale, a power of two           */
/* 2^(code - 127); there is no tensor scale.                                 */
/* ------------------------------------------------------------------------ */

/* Value of an E8M0 code: 2^(code - 127); code 255 is NaN. */
double oracle_e8m0_value(int code) {
    if (code == 255) return NAN;
    double v = 1.0;
    for (int k = 127; k < code; ++k) v *= 2.0;
    for (int k = code; k < 127; ++k) v /= 2.0;
    return v;
}

/* The block's shared exponent: floor(log2(amax)) less the largest E2M1
 * exponent (2, as 6 = 1.5 x 2^2), clamped to E8M0's [-127, 127]; an
 * all-zero block takes -127. */
int oracle_mxfp4_shared_exp(float amax) {
    if (amax == 0.0f) return -127;
    double a = amax;
    int e = 0;
    while (a >= 2.0) { a /= 2.0; ++e; }
    while (a < 1.0) { a *= 2.0; --e; }
    int se = e - 2;
    if (se < -127) se = -127;
    if (se > 127) se = 127;
    return se;
}

/* Quantize a bf16 rows x cols tensor to MXFP4: per block of 32 along the
 * blocked dim, se = oracle_mxfp4_shared_exp(block amax), scale code se + 127,
 * y = |x| * 2^-se (one fp32 multiplication by that power of two), code =
 * sign | E2M1(y) rounded as for NVFP4 (nearest, or stochastic with the same
 * random bits per source element).  Orientation and return values as for
 * NVFP4; codes OR x OC/2 bytes, scales OR x OC/32 bytes; needs OC % 32 == 0;
 * sel, n_sel as for NVFP4. */
int oracle_quantize_mxfp4(const uint16_t* x, int64_t rows, int64_t cols, int orient, int rnd,
                          uint64_t seed, uint64_t stream_id, uint8_t* codes, uint8_t* scales,
                          const int64_t* sel, int64_t n_sel) {
    int64_t OR = orient == 0 ? rows : cols, OC = orient == 0 ? cols : rows;
    if (OC % 32 != 0) return 2;
    float amax;
    if (oracle_amax_bf16(x, rows * cols, &amax)) return 1;
    int64_t nb = OC / 32;
    int64_t nout = sel ? n_sel : OR;
    for (int64_t ii = 0; ii < nout; ++ii) {
        int64_t i = sel ? sel[ii] : ii;
        for (int64_t b = 0; b < nb; ++b) {
            float xs[32];
            uint64_t es[32];
            float ab = 0.0f;
            for (int k = 0; k < 32; ++k) {
                es[k] = (uint64_t)src_index(orient, rows, cols, i, b * 32 + k);
                xs[k] = bf16_to_float(x[es[k]]);
                if (fabsf(xs[k]) > ab) ab = fabsf(xs[k]);
            }
            int se = oracle_mxfp4_shared_exp(ab);
            scales[ii * nb + b] = (uint8_t)(se + 127);
            float inv = (float)oracle_e8m0_value(127 - se);   /* 2^-se, exact in fp32 */
            for (int k = 0; k < 32; ++k) {
                int sign = signbit(xs[k]) ? 8 : 0;
                float y = fabsf(xs[k]) * inv;
                int mag = rnd == 0 ? oracle_e2m1_rtn(y)
                                   : oracle_e2m1_sr(y, oracle_sr_bits(seed, stream_id, es[k]));
                int code = sign | mag;
                int64_t col = b * 32 + k;
                uint8_t* byte = &codes[ii * (OC / 2) + col / 2];
                if ((col & 1) == 0) *byte = (uint8_t)((*byte & 0xf0) | code);
                else *byte = (uint8_t)((*byte & 0x0f) | (code << 4));
            }
        }
    }
    return 0;
}

/* Dequantize MXFP4 (OR x OC) into fp64: value(code) * 2^(scale - 127). */
void oracle_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, int64_t OR, int64_t OC, double* out) {
    for (int64_t i = 0; i < OR; ++i)
        for (int64_t k = 0; k < OC; ++k) {
            uint8_t byte = codes[i * (OC / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            out[i * OC + k] = oracle_e2m1_value(code) * oracle_e8m0_value(scales[i * (OC / 32) + k / 32]);
        }
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 with one fp32 scale per tensor                                   */
/* ------------------------------------------------------------------------ */

float oracle_fp8_tensor_scale(float amax) {
    if (amax == 0.0f) return 1.0f;
    return amax / 448.0f;
}

/* Quantize a bf16 rows x cols tensor to E4M3 codes with one tensor scale s
 * (x ~ code * s).  Orientation, rounding and return values as for NVFP4;
 * codes is OR x OC bytes; sel, n_sel as for NVFP4. */
int oracle_quantize_fp8_at(const uint16_t* x, int64_t rows, int64_t cols, int orient, int rnd,
                           uint64_t seed, uint64_t stream_id, const float* s_in, uint64_t index_base,
                           uint8_t* codes, float* s_out, const int64_t* sel, int64_t n_sel);
int oracle_quantize_fp8(const uint16_t* x, int64_t rows, int64_t cols, int orient, int rnd,
                        uint64_t seed, uint64_t stream_id, const float* s_in,
                        uint8_t* codes, float* s_out, const int64_t* sel, int64_t n_sel) {
    return oracle_quantize_fp8_at(x, rows, cols, orient, rnd, seed, stream_id, s_in, 0, codes, s_out, sel, n_sel);
}

/* The same for a part of a larger tensor starting at element index_base of it
 * (as oracle_quantize_nvfp4_at). */
int oracle_quantize_fp8_at(const uint16_t* x, int64_t rows, int64_t cols, int orient, int rnd,
                           uint64_t seed, uint64_t stream_id, const float* s_in, uint64_t index_base,
                           uint8_t* codes, float* s_out, const int64_t* sel, int64_t n_sel) {
    int64_t OR = orient == 0 ? rows : cols, OC = orient == 0 ? cols : rows;
    float amax;
    if (oracle_amax_bf16(x, rows * cols, &amax)) return 1;
    float s = s_in ? *s_in : oracle_fp8_tensor_scale(amax);
    *s_out = s;
    float inv = 1.0f / s;
    int64_t nout = sel ? n_sel : OR;
    for (int64_t ii = 0; ii < nout; ++ii)
        for (int64_t k = 0; k < OC; ++k) {
            int64_t i = sel ? sel[ii] : ii;
            uint64_t e = (uint64_t)src_index(orient, rows, cols, i, k);
            float xv = bf16_to_float(x[e]);
            int sign = signbit(xv) ? 0x80 : 0;
            int mag = 0;
            if (xv != 0.0f) {
                float y = fabsf(xv) * inv;
                mag = rnd == 0 ? oracle_e4m3_rtn(y)
                               : oracle_e4m3_sr(y, oracle_sr_bits(seed, stream_id, index_base + e));
            }
            codes[ii * OC + k] = (uint8_t)(sign | mag);
        }
    return 0;
}

void oracle_dequant_fp8(const uint8_t* codes, float s, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_value(codes[i]) * (double)s;
}

/* E5M2 with one tensor scale s = amax / 57344 (1 for an all-zero tensor) or
 * *s_in: code = sign | E5M2(|x| * (1/s)), nearest-even saturating (RTN) or
 * stochastic with the element's 16 Philox bits (SR).  Orientation, row
 * selection and return values as for oracle_quantize_fp8. */
float oracle_e5m2_tensor_scale(float amax) {
    if (amax == 0.0f) return 1.0f;
    return amax / 57344.0f;
}

int oracle_quantize_e5m2(const uint16_t* x, int64_t rows, int64_t cols, int orient, int rnd,
                         uint64_t seed, uint64_t stream_id, const float* s_in,
                         uint8_t* codes, float* s_out, const int64_t* sel, int64_t n_sel) {
    int64_t OR = orient == 0 ? rows : cols, OC = orient == 0 ? cols : rows;
    float amax;
    if (oracle_amax_bf16(x, rows * cols, &amax)) return 1;
    float s = s_in ? *s_in : oracle_e5m2_tensor_scale(amax);
    *s_out = s;
    float inv = 1.0f / s;
    int64_t nout = sel ? n_sel : OR;
    for (int64_t ii = 0; ii < nout; ++ii)
        for (int64_t k = 0; k < OC; ++k) {
            int64_t i = sel ? sel[ii] : ii;
            uint64_t e = (uint64_t)src_index(orient, rows, cols, i, k);
            float xv = bf16_to_float(x[e]);
            int sign = signbit(xv) ? 0x80 : 0;
            int mag = 0;
            if (xv != 0.0f) {
                float y = fabsf(xv) * inv;
                mag = rnd == 0 ? oracle_e5m2_rtn(y)
                               : oracle_e5m2_sr(y, oracle_sr_bits(seed, stream_id, e));
            }
            codes[ii * OC + k] = (uint8_t)(sign | mag);
        }
    return 0;
}

void oracle_dequant_e5m2(const uint8_t* codes, float s, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e5m2_value(codes[i]) * (double)s;
}

/* ------------------------------------------------------------------------ */
/* Statistics (SNIP's periodic statistics on one tensor)                     */
/* ------------------------------------------------------------------------ */

/* Slots of the raw statistics vector. */
enum {
    ST_SUM_X2 = 0,      /* ||A||^2                                          */
    ST_NVFP4_ERR2 = 1,  /* ||Q_nvfp4(A) - A||^2 under the given rounding     */
    ST_FP8_ERR2 = 2,    /* ||Q_fp8(A) - A||^2 under the given rounding       */
    ST_NVFP4_SRVAR = 3, /* sum over elements of (hi-|y|)(|y|-lo) q^2, NVFP4  */
    ST_FP8_SRVAR = 4,   /* the same on the FP8 grid                          */
    ST_AMAX = 5,        /* max |A|                                           */
    ST_COUNT = 6,       /* number of elements                                */
    ST_N = 8
};

/* Largest grid value <= y and the next one, for the expected-variance sum. */
static void e2m1_bracket(float y, double* lo, double* hi) {
    int c = 0;
    for (int k = 0; k <= 7; ++k)
        if (oracle_e2m1_value(k) <= (double)y) c = k;
    *lo = oracle_e2m1_value(c);
    *hi = c < 7 ? oracle_e2m1_value(c + 1) : *lo;
}
static void e4m3_bracket(float y, double* lo, double* hi) {
    int c = e4m3_floor_code((double)y);
    *lo = e4m3_table[c];
    *hi = c < 0x7e ? e4m3_table[c + 1] : *lo;
}

/* One pass of statistics over a bf16 rows x cols tensor (blocks of 16 along
 * cols, the tensor's own rounding rnd with (seed, stream_id) for SR).
 * out[ST_N] receives the raw sums; block_err_nvfp4 / block_err_fp8
 * (nullable, rows x cols/16) receive per-block squared errors.
 * Returns 0, 1 for non-finite input, 2 for a shape error. */
int oracle_quant_stats_at(const uint16_t* x, int64_t rows, int64_t cols, int rnd, uint64_t seed,
                          uint64_t stream_id, const float* g_in, const float* s_in, uint64_t index_base,
                          double* out, double* block_err_nvfp4, double* block_err_fp8);
int oracle_quant_stats(const uint16_t* x, int64_t rows, int64_t cols, int rnd,
                       uint64_t seed, uint64_t stream_id, double* out,
                       double* block_err_nvfp4, double* block_err_fp8) {
    return oracle_quant_stats_at(x, rows, cols, rnd, seed, stream_id, NULL, NULL, 0, out, block_err_nvfp4,
                                 block_err_fp8);
}

/* The statistics of a part of a larger tensor (rows starting at element
 * index_base of it) under the whole tensor's scales g_in, s_in (NULL: this
 * part's own): the sums of the parts are the whole tensor's; out[ST_AMAX] is
 * this part's amax (the whole tensor's is their maximum). */
int oracle_quant_stats_at(const uint16_t* x, int64_t rows, int64_t cols, int rnd, uint64_t seed,
                          uint64_t stream_id, const float* g_in, const float* s_in, uint64_t index_base,
                          double* out, double* block_err_nvfp4, double* block_err_fp8) {
    if (cols % 16 != 0) return 2;
    int64_t n = rows * cols;
    uint8_t* c4 = (uint8_t*)calloc((size_t)(n / 2 + 1), 1);
    uint8_t* s4 = (uint8_t*)calloc((size_t)(n / 16 + 1), 1);
    uint8_t* c8 = (uint8_t*)calloc((size_t)(n + 1), 1);
    double* bl4 = (double*)calloc((size_t)(n / 16 + 1), sizeof(double));
    if (!c4 || !s4 || !c8 || !bl4) { free(c4); free(s4); free(c8); free(bl4); return 3; }
    float g, s;
    int st = oracle_quantize_nvfp4_at(x, rows, cols, 0, rnd, seed, stream_id, g_in, index_base, c4, s4, &g, bl4,
                                      NULL, 0);
    if (st == 0)
        st = oracle_quantize_fp8_at(x, rows, cols, 0, rnd, seed, stream_id, s_in, index_base, c8, &s, NULL, 0);
    if (st != 0) { free(c4); free(s4); free(c8); free(bl4); return st; }
    for (int k = 0; k < ST_N; ++k) out[k] = 0.0;
    float amax;
    oracle_amax_bf16(x, n, &amax);
    out[ST_AMAX] = amax;
    out[ST_COUNT] = (double)n;
    float inv8 = 1.0f / s;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t b = 0; b < cols / 16; ++b) {
            int sb = s4[i * (cols / 16) + b];
            float p = (float)oracle_e4m3_value(sb) * g;
            double q4 = oracle_e4m3_value(sb) * (double)g;
            double e8 = 0.0;
            for (int k = 0; k < 16; ++k) {
                int64_t e = i * cols + b * 16 + k;
                double xv = (double)bf16_to_float(x[e]);
                out[ST_SUM_X2] += xv * xv;
                /* FP8 error */
                double xh8 = oracle_e4m3_value(c8[e]) * (double)s;
                e8 += (xh8 - xv) * (xh8 - xv);
                /* expected SR variance, both grids, in units of x */
                if (xv != 0.0) {
                    double lo, hi;
                    if (p != 0.0f) {
                        float y4 = fabsf((float)xv) * (1.0f / p);
                        if (y4 < 6.0f) {
                            e2m1_bracket(y4, &lo, &hi);
                            out[ST_NVFP4_SRVAR] += (hi - y4) * (y4 - lo) * q4 * q4;
                        }
                    }
                    float y8 = fabsf((float)xv) * inv8;
                    if (y8 < 448.0f) {
                        e4m3_bracket(y8, &lo, &hi);
                        out[ST_FP8_SRVAR] += (hi - y8) * (y8 - lo) * (double)s * (double)s;
                    }
                }
            }
            out[ST_NVFP4_ERR2] += bl4[i * (cols / 16) + b];
            out[ST_FP8_ERR2] += e8;
            if (block_err_nvfp4) block_err_nvfp4[i * (cols / 16) + b] = bl4[i * (cols / 16) + b];
            if (block_err_fp8) block_err_fp8[i * (cols / 16) + b] = e8;
        }
    free(c4); free(s4); free(c8); free(bl4);
    return 0;
}
