/*
 * qpo.c — scalar CPU oracle (see qpo.h for scope and citations).
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU baseline, never by the product library.
 *
 * Compile with -ffp-contract=off and without fast-math: every f32 operation
 * below is rounded on its own.
 *
 * Block layouts (GGUF reading; the pages name the types, the workload
 * definition gives field sizes and the value formulas):
 *
 *   Q8_0  32 values, 34 B:  d:f16 | q:int8[32]               value = d*q
 *   Q4_K 256 values, 144 B: d:f16 | dmin:f16 | scales:u8[12] | qs:u8[128]
 *         eight sub-blocks of 32 values, each with a 6-bit scale sc and a
 *         6-bit min m;                                       value = d*sc*q - dmin*m
 *   Q2_K 256 values, 84 B:  scales:u8[16] | qs:u8[64] | d:f16 | dmin:f16
 *         sixteen sub-blocks of 16 values; scales[s] low nibble = sc,
 *         high nibble = m;                                   value = d*sc*q - dmin*m
 *   Q6_K 256 values, 210 B: ql:u8[128] | qh:u8[64] | scales:i8[16] | d:f16
 *         sixteen sub-blocks of 16 values;                   value = d*s*(q-32)
 *   Q5_K 256 values, 176 B: d:f16 | dmin:f16 | scales:u8[12] | qh:u8[32] |
 *         qs:u8[128]; sub-blocks, scales and mins as in Q4_K; each q has a
 *         fifth (high) bit held in the qh plane;             value = d*sc*q - dmin*m
 *   F16     1 value,   2 B: the fp16 weight itself;          value = that fp16
 * (Q5_K and F16 are in the page's list of types the f32 dequant has device
 * kernels for, "Qwen3.5 batched prefill has no f32 dequant for IQ2_XXS,
 * IQ3_S, IQ3_XXS, Q2_K", section Cause.)
 */
#include "qpo.h"

#include <fenv.h>
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int qpo_block_info(int type, int64_t *qk, int64_t *block_bytes) {
    switch (type) {
    case QPO_Q8_0: *qk = 32;  *block_bytes = 34;  return 0;
    case QPO_Q4_K: *qk = 256; *block_bytes = 144; return 0;
    case QPO_Q2_K: *qk = 256; *block_bytes = 84;  return 0;
    case QPO_Q6_K: *qk = 256; *block_bytes = 210; return 0;
    case QPO_Q5_K: *qk = 256; *block_bytes = 176; return 0;
    case QPO_F16:  *qk = 1;   *block_bytes = 2;   return 0;
    default: return -1;
    }
}

int qpo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void qpo_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------- fp16 --- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Written from the definition: a normal number is (1024+f)*2^(e-25), a
 * subnormal f*2^-24.  Both products are exact in binary32. */
float qpo_f16_to_f32(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    float mag;
    if (e == 0)
        mag = ldexpf((float)f, -24);
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexpf((float)(1024 + f), e - 25);
    return sign ? -mag : mag;
}

/* Encode a magnitude that is exactly representable in binary16 (or is 2^16,
 * the first value past the largest finite one). */
static uint16_t encode_exact_f16(double a) {
    if (a == 0.0) return 0;
    if (a < ldexp(1.0, -14))                    /* subnormal: a = f * 2^-24 */
        return (uint16_t)(a * ldexp(1.0, 24));
    int ex;
    frexp(a, &ex);                              /* a = m * 2^ex, m in [0.5,1) */
    const int e = ex - 1;                       /* a in [2^e, 2^(e+1)) */
    if (e > 15) return 0x7c00;                  /* overflow -> inf */
    const double frac = a * ldexp(1.0, 10 - e) - 1024.0;   /* exact integer */
    return (uint16_t)(((e + 15) << 10) | (int)frac);
}

/* Round to the nearest binary16 value, ties to even: scale |f| so that the
 * binary16 quantum at its exponent becomes 1, round that to the nearest
 * integer in the default (to-nearest-even) mode, and scale back.  All of it is
 * exact in double except the one intended rounding. */
uint16_t qpo_f32_to_f16(float f) {
    const uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f)) return (uint16_t)(sign | 0x7e00);
    const double a = fabs((double)f);
    if (isinf(f)) return (uint16_t)(sign | 0x7c00);
    int quantum_exp;                            /* quantum = 2^quantum_exp */
    if (a < ldexp(1.0, -14)) {
        quantum_exp = -24;
    } else {
        int ex;
        frexp(a, &ex);
        quantum_exp = (ex - 1) - 10;
    }
    const int saved = fegetround();
    fesetround(FE_TONEAREST);
    const double n = nearbyint(ldexp(a, -quantum_exp));
    fesetround(saved);
    const double r = ldexp(n, quantum_exp);
    if (r >= 65536.0) return (uint16_t)(sign | 0x7c00);   /* past 65504 -> inf */
    return (uint16_t)(sign | encode_exact_f16(r));
}

void qpo_f16_to_f32_array(const uint16_t *h, int64_t n, float *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = qpo_f16_to_f32(h[i]);
}

void qpo_f32_to_f16_array(const float *f, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = qpo_f32_to_f16(f[i]);
}

/* ----------------------------------------------------------- decoding --- */

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Q8_0: value v = d * q[v]. */
static float decode_q8_0(const uint8_t *b, int v) {
    const float d = qpo_f16_to_f32(rd16(b));
    const float q = (float)(int8_t)b[2 + v];
    return d * q;
}

/* Q4_K 6-bit scale/min of sub-block s (0..7) from the 12 packed bytes.
 * Sub-blocks 0-3 keep sc and m in the low six bits of bytes s and s+4.
 * Sub-blocks 4-7 keep their low four bits in the nibbles of byte s+4
 * (sc low, m high) and their top two bits in the top two bits of bytes
 * s-4 (for sc) and s (for m). */
static void q4_k_scale_min(const uint8_t *scales, int s, int *sc, int *m) {
    if (s < 4) {
        *sc = scales[s] & 63;
        *m = scales[s + 4] & 63;
    } else {
        *sc = (scales[s + 4] & 0x0f) | ((scales[s - 4] >> 6) << 4);
        *m = (scales[s + 4] >> 4) | ((scales[s] >> 6) << 4);
    }
}

/* Q4_K: value v lies in sub-block s = v/32 and 64-value group g = v/64; its
 * 4-bit q is the low nibble of qs[32g + v%32] for the first 32 values of the
 * group and the high nibble of the same byte for the last 32. */
static float decode_q4_k(const uint8_t *b, int v) {
    const float d = qpo_f16_to_f32(rd16(b + 0));
    const float dmin = qpo_f16_to_f32(rd16(b + 2));
    const uint8_t *scales = b + 4;
    const uint8_t *qs = b + 16;
    const int s = v / 32, g = v / 64;
    int sc, m;
    q4_k_scale_min(scales, s, &sc, &m);
    const uint8_t byte = qs[32 * g + v % 32];
    const int q = (v % 64 < 32) ? (byte & 0x0f) : (byte >> 4);
    const float dl = d * (float)sc;
    const float ml = dmin * (float)m;
    const float dq = dl * (float)q;
    return dq - ml;
}

/* Q2_K: value v = 128n + 32j + l (l < 32) takes bits 2j..2j+1 of qs[32n + l];
 * its sub-block is s = v/16 with scale byte scales[s]. */
static float decode_q2_k(const uint8_t *b, int v) {
    const uint8_t *scales = b + 0;
    const uint8_t *qs = b + 16;
    const float d = qpo_f16_to_f32(rd16(b + 80));
    const float dmin = qpo_f16_to_f32(rd16(b + 82));
    const int n = v / 128, j = (v % 128) / 32, l = v % 32;
    const int q = (qs[32 * n + l] >> (2 * j)) & 3;
    const int s = v / 16;
    const int sc = scales[s] & 0x0f;
    const int m = scales[s] >> 4;
    const float dl = d * (float)sc;
    const float ml = dmin * (float)m;
    const float dq = dl * (float)q;
    return dq - ml;
}

/* Q6_K: value v = 128n + 32j + l (l < 32).  The low four bits of its 6-bit q
 * are a nibble of ql[64n + l + 32*(j&1)] (low nibble for j < 2, high for
 * j >= 2); the high two bits are bits 2j..2j+1 of qh[32n + l].  Its sub-block
 * is s = v/16 with signed scale scales[s]. */
static float decode_q6_k(const uint8_t *b, int v) {
    const uint8_t *ql = b + 0;
    const uint8_t *qh = b + 128;
    const int8_t *scales = (const int8_t *)(b + 192);
    const float d = qpo_f16_to_f32(rd16(b + 208));
    const int n = v / 128, j = (v % 128) / 32, l = v % 32;
    const uint8_t lbyte = ql[64 * n + l + 32 * (j & 1)];
    const int lo = (j < 2) ? (lbyte & 0x0f) : (lbyte >> 4);
    const int hi = (qh[32 * n + l] >> (2 * j)) & 3;
    const int q = lo | (hi << 4);
    const int s = v / 16;
    const float dl = d * (float)scales[s];
    return dl * (float)(q - 32);
}

/* Q5_K: value v lies in sub-block s = v/32 and 64-value group g = v/64; the
 * low four bits of its 5-bit q are the Q4_K nibble (low nibble of
 * qs[32g + v%32] for the first 32 values of the group, high nibble for the
 * last 32) and its fifth bit is bit s of qh[v%32]. */
static float decode_q5_k(const uint8_t *b, int v) {
    const float d = qpo_f16_to_f32(rd16(b + 0));
    const float dmin = qpo_f16_to_f32(rd16(b + 2));
    const uint8_t *scales = b + 4;
    const uint8_t *qh = b + 16;
    const uint8_t *qs = b + 48;
    const int s = v / 32, g = v / 64, l = v % 32;
    int sc, m;
    q4_k_scale_min(scales, s, &sc, &m);
    const uint8_t byte = qs[32 * g + l];
    const int lo = (v % 64 < 32) ? (byte & 0x0f) : (byte >> 4);
    const int q = lo | (((qh[l] >> s) & 1) << 4);
    const float dl = d * (float)sc;
    const float ml = dmin * (float)m;
    const float dq = dl * (float)q;
    return dq - ml;
}

/* F16: the block is one fp16 weight; its value is that number. */
static float decode_f16(const uint8_t *b, int v) {
    (void)v;
    return qpo_f16_to_f32(rd16(b));
}

float qpo_decode_value(int type, const uint8_t *block, int v) {
    switch (type) {
    case QPO_Q8_0: return decode_q8_0(block, v);
    case QPO_Q4_K: return decode_q4_k(block, v);
    case QPO_Q2_K: return decode_q2_k(block, v);
    case QPO_Q6_K: return decode_q6_k(block, v);
    case QPO_Q5_K: return decode_q5_k(block, v);
    case QPO_F16: return decode_f16(block, v);
    default: return NAN;
    }
}

/* ------------------------------------------------------------ dequant --- */

/* Row r holds nb = ceil(cols/QK) whole blocks, back to back; value c of row r
 * is value c%QK of block c/QK.  Only the first `cols` values are written: the
 * padding values of a partial last block are never decoded into the output. */
int qpo_dequant_f32(int type, const void *blocks, int64_t rows, int64_t cols, float *out) {
    int64_t qk, bb;
    if (qpo_block_info(type, &qk, &bb)) return -1;
    const int64_t nb = (cols + qk - 1) / qk;
    const uint8_t *base = (const uint8_t *)blocks;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            const uint8_t *blk = base + (r * nb + c / qk) * bb;
            out[r * cols + c] = qpo_decode_value(type, blk, (int)(c % qk));
        }
    }
    return 0;
}

/* The f16 copy is made from the f32 result (issue #4952 §Cause, f16 mode). */
int qpo_dequant_f16(int type, const void *blocks, int64_t rows, int64_t cols, uint16_t *out) {
    int64_t qk, bb;
    if (qpo_block_info(type, &qk, &bb)) return -1;
    const int64_t nb = (cols + qk - 1) / qk;
    const uint8_t *base = (const uint8_t *)blocks;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            const uint8_t *blk = base + (r * nb + c / qk) * bb;
            out[r * cols + c] = qpo_f32_to_f16(qpo_decode_value(type, blk, (int)(c % qk)));
        }
    }
    return 0;
}

/* --------------------------------------------------------------- GEMM --- */

void qpo_gemm_f64(const uint16_t *X, const float *W, int64_t T, int64_t out, int64_t in,
                  const int64_t *rows, int64_t nrows, double *Y, double *A) {
    if (!rows) nrows = T;
    /* The selected X rows, widened to double once. */
    double *xd = (double *)malloc((size_t)(nrows * in) * sizeof(double));
    if (!xd) return;
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t t = rows ? rows[i] : i;
        for (int64_t k = 0; k < in; ++k) xd[i * in + k] = (double)qpo_f16_to_f32(X[t * in + k]);
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < nrows * out; ++p) {
        const int64_t i = p / out, o = p % out;
        const double *x = xd + i * in;
        const float *w = W + o * in;
        double y = 0.0, a = 0.0;
        for (int64_t k = 0; k < in; ++k) {
            const double wv = (double)w[k];
            y += x[k] * wv;
            a += fabs(x[k]) * fabs(wv);
        }
        Y[p] = y;
        A[p] = a;
    }
    free(xd);
}
