/*
 * synth.c — seeded synthetic inputs for the tests and the benchmark.
 *
 * This module only draws random numbers and places them at the byte offsets
 * of each block format.  It holds none of the method's arithmetic (no
 * decoding, no scale unpacking, no GEMM).  Both the CPU oracle and the CUDA
 * path are fed the bytes it writes.
 *
 * Random source: splitmix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used counter-based: draw i of
 * a stream with key K is mix(K + (i+1)*GAMMA), so every block or value can be
 * generated independently and in parallel with identical results.
 *
 * Distributions (per block type; d and dmin are fp16 values snapped from a
 * uniform draw in [1e-3, 1e-2)):
 *   Q8_0: d; 32 int8 q uniform on [-127, 127].
 *   Q4_K: d, dmin; 12 scale bytes and 128 qs bytes uniform, so every packed
 *         6-bit scale/min is uniform on [0, 63] and every 4-bit q on [0, 15].
 *   Q2_K: 16 scale bytes and 64 qs bytes uniform (4-bit scale/min uniform on
 *         [0, 15], 2-bit q on [0, 3]); d, dmin.
 *   Q6_K: 128 ql and 64 qh bytes uniform (6-bit q uniform on [0, 63]);
 *         16 int8 scales uniform on [-127, 127]; d.
 *   Q5_K: d, dmin; 12 scale bytes, 32 qh bytes and 128 qs bytes uniform
 *         (6-bit scale/min uniform on [0, 63], 5-bit q on [0, 31]).
 *   F16:  one weight per block, standard normal snapped to fp16.
 *   X:    standard normal (Box-Muller), snapped to fp16.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

/* Stream key of tensor `tensor` under `seed`. */
uint64_t synth_key(uint64_t seed, uint64_t tensor) {
    return mix64(mix64(seed + GAMMA) + (tensor + 1) * 0xD1B54A32D192ED03ULL);
}

/* Nearest fp16 bit pattern to x (round half away from zero); x is a finite
 * sample well inside the fp16 range.  Used only to put samples on the fp16
 * grid. */
static uint16_t snap_f16(double x) {
    uint16_t sign = 0;
    if (x < 0) { sign = 0x8000; x = -x; }
    if (x == 0.0) return sign;
    if (x < 6.103515625e-05) {                 /* below 2^-14: multiples of 2^-24 */
        long n = (long)floor(x * 16777216.0 + 0.5);
        return (uint16_t)(sign | (uint16_t)n); /* n == 1024 encodes 2^-14 */
    }
    int ex;
    double m = frexp(x, &ex);                  /* x = m*2^ex, m in [0.5, 1) */
    long mant = (long)floor(m * 2048.0 + 0.5); /* 1024..2048 */
    if (mant == 2048) { mant = 1024; ex += 1; }
    int biased = ex - 1 + 15;
    if (biased >= 31) return (uint16_t)(sign | 0x7bff);
    return (uint16_t)(sign | (uint16_t)(biased << 10) | (uint16_t)(mant - 1024));
}

static inline double unit53(uint64_t z) { return (double)(z >> 11) * (1.0 / 9007199254740992.0); }

static inline void put16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }

static uint16_t scale_sample(uint64_t z) { return snap_f16(1e-3 + 9e-3 * unit53(z)); }

/* int8 uniform on [-127, 127] from a 16-bit slice. */
static inline uint8_t int8_sym(uint32_t u16) { return (uint8_t)(int8_t)((int)((u16 * 255u) >> 16) - 127); }

/* Fill n bytes from consecutive draws starting at draw index i0. */
static void fill_bytes(uint64_t key, uint64_t i0, uint8_t *p, int n) {
    for (int k = 0; k < n; k += 8) {
        uint64_t z = draw(key, i0 + (uint64_t)(k / 8));
        for (int b = 0; b < 8 && k + b < n; ++b) p[k + b] = (uint8_t)(z >> (8 * b));
    }
}

/* Draws per block: fixed strides so block b never overlaps block b+1. */
#define STRIDE 64

void synth_blocks(int type, uint64_t key, int64_t nblocks, uint8_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
        const uint64_t i0 = (uint64_t)b * STRIDE;
        if (type == 8) {                         /* Q8_0, 34 B */
            uint8_t *p = out + b * 34;
            put16(p, scale_sample(draw(key, i0)));
            for (int v = 0; v < 32; v += 4) {
                uint64_t z = draw(key, i0 + 1 + (uint64_t)(v / 4));
                for (int u = 0; u < 4; ++u) p[2 + v + u] = int8_sym((uint32_t)(z >> (16 * u)) & 0xffffu);
            }
        } else if (type == 12) {                 /* Q4_K, 144 B */
            uint8_t *p = out + b * 144;
            put16(p + 0, scale_sample(draw(key, i0)));
            put16(p + 2, scale_sample(draw(key, i0 + 1)));
            fill_bytes(key, i0 + 2, p + 4, 140);
        } else if (type == 10) {                 /* Q2_K, 84 B */
            uint8_t *p = out + b * 84;
            fill_bytes(key, i0 + 2, p, 80);
            put16(p + 80, scale_sample(draw(key, i0)));
            put16(p + 82, scale_sample(draw(key, i0 + 1)));
        } else if (type == 13) {                 /* Q5_K, 176 B */
            uint8_t *p = out + b * 176;
            put16(p + 0, scale_sample(draw(key, i0)));
            put16(p + 2, scale_sample(draw(key, i0 + 1)));
            fill_bytes(key, i0 + 2, p + 4, 172);
        } else if (type == 1) {                  /* F16, 2 B */
            const uint64_t z = draw(key, i0);
            const double u1 = ((double)(z >> 32) + 1.0) * (1.0 / 4294967296.0);
            const double u2 = (double)(z & 0xffffffffu) * (1.0 / 4294967296.0);
            put16(out + b * 2, snap_f16(sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2)));
        } else if (type == 14) {                 /* Q6_K, 210 B */
            uint8_t *p = out + b * 210;
            fill_bytes(key, i0 + 2, p, 192);
            for (int s = 0; s < 16; s += 4) {
                uint64_t z = draw(key, i0 + 40 + (uint64_t)(s / 4));
                for (int u = 0; u < 4; ++u) p[192 + s + u] = int8_sym((uint32_t)(z >> (16 * u)) & 0xffffu);
            }
            put16(p + 208, scale_sample(draw(key, i0)));
        }
    }
}

/* Blocks whose quant, scale and min bytes are all uniform random bytes, so
 * every bit pattern of every field occurs (int8 q = -128 in Q8_0, int8 scale
 * = -128 in Q6_K, 6-bit scales and mins with their top bits set, ...), while
 * the fp16 d and dmin fields are drawn as in synth_blocks, which keeps every
 * weight finite.  F16 blocks are drawn as in synth_blocks. */
void synth_blocks_anybits(int type, uint64_t key, int64_t nblocks, uint8_t *out) {
    if (type == 1) {
        synth_blocks(type, key, nblocks, out);
        return;
    }
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
        const uint64_t i0 = (uint64_t)b * STRIDE;
        if (type == 8) {                         /* Q8_0: d | q[32] */
            uint8_t *p = out + b * 34;
            fill_bytes(key, i0 + 2, p + 2, 32);
            put16(p, scale_sample(draw(key, i0)));
        } else if (type == 12 || type == 13) {   /* Q4_K, Q5_K: d | dmin | ... */
            const int bb = type == 12 ? 144 : 176;
            uint8_t *p = out + b * bb;
            fill_bytes(key, i0 + 2, p + 4, bb - 4);
            put16(p + 0, scale_sample(draw(key, i0)));
            put16(p + 2, scale_sample(draw(key, i0 + 1)));
        } else if (type == 10) {                 /* Q2_K: ... | d | dmin */
            uint8_t *p = out + b * 84;
            fill_bytes(key, i0 + 2, p, 80);
            put16(p + 80, scale_sample(draw(key, i0)));
            put16(p + 82, scale_sample(draw(key, i0 + 1)));
        } else if (type == 14) {                 /* Q6_K: ql | qh | scales | d */
            uint8_t *p = out + b * 210;
            fill_bytes(key, i0 + 2, p, 208);
            put16(p + 208, scale_sample(draw(key, i0)));
        }
    }
}

/* n standard-normal fp16 values (Box-Muller, one value per draw: the upper 32
 * bits give u1 in (0,1], the lower 32 bits u2 in [0,1)). */
void synth_normal_f16(uint64_t key, int64_t n, uint16_t *out) {
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t z = draw(key, (uint64_t)i);
        double u1 = ((double)(z >> 32) + 1.0) * (1.0 / 4294967296.0);
        double u2 = (double)(z & 0xffffffffu) * (1.0 / 4294967296.0);
        out[i] = snap_f16(sqrt(-2.0 * log(u1)) * cos(two_pi * u2));
    }
}

/* n raw random bytes (used for guard-band and fuzz tests). */
void synth_bytes(uint64_t key, int64_t n, uint8_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < (n + 4095) / 4096; ++c) {
        int64_t lo = c * 4096, len = (n - lo < 4096) ? n - lo : 4096;
        fill_bytes(key, (uint64_t)lo / 8, out + lo, (int)len);
    }
}
