// gemv.cu — the decode-side projection over the same weight blocks:
//   Y[t, o] = sum_k X[t, k] * W[o, k]      0 <= t < T <= 8
// for a handful of token rows: the serial path one token at a time ("QK-norm
// models take the FP16 batched prefill when it fits", §What changes: the
// serial prefill is one forward per prompt token) and the decode GEMVs that
// run over the same block types ("Qwen3.5 batched prefill has no f32 dequant
// for IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", §Cause).  W is the exact f32 dequant
// for the K-quants (their codes are multiplied as they are and the scales
// applied in f32, below) and the fp16 weights of the f16 dequant for Q8_0
// and F16; the sums are f32.
//
// Meant to be bound by HBM on W (every weight byte is read once), which puts
// the integer pipe on a budget of one to two instructions per weight value:
// the lanes only isolate code bits, and the dot products run on the tensor
// cores with the warp-level mma.sync m16n8k16.  The MMA's A operand is 16
// weight rows x 16 K values in fp16, B is X (8 columns), D = f32.
//
// Two persistent CTAs per SM take 16-row blocks b, b + gridDim.x, ... of the
// launch.  A producer warp streams each block's rows through a ring of
// shared-memory tiles with 2-D TMA copies: a tile is the 16 rows x S steps
// (S x 256 values) of one K range, as the 16-byte aligned cover of that range
// in every row (up to 2 KB per row, so that the copies are long).  Eight
// consumer warps split the tiles: with S < 8 (Q8_0, F16), warp w takes step
// w % S of every tile its team w / S is given (the teams take a block's tiles
// in turn); with S >= 8, warp w takes steps w, w + 8, ... of every tile.
// Every consumer warp waits for and releases every tile.  Measured on
// the 8B-shaped layer's weights at T = 1, two such CTAs per SM stream 13%
// faster than one with twice the warps and ring.  A step is 256 values of
// weight rows g and g + 8 for lane (g, c) (g = lane / 4, c = lane % 4): the
// K-quants in the sub-block group layout described with their steps below;
// Q8_0 and F16 with the exact run decoders of qp_runs.cuh (runs 2c, 2c + 1
// rounded to fp16, B = the token rows, the MMA's K order permuted alike in
// A and B so that K slots 2c, 2c + 1, 2c + 8, 2c + 9 hold values 4i .. 4i + 3
// of lane c's run in MMA i).  Steps past the row's end contribute zeros.  At
// a block's end the consumer warps' 16 x 8 partial tiles are summed through
// shared memory in warp order, so results are deterministic: for the
// K-quants at T <= 4 by the warp that completes the block's arrival count
// (no barrier), otherwise behind a named barrier over the consumers only.
//
// Weights whose row pitch is not a multiple of 16 bytes (which a TMA tensor
// cannot describe) are staged instead by 16 bulk copies a tile, one per row.
//
// Every wait is bounded; on expiry the kernel records an error bit and stops
// (the consumers still meet at every block's barrier), and the producer
// waits for its copies in flight before the CTA exits.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qp_decode.cuh"
#include "qp_internal.h"
#include "qp_ptx.cuh"
#include "qp_runs.cuh"
#include "qp_sync.cuh"

namespace qp {
namespace {

using namespace runs;

// Bytes per block and 32-value runs per block (F16: a "block" of 32 values)
// for the types decoded through the generic run decoders.
template <int TYPE> struct Geom;
template <> struct Geom<kQ8_0> { static constexpr int BB = 34, RPB = 1; };
template <> struct Geom<kF16> { static constexpr int BB = 64, RPB = 1; };

// One run's 32 weights as 16 fp16 pairs (values 2p, 2p + 1 in word p).
template <int TYPE>
__device__ __forceinline__ void run_f16(const typename RawOf<TYPE>::T &raw, int t, uint32_t (&h)[16]) {
    if constexpr (TYPE == kF16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            h[4 * i] = raw.a[i].x;
            h[4 * i + 1] = raw.a[i].y;
            h[4 * i + 2] = raw.a[i].z;
            h[4 * i + 3] = raw.a[i].w;
        }
    } else {
        pair_t y[16];
        raw.decode(t, y);
#pragma unroll
        for (int p = 0; p < 16; ++p) h[p] = f2h2(y[p]);
    }
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------- K-quant steps on the raw codes --
// The K-quant weights are never formed.  An MMA's A operand holds the raw
// quantized codes of 16 rows: each code u (a small unsigned integer) sits in
// the low bits of its fp16 field, which is then the subnormal u * 2^-24,
// exactly.  Within one sub-block of a row the value formulas of the K-quant
// page ("Q2_K", "Q4_K", "Q5_K", "Q6_K" sections) are affine in u:
//   w = alpha * (u * 2^-24) + beta,
//   Q2_K, Q4_K, Q5_K: alpha = d * sc * 2^24, beta = -(dmin * m);
//   Q6_K:             alpha = d * s * 2^24,  beta = -32 * d * s.
// So a sub-block's share of a dot product is alpha * D + beta * SX, where
// D = sum_k X[k] * A[k] comes from the tensor cores and SX = sum_k X[k] from
// one more MMA whose A is all ones.  alpha * u * 2^-24 and beta are the
// exact factors of the f32 dequant (d * sc * u and dmin * m need at most 24
// significant bits), so each weight behind the sums is the exact f32 value:
// a one-hot X row returns it bit for bit.
//
// The scales are applied per (row, sub-block, token) with a group layout: an
// MMA's 16 K slots belong to NSB consecutive sub-blocks, and its 8 N columns
// to (token, sub-block) pairs.  K slot pair p (slots 2p, 2p + 1) holds
// sub-block p % NSB of the group, values i * 16 / NSB + 2 * (p / NSB) + {0, 1}
// of it in the group's MMA i (NSB = 1 and 2: pairs c and c + 4 hold values
// 16i / NSB + 4 (c / (2 / NSB)) + {0, 1} and {2, 3} of their sub-block, so that
// a lane's four X values are one 8-byte load); column n is token n / NSB
// restricted to
// sub-block n % NSB (zero in the other sub-blocks' slots), so column n of D
// sums one sub-block of one token.  NSB = 8 / T rounded up to a power of
// two: at T = 1 one MMA spans eight sub-blocks and the scales cost two f32x2
// fmas per lane per eight MMAs.  Lane (g, c) holds A of rows g, g + 8 in K
// pairs c and c + 4, B of column g, and D of columns 2c, 2c + 1.

constexpr uint32_t kOnesH2 = 0x3C003C00u;   // fp16 1.0 twice

// X beyond a lane's column reads as zeros from here (a step's offsets stay
// below 256 values).
__device__ __align__(16) uint16_t g_zero_x[256];

__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint32_t lds16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }
__device__ __forceinline__ uint32_t lds8(const uint8_t *p) { return *p; }
__device__ __forceinline__ uint2 ldx64(const uint16_t *p) { return __ldg(reinterpret_cast<const uint2 *>(p)); }
__device__ __forceinline__ uint4 ldx128(const uint16_t *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ uint32_t word_of(const uint4 &v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

// Bytes 2h, 2h + 1 of w into the low bytes of two fp16 fields.
__device__ __forceinline__ uint32_t spread(uint32_t w, int h) { return __byte_perm(w, 0u, h ? 0x4342 : 0x4140); }

// 2^e as a float, for small integer e (exact scaling).
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

template <int NSB>
struct LaneMap {
    int c;
    int j0, j1;    // sub-block (within the group) of K pairs c and c + 4
    int jg, tg;    // column g: its sub-block and token
    int jn;        // D columns 2c, 2c + 1: sub-blocks jn, jn + 1 (NSB > 1), or jn for both (NSB = 1)
    __device__ __forceinline__ LaneMap(int g, int c_)
        : c(c_), j0(c_ % NSB), j1((c_ + 4) % NSB), jg(g % NSB), tg(g / NSB), jn((2 * c_) % NSB) {}
};

// The value B words of the lane in MMA i of a group, from the column-g
// sub-block chunk at xa (pair c) and xb (pair c + 4) (zeros where the lane's
// pair is not in column g's sub-block): for NSB >= 4 word i * 8 / NSB +
// (p / NSB) of it, for NSB <= 2 the four values from 16i / NSB +
// 4 (c / (2 / NSB)) in one load.
template <int NSB>
struct XWords {
    uint4 qa, qb;
    __device__ __forceinline__ void get(const uint16_t *xa, const uint16_t *xb, int i, int c, uint32_t &b0,
                                        uint32_t &b1) {
        if constexpr (NSB == 8) {                       // words i, i
            if (i % 4 == 0) {
                qa = ldx128(xa + 2 * i);
                qb = ldx128(xb + 2 * i);
            }
            b0 = word_of(qa, i % 4);
            b1 = word_of(qb, i % 4);
        } else if constexpr (NSB == 4) {                // words 2i, 2i + 1 (xa = xb)
            if (i % 2 == 0) qa = ldx128(xa + 4 * i);
            b0 = word_of(qa, 2 * (i % 2));
            b1 = word_of(qa, 2 * (i % 2) + 1);
        } else if constexpr (NSB == 2) {                // values 8i + 4(c/2) .. + 3 (xa = xb)
            const uint2 v = ldx64(xa + 8 * i + 4 * (c >> 1));
            b0 = v.x;
            b1 = v.y;
        } else {                                        // values 16i + 4c .. 16i + 4c + 3 (xa = xb)
            const uint2 v = ldx64(xa + 16 * i + 4 * c);
            b0 = v.x;
            b1 = v.y;
        }
    }
};

// ---- Q2_K (84-byte superblocks: scales[16], qs[64], d, dmin): value v of
// sub-block s is crumb (s % 8) / 2 of qs[32 (s / 8) + 16 (s % 2) + v], the
// crumb kept in place in its byte (code u * 4^crumb); scale byte s holds sc
// (low nibble) and m (high nibble).  Pairs c and c + 4 always read the same
// 16 qs bytes of a group.
template <int NSB>
struct Q2Codes {
    static constexpr int SBV = 16, NSUB = 16;
    uint32_t w[NSB == 1 ? 1 : (NSB == 2 ? 2 : 4)];
    uint32_t m0, m1;
    __device__ __forceinline__ void load(const uint8_t *sb, int gm, int c) {
        constexpr uint32_t M = 0x00030003u;
        if constexpr (NSB == 8) {                       // s = 8gm + c, 8gm + c + 4
            const uint8_t *q = sb + 16 + 32 * gm + 16 * (c & 1);
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = lds32(q + 4 * k);
            m0 = M << (2 * (c >> 1));
            m1 = m0 << 4;
        } else if constexpr (NSB == 4) {                // s = 4gm + c
            const uint8_t *q = sb + 16 + 32 * (gm >> 1) + 16 * (c & 1);
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = lds32(q + 4 * k);
            m0 = m1 = M << (2 * (2 * (gm & 1) + (c >> 1)));
        } else if constexpr (NSB == 2) {                // s = 2gm + c % 2, values 8i + 4(c/2) .. + 3
            const uint8_t *q = sb + 16 + 32 * (gm >> 2) + 16 * (c & 1) + 4 * (c >> 1);
            w[0] = lds32(q);
            w[1] = lds32(q + 8);
            m0 = m1 = M << (2 * (gm & 3));
        } else {                                        // s = gm, values 4c .. 4c + 3
            w[0] = lds32(sb + 16 + 32 * (gm >> 3) + 16 * (gm & 1) + 4 * c);
            m0 = m1 = M << (2 * ((gm & 7) >> 1));
        }
    }
    __device__ __forceinline__ uint32_t pair(int i, int p) const {
        if constexpr (NSB == 8) return spread(w[i >> 1], i & 1) & (p ? m1 : m0);
        else if constexpr (NSB == 4) return spread(w[i], p) & m0;
        else if constexpr (NSB == 2) return spread(w[i], p) & m0;
        else return spread(w[0], p) & m0;
    }
};

// Q2_K alpha / beta of the lane's D columns in group gm for one row.
template <int NSB>
__device__ __forceinline__ void q2_scales(const uint8_t *sb, float d, float ndmin, int gm, const LaneMap<NSB> &L,
                                          pair_t &al, pair_t &be) {
    const int s0 = gm * NSB + L.jn;                     // even when NSB > 1
    const int crumb = (s0 & 7) >> 1;
    const float dsc = d * pow2f(24 - 2 * crumb);        // exact
    if constexpr (NSB > 1) {
        const uint32_t sw = lds16(sb + s0);
        const uint32_t scw = sw & 0x0F0Fu, mw = (sw >> 4) & 0x0F0Fu;
        const pair_t nbias = pk2(-8388608.0f, -8388608.0f);
        const pair_t sc = fadd2(pk2(bias_float<0>(scw), bias_float<1>(scw)), nbias);   // exact
        const pair_t m = fadd2(pk2(bias_float<0>(mw), bias_float<1>(mw)), nbias);
        al = fmul2(pk2(dsc, dsc), sc);
        be = fmul2(pk2(ndmin, ndmin), m);
    } else {
        const uint32_t b = lds8(sb + s0);
        const float a = dsc * u2f_exact(b & 15u), n = ndmin * u2f_exact(b >> 4);
        al = pk2(a, a);
        be = pk2(n, n);
    }
}

// ---- Q6_K (210-byte superblocks: ql[128], qh[64], scales[16] int8, d):
// value v of sub-block s (half n = s / 8, j = (s % 8) / 2, l = 16 (s % 2) + v)
// is the low (j < 2) or high nibble of ql[64n + 32 (j % 2) + l] plus crumb j
// of qh[32n + l] as bits 4..5: the 6-bit code u (value d * s * (u - 32)).
// A superblock starts 2 bytes past a 4-byte boundary when its offset in the
// stage is; MIS = 0: aligned, 1: 2 bytes past, 2: per lane (shift `sh`).
// Words are then read from the aligned address 2 bytes early and realigned;
// every read stays inside the superblock.
template <int MIS, int N>
__device__ __forceinline__ void q6_words(const uint8_t *p, uint32_t sh, uint32_t (&w)[N]) {
    if constexpr (MIS == 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) w[k] = lds32(p + 4 * k);
    } else {
        const uint8_t *a = p - (MIS == 1 ? 2 : static_cast<int>(sh >> 3));
        const uint32_t s = MIS == 1 ? 16u : sh;
        uint32_t t[N + 1];
#pragma unroll
        for (int k = 0; k <= N; ++k) t[k] = lds32(a + 4 * k);
#pragma unroll
        for (int k = 0; k < N; ++k) w[k] = __funnelshift_r(t[k], t[k + 1], s);
    }
}

// Four 6-bit codes (one per byte) from a ql word (nibble half `hi`) and a qh
// word (crumb j).
__device__ __forceinline__ uint32_t q6_code_word(uint32_t wl, uint32_t wh, int hi, int j) {
    return ((hi ? wl >> 4 : wl) & 0x0F0F0F0Fu) | (((wh >> (2 * j)) << 4) & 0x30303030u);
}

template <int NSB, int MIS>
struct Q6Codes {
    static constexpr int SBV = 16, NSUB = 16;
    static constexpr int NW = NSB == 1 ? 1 : (NSB == 2 ? 2 : 4);
    uint32_t u0[NW], u1[NSB == 8 ? 4 : 1];
    __device__ __forceinline__ void load(const uint8_t *sb, uint32_t sh, int gm, int c) {
        if constexpr (NSB == 8) {
            // s = 8gm + c (low nibbles, crumb c/2) and 8gm + c + 4 (high nibbles,
            // crumb c/2 + 2): the same 16 ql and 16 qh bytes
            uint32_t wl[4], wh[4];
            q6_words<MIS, 4>(sb + 64 * gm + 16 * c, sh, wl);
            q6_words<MIS, 4>(sb + 128 + 32 * gm + 16 * (c & 1), sh, wh);
            const int j = c >> 1;
            const uint32_t keep = 0x33333333u << (2 * j);      // crumbs j and j + 2 of every byte
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t hm = wh[k] & keep;
                u0[k] = (wl[k] & 0x0F0F0F0Fu) | ((hm << (4 - 2 * j)) & 0xF0F0F0F0u);
                u1[k] = ((wl[k] >> 4) & 0x0F0F0F0Fu) | ((hm >> (2 * j)) & 0xF0F0F0F0u);
            }
        } else if constexpr (NSB == 4) {                       // s = 4gm + c
            uint32_t wl[4], wh[4];
            q6_words<MIS, 4>(sb + 64 * (gm >> 1) + 16 * c, sh, wl);
            q6_words<MIS, 4>(sb + 128 + 32 * (gm >> 1) + 16 * (c & 1), sh, wh);
            const int j = 2 * (gm & 1) + (c >> 1);
#pragma unroll
            for (int k = 0; k < 4; ++k) u0[k] = q6_code_word(wl[k], wh[k], gm & 1, j);
        } else if constexpr (NSB == 2) {                       // s = 2gm + c % 2, values 8i + 4(c/2) .. + 3
            const int l0 = 16 * (c & 1) + 4 * (c >> 1);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                uint32_t wl[1], wh[1];
                q6_words<MIS, 1>(sb + 64 * (gm >> 2) + 32 * (gm & 1) + l0 + 8 * i, sh, wl);
                q6_words<MIS, 1>(sb + 128 + 32 * (gm >> 2) + l0 + 8 * i, sh, wh);
                u0[i] = q6_code_word(wl[0], wh[0], (gm & 3) >= 2, gm & 3);
            }
        } else {                                               // s = gm, values 4c .. 4c + 3
            const int n = gm >> 3, j = (gm & 7) >> 1, l0 = 16 * (gm & 1) + 4 * c;
            uint32_t wl[1], wh[1];
            q6_words<MIS, 1>(sb + 64 * n + 32 * (j & 1) + l0, sh, wl);
            q6_words<MIS, 1>(sb + 128 + 32 * n + l0, sh, wh);
            u0[0] = q6_code_word(wl[0], wh[0], j >= 2, j);
        }
    }
    __device__ __forceinline__ uint32_t pair(int i, int p) const {
        if constexpr (NSB == 8) return spread(p ? u1[i >> 1] : u0[i >> 1], i & 1);
        else if constexpr (NSB == 4) return spread(u0[i], p);
        else if constexpr (NSB == 2) return spread(u0[i], p);
        else return spread(u0[0], p);
    }
};

template <int NSB>
__device__ __forceinline__ void q6_scales(const uint8_t *sb, float d24, int gm, const LaneMap<NSB> &L, pair_t &al,
                                          pair_t &be) {
    const int s0 = gm * NSB + L.jn;
    const pair_t m32 = pk2(-1.9073486328125e-06f, -1.9073486328125e-06f);   // -32 * 2^-24
    if constexpr (NSB > 1) {
        const uint32_t sx = lds16(sb + 192 + s0) ^ 0x8080u;                // int8 + 128
        const pair_t nb = pk2(-8388736.0f, -8388736.0f);                  // -(2^23 + 128)
        const pair_t s = fadd2(pk2(bias_float<0>(sx), bias_float<1>(sx)), nb);   // exact
        al = fmul2(pk2(d24, d24), s);                                      // d * s * 2^24, exact
    } else {
        const float s = static_cast<float>(static_cast<int8_t>(lds8(sb + 192 + s0)));
        const float a = d24 * s;
        al = pk2(a, a);
    }
    be = fmul2(al, m32);                                                   // -32 * d * s, exact
}

// ---- Q4_K / Q5_K (144- / 176-byte superblocks, 16-byte aligned in the
// stage: d, dmin, 12 bytes of packed 6-bit (sc, m), Q5_K's qh[32], qs[128]):
// value v of sub-block s (32 values) is the low (s even) or high nibble of
// qs[32 (s / 2) + v], Q5_K's fifth bit being bit s of qh[v].
template <int TYPE, int NSB>
struct K4Codes {
    static constexpr bool Q5 = TYPE == kQ5_K;
    static constexpr int QS = Q5 ? 48 : 16;
    static constexpr int SBV = 32, NSUB = 8;
    const uint8_t *q0, *q1, *qh;   // qs words of pairs c and c + 4 (MMA i reads word i * 8 / NSB + ...)
    int hi, s0, s1;                // nibble half; sub-blocks of the pairs (Q5_K's qh bit)
    __device__ __forceinline__ void load(const uint8_t *sb, int gm, int c) {
        qh = sb + 16;
        if constexpr (NSB == 8) {                       // s = c, c + 4
            q0 = sb + QS + 32 * (c >> 1);
            q1 = q0 + 64;
            hi = c & 1;
            s0 = c;
            s1 = c + 4;
        } else if constexpr (NSB == 4) {                // s = 4gm + c
            q0 = q1 = sb + QS + 64 * gm + 32 * (c >> 1);
            hi = c & 1;
            s0 = s1 = 4 * gm + c;
        } else if constexpr (NSB == 2) {                // s = 2gm + c % 2
            q0 = q1 = sb + QS + 32 * gm;
            hi = c & 1;
            s0 = s1 = 2 * gm + (c & 1);
        } else {                                        // s = gm
            q0 = q1 = sb + QS + 32 * (gm >> 1);
            hi = gm & 1;
            s0 = s1 = gm;
        }
    }
    // the codes of qs word k (and qh word k) of pair p, one per byte
    __device__ __forceinline__ uint32_t codes(int k, int p) const {
        const uint32_t w = lds32((p ? q1 : q0) + 4 * k);
        uint32_t u = (hi ? w >> 4 : w) & 0x0F0F0F0Fu;
        if constexpr (Q5) u |= ((lds32(qh + 4 * k) >> (p ? s1 : s0)) & 0x01010101u) << 4;
        return u;
    }
    __device__ __forceinline__ uint32_t pair(int i, int p, int c) const {
        if constexpr (NSB == 8) return spread(codes(i >> 1, p), i & 1);          // values 2i, 2i + 1
        else if constexpr (NSB == 4) return spread(codes(i, 0), p);              // 4i + 2p ..
        else if constexpr (NSB == 2) return spread(codes(2 * i + (c >> 1), 0), p);   // 8i + 4(c/2) + 2p ..
        else return spread(codes(4 * i + c, 0), p);                             // 16i + 4c + 2p ..
    }
};

// The 6-bit (sc, m) of sub-block t from the packed scale bytes (hd.y, hd.z,
// hd.w = bytes 4..15 of the superblock).
__device__ __forceinline__ void k4_sm(const uint4 &hd, int t, uint32_t &sc, uint32_t &m) {
    const int sh = 8 * (t & 3);
    const uint32_t ys = hd.y >> sh, zs = hd.z >> sh, ws = hd.w >> sh;
    sc = t < 4 ? (ys & 63u) : ((ws & 15u) | ((ys >> 6 & 3u) << 4));
    m = t < 4 ? (zs & 63u) : (((ws >> 4) & 15u) | ((zs >> 6 & 3u) << 4));
}

template <int NSB>
__device__ __forceinline__ void k4_scales(const uint4 &hd, float d24, float ndmin, int gm, const LaneMap<NSB> &L,
                                          pair_t &al, pair_t &be) {
    const int t0 = gm * NSB + L.jn;
    uint32_t sc0, m0;
    k4_sm(hd, t0, sc0, m0);
    if constexpr (NSB > 1) {
        uint32_t sc1, m1;
        k4_sm(hd, t0 + 1, sc1, m1);
        al = fmul2(pk2(d24, d24), pk2(u2f_exact(sc0), u2f_exact(sc1)));      // d * sc * 2^24, exact
        be = fmul2(pk2(ndmin, ndmin), pk2(u2f_exact(m0), u2f_exact(m1)));   // -(dmin * m), exact
    } else {
        const float a = d24 * u2f_exact(sc0), n = ndmin * u2f_exact(m0);
        al = pk2(a, a);
        be = pk2(n, n);
    }
}

// Per-row, per-superblock header values.
template <int TYPE> struct RowHead;
template <> struct RowHead<kQ2_K> {
    float d24, ndmin;   // d (scaled per group by the crumb), -dmin
    __device__ __forceinline__ explicit RowHead(const uint8_t *sb) {
        const uint32_t dd = lds32(sb + 80);
        d24 = h2f(dd);
        ndmin = -h2f(dd >> 16);
    }
};
template <> struct RowHead<kQ6_K> {
    float d24;
    __device__ __forceinline__ explicit RowHead(const uint8_t *sb) { d24 = h2f(lds16(sb + 208)) * 16777216.0f; }
};
template <int TYPE> struct K4Head {
    uint4 hd;
    float d24, ndmin;
    __device__ __forceinline__ explicit K4Head(const uint8_t *sb) {
        hd = *reinterpret_cast<const uint4 *>(sb);
        d24 = h2f(hd.x) * 16777216.0f;
        ndmin = -h2f(hd.x >> 16);
    }
};
template <> struct RowHead<kQ4_K> : K4Head<kQ4_K> {
    __device__ __forceinline__ explicit RowHead(const uint8_t *sb) : K4Head<kQ4_K>(sb) {}
};
template <> struct RowHead<kQ5_K> : K4Head<kQ5_K> {
    __device__ __forceinline__ explicit RowHead(const uint8_t *sb) : K4Head<kQ5_K>(sb) {}
};

// mma.sync without `volatile`: a pure function of its registers, so loads
// around it may be merged and scheduled freely.
__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int TYPE, int NSB, int MIS> struct CodesOf;
template <int NSB, int MIS> struct CodesOf<kQ2_K, NSB, MIS> { using T = Q2Codes<NSB>; };
template <int NSB, int MIS> struct CodesOf<kQ6_K, NSB, MIS> { using T = Q6Codes<NSB, MIS>; };
template <int NSB, int MIS> struct CodesOf<kQ4_K, NSB, MIS> { using T = K4Codes<kQ4_K, NSB>; };
template <int NSB, int MIS> struct CodesOf<kQ5_K, NSB, MIS> { using T = K4Codes<kQ5_K, NSB>; };

template <int TYPE, int NSB, int MIS>
__device__ __forceinline__ void load_codes(typename CodesOf<TYPE, NSB, MIS>::T &q, const uint8_t *sb, uint32_t sh,
                                           int gm, int c) {
    if constexpr (TYPE == kQ6_K) q.load(sb, sh, gm, c);
    else q.load(sb, gm, c);
}

template <int TYPE, int NSB, int MIS>
__device__ __forceinline__ uint32_t code_pair(const typename CodesOf<TYPE, NSB, MIS>::T &q, int i, int p, int c) {
    if constexpr (TYPE == kQ4_K || TYPE == kQ5_K) return q.pair(i, p, c);
    else return q.pair(i, p);
}

template <int TYPE, int NSB>
__device__ __forceinline__ void group_scales(const uint8_t *sb, const RowHead<TYPE> &h, int gm,
                                             const LaneMap<NSB> &L, pair_t &al, pair_t &be) {
    if constexpr (TYPE == kQ2_K) q2_scales<NSB>(sb, h.d24, h.ndmin, gm, L, al, be);
    else if constexpr (TYPE == kQ6_K) q6_scales<NSB>(sb, h.d24, gm, L, al, be);
    else k4_scales<NSB>(h.hd, h.d24, h.ndmin, gm, L, al, be);
}

// NSB = 1: the factors of rows g and g + 8 (the same sub-block gm) computed
// together in f32 pairs, the same exact operations as group_scales per row;
// each row's alpha and beta then fill both of its D columns (the tokens).
template <int TYPE>
__device__ __forceinline__ void row_pair_scales(const uint8_t *r0, const uint8_t *r1, const RowHead<TYPE> &h0,
                                                const RowHead<TYPE> &h1, int gm, pair_t &al0, pair_t &be0,
                                                pair_t &al1, pair_t &be1) {
    const pair_t nbias = pk2(-8388608.0f, -8388608.0f);
    pair_t a, n;
    if constexpr (TYPE == kQ2_K) {
        const float p2 = pow2f(24 - 2 * ((gm & 7) >> 1));                  // the crumb's 4^-crumb
        const uint32_t w = lds8(r0 + gm) | (lds8(r1 + gm) << 8);           // the rows' scale bytes
        const uint32_t scw = w & 0x0F0Fu, mw = (w >> 4) & 0x0F0Fu;
        const pair_t sc = fadd2(pk2(bias_float<0>(scw), bias_float<1>(scw)), nbias);   // exact
        const pair_t m = fadd2(pk2(bias_float<0>(mw), bias_float<1>(mw)), nbias);
        a = fmul2(pk2(h0.d24 * p2, h1.d24 * p2), sc);                      // exact
        n = fmul2(pk2(h0.ndmin, h1.ndmin), m);                             // -(dmin * m), exact
    } else if constexpr (TYPE == kQ6_K) {
        const uint32_t sx = (lds8(r0 + 192 + gm) | (lds8(r1 + 192 + gm) << 8)) ^ 0x8080u;   // int8 + 128
        const pair_t sv = fadd2(pk2(bias_float<0>(sx), bias_float<1>(sx)), pk2(-8388736.0f, -8388736.0f));
        a = fmul2(pk2(h0.d24, h1.d24), sv);                                // d * s * 2^24, exact
        n = fmul2(a, pk2(-1.9073486328125e-06f, -1.9073486328125e-06f)); // -32 * d * s, exact
    } else {
        uint32_t sc0, m0, sc1, m1;
        k4_sm(h0.hd, gm, sc0, m0);
        k4_sm(h1.hd, gm, sc1, m1);
        const pair_t sc = fadd2(pk2(__uint_as_float(0x4B000000u | sc0), __uint_as_float(0x4B000000u | sc1)), nbias);
        const pair_t m = fadd2(pk2(__uint_as_float(0x4B000000u | m0), __uint_as_float(0x4B000000u | m1)), nbias);
        a = fmul2(pk2(h0.d24, h1.d24), sc);                                // d * sc * 2^24, exact
        n = fmul2(pk2(h0.ndmin, h1.ndmin), m);                             // -(dmin * m), exact
    }
    float a0, a1, n0, n1;
    unpk2(a, a0, a1);
    unpk2(n, n0, n1);
    al0 = pk2(a0, a0);
    be0 = pk2(n0, n0);
    al1 = pk2(a1, a1);
    be1 = pk2(n1, n1);
}

// One step (one superblock of rows g and g + 8, at r0 and r1 in the stage)
// of a K-quant: for each group of NSB sub-blocks, the SX MMA(s), the value
// MMAs, and acc += alpha * D + beta * SX for the lane's two D columns of each
// row.  xa, xb, xg: the step's X values of the lane's value-B pairs and of
// its column, or the zero page.
template <int TYPE, int NSB, int MIS>
__device__ __forceinline__ void step_codes(const uint8_t *r0, const uint8_t *r1, uint32_t sh, const LaneMap<NSB> &L,
                                           const uint16_t *xa, const uint16_t *xb, const uint16_t *xg,
                                           pair_t (&acc)[2]) {
    using Q = typename CodesOf<TYPE, NSB, MIS>::T;
    constexpr int SBV = Q::SBV, GROUPS = Q::NSUB / NSB, MMAS = NSB * SBV / 16;
    const RowHead<TYPE> h0(r0), h1(r1);
#pragma unroll
    for (int gm = 0; gm < GROUPS; ++gm) {
        const int xo = SBV * (gm * NSB + L.jg);        // column g's sub-block in the step's X
        // two accumulators for the value MMAs (alternating), so that their
        // dependency chain is half as long
        float D[4] = {0.0f, 0.0f, 0.0f, 0.0f}, E[4] = {0.0f, 0.0f, 0.0f, 0.0f}, S[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int hh = 0; hh < SBV / 16; ++hh) {
            // A is all ones, so any K order that covers the sub-block's 16
            // values once does: lane c takes values 4c .. 4c + 3 in one load
            // (at NSB = 1 the same load as its value MMA's)
            const uint2 v = ldx64(xg + xo + 16 * hh + 4 * L.c);
            mma_acc(S, kOnesH2, kOnesH2, kOnesH2, kOnesH2, v.x, v.y);
        }
        Q q0, q1;
        load_codes<TYPE, NSB, MIS>(q0, r0, sh, gm, L.c);
        load_codes<TYPE, NSB, MIS>(q1, r1, sh, gm, L.c);
        XWords<NSB> xw;
#pragma unroll
        for (int i = 0; i < MMAS; ++i) {
            uint32_t b0, b1;
            xw.get(xa + xo, xb + xo, i, L.c, b0, b1);
            mma_acc(i % 2 ? E : D, code_pair<TYPE, NSB, MIS>(q0, i, 0, L.c), code_pair<TYPE, NSB, MIS>(q1, i, 0, L.c),
                    code_pair<TYPE, NSB, MIS>(q0, i, 1, L.c), code_pair<TYPE, NSB, MIS>(q1, i, 1, L.c), b0, b1);
        }
        if constexpr (MMAS > 1) {
#pragma unroll
            for (int k = 0; k < 4; ++k) D[k] += E[k];
        }
        pair_t al0, be0, al1, be1;
        if constexpr (NSB == 1) {
            row_pair_scales<TYPE>(r0, r1, h0, h1, gm, al0, be0, al1, be1);
        } else {
            group_scales<TYPE, NSB>(r0, h0, gm, L, al0, be0);
            group_scales<TYPE, NSB>(r1, h1, gm, L, al1, be1);
        }
        acc[0] = ffma2(al0, pk2(D[0], D[1]), ffma2(be0, pk2(S[0], S[1]), acc[0]));
        acc[1] = ffma2(al1, pk2(D[2], D[3]), ffma2(be1, pk2(S[2], S[3]), acc[1]));
    }
}

constexpr int ROWS = 16;                      // weight rows per block (the MMA's M)
constexpr int STEP_VALUES = 256;              // values of a row per step (8 runs)
constexpr int NC = 8;                         // consumer warps per CTA
constexpr int GEMV_THREADS = (NC + 1) * 32;   // + the producer warp

// A step's bytes per row (STEP), steps per tile (S), the staged row pitch
// (PITCH: the TMA box width, an odd multiple of 16 bytes at least the
// 16-byte aligned cover of S steps wherever they start, so that 16-byte
// loads of the rows of a load phase hit different bank groups) and the ring
// depth NST (tiles, 80-95 KB in all: two CTAs share an SM).
template <int TYPE> struct Stage;
template <> struct Stage<kQ4_K> { static constexpr int STEP = 144, S = 8, PITCH = 1168, NST = 5; };
template <> struct Stage<kQ5_K> { static constexpr int STEP = 176, S = 8, PITCH = 1424, NST = 4; };
template <> struct Stage<kQ2_K> { static constexpr int STEP = 84, S = 16, PITCH = 1360, NST = 4; };
template <> struct Stage<kQ6_K> { static constexpr int STEP = 210, S = 8, PITCH = 1712, NST = 3; };
template <> struct Stage<kQ8_0> { static constexpr int STEP = 272, S = 4, PITCH = 1104, NST = 5; };
template <> struct Stage<kF16> { static constexpr int STEP = 512, S = 2, PITCH = 1040, NST = 5; };

template <int TYPE> __host__ __device__ constexpr int tile_bytes() { return ROWS * Stage<TYPE>::PITCH; }
template <int TYPE> __host__ __device__ constexpr int gemv_smem() { return Stage<TYPE>::NST * tile_bytes<TYPE>(); }

// A launch runs up to kMaxGroup projections of one type over the same T
// token rows.  Their 16-row blocks are numbered projection after projection;
// CTA b takes blocks b, b + gridDim.x, ...  A block's sums do not depend on
// which CTA computes it or what shares the launch.
struct GemvGroup {
    const uint8_t *W;
    const uint16_t *X;
    float *Y;
    int64_t row_bytes;
    int out_f, in_f, blk_end;      // blk_end: one past the projection's last block
    int use_tma;                   // tmW describes W (its row pitch is a multiple of 16 bytes)
};
struct GemvParams {
    CUtensorMap tmW[kMaxGroup];    // W as [out_f rows x row_bytes / 8] 64-bit words, box PITCH / 8 x 16
    GemvGroup g[kMaxGroup];
    int n, T;
    uint32_t *err;
    uint64_t limit_ns;
    int inject_stall;              // test hook: each CTA's producer arms ring tile n but leaves its copy out
};

// Block b of the launch: its projection, first weight row, steps per row
// and tiles.  A CTA's blocks only increase, so the projection search starts
// at the previous block's (k).
struct BlockLoc {
    int grp, m0, nsteps, ntiles;
};

template <int TYPE>
__device__ __forceinline__ BlockLoc block_loc(const GemvParams &gp, int b, int &k) {
    while (k < gp.n - 1 && b >= gp.g[k].blk_end) ++k;
    const int nsteps = (gp.g[k].in_f + STEP_VALUES - 1) / STEP_VALUES;
    return {k, (b - (k ? gp.g[k - 1].blk_end : 0)) * ROWS, nsteps, (nsteps + Stage<TYPE>::S - 1) / Stage<TYPE>::S};
}

template <int TYPE> constexpr bool kIsKQuant = TYPE == kQ2_K || TYPE == kQ4_K || TYPE == kQ5_K || TYPE == kQ6_K;

// NSB: sub-blocks per K-quant MMA (8 / T rounded up to a power of two); 1
// for Q8_0 and F16, whose columns are the token rows.
template <int TYPE, int NSB>
__global__ void __launch_bounds__(GEMV_THREADS, 2) gemv_kernel(const __grid_constant__ GemvParams gp) {
    using G = Geom<TYPE>;
    using S = Stage<TYPE>;
    using Raw = typename RawOf<TYPE>::T;
    constexpr int TILE = tile_bytes<TYPE>();
    // S < NC: teams of S warps take whole tiles in turn; S >= NC: every warp
    // takes S / NC steps of every tile
    constexpr int TEAMS = S::S >= NC ? 1 : NC / S::S;     // tiles in work at once
    constexpr int SPW = S::S >= NC ? S::S / NC : 1;       // steps per warp and tile
    static_assert(S::S >= NC ? S::S % NC == 0 : NC % S::S == 0, "steps per tile");
    extern __shared__ __align__(128) uint8_t ring[];
    // Block end.  K-quants with NSB >= 2: no barrier; each warp publishes its
    // partial tile and counts itself in, and the warp that completes a
    // block's count sums the eight tiles.  NBUF = NST + 1 buffers: a warp
    // reaches block B only once every warp has released the first tile of
    // block B - NBUF + 1 (B's first tile reuses the slot of a tile NST
    // earlier, and every block has at least one tile), that is, once every
    // warp, the summing one included, is done with block B - NBUF.  Else
    // (Q8_0, F16, and K-quants at NSB = 1, whose tiles would not fit beside
    // the ring): one named barrier per block over two buffers.
    constexpr bool LAST_SUMS = kIsKQuant<TYPE> && NSB >= 2;
    constexpr int NBUF = LAST_SUMS ? S::NST + 1 : 2;
    __shared__ float part[NBUF][NC][ROWS][8 / NSB];       // each consumer warp's 16 weight rows x tokens
    __shared__ uint32_t arrivals[NBUF];                   // warps counted in, over every use of the buffer
    __shared__ __align__(8) uint64_t full[S::NST], empty[S::NST];
    __shared__ uint32_t stop_word, drain_failed;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Stop stop{&stop_word, 0u};
    if (threadIdx.x == 0) {
        for (int s = 0; s < S::NST; ++s) {
            mbar_init(&full[s], 1);                       // the producer's arrive + the bytes
            mbar_init(&empty[s], NC);                     // every consumer warp, whichever team reads it
        }
        stop_word = 0u;
        drain_failed = 0u;
        for (int k = 0; k < NBUF; ++k) arrivals[k] = 0u;
        for (int k = 0; k < gp.n; ++k)
            if (gp.g[k].use_tma) prefetch_tensormap(&gp.tmW[k]);
        mbar_fence_init();
    }
    __syncthreads();
    grid_launch_dependents();                             // the next grid may launch; it still waits for this one
    const int nblk = gp.g[gp.n - 1].blk_end;

    if (warp == NC) {
        // ------------------------------------------------------------ producer --
        // Block-quantized weights are streamed before the previous grid has
        // finished (no kernel of this library writes them): the first NST
        // tiles, whose slots are free, fill the ring while it drains.  The
        // producer waits for that grid before its first wait on a slot, which
        // needs consumers past their own dependency wait, so the time limit
        // never runs while the previous grid does.  F16 weights may be such a
        // kernel's output: their producer waits first.
        // The first NST tiles go out one at a time, each once the one before
        // it has landed (a wait on copies only, so it too ends while the
        // previous grid runs): every CTA's first tile then reaches the SM
        // without the rest of all CTAs' prefill in the DRAM queues beside it,
        // and the consumers start sooner.  Past the prefill, tiles go out as
        // slots free up, several in flight.
        if constexpr (TYPE == kF16) grid_dependency_wait();
        // The CTA's tiles in order: block after block, each block's tiles
        // 0 .. ntiles - 1; tile n goes to slot n % NST.
        int n = 0, kp = 0;
        bool ok = true;
        for (int b = blockIdx.x; ok && b < nblk; b += gridDim.x) {
            const BlockLoc L = block_loc<TYPE>(gp, b, kp);
            const GemvGroup &P = gp.g[L.grp];
            for (int j = 0; j < L.ntiles; ++j, ++n) {
                const int s = n % S::NST;
                if (TYPE != kF16 && n == S::NST) grid_dependency_wait();
                if (n > 0 && n < S::NST &&
                    !wait_phase_warp(&full[n - 1], 0u, gp.limit_ns, stop, gp.err, kErrTimeoutGemv)) {
                    ok = false;
                    break;
                }
                if (!wait_phase_warp(&empty[s], ((n / S::NST) & 1) ^ 1u, gp.limit_ns, stop, gp.err,
                                     kErrTimeoutGemv)) {
                    ok = false;
                    break;
                }
                uint8_t *const slot = ring + s * TILE;
                const int64_t off = static_cast<int64_t>(j) * S::S * S::STEP;   // the tile's first byte in a row
                const bool drop = n == gp.inject_stall;   // test hook: the tile's copy left out
                if (P.use_tma) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[s], TILE);
                        if (!drop)
                            tma_load_2d(slot, &gp.tmW[L.grp], &full[s],
                                        static_cast<int32_t>((off & ~int64_t(15)) >> 3), L.m0);
                    }
                } else if (lane < ROWS) {
                    // row m0 + lane: the 16-byte aligned cover of its S steps
                    uint32_t bytes = 0;
                    const uint8_t *a0 = nullptr;
                    uint8_t *dst = slot + lane * S::PITCH;
                    if (L.m0 + lane < P.out_f) {
                        const uint8_t *row = P.W + static_cast<int64_t>(L.m0 + lane) * P.row_bytes;
                        const uint8_t *start = row + off;
                        const int64_t left = P.row_bytes - off;
                        const uint8_t *end = start + (left < int64_t(S::S) * S::STEP ? left : int64_t(S::S) * S::STEP);
                        const uint8_t *w_end = P.W + static_cast<int64_t>(P.out_f) * P.row_bytes;
                        a0 = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(start) & ~uintptr_t(15));
                        const uint8_t *a1 = reinterpret_cast<const uint8_t *>(
                            (reinterpret_cast<uintptr_t>(end) + 15) & ~uintptr_t(15));
                        if (a1 > w_end) {   // only the last row's last tile: its last bytes by plain loads
                            a1 = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(w_end) & ~uintptr_t(15));
                            if (a1 < a0) a1 = a0;
                            for (const uint8_t *p = a1; p < end; ++p) dst[p - a0] = *p;
                        }
                        bytes = static_cast<uint32_t>(a1 - a0);
                    }
                    const uint32_t total = __reduce_add_sync(0x0000ffffu, bytes);
                    __syncwarp(0x0000ffffu);              // the plain stores above precede the arrive
                    if (lane == 0) mbar_arrive_expect_tx(&full[s], total);
                    if (bytes && !drop) bulk_load(dst, a0, bytes, &full[s]);
                }
                __syncwarp();
            }
        }
        // the copies issued land before the CTA's shared memory goes
        if (lane == 0) {
            bool drained = true;
            for (int m = n - S::NST < 0 ? 0 : n - S::NST; m < n; ++m)
                if (m != gp.inject_stall)                 // a dropped tile has no copy to wait for
                    drained = wait_drain(&full[m % S::NST], static_cast<uint32_t>((m / S::NST) & 1), gp.limit_ns) &&
                              drained;
            if (!drained) {
                drain_failed = 1u;
                atomicOr(gp.err, kErrTimeoutGemv);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers --
        grid_dependency_wait();                           // X, Y: the previous grid's memory operations are done
        const int g = lane >> 2, c = lane & 3;
        const int team = S::S >= NC ? 0 : warp / S::S;    // this warp's team
        const int sl = S::S >= NC ? warp : warp % S::S;   // ... and first step within a tile
        const int T = gp.T;
        const bool tok = g < T;                           // Q8_0, F16: this lane's B column is a token row
        const LaneMap<NSB> lm(g, c);                      // K-quants: the group layout
        const bool pa = lm.j0 == lm.jg && lm.tg < T, pb = lm.j1 == lm.jg && lm.tg < T, pg = lm.tg < T;
        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f}, e[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        pair_t acc[2] = {pk2(0.0f, 0.0f), pk2(0.0f, 0.0f)};
        bool live = true;
        int n0 = 0;                                       // the block's first tile in the CTA's sequence
        int nb = 0;                                       // blocks done (partial-tile buffer nb % 2)
        int kp = 0;                                       // the current block's projection
        for (int b = blockIdx.x; b < nblk; b += gridDim.x) {
            const BlockLoc L = block_loc<TYPE>(gp, b, kp);
            const GemvGroup &P = gp.g[L.grp];
            // rows g, g + 8: the row's start modulo 16 (0 when staged by TMA)
            const int base0 = P.use_tma ? 0
                                        : static_cast<int>((reinterpret_cast<uintptr_t>(P.W) +
                                                            static_cast<uint64_t>(L.m0 + g) * P.row_bytes) & 15);
            const int base1 = P.use_tma ? 0
                                        : static_cast<int>((reinterpret_cast<uintptr_t>(P.W) +
                                                            static_cast<uint64_t>(L.m0 + g + 8) * P.row_bytes) & 15);
            const uint16_t *xrow = P.X + static_cast<int64_t>(tok ? g : 0) * P.in_f;
            const uint16_t *xcol = P.X + static_cast<int64_t>(pg ? lm.tg : 0) * P.in_f;
            for (int j = 0; j < L.ntiles; ++j) {
                // Every consumer warp waits for every tile and releases it, also
                // the tiles another team reads: a warp that skipped ring rounds
                // could meet a slot's barrier two phases on, where a parity wait
                // no longer tells the phases apart.
                const int n = n0 + j, s = n % S::NST;
                live = live && wait_phase_warp(&full[s], static_cast<uint32_t>((n / S::NST) & 1), gp.limit_ns, stop,
                                               gp.err, kErrTimeoutGemv);
                if (!live) continue;
                // this warp's steps of the tile: sl, sl + NC, ...
#pragma unroll
                for (int us = 0; us < SPW; ++us) {
                    const int sq = sl + us * NC;          // step of the tile
                    const int q = j * S::S + sq;          // ... and of the row
                    if (j % TEAMS == team && q < L.nsteps) {
                        const int off = j * S::S * S::STEP;
                        const uint8_t *slot = ring + s * TILE;
                        const uint8_t *src0 = slot + g * S::PITCH + ((base0 + off) & 15) + sq * S::STEP;
                        const uint8_t *src1 = slot + (g + 8) * S::PITCH + ((base1 + off) & 15) + sq * S::STEP;
                        if constexpr (kIsKQuant<TYPE>) {
                            const uint16_t *xs = xcol + 256 * q;
                            const uint16_t *xa = pa ? xs : g_zero_x, *xb = pb ? xs : g_zero_x;
                            const uint16_t *xg = pg ? xs : g_zero_x;
                            if constexpr (TYPE == kQ6_K) {
                                // rows g and g + 8 start alike modulo 4 (8 row pitches apart);
                                // with TMA tiles every row of the step does
                                const uint32_t sh = (smem_u32(src0) & 2u) ? 16u : 0u;
                                if (__all_sync(0xffffffffu, sh != 0u))
                                    step_codes<TYPE, NSB, 1>(src0, src1, sh, lm, xa, xb, xg, acc);
                                else if (!__any_sync(0xffffffffu, sh != 0u))
                                    step_codes<TYPE, NSB, 0>(src0, src1, sh, lm, xa, xb, xg, acc);
                                else
                                    step_codes<TYPE, NSB, 2>(src0, src1, sh, lm, xa, xb, xg, acc);
                            } else {
                                step_codes<TYPE, NSB, 0>(src0, src1, 0u, lm, xa, xb, xg, acc);
                            }
                        } else {
                            const int nruns = (P.in_f + 31) / 32;
                            const bool row0 = L.m0 + g < P.out_f, row1 = L.m0 + g + 8 < P.out_f;
#pragma unroll
                            for (int rho = 0; rho < 2; ++rho) {
                                const int t = 2 * c + rho;        // this lane's run of the step
                                const int jr = 8 * q + t;         // ... and of the row
                                const bool valid = jr < nruns;
                                uint32_t h0[16], h1[16];
                                if (valid && row0) {
                                    Raw raw;
                                    raw.template load<Smem>(src0 + (t / G::RPB) * G::BB, t % G::RPB);
                                    run_f16<TYPE>(raw, t % G::RPB, h0);
                                } else {
#pragma unroll
                                    for (int p = 0; p < 16; ++p) h0[p] = 0u;
                                }
                                if (valid && row1) {
                                    Raw raw;
                                    raw.template load<Smem>(src1 + (t / G::RPB) * G::BB, t % G::RPB);
                                    run_f16<TYPE>(raw, t % G::RPB, h1);
                                } else {
#pragma unroll
                                    for (int p = 0; p < 16; ++p) h1[p] = 0u;
                                }
                                const uint4 *xv = reinterpret_cast<const uint4 *>(xrow + 32 * jr);
                                float (&dr)[4] = rho ? e : d;
#pragma unroll
                                for (int u = 0; u < 4; ++u) {     // 8 values of X per 16-byte load: two MMAs
                                    const uint4 x = tok && valid ? __ldg(xv + u) : make_uint4(0u, 0u, 0u, 0u);
                                    mma_16816(dr, h0[4 * u], h1[4 * u], h0[4 * u + 1], h1[4 * u + 1], x.x, x.y);
                                    mma_16816(dr, h0[4 * u + 2], h1[4 * u + 2], h0[4 * u + 3], h1[4 * u + 3], x.z, x.w);
                                }
                            }
                        }
                    }
                }
                __syncwarp();                             // the tile is read before it is released
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            n0 += L.ntiles;
            // block end: D rows g, g + 8 (weight rows), columns 2c, 2c + 1 (token
            // n / NSB, sub-block n % NSB)
            float v[4];
            if constexpr (kIsKQuant<TYPE>) {
                unpk2(acc[0], v[0], v[1]);
                unpk2(acc[1], v[2], v[3]);
                acc[0] = acc[1] = pk2(0.0f, 0.0f);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[k] = d[k] + e[k];
                    d[k] = e[k] = 0.0f;
                }
            }
            // The sub-block columns of a token are summed in the warp (fixed
            // shuffle order), the warps' tiles through shared memory in warp
            // order.  The tiles are double buffered: a warp writes the next
            // block's tile into the other buffer, and it reaches the block
            // after that only past the next block's barrier, which this
            // block's readers reach after their reads; so one barrier a block.
            const int buf = nb % NBUF;
            float (&pw)[ROWS][8 / NSB] = part[buf][warp];
            if constexpr (NSB == 1) {
                pw[g][2 * c] = v[0];
                pw[g][2 * c + 1] = v[1];
                pw[g + 8][2 * c] = v[2];
                pw[g + 8][2 * c + 1] = v[3];
            } else {
                float y0 = v[0] + v[1], y1 = v[2] + v[3];     // token 2c / NSB, rows g and g + 8
#pragma unroll
                for (int m = 1; m < NSB / 2; m <<= 1) {      // the lanes c of one token
                    y0 += __shfl_xor_sync(0xffffffffu, y0, m);
                    y1 += __shfl_xor_sync(0xffffffffu, y1, m);
                }
                if ((c & (NSB / 2 - 1)) == 0) {
                    pw[g][2 * c / NSB] = y0;
                    pw[g + 8][2 * c / NSB] = y1;
                }
            }
            if constexpr (LAST_SUMS) {
                __syncwarp();                             // the warp's tile stores precede lane 0's release
                uint32_t before = 0u;
                if (lane == 0) {
                    __threadfence_block();
                    before = atomicAdd(&arrivals[buf], 1u);
                    __threadfence_block();
                }
                before = __shfl_sync(0xffffffffu, before, 0);
                __syncwarp();                             // lane 0's acquire precedes the warp's reads
                if (before == static_cast<uint32_t>(NC * (nb / NBUF + 1) - 1)) {
                    for (int o = lane; o < ROWS * (8 / NSB); o += 32) {
                        const int tt = o / ROWS, r = o % ROWS;
                        float y = 0.0f;
#pragma unroll
                        for (int w = 0; w < NC; ++w) y += part[buf][w][r][tt];
                        if (tt < T && L.m0 + r < P.out_f) P.Y[static_cast<int64_t>(tt) * P.out_f + L.m0 + r] = y;
                    }
                }
            } else {
                named_barrier_sync(1, NC * 32);
                for (int o = threadIdx.x; o < ROWS * (8 / NSB); o += NC * 32) {
                    const int tt = o / ROWS, r = o % ROWS;    // consecutive threads: consecutive rows of Y
                    float y = 0.0f;
#pragma unroll
                    for (int w = 0; w < NC; ++w) y += part[buf][w][r][tt];
                    if (tt < T && L.m0 + r < P.out_f) P.Y[static_cast<int64_t>(tt) * P.out_f + L.m0 + r] = y;
                }
            }
            ++nb;
        }
    }
    __syncthreads();
    if (drain_failed) pause_ns(200000ull);
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// W as a 2-D tensor of 64-bit words [out_f rows x row_bytes / 8], box
// pitch / 8 words x 16 rows, no swizzle; reads outside it are zero-filled.
bool encode_w(void *encode_fn, const void *W, int64_t row_bytes, int64_t out_f, int pitch, CUtensorMap *map) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / 8), static_cast<cuuint64_t>(out_f)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(pitch / 8), static_cast<cuuint32_t>(ROWS)};
    const cuuint32_t estr[2] = {1, 1};
    return reinterpret_cast<EncodeFn>(encode_fn)(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(W), dims,
                                                 strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                                 CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Persistent grid: two CTAs per SM, at most one per 16-row block; each CTA's
// ring runs on from one block into its next, across the projections of the
// launch.  Launched with programmatic stream serialization (the kernel waits
// for the previous grid before it reads or writes).
template <int TYPE, int NSB>
cudaError_t launch_nsb(const GemvArgs *a, int n, cudaStream_t stream, const LaunchEnv &env) {
    auto kern = gemv_kernel<TYPE, NSB>;
    constexpr int smem = gemv_smem<TYPE>();
    static std::atomic<int> smem_set[kMaxDevices];        // the opt-in holds per device
    if (!smem_set[env.device].load()) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        smem_set[env.device].store(1);
    }
    GemvParams gp;
    memset(&gp, 0, sizeof(gp));
    int64_t blocks = 0;
    for (int i = 0; i < n; ++i) {
        blocks += (a[i].out_f + ROWS - 1) / ROWS;
        if (blocks > INT32_MAX) return cudaErrorInvalidValue;
        // TMA tiles need a row pitch that is a multiple of 16 bytes (and a
        // 16-byte aligned base, which the C ABI already requires)
        const bool tma = a[i].row_bytes % 16 == 0 && env.encode_fn &&
                         encode_w(env.encode_fn, a[i].W, a[i].row_bytes, a[i].out_f, Stage<TYPE>::PITCH, &gp.tmW[i]);
        gp.g[i] = GemvGroup{static_cast<const uint8_t *>(a[i].W), a[i].X, a[i].Y, a[i].row_bytes,
                            static_cast<int>(a[i].out_f), static_cast<int>(a[i].in_f), static_cast<int>(blocks),
                            tma ? 1 : 0};
    }
    gp.n = n;
    gp.T = static_cast<int>(a[0].T);
    gp.err = env.err;
    gp.limit_ns = env.wait_limit_ns;
    gp.inject_stall = env.inject_stall;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(blocks < 2 * env.num_sms ? blocks : 2 * env.num_sms), 1, 1);
    cfg.blockDim = dim3(GEMV_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, gp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// The K-quants take NSB = 8 / T rounded up to a power of two (8 / NSB token
// columns per MMA); Q8_0 and F16 one column per token.
template <int TYPE>
cudaError_t launch_typed(const GemvArgs *a, int n, cudaStream_t stream, const LaunchEnv &env) {
    if constexpr (kIsKQuant<TYPE>) {
        const int64_t T = a[0].T;
        if (T == 1) return launch_nsb<TYPE, 8>(a, n, stream, env);
        if (T == 2) return launch_nsb<TYPE, 4>(a, n, stream, env);
        if (T <= 4) return launch_nsb<TYPE, 2>(a, n, stream, env);
    }
    return launch_nsb<TYPE, 1>(a, n, stream, env);
}

}  // namespace

cudaError_t launch_decode_gemv(int type, const GemvArgs *a, int n, cudaStream_t stream, const LaunchEnv &env) {
    if (n < 1 || n > kMaxGroup) return cudaErrorInvalidValue;
    switch (type) {
    case kQ8_0: return launch_typed<kQ8_0>(a, n, stream, env);
    case kQ2_K: return launch_typed<kQ2_K>(a, n, stream, env);
    case kQ4_K: return launch_typed<kQ4_K>(a, n, stream, env);
    case kQ5_K: return launch_typed<kQ5_K>(a, n, stream, env);
    case kQ6_K: return launch_typed<kQ6_K>(a, n, stream, env);
    case kF16: return launch_typed<kF16>(a, n, stream, env);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qp
