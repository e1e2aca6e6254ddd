// qp_runs.cuh — decoders of one 32-value run of a block-quantized weight row
// (shared by the standalone dequant kernels and the decode GEMV).
//
// Run t (0..7) of a K-quant superblock is values 32t..32t+31; a Q8_0 block
// is one run.  load() fetches the run's raw bytes (issued one loop step ahead
// of their use by the callers), decode() turns them into 16 f32 pairs with
// the exact one-rounding arithmetic of qp_decode.cuh: bit for bit the value
// formula evaluated with separately rounded f32 operations.  Block fields are
// read straight from global memory with loads no wider than the block's
// alignment (Q4_K and Q5_K blocks are 16-byte aligned, Q2_K 4-byte, Q6_K and
// Q8_0 2-byte; 2-byte aligned runs are assembled from aligned words).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "qp_decode.cuh"
#include "qp_internal.h"

namespace qp {
namespace runs {

// Where a run's bytes are read from: global memory through the read-only
// path (the dequant kernels), or a copy staged in shared memory that keeps
// the bytes' alignment modulo 16 (the decode GEMV).
struct Gmem {
    __device__ __forceinline__ static uint32_t u16(const uint8_t *p) {
        return __ldg(reinterpret_cast<const unsigned short *>(p));
    }
    __device__ __forceinline__ static uint32_t u32(const uint8_t *p) {
        return __ldg(reinterpret_cast<const unsigned int *>(p));
    }
    __device__ __forceinline__ static uint4 u128(const uint8_t *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
};
// Shared-memory loads are issued as ld.shared on the 32-bit shared address:
// the callers' pointers are generic (derived through aligned integer
// arithmetic), and a generic load would take the slower global-memory path.
struct Smem {
    __device__ __forceinline__ static uint32_t a32(const uint8_t *p) {
        return static_cast<uint32_t>(__cvta_generic_to_shared(p));
    }
    __device__ __forceinline__ static uint32_t u16(const uint8_t *p) {
        unsigned short v;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a32(p)));
        return v;
    }
    __device__ __forceinline__ static uint32_t u32(const uint8_t *p) {
        uint32_t v;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a32(p)));
        return v;
    }
    __device__ __forceinline__ static uint4 u128(const uint8_t *p) {
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a32(p)));
        return v;
    }
};

// Raw bytes of one lane's run, loaded one loop step ahead of their decode.
// Two-byte aligned runs (Q6_K, Q8_0) are fetched as aligned words starting
// up to 2 bytes early (never before the block array, which is 16-byte
// aligned) and realigned when decoded; every load stays inside
// [run start - 2, run end).
struct Span32 {
    uint32_t a[9];
    uint32_t sh;                                          // 0 or 16: realignment shift
    template <class M = Gmem>
    __device__ __forceinline__ void load(const uint8_t *p) {
        const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p) & 2u);
        const uint8_t *q = p - mis;
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = M::u32(q + 4 * k);
        a[8] = mis ? M::u16(p + 30) : 0u;
        sh = mis ? 16u : 0u;
    }
    __device__ __forceinline__ uint32_t word(int k) const { return __funnelshift_r(a[k], a[k + 1], sh); }
};

// ---------------------------------------------------------- per-type runs --
// Run t (0..7) of the superblock at b: values 32t..32t+31, decoded to 16 f32
// pairs.

// Q4_K: run t is sub-block t: the low (t even) or high nibbles of
// qs[32(t/2) .. +31]; its 6-bit scale/min are unpacked from the 12 scale
// bytes (t < 4: low 6 bits of bytes t and t+4; t >= 4: nibbles of byte t+4
// plus the top two bits of bytes t-4 and t).
struct RawQ4K {
    uint4 hd, q0, q1;
    template <class M = Gmem>
    __device__ __forceinline__ void load(const uint8_t *b, int t) {
        hd = M::u128(b);    // d, dmin, scales[0..11]
        q0 = M::u128(b + 16 + 32 * (t >> 1));
        q1 = M::u128(b + 32 + 32 * (t >> 1));
    }
    __device__ __forceinline__ void decode(int t, pair_t (&y)[16]) const {
        const int sh = 8 * (t & 3);
        const uint32_t ys = hd.y >> sh, zs = hd.z >> sh, ws = hd.w >> sh;
        const uint32_t sc = t < 4 ? (ys & 63u) : ((ws & 15u) | ((ys >> 6 & 3u) << 4));
        const uint32_t m = t < 4 ? (zs & 63u) : (((ws >> 4) & 15u) | ((zs >> 6 & 3u) << 4));
        const float dl = __fmul_rn(h2f(hd.x), u2f_exact(sc));
        const float nml = -__fmul_rn(h2f(hd.x >> 16), u2f_exact(m));
        const pair_t dl2 = pk2(dl, dl), nml2 = pk2(nml, nml);
        const int nsh = 4 * (t & 1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) affine4((w[k] >> nsh) & 0x0F0F0F0Fu, dl2, nml2, y[2 * k], y[2 * k + 1]);
    }
};

// Q5_K: Q4_K's fields and nibble order, plus a 32-byte plane qh before qs
// holding each value's fifth bit: run t (sub-block t) takes bit t of
// qh[0..31].  q <= 31 still fits the exact byte-to-float step.
struct RawQ5K {
    uint4 hd, h0, h1, q0, q1;
    template <class M = Gmem>
    __device__ __forceinline__ void load(const uint8_t *b, int t) {
        hd = M::u128(b);    // d, dmin, scales[0..11]
        h0 = M::u128(b + 16);
        h1 = M::u128(b + 32);
        q0 = M::u128(b + 48 + 32 * (t >> 1));
        q1 = M::u128(b + 64 + 32 * (t >> 1));
    }
    __device__ __forceinline__ void decode(int t, pair_t (&y)[16]) const {
        const int sh = 8 * (t & 3);
        const uint32_t ys = hd.y >> sh, zs = hd.z >> sh, ws = hd.w >> sh;
        const uint32_t sc = t < 4 ? (ys & 63u) : ((ws & 15u) | ((ys >> 6 & 3u) << 4));
        const uint32_t m = t < 4 ? (zs & 63u) : (((ws >> 4) & 15u) | ((zs >> 6 & 3u) << 4));
        const float dl = __fmul_rn(h2f(hd.x), u2f_exact(sc));
        const float nml = -__fmul_rn(h2f(hd.x >> 16), u2f_exact(m));
        const pair_t dl2 = pk2(dl, dl), nml2 = pk2(nml, nml);
        const int nsh = 4 * (t & 1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint32_t h[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k)
            affine4(((w[k] >> nsh) & 0x0F0F0F0Fu) | (((h[k] >> t) & 0x01010101u) << 4), dl2, nml2, y[2 * k],
                    y[2 * k + 1]);
    }
};

// Q2_K: value 128n + 32j + l takes bits 2j..2j+1 of qs[32n + l]; run t has
// n = t/4, j = t%4, sub-blocks 2t (l < 16) and 2t+1, scale bytes scales[2t],
// scales[2t+1] (sc low nibble, m high nibble).
struct RawQ2K {
    uint32_t w[8], sb, dd;
    template <class M = Gmem>
    __device__ __forceinline__ void load(const uint8_t *b, int t) {
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = M::u32(b + 16 + 32 * (t >> 2) + 4 * k);
        sb = M::u32(b + 4 * (t >> 1));
        dd = M::u32(b + 80);                                // d | dmin << 16
    }
    __device__ __forceinline__ void decode(int t, pair_t (&y)[16]) const {
        const uint32_t sbt = sb >> (16 * (t & 1));         // scales[2t] | scales[2t+1] << 8
        const float d = h2f(dd), dmin = h2f(dd >> 16);
        const int sh = 2 * (t & 3);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint32_t s = (sbt >> (8 * half)) & 0xffu;
            const float dl = __fmul_rn(d, u2f_exact(s & 15u));
            const float nml = -__fmul_rn(dmin, u2f_exact(s >> 4));
            const pair_t dl2 = pk2(dl, dl), nml2 = pk2(nml, nml);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = 4 * half + k;
                affine4((w[i] >> sh) & 0x03030303u, dl2, nml2, y[2 * i], y[2 * i + 1]);
            }
        }
    }
};

// Q6_K: value 128n + 32j + l has low four bits = a nibble (low for j < 2,
// high for j >= 2) of ql[64n + l + 32(j&1)] and high two bits = bits
// 2j..2j+1 of qh[32n + l]; run t has n = t/4, j = t%4, sub-blocks 2t and
// 2t+1 with int8 scales.  y = d*s*(q - 32), an exact product.
struct RawQ6K {
    Span32 ql, qh;
    uint32_t sb, db;
    template <class M = Gmem>
    __device__ __forceinline__ void load(const uint8_t *b, int t) {
        ql.template load<M>(b + 64 * (t >> 2) + 32 * (t & 1));
        qh.template load<M>(b + 128 + 32 * (t >> 2));
        sb = M::u16(b + 192 + 2 * t);                       // two int8 scales
        db = M::u16(b + 208);
    }
    __device__ __forceinline__ void decode(int t, pair_t (&y)[16]) const {
        const int j = t & 3;
        const float d = h2f(db);
        const pair_t nbias2 = pk2(-8388640.0f, -8388640.0f);   // -(2^23 + 32)
        const int nsh = j >= 2 ? 4 : 0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint32_t s = (sb >> (8 * half)) & 0xffu;
            const float dl = __fmul_rn(d, __fsub_rn(u2f_exact(s ^ 0x80u), 128.0f));   // exact int8 value
            const pair_t dl2 = pk2(dl, dl);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = 4 * half + k;
                const uint32_t u =
                    ((ql.word(i) >> nsh) & 0x0F0F0F0Fu) | (((qh.word(i) >> (2 * j)) << 4) & 0x30303030u);
                scaled4(u, dl2, nbias2, y[2 * i], y[2 * i + 1]);
            }
        }
    }
};

// Q8_0: one block = one run of 32 values; q + 128 = byte ^ 0x80.
struct RawQ80 {
    Span32 q;
    uint32_t db;
    template <class M = Gmem>
    __device__ __forceinline__ void load(const uint8_t *b, int) {
        q.template load<M>(b + 2);
        db = M::u16(b);
    }
    __device__ __forceinline__ void decode(int, pair_t (&y)[16]) const {
        const float d = h2f(db);
        const pair_t d2 = pk2(d, d), nbias2 = pk2(-8388736.0f, -8388736.0f);   // -(2^23 + 128)
#pragma unroll
        for (int k = 0; k < 8; ++k) scaled4(q.word(k) ^ 0x80808080u, d2, nbias2, y[2 * k], y[2 * k + 1]);
    }
};

// F16: 32 consecutive fp16 weights (64 bytes, 16-byte aligned), widened
// exactly.  (Used by the decode GEMV, which walks F16 rows 32 values at a
// time; the dequant kernels convert F16 with a flat kernel of their own.)
struct RawF16 {
    uint4 a[4];
    template <class M = Gmem>
    __device__ __forceinline__ void load(const uint8_t *b, int) {
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = M::u128(b + 16 * i);
    }
    __device__ __forceinline__ void decode(int, pair_t (&y)[16]) const {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) y[4 * i + k] = pk2(h2f(w[k]), h2f(w[k] >> 16));
        }
    }
};

template <int TYPE> struct RawOf;
template <> struct RawOf<kQ4_K> { using T = RawQ4K; };
template <> struct RawOf<kQ5_K> { using T = RawQ5K; };
template <> struct RawOf<kQ2_K> { using T = RawQ2K; };
template <> struct RawOf<kQ6_K> { using T = RawQ6K; };
template <> struct RawOf<kQ8_0> { using T = RawQ80; };
template <> struct RawOf<kF16> { using T = RawF16; };

}  // namespace runs
}  // namespace qp
