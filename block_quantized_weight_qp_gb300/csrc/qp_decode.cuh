// qp_decode.cuh — exact per-value arithmetic shared by the dequant kernels
// and the fused GEMM's decode warps.
//
// A quantized field q (a small unsigned integer held in one byte of a 32-bit
// word) becomes the float 2^23 + q by placing the byte in the low mantissa
// bits of 2^23 (0x4B000000) with one byte permute; subtracting 2^23 (or
// 2^23 + offset) is exact.  The weight is then one fma / mul whose product is
// exact for these formats (at most 24 significant bits), so each value is
// rounded once in f32, as the value formula evaluated with separately rounded
// f32 operations would be.  f16 results are round-to-nearest-even of that f32.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace qp {

// fp16 bits (low half of h) -> f32, exact.
__device__ __forceinline__ float h2f(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xffffu)));
}

// A pair of f32 values processed together: packed f32x2 instructions
// (sm_100+) by default, plain scalar f32 operations with QP_SCALAR_PAIRS.
// Either way every operation is an individually rounded IEEE f32 op.
#ifndef QP_SCALAR_PAIRS
using pair_t = uint64_t;

__device__ __forceinline__ pair_t pk2(float lo, float hi) {
    pair_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ pair_t fadd2(pair_t a, pair_t b) {
    pair_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ pair_t fmul2(pair_t a, pair_t b) {
    pair_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ pair_t ffma2(pair_t a, pair_t b, pair_t c) {
    pair_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Round a packed float pair to a packed half pair (round to nearest even).
__device__ __forceinline__ uint32_t f2h2(pair_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}
#else
struct pair_t {
    float x, y;
};

__device__ __forceinline__ pair_t pk2(float lo, float hi) { return {lo, hi}; }
__device__ __forceinline__ pair_t fadd2(pair_t a, pair_t b) { return {__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y)}; }
__device__ __forceinline__ pair_t fmul2(pair_t a, pair_t b) { return {__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y)}; }
__device__ __forceinline__ pair_t ffma2(pair_t a, pair_t b, pair_t c) {
    return {__fmaf_rn(a.x, b.x, c.x), __fmaf_rn(a.y, b.y, c.y)};
}
__device__ __forceinline__ uint32_t f2h2(pair_t v) {
    const __half2 h = __floats2half2_rn(v.x, v.y);
    return *reinterpret_cast<const uint32_t *>(&h);
}
#endif

// Byte i (< 2^8) of u -> the float 2^23 + byte, exactly: the byte becomes the
// low mantissa bits of 2^23 (0x4B000000).
template <int I>
__device__ __forceinline__ float bias_float(uint32_t u) {
    return __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440 + I));
}

// Byte permute with a selector computed at run time.  __byte_perm ignores
// bit 3 of each selector nibble, so for a run-time selector the compiler
// clears those bits first, an extra instruction per permute; the selectors
// used here never set them (nibbles 0..7), so the PTX permute takes them as
// they are.
__device__ __forceinline__ uint32_t prmt_sel(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// hi32(a * b) + c: one integer multiply-add.
__device__ __forceinline__ uint32_t mad_hi(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Unpack a pair into two floats.
#ifndef QP_SCALAR_PAIRS
__device__ __forceinline__ void unpk2(pair_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
#else
__device__ __forceinline__ void unpk2(pair_t v, float &lo, float &hi) {
    lo = v.x;
    hi = v.y;
}
#endif

// Four small integers (the bytes of u) -> four weights, as two f32 pairs.
//   affine: y = fma(dl, byte, -ml)      (dl*byte exact)
//   scaled: y = dl * (byte + nbias)     (nbias = -(2^23 + offset); product exact)
__device__ __forceinline__ void affine4(uint32_t u, pair_t dl2, pair_t nml2, pair_t &y01, pair_t &y23) {
    const pair_t nbias = pk2(-8388608.0f, -8388608.0f);
    const pair_t q01 = fadd2(pk2(bias_float<0>(u), bias_float<1>(u)), nbias);   // exact
    const pair_t q23 = fadd2(pk2(bias_float<2>(u), bias_float<3>(u)), nbias);
    y01 = ffma2(dl2, q01, nml2);
    y23 = ffma2(dl2, q23, nml2);
}

__device__ __forceinline__ void scaled4(uint32_t u, pair_t dl2, pair_t nbias2, pair_t &y01, pair_t &y23) {
    y01 = fmul2(dl2, fadd2(pk2(bias_float<0>(u), bias_float<1>(u)), nbias2));
    y23 = fmul2(dl2, fadd2(pk2(bias_float<2>(u), bias_float<3>(u)), nbias2));
}

// The same, rounded to four fp16 (two half2 words).
__device__ __forceinline__ uint2 word_affine(uint32_t u, pair_t dl2, pair_t nml2) {
    pair_t a, b;
    affine4(u, dl2, nml2, a, b);
    return make_uint2(f2h2(a), f2h2(b));
}

__device__ __forceinline__ uint2 word_scaled(uint32_t u, pair_t dl2, pair_t nbias2) {
    pair_t a, b;
    scaled4(u, dl2, nbias2, a, b);
    return make_uint2(f2h2(a), f2h2(b));
}

// The fp16 value tables of two Q2_K sub-blocks whose scale bytes are the
// low two bytes of sw (scale = low nibble, min = high nibble): entry q of
// sub-block k is RN_f16(fma(d * sc_k, q, -(dmin * m_k))), q = 0..3 -- the
// f32 operations of the value formula, each rounded once, then the fp16
// rounding -- held byte-planar (plo[k]: the low bytes of entries 0..3,
// phi[k]: the high bytes) so that byte permutes select entries.  Both
// sub-blocks go through the same operations on f32 pairs.
__device__ __forceinline__ uint32_t h2_of(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void q2k_tables(uint32_t sw, float d, float dmin, uint32_t (&plo)[2],
                                           uint32_t (&phi)[2]) {
    const pair_t nbias = pk2(-8388608.0f, -8388608.0f);
    const uint32_t scw = sw & 0x0F0Fu, mw = (sw >> 4) & 0x0F0Fu;
    const pair_t sc2 = fadd2(pk2(bias_float<0>(scw), bias_float<1>(scw)), nbias);   // exact
    const pair_t m2 = fadd2(pk2(bias_float<0>(mw), bias_float<1>(mw)), nbias);
    const pair_t dl2 = fmul2(pk2(d, d), sc2);
    const pair_t nml2 = fmul2(pk2(-dmin, -dmin), m2);      // = -(dmin * m): rounding is sign-symmetric
    float x[4], y[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) unpk2(ffma2(dl2, pk2(static_cast<float>(q), static_cast<float>(q)), nml2), x[q], y[q]);
    const uint32_t a01 = h2_of(x[0], x[1]), a23 = h2_of(x[2], x[3]);
    const uint32_t b01 = h2_of(y[0], y[1]), b23 = h2_of(y[2], y[3]);
    plo[0] = __byte_perm(a01, a23, 0x6420);
    phi[0] = __byte_perm(a01, a23, 0x7531);
    plo[1] = __byte_perm(b01, b23, 0x6420);
    phi[1] = __byte_perm(b01, b23, 0x7531);
}

// Small integer (< 2^23) -> float, exactly.
__device__ __forceinline__ float u2f_exact(uint32_t v) {
    return __fsub_rn(__uint_as_float(0x4B000000u | v), 8388608.0f);
}

}  // namespace qp
