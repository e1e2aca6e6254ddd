// dequant.cu — block-quantized weight -> dense f32 / f16 (the per-type
// dequantize-to-f32 step of "Qwen3.5 batched prefill has no f32 dequant for
// IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", §Cause; the f16 copy built from it).
//
// HBM-bound.  One warp decodes one 256-value group (one K-quant superblock, or
// eight Q8_0 blocks) per step of a grid-stride loop, two groups per loop
// iteration so that both groups' loads are in flight together; lane l owns
// values 8l..8l+7 of the group, so a warp writes 1 KiB (f32) or 512 B (f16)
// of one output row with two / one 16-byte stores per lane.  Block fields are
// read straight from global memory with loads no wider than the block's
// alignment (Q4_K blocks are 16-byte aligned, Q2_K 4-byte, Q6_K and Q8_0
// 2-byte; 2-byte aligned runs are assembled from aligned words).  The
// (row, block) position of a warp's group is divided out once and then
// stepped.
//
// Arithmetic (qp_decode.cuh): every field is widened exactly and each value
// is one fma / mul with an exact product, i.e. one f32 rounding — the same
// bits as the value formula evaluated with separately rounded f32 operations
// (the CPU oracle).  f16 output is round-to-nearest-even of that f32.
//
// Tail guard: a lane writes only columns < cols; the padding values of a
// partial last block are decoded but never stored.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qp_decode.cuh"
#include "qp_internal.h"

namespace qp {
namespace {

__device__ __forceinline__ uint32_t ldg16(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned short *>(p));
}

__device__ __forceinline__ uint32_t ldg32(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}

// 8 bytes starting at a 2-byte aligned address, as two little-endian words;
// every load stays inside those 8 bytes or the 2 bytes just before them.
__device__ __forceinline__ void ld8_a2(const uint8_t *p, uint32_t &lo, uint32_t &hi) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if ((a & 2u) == 0) {
        lo = ldg32(p);
        hi = ldg32(p + 4);
    } else {
        const uint32_t w0 = ldg32(p - 2), w1 = ldg32(p + 2), t = ldg16(p + 6);
        lo = __funnelshift_r(w0, w1, 16);
        hi = __funnelshift_r(w1, t, 16);
    }
}

// ---------------------------------------------------------- per-type lanes --
// Values 8l..8l+7 of the group whose first (or only) block starts at b, as
// four f32 pairs.

// Q4_K: sub-block s = l/4; the lane's 8 quants are the low (l%8 < 4) or high
// nibbles of qs[32(l/8) + 8(l%4) ..]; 6-bit scale/min of s unpacked from the
// 12 scale bytes (s < 4: low 6 bits of bytes s and s+4; s >= 4: nibbles of
// byte s+4 plus the top two bits of bytes s-4 and s).
__device__ __forceinline__ void lane_q4_k(const uint8_t *b, int lane, pair_t (&y)[4]) {
    const uint4 hd = __ldg(reinterpret_cast<const uint4 *>(b));   // d, dmin, scales[0..11]
    const uint2 q = __ldg(reinterpret_cast<const uint2 *>(b + 16 + 32 * (lane >> 3) + 8 * (lane & 3)));
    const int s = lane >> 2;
    const int sh = 8 * (s & 3);
    const uint32_t ys = hd.y >> sh, zs = hd.z >> sh, ws = hd.w >> sh;
    const uint32_t sc = s < 4 ? (ys & 63u) : ((ws & 15u) | ((ys >> 6 & 3u) << 4));
    const uint32_t m = s < 4 ? (zs & 63u) : (((ws >> 4) & 15u) | ((zs >> 6 & 3u) << 4));
    const float dl = __fmul_rn(h2f(hd.x), u2f_exact(sc));
    const float nml = -__fmul_rn(h2f(hd.x >> 16), u2f_exact(m));
    const pair_t dl2 = pk2(dl, dl), nml2 = pk2(nml, nml);
    const int nsh = (lane & 4) ? 4 : 0;
    affine4((q.x >> nsh) & 0x0F0F0F0Fu, dl2, nml2, y[0], y[1]);
    affine4((q.y >> nsh) & 0x0F0F0F0Fu, dl2, nml2, y[2], y[3]);
}

// Q2_K: value 128n + 32j + l' takes bits 2j..2j+1 of qs[32n + l']; lane l has
// n = l/16, j = (l/4)%4, l' = 8(l%4).., sub-block s = l/2 with scale byte
// scales[s] (sc low nibble, m high nibble).
__device__ __forceinline__ void lane_q2_k(const uint8_t *b, int lane, pair_t (&y)[4]) {
    const int n = lane >> 4, j = (lane >> 2) & 3, s = lane >> 1;
    const uint32_t q0 = ldg32(b + 16 + 32 * n + 8 * (lane & 3));
    const uint32_t q1 = ldg32(b + 20 + 32 * n + 8 * (lane & 3));
    const uint32_t scb = (ldg32(b + 4 * (s >> 2)) >> (8 * (s & 3))) & 0xffu;
    const uint32_t dd = ldg32(b + 80);                                // d | dmin << 16
    const float dl = __fmul_rn(h2f(dd), u2f_exact(scb & 15u));
    const float nml = -__fmul_rn(h2f(dd >> 16), u2f_exact(scb >> 4));
    const pair_t dl2 = pk2(dl, dl), nml2 = pk2(nml, nml);
    affine4((q0 >> (2 * j)) & 0x03030303u, dl2, nml2, y[0], y[1]);
    affine4((q1 >> (2 * j)) & 0x03030303u, dl2, nml2, y[2], y[3]);
}

// Q6_K: value 128n + 32j + l' has low four bits = a nibble (low for j < 2,
// high for j >= 2) of ql[64n + l' + 32(j&1)] and high two bits = bits
// 2j..2j+1 of qh[32n + l']; sub-block s = l/2 has an int8 scale.
__device__ __forceinline__ void lane_q6_k(const uint8_t *b, int lane, pair_t (&y)[4]) {
    const int n = lane >> 4, j = (lane >> 2) & 3, l0 = 8 * (lane & 3), s = lane >> 1;
    uint32_t l_lo, l_hi, h_lo, h_hi;
    ld8_a2(b + 64 * n + l0 + 32 * (j & 1), l_lo, l_hi);
    ld8_a2(b + 128 + 32 * n + l0, h_lo, h_hi);
    const uint32_t sb = __ldg(b + 192 + s);                              // int8 scale, as a byte
    const float sf = __fsub_rn(u2f_exact(sb ^ 0x80u), 128.0f);           // exact int8 value
    const float dl = __fmul_rn(h2f(ldg16(b + 208)), sf);
    const pair_t dl2 = pk2(dl, dl), nbias2 = pk2(-8388640.0f, -8388640.0f);   // -(2^23 + 32)
    const int nsh = j >= 2 ? 4 : 0;
    const uint32_t u0 = ((l_lo >> nsh) & 0x0F0F0F0Fu) | (((h_lo >> (2 * j)) << 4) & 0x30303030u);
    const uint32_t u1 = ((l_hi >> nsh) & 0x0F0F0F0Fu) | (((h_hi >> (2 * j)) << 4) & 0x30303030u);
    scaled4(u0, dl2, nbias2, y[0], y[1]);
    scaled4(u1, dl2, nbias2, y[2], y[3]);
}

// Q8_0: lane l takes values 8(l%4)..+7 of the block at b; q + 128 = byte ^ 0x80.
__device__ __forceinline__ void lane_q8_0(const uint8_t *b, int lane, pair_t (&y)[4]) {
    uint32_t q0, q1;
    ld8_a2(b + 2 + 8 * (lane & 3), q0, q1);
    const float d = h2f(ldg16(b));
    const pair_t d2 = pk2(d, d), nbias2 = pk2(-8388736.0f, -8388736.0f);     // -(2^23 + 128)
    scaled4(q0 ^ 0x80808080u, d2, nbias2, y[0], y[1]);
    scaled4(q1 ^ 0x80808080u, d2, nbias2, y[2], y[3]);
}

// ------------------------------------------------------------------ store --

__device__ __forceinline__ void store8(float *out, int64_t cols, int64_t row, int64_t col0, const pair_t (&y)[4]) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpk2(y[i], v[2 * i], v[2 * i + 1]);
    float *p = out + row * cols + col0;
    if (col0 + 8 <= cols && (cols & 3) == 0) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (col0 + i < cols) p[i] = v[i];
    }
}

__device__ __forceinline__ void store8(uint16_t *out, int64_t cols, int64_t row, int64_t col0,
                                       const pair_t (&y)[4]) {
    uint16_t *p = out + row * cols + col0;
    const uint32_t h0 = f2h2(y[0]), h1 = f2h2(y[1]), h2 = f2h2(y[2]), h3 = f2h2(y[3]);
    if (col0 + 8 <= cols && (cols & 7) == 0) {
        __stcs(reinterpret_cast<uint4 *>(p), make_uint4(h0, h1, h2, h3));
    } else {
        const uint32_t h[4] = {h0, h1, h2, h3};
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (col0 + i < cols) p[i] = static_cast<uint16_t>(h[i >> 1] >> (16 * (i & 1)));
    }
}

// ----------------------------------------------------------------- kernel --

// Position of a lane's values: block index, its (row, block-in-row), stepped
// by a grid stride whose (rows, blocks) split was divided out on the host.
struct Cursor {
    int64_t blk, row, kb;
    __device__ __forceinline__ void step(int64_t dblk, int64_t drow, int64_t dkb, int64_t nb) {
        blk += dblk;
        row += drow;
        kb += dkb;
        if (kb >= nb) {
            kb -= nb;
            ++row;
        }
    }
};

template <int TYPE>
__device__ __forceinline__ void decode_lane(const uint8_t *p, int lane, pair_t (&y)[4]) {
    if constexpr (TYPE == kQ4_K) lane_q4_k(p, lane, y);
    else if constexpr (TYPE == kQ2_K) lane_q2_k(p, lane, y);
    else if constexpr (TYPE == kQ6_K) lane_q6_k(p, lane, y);
    else lane_q8_0(p, lane, y);
}

template <int TYPE, typename OutT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ blocks, int64_t cols, int64_t nb,
                                                      int64_t nblocks, int64_t drow, int64_t dkb,
                                                      OutT *__restrict__ out) {
    constexpr int QK = TYPE == kQ8_0 ? 32 : 256;
    constexpr int BB = TYPE == kQ8_0 ? 34 : (TYPE == kQ4_K ? 144 : (TYPE == kQ2_K ? 84 : 210));
    constexpr int BPG = TYPE == kQ8_0 ? 8 : 1;                // blocks per group
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t g0 = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t dblk = warps * BPG;                         // blocks per grid stride
    // the lane's block: the group's block, or (Q8_0) block l/4 of the group
    Cursor a;
    a.blk = g0 * BPG + (TYPE == kQ8_0 ? (lane >> 2) : 0);
    a.row = a.blk / nb;
    a.kb = a.blk - a.row * nb;
    const int v0 = TYPE == kQ8_0 ? 8 * (lane & 3) : 8 * lane;
    while (__any_sync(0xffffffffu, a.blk < nblocks)) {
        Cursor b = a;
        b.step(dblk, drow, dkb, nb);
        const bool a_ok = a.blk < nblocks, b_ok = b.blk < nblocks;
        pair_t ya[4], yb[4];
        if (a_ok) decode_lane<TYPE>(blocks + a.blk * BB, lane, ya);
        if (b_ok) decode_lane<TYPE>(blocks + b.blk * BB, lane, yb);
        if (a_ok && a.kb * QK + v0 < cols) store8(out, cols, a.row, a.kb * QK + v0, ya);
        if (b_ok && b.kb * QK + v0 < cols) store8(out, cols, b.row, b.kb * QK + v0, yb);
        a = b;
        a.step(dblk, drow, dkb, nb);
    }
}

template <int TYPE, typename OutT>
cudaError_t launch(const void *blocks, int64_t rows, int64_t cols, OutT *out, cudaStream_t stream, int num_sms) {
    const int64_t qk = TYPE == kQ8_0 ? 32 : 256;
    const int64_t nb = (cols + qk - 1) / qk;
    const int64_t nblocks = rows * nb;
    const int64_t ngroups = TYPE == kQ8_0 ? (nblocks + 7) / 8 : nblocks;
    // one resident wave of 256-thread blocks, at least two groups per warp
    static int per_sm = 0;
    if (per_sm == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dequant_kernel<TYPE, OutT>, 256, 0) != cudaSuccess ||
            n < 1)
            n = 1;
        per_sm = n;
    }
    const int64_t want = (ngroups + 15) / 16;
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
    const int64_t dblk = static_cast<int64_t>(grid) * 8 * (TYPE == kQ8_0 ? 8 : 1);
    dequant_kernel<TYPE, OutT><<<grid, 256, 0, stream>>>(static_cast<const uint8_t *>(blocks), cols, nb, nblocks,
                                                         dblk / nb, dblk % nb, out);
    return cudaGetLastError();
}

template <typename OutT>
cudaError_t dispatch(int type, const void *blocks, int64_t rows, int64_t cols, OutT *out, cudaStream_t stream,
                     int num_sms) {
    switch (type) {
    case kQ8_0: return launch<kQ8_0>(blocks, rows, cols, out, stream, num_sms);
    case kQ2_K: return launch<kQ2_K>(blocks, rows, cols, out, stream, num_sms);
    case kQ4_K: return launch<kQ4_K>(blocks, rows, cols, out, stream, num_sms);
    case kQ6_K: return launch<kQ6_K>(blocks, rows, cols, out, stream, num_sms);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_dequant_f32(int type, const void *blocks, int64_t rows, int64_t cols, float *out,
                               cudaStream_t stream, int num_sms) {
    return dispatch(type, blocks, rows, cols, out, stream, num_sms);
}

cudaError_t launch_dequant_f16(int type, const void *blocks, int64_t rows, int64_t cols, uint16_t *out,
                               cudaStream_t stream, int num_sms) {
    return dispatch(type, blocks, rows, cols, out, stream, num_sms);
}

}  // namespace qp
