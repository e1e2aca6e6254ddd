// dequant.cu — block-quantized weight -> dense f32 / f16 (the per-type
// dequantize-to-f32 step of "Qwen3.5 batched prefill has no f32 dequant for
// IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", §Cause; the f16 copy built from it).
//
// HBM-bound.  One warp decodes one 256-value group (one K-quant superblock, or
// eight Q8_0 blocks) per iteration of a grid-stride loop; lane l owns values
// 8l..8l+7 of the group, so a warp writes 1 KiB (f32) or 512 B (f16) of one
// output row with two / one 16-byte stores per lane.  Block fields are read
// straight from global memory with loads no wider than the block's alignment
// (Q4_K blocks are 16-byte aligned, Q2_K 4-byte, Q6_K and Q8_0 2-byte).
//
// Arithmetic: every field is widened exactly (fp16 -> f32, small ints ->
// f32) and the value formula is evaluated with explicitly rounded f32
// operations (__fmul_rn / __fsub_rn); this translation unit is also built with
// -fmad=false.  The products d*sc, dmin*m and dl*q are exact for these
// formats, so each value carries exactly one rounding: the same bits as the
// CPU oracle.  The f16 output is cvt.rn (round to nearest even) of that f32.
//
// Tail guard: a lane writes only columns < cols; the padding values of a
// partial last block are decoded but never stored.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qp_internal.h"

namespace qp {
namespace {

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xffffu)));
}

__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned short *>(p));
}

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}

// 8 consecutive bytes starting at a 2-byte aligned address, as two words.
__device__ __forceinline__ void ld_8_from_2aligned(const uint8_t *p, uint32_t &lo, uint32_t &hi) {
    const uint32_t a = ld_u16(p), b = ld_u16(p + 2), c = ld_u16(p + 4), d = ld_u16(p + 6);
    lo = a | (b << 16);
    hi = c | (d << 16);
}

__device__ __forceinline__ uint32_t byte_of(uint32_t lo, uint32_t hi, int i) {
    return ((i < 4 ? lo : hi) >> (8 * (i & 3))) & 0xffu;
}

// Byte k (0..11) of the three scale words of a Q4_K block.
__device__ __forceinline__ uint32_t scale_byte(uint32_t w0, uint32_t w1, uint32_t w2, int k) {
    const uint32_t w = k < 4 ? w0 : (k < 8 ? w1 : w2);
    return (w >> (8 * (k & 3))) & 0xffu;
}

// ---------------------------------------------------------- per-type lanes --
// Each fills y[0..7] with values v0..v0+7 of the group and returns the
// output row and first column they belong to (row < 0: nothing to write).

struct LaneOut {
    int64_t row;
    int64_t col0;
};

// (row, block-in-row) of flat block index g: 32-bit division when the block
// count fits (the host picks), 64-bit otherwise.
template <bool WIDE>
__device__ __forceinline__ void split(int64_t g, int64_t nb, int64_t &row, int64_t &kb) {
    if constexpr (WIDE) {
        row = g / nb;
        kb = g - row * nb;
    } else {
        const uint32_t q = static_cast<uint32_t>(g) / static_cast<uint32_t>(nb);
        row = q;
        kb = static_cast<uint32_t>(g) - q * static_cast<uint32_t>(nb);
    }
}

template <bool WIDE>
__device__ __forceinline__ LaneOut lane_q4_k(const uint8_t *blocks, int64_t group, int64_t nb, int lane,
                                             float (&y)[8]) {
    const uint8_t *b = blocks + group * 144;
    const uint4 h = __ldg(reinterpret_cast<const uint4 *>(b));     // d, dmin, scales[0..11]
    const int s = lane >> 2;                                       // sub-block of 32
    const int g = lane >> 3;                                       // group of 64
    const int l0 = 8 * (lane & 3);
    const bool high = (lane & 7) >= 4;
    const uint2 qv = __ldg(reinterpret_cast<const uint2 *>(b + 16 + 32 * g + l0));
    uint32_t sc, m;
    if (s < 4) {
        sc = scale_byte(h.y, h.z, h.w, s) & 63u;
        m = scale_byte(h.y, h.z, h.w, s + 4) & 63u;
    } else {
        const uint32_t packed = scale_byte(h.y, h.z, h.w, s + 4);
        sc = (packed & 15u) | ((scale_byte(h.y, h.z, h.w, s - 4) >> 6) << 4);
        m = (packed >> 4) | ((scale_byte(h.y, h.z, h.w, s) >> 6) << 4);
    }
    const float d = f16_bits_to_f32(h.x), dmin = f16_bits_to_f32(h.x >> 16);
    const float dl = __fmul_rn(d, static_cast<float>(sc));
    const float ml = __fmul_rn(dmin, static_cast<float>(m));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t q = (byte_of(qv.x, qv.y, i) >> (high ? 4 : 0)) & 15u;
        y[i] = __fsub_rn(__fmul_rn(dl, static_cast<float>(q)), ml);
    }
    int64_t row, kb;
    split<WIDE>(group, nb, row, kb);
    return {row, kb * 256 + 8 * lane};
}

template <bool WIDE>
__device__ __forceinline__ LaneOut lane_q2_k(const uint8_t *blocks, int64_t group, int64_t nb, int lane,
                                             float (&y)[8]) {
    const uint8_t *b = blocks + group * 84;                        // 4-byte aligned
    const int n = lane >> 4, j = (lane & 15) >> 2, l0 = 8 * (lane & 3), s = lane >> 1;
    const uint32_t q0 = ld_u32(b + 16 + 32 * n + l0), q1 = ld_u32(b + 16 + 32 * n + l0 + 4);
    const uint32_t scw = ld_u32(b + 4 * (s >> 2));
    const uint32_t scb = (scw >> (8 * (s & 3))) & 0xffu;
    const uint32_t dd = ld_u32(b + 80);                            // d | dmin << 16
    const float d = f16_bits_to_f32(dd), dmin = f16_bits_to_f32(dd >> 16);
    const float dl = __fmul_rn(d, static_cast<float>(scb & 15u));
    const float ml = __fmul_rn(dmin, static_cast<float>(scb >> 4));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t q = (byte_of(q0, q1, i) >> (2 * j)) & 3u;
        y[i] = __fsub_rn(__fmul_rn(dl, static_cast<float>(q)), ml);
    }
    int64_t row, kb;
    split<WIDE>(group, nb, row, kb);
    return {row, kb * 256 + 8 * lane};
}

template <bool WIDE>
__device__ __forceinline__ LaneOut lane_q6_k(const uint8_t *blocks, int64_t group, int64_t nb, int lane,
                                             float (&y)[8]) {
    const uint8_t *b = blocks + group * 210;                       // 2-byte aligned
    const int n = lane >> 4, j = (lane & 15) >> 2, l0 = 8 * (lane & 3), s = lane >> 1;
    uint32_t l_lo, l_hi, h_lo, h_hi;
    ld_8_from_2aligned(b + 64 * n + l0 + 32 * (j & 1), l_lo, l_hi);
    ld_8_from_2aligned(b + 128 + 32 * n + l0, h_lo, h_hi);
    const int32_t sc = static_cast<int8_t>(__ldg(b + 192 + s));
    const float d = f16_bits_to_f32(ld_u16(b + 208));
    const float dl = __fmul_rn(d, static_cast<float>(sc));
    const int lshift = j < 2 ? 0 : 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = (byte_of(l_lo, l_hi, i) >> lshift) & 15u;
        const uint32_t hi = (byte_of(h_lo, h_hi, i) >> (2 * j)) & 3u;
        const int32_t q = static_cast<int32_t>(lo | (hi << 4)) - 32;
        y[i] = __fmul_rn(dl, static_cast<float>(q));
    }
    int64_t row, kb;
    split<WIDE>(group, nb, row, kb);
    return {row, kb * 256 + 8 * lane};
}

// Q8_0 groups hold eight consecutive blocks of the flat block array; lane l
// takes values 8(l%4)..+7 of block 8*group + l/4.
template <bool WIDE>
__device__ __forceinline__ LaneOut lane_q8_0(const uint8_t *blocks, int64_t group, int64_t nb, int64_t nblocks,
                                             int lane, float (&y)[8]) {
    const int64_t blk = group * 8 + (lane >> 2);
    if (blk >= nblocks) return {-1, 0};
    const uint8_t *b = blocks + blk * 34;                          // 2-byte aligned
    const int v0 = 8 * (lane & 3);
    uint32_t q_lo, q_hi;
    ld_8_from_2aligned(b + 2 + v0, q_lo, q_hi);
    const float d = f16_bits_to_f32(ld_u16(b));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int32_t q = static_cast<int8_t>(byte_of(q_lo, q_hi, i));
        y[i] = __fmul_rn(d, static_cast<float>(q));
    }
    int64_t row, kb;
    split<WIDE>(blk, nb, row, kb);
    return {row, kb * 32 + v0};
}

// ------------------------------------------------------------------ store --

__device__ __forceinline__ void store8(float *out, int64_t cols, LaneOut o, const float (&y)[8]) {
    if (o.row < 0 || o.col0 >= cols) return;
    float *p = out + o.row * cols + o.col0;
    if (o.col0 + 8 <= cols && (cols & 3) == 0) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(y[0], y[1], y[2], y[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(y[4], y[5], y[6], y[7]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (o.col0 + i < cols) p[i] = y[i];
    }
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void store8(uint16_t *out, int64_t cols, LaneOut o, const float (&y)[8]) {
    if (o.row < 0 || o.col0 >= cols) return;
    uint16_t *p = out + o.row * cols + o.col0;
    if (o.col0 + 8 <= cols && (cols & 7) == 0) {
        *reinterpret_cast<uint4 *>(p) =
            make_uint4(pack_h2(y[0], y[1]), pack_h2(y[2], y[3]), pack_h2(y[4], y[5]), pack_h2(y[6], y[7]));
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (o.col0 + i < cols) p[i] = __half_as_ushort(__float2half_rn(y[i]));
    }
}

// ----------------------------------------------------------------- kernel --

template <int TYPE, bool WIDE>
__device__ __forceinline__ LaneOut decode_group(const uint8_t *blocks, int64_t g, int64_t nb, int64_t nblocks,
                                                int lane, float (&y)[8]) {
    if constexpr (TYPE == kQ4_K) return lane_q4_k<WIDE>(blocks, g, nb, lane, y);
    else if constexpr (TYPE == kQ2_K) return lane_q2_k<WIDE>(blocks, g, nb, lane, y);
    else if constexpr (TYPE == kQ6_K) return lane_q6_k<WIDE>(blocks, g, nb, lane, y);
    else return lane_q8_0<WIDE>(blocks, g, nb, nblocks, lane, y);
}

// Grid-stride over groups, two groups per warp per iteration so that the
// loads of both are in flight before either is stored.
template <int TYPE, bool WIDE, typename OutT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ blocks, int64_t rows, int64_t cols,
                                                      int64_t nb, OutT *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t nblocks = rows * nb;
    const int64_t ngroups = TYPE == kQ8_0 ? (nblocks + 7) / 8 : nblocks;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    int64_t g = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (; g + warps < ngroups; g += 2 * warps) {
        float y0[8], y1[8];
        const LaneOut o0 = decode_group<TYPE, WIDE>(blocks, g, nb, nblocks, lane, y0);
        const LaneOut o1 = decode_group<TYPE, WIDE>(blocks, g + warps, nb, nblocks, lane, y1);
        store8(out, cols, o0, y0);
        store8(out, cols, o1, y1);
    }
    if (g < ngroups) {
        float y[8];
        const LaneOut o = decode_group<TYPE, WIDE>(blocks, g, nb, nblocks, lane, y);
        store8(out, cols, o, y);
    }
}

template <int TYPE, typename OutT>
cudaError_t launch(const void *blocks, int64_t rows, int64_t cols, OutT *out, cudaStream_t stream, int num_sms) {
    const int64_t qk = TYPE == kQ8_0 ? 32 : 256;
    const int64_t nb = (cols + qk - 1) / qk;
    const int64_t ngroups = TYPE == kQ8_0 ? (rows * nb + 7) / 8 : rows * nb;
    const int64_t want = (ngroups + 7) / 8;                         // 8 warps per block
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;          // 8 blocks of 256 threads per SM
    const int grid = static_cast<int>(want < cap ? want : cap);
    if (rows * nb + 8 < (int64_t(1) << 32))
        dequant_kernel<TYPE, false, OutT><<<grid, 256, 0, stream>>>(static_cast<const uint8_t *>(blocks), rows, cols,
                                                                    nb, out);
    else
        dequant_kernel<TYPE, true, OutT><<<grid, 256, 0, stream>>>(static_cast<const uint8_t *>(blocks), rows, cols,
                                                                   nb, out);
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
