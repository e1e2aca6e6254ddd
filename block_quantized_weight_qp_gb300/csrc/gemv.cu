// gemv.cu — the decode-side projection over the same weight blocks:
//   Y[t, o] = sum_k X[t, k] * W[o, k]      0 <= t < T <= 8
// for a handful of token rows: the serial path one token at a time ("QK-norm
// models take the FP16 batched prefill when it fits", §What changes: the
// serial prefill is one forward per prompt token) and the decode GEMVs that
// run over the same block types ("Qwen3.5 batched prefill has no f32 dequant
// for IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", §Cause).
//
// Bound by HBM on W: every weight byte is read once.  One warp owns one
// weight row at a time; its lanes walk the row's 32-value runs (lane j takes
// runs j, j + 32, ...) keeping DEPTH runs' raw bytes in flight (a register
// ring, unrolled so it stays in registers), decode them (qp_runs.cuh: the
// exact f32 weights, bit for bit those of qp_dequant_f32), and fold them
// into T dot products with the token rows in f32 (packed f32x2 fma).  The lanes' partial sums are combined by a fixed
// butterfly, so results are deterministic.  X is staged once per CTA in
// shared memory -- as f32 when T * in_f * 4.5 bytes fit in 200 KiB, else as
// f16, widened on use -- with 16 bytes of padding after every 128 bytes, so
// the eight lanes of a 16-byte load phase hit eight different bank groups.
#include <cstdint>
#include <mutex>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qp_decode.cuh"
#include "qp_internal.h"
#include "qp_runs.cuh"

#ifndef QP_GEMV_NW
#define QP_GEMV_NW 4          // warps per CTA while several CTAs share an SM
#endif
#ifndef QP_GEMV_DEPTH
#define QP_GEMV_DEPTH 4       // runs in flight per lane at QP_GEMV_NW warps
#endif
#ifndef QP_GEMV_DEPTH_WIDE
#define QP_GEMV_DEPTH_WIDE 2  // runs in flight per lane at 16 warps
#endif

namespace qp {
namespace {

using namespace runs;


// Bytes per block and 32-value runs per block (F16: a "block" of 32 values).
template <int TYPE> struct Geom;
template <> struct Geom<kQ4_K> { static constexpr int BB = 144, RPB = 8; };
template <> struct Geom<kQ5_K> { static constexpr int BB = 176, RPB = 8; };
template <> struct Geom<kQ2_K> { static constexpr int BB = 84, RPB = 8; };
template <> struct Geom<kQ6_K> { static constexpr int BB = 210, RPB = 8; };
template <> struct Geom<kQ8_0> { static constexpr int BB = 34, RPB = 1; };
template <> struct Geom<kF16> { static constexpr int BB = 64, RPB = 1; };

// Staged X: row t, value k at byte t * pitch + addr(k), where every 128 bytes
// of values are followed by 16 bytes of padding.
template <bool XF32> struct XLayout {
    static constexpr int ESZ = XF32 ? 4 : 2;
    static constexpr int PER128 = 128 / ESZ;          // values per padded 144-byte stretch
    __host__ __device__ static int64_t pitch(int in_f) {
        return static_cast<int64_t>((in_f + PER128 - 1) / PER128) * 144;
    }
    __device__ static uint32_t addr(int k) { return static_cast<uint32_t>((k / PER128) * 144 + (k % PER128) * ESZ); }
};

// NW warps per CTA: 4, so that small projections still spread over all SMs,
// or 16 when the staged X is so large that one CTA fills an SM's shared
// memory.  DEPTH runs in flight per lane: 4, or 2 with 16 warps (whose
// threads have half the registers each).
// TT = the token rows the kernel is compiled for (1, 2, 4 or 8); a call with
// T < TT stages rows T..TT-1 of X as zeros and writes only rows < T.
template <int TYPE, bool XF32, int NW, int TT>
__global__ void __launch_bounds__(NW * 32) gemv_kernel(const uint8_t *__restrict__ W, int64_t row_bytes, int out_f,
                                                         int in_f, const uint16_t *__restrict__ X, int T,
                                                         float *__restrict__ Y) {
    using G = Geom<TYPE>;
    using L = XLayout<XF32>;
    using Raw = typename RawOf<TYPE>::T;
    constexpr int DEPTH = NW >= 16 ? QP_GEMV_DEPTH_WIDE : QP_GEMV_DEPTH;
    extern __shared__ __align__(16) uint8_t xs[];
    const int64_t pitch = L::pitch(in_f);

    // ---- stage X (TT x in_f fp16, in_f % 32 == 0; rows >= T zero): 8 values per thread and step
    const int n8 = TT * in_f / 8;
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
        const int t = (8 * i) / in_f, k = (8 * i) % in_f;
        const uint4 v = t < T ? __ldg(reinterpret_cast<const uint4 *>(X) + i) : make_uint4(0u, 0u, 0u, 0u);
        uint8_t *dst = xs + t * pitch + L::addr(k);   // 8 values never straddle a pad
        if constexpr (XF32) {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            float4 *d = reinterpret_cast<float4 *>(dst);
            d[0] = make_float4(h2f(w[0]), h2f(w[0] >> 16), h2f(w[1]), h2f(w[1] >> 16));
            d[1] = make_float4(h2f(w[2]), h2f(w[2] >> 16), h2f(w[3]), h2f(w[3] >> 16));
        } else {
            *reinterpret_cast<uint4 *>(dst) = v;
        }
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nruns = in_f / 32;
    for (int r = blockIdx.x * NW + warp; r < out_f; r += gridDim.x * NW) {
        const uint8_t *row = W + static_cast<int64_t>(r) * row_bytes;
        pair_t acc[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[t] = pk2(0.0f, 0.0f);
        Raw ring[DEPTH];
#pragma unroll
        for (int d = 0; d < DEPTH; ++d) {
            const int j = lane + 32 * d;
            if (j < nruns) ring[d].load(row + static_cast<int64_t>(j / G::RPB) * G::BB, j % G::RPB);
        }
        for (int j0 = lane; j0 < nruns; j0 += 32 * DEPTH) {
#pragma unroll
          for (int d = 0; d < DEPTH; ++d) {
            const int j = j0 + 32 * d;
            if (j >= nruns) break;
            pair_t y[16];
            ring[d].decode(j % G::RPB, y);
            const int jn = j + 32 * DEPTH;
            if (jn < nruns) ring[d].load(row + static_cast<int64_t>(jn / G::RPB) * G::BB, jn % G::RPB);
            const uint32_t xa = L::addr(32 * j);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                const uint8_t *xr = xs + t * pitch + xa;
#pragma unroll
                for (int q = 0; q < 8; ++q) {          // 4 values per 16-byte load (f32), 8 (f16)
                    if constexpr (XF32) {
                        const float4 v = *reinterpret_cast<const float4 *>(xr + 16 * q);
                        acc[t] = ffma2(y[2 * q], pk2(v.x, v.y), acc[t]);
                        acc[t] = ffma2(y[2 * q + 1], pk2(v.z, v.w), acc[t]);
                    } else if (q < 4) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(xr + 16 * q);
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            acc[t] = ffma2(y[4 * q + u], pk2(h2f(w[u]), h2f(w[u] >> 16)), acc[t]);
                    }
                }
            }
          }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            float lo, hi;
            unpk2(acc[t], lo, hi);
            float v = lo + hi;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == t && t < T) Y[static_cast<int64_t>(t) * out_f + r] = v;
        }
    }
}

// Resident CTAs per SM of one kernel instantiation at one shared-memory size,
// cached: the decode GEMVs are microsecond kernels, and querying the
// occupancy on every call would cost more host time than the kernel takes.
struct OccCache {
    int smem[8] = {};
    int per_sm[8] = {};
    int n = 0;
};

template <int TYPE, bool XF32, int NW, int TT>
cudaError_t launch_nw(const void *W, int64_t row_bytes, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                      float *Y, cudaStream_t stream, int num_sms, int smem) {
    auto kern = gemv_kernel<TYPE, XF32, NW, TT>;
    static OccCache cache;
    static std::mutex mu;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < cache.n; ++i)
            if (cache.smem[i] == smem) per_sm = cache.per_sm[i];
        if (per_sm == 0) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
            if (e != cudaSuccess) return e;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem) != cudaSuccess ||
                per_sm < 1) {
                cudaGetLastError();
                per_sm = 1;
            }
            const int slot = cache.n < 8 ? cache.n++ : 7;
            cache.smem[slot] = smem;
            cache.per_sm[slot] = per_sm;
        }
    }
    const int64_t want = (out_f + NW - 1) / NW;
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    const int grid = static_cast<int>(want < cap ? want : cap);
    kern<<<grid, NW * 32, smem, stream>>>(static_cast<const uint8_t *>(W), row_bytes, static_cast<int>(out_f),
                                          static_cast<int>(in_f), X, static_cast<int>(T), Y);
    return cudaGetLastError();
}

// Staged X as f32 when it fits in 200 KiB, else as f16; 16 warps a CTA when
// the staging leaves room for one CTA per SM, QP_GEMV_NW otherwise.
template <int TYPE, int TT, bool XF32>
cudaError_t launch_x(const void *W, int64_t row_bytes, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                     float *Y, cudaStream_t stream, int num_sms) {
    const int smem = static_cast<int>(TT * XLayout<XF32>::pitch(static_cast<int>(in_f)));
    if (smem > 116 * 1024)
        return launch_nw<TYPE, XF32, 16, TT>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms, smem);
    return launch_nw<TYPE, XF32, QP_GEMV_NW, TT>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms, smem);
}

template <int TYPE, int TT>
cudaError_t launch_tt(const void *W, int64_t row_bytes, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                      float *Y, cudaStream_t stream, int num_sms) {
    if (TT * XLayout<true>::pitch(static_cast<int>(in_f)) <= 200 * 1024)
        return launch_x<TYPE, TT, true>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    return launch_x<TYPE, TT, false>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
}

template <int TYPE>
cudaError_t launch_t(const void *W, int64_t row_bytes, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                     float *Y, cudaStream_t stream, int num_sms) {
    if (T <= 1) return launch_tt<TYPE, 1>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    if (T <= 2) return launch_tt<TYPE, 2>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    if (T <= 4) return launch_tt<TYPE, 4>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    return launch_tt<TYPE, 8>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
}

}  // namespace

cudaError_t launch_decode_gemv(int type, const void *W, int64_t row_bytes, int64_t out_f, int64_t in_f,
                               const uint16_t *X, int64_t T, float *Y, cudaStream_t stream, int num_sms) {
    switch (type) {
    case kQ8_0: return launch_t<kQ8_0>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    case kQ2_K: return launch_t<kQ2_K>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    case kQ4_K: return launch_t<kQ4_K>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    case kQ5_K: return launch_t<kQ5_K>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    case kQ6_K: return launch_t<kQ6_K>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    case kF16: return launch_t<kF16>(W, row_bytes, out_f, in_f, X, T, Y, stream, num_sms);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qp
