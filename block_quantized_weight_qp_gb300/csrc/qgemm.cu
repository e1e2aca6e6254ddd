// qgemm.cu — the batched-prefill projection Y[T x out] = X[T x in] * W16^T
// on the sm_103a tensor cores ("QK-norm models take the FP16 batched prefill
// when it fits", §What changes: one GEMM per projection over a prompt chunk;
// "Qwen3.5 batched prefill has no f32 dequant for IQ2_XXS, IQ3_S, IQ3_XXS,
// Q2_K", §Cause: the weights are the per-type dequantized blocks, and the f16
// mode works from an f16 copy of them).
//
// Two modes share one persistent, warp-specialized kernel:
//   FUSED  W is block-quantized.  TMA stages one superblock-wide slice of 128
//          weight rows (raw bytes) into shared memory; four dequant warps
//          decode it row by row into fp16, written straight into the
//          128-byte-swizzled K-major layout the tensor cores read.
//   F16W   W is a dense fp16 weight (the cached mode), staged by TMA.
// Roles (one CTA per SM, tiles 128 weight rows x 256 tokens, K step 64):
//   warp 0      TMA producer (X tiles; quantized slices or fp16 W tiles)
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16,
//               M=128 (weight rows) N=256 (tokens) K=16, fp32 accumulators
//               in TMEM, double buffered (2 x 256 columns)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, fp32 stores of Y
//               (each warp owns the 32 TMEM lanes its warp index selects)
//   warps 6-9   dequant (FUSED only), thread i owns weight row i of the tile
//
// Exactness of the fused decode: every field is widened exactly, the int ->
// float step is the exponent-bias trick (OR the integer into the mantissa of
// 2^23, subtract 2^23), and the value is one fma / mul whose product is exact
// (d*sc*q, d*s*(q-32) and d*q need at most 24 significant bits), so each value
// carries a single f32 rounding; cvt.rn.f16x2 then rounds to fp16.  The fp16
// weights are therefore bitwise those of the standalone f16 dequant, and the
// fused and cached modes give bitwise equal Y.
//
// Every wait on an mbarrier is bounded by a time limit; on expiry the kernel
// latches an error bit in the device error word, makes every role stop,
// lets copies in flight land, frees its TMEM and returns.
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qp_internal.h"
#include "qp_ptx.cuh"

namespace qp {
namespace {

constexpr int BM = 128;                       // weight rows per tile (MMA M)
constexpr int BN = 256;                       // tokens per tile (MMA N)
constexpr int BK = 64;                        // K per pipeline stage (one 128-B swizzle row)
constexpr int SB = 256;                       // K per quantized slice (one superblock)
constexpr int X_STAGE_BYTES = BN * BK * 2;    // 32 KiB
constexpr int W_STAGE_BYTES = BM * BK * 2;    // 16 KiB
constexpr int TMEM_COLS = 2 * BN;             // two fp32 accumulators of 256 columns
constexpr int QSTAGES = 2;                    // quantized slices in flight
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);

// Geometry of one quantized slice: SB_BYTES bytes of one row cover 256
// values; the TMA box (BOX bytes wide, a multiple of 16) starts at the slice
// start rounded down to 16 bytes, so the slice begins REM = start % 16 bytes
// into each smem row.
template <int TYPE> struct QFmt;
template <> struct QFmt<kQ4_K> { static constexpr int SB_BYTES = 144, BOX = 144; };
template <> struct QFmt<kQ2_K> { static constexpr int SB_BYTES = 84, BOX = 96; };
template <> struct QFmt<kQ6_K> { static constexpr int SB_BYTES = 210, BOX = 224; };
template <> struct QFmt<kQ8_0> { static constexpr int SB_BYTES = 272, BOX = 272; };  // 8 blocks
template <> struct QFmt<0> { static constexpr int SB_BYTES = 0, BOX = 0; };            // fp16 weight

template <int TYPE> struct Cfg {
    static constexpr bool FUSED = TYPE != 0;
    static constexpr int STAGES = FUSED ? 3 : 4;
    static constexpr int THREADS = FUSED ? 320 : 192;
    static constexpr int Q_SLOT_BYTES = FUSED ? BM * QFmt<TYPE>::BOX : 0;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_W = OFF_X + STAGES * X_STAGE_BYTES;
    static constexpr int OFF_Q = OFF_W + STAGES * W_STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_Q + (FUSED ? QSTAGES * Q_SLOT_BYTES : 0);
    // barriers: full[S], empty[S], qfull[Q], qempty[Q], accfull[2], accempty[2], done
    static constexpr int NBAR = 2 * STAGES + 2 * QSTAGES + 5;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
    static_assert(OFF_Q % 1024 == 0 && Q_SLOT_BYTES % 16 == 0, "alignment");
};

struct Shared {
    uint64_t *full, *empty, *qfull, *qempty, *accfull, *accempty, *done;
    uint32_t *tmem_base;
    volatile uint32_t *abort_flag;
};

// Bounded wait on a barrier phase.  Returns false (and stops every role of
// this CTA) when the limit passes or another role already gave up.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                           volatile uint32_t *abort_flag, uint32_t *err, uint32_t errbit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort_flag = 1u;
                atomicOr(err, errbit);
                return false;
            }
        }
    }
}

// Warp-uniform form for roles whose every lane reads the guarded data.
__device__ __forceinline__ bool wait_phase_warp(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                                volatile uint32_t *abort_flag, uint32_t *err, uint32_t errbit) {
    const bool ok = wait_phase(bar, parity, limit_ns, abort_flag, err, errbit);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void advance(int &stage, uint32_t &phase, int n) {
    if (++stage == n) {
        stage = 0;
        phase ^= 1u;
    }
}

// --------------------------------------------------------- fused decoding --

// fp16 bits (low half of h) -> f32, exact.
__device__ __forceinline__ float h2f(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xffffu)));
}

// Four small unsigned integers held in the bytes of u (each < 2^8) -> the
// floats 2^23 + byte, exactly: the byte is placed in the low mantissa bits of
// 2^23 (0x4B000000).
__device__ __forceinline__ void bias_floats(uint32_t u, float &f0, float &f1, float &f2, float &f3) {
    f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440));
    f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441));
    f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442));
    f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// y = dl*q - ml for the 8 quant values held in the bytes of (u0, u1), packed
// to 4 x half2.  dl*q is exact, so the fma rounds once.
__device__ __forceinline__ uint4 chunk_affine(uint32_t u0, uint32_t u1, float dl, float ml) {
    float f[8];
    bias_floats(u0, f[0], f[1], f[2], f[3]);
    bias_floats(u1, f[4], f[5], f[6], f[7]);
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fmaf_rn(dl, __fsub_rn(f[i], 8388608.0f), -ml);
    return make_uint4(pack_half2(y[0], y[1]), pack_half2(y[2], y[3]), pack_half2(y[4], y[5]),
                      pack_half2(y[6], y[7]));
}

// y = dl*(byte - off) for the 8 bytes of (u0, u1); the product is exact.
__device__ __forceinline__ uint4 chunk_scaled(uint32_t u0, uint32_t u1, float dl, float bias) {
    float f[8];
    bias_floats(u0, f[0], f[1], f[2], f[3]);
    bias_floats(u1, f[4], f[5], f[6], f[7]);
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(dl, __fsub_rn(f[i], bias));
    return make_uint4(pack_half2(y[0], y[1]), pack_half2(y[2], y[3]), pack_half2(y[4], y[5]),
                      pack_half2(y[6], y[7]));
}

// Store 16-byte chunk c (k = 8c..8c+7) of row `row` into a 128-B swizzled
// K-major tile: physical chunk = c XOR (row mod 8).
__device__ __forceinline__ void st_chunk(uint8_t *tile, int row, int c, uint4 v) {
    *reinterpret_cast<uint4 *>(tile + row * 128 + ((c ^ (row & 7)) << 4)) = v;
}

// Word k (4 bytes at byte offset rem + 4k) of a row whose aligned start is
// `base`; `rem` is even and uniform across the CTA for a given slice.
__device__ __forceinline__ uint32_t ld_word_at(const uint32_t *base, int rem, int k) {
    const int w = (rem >> 2) + k;
    if ((rem & 3) == 0) return base[w];
    return __funnelshift_r(base[w], base[w + 1], 16);
}

// Per-superblock state of one dequant thread (decoded scales).
template <int TYPE> struct SbState;

template <> struct SbState<kQ4_K> {
    float dl[8], ml[8];
    __device__ __forceinline__ void load(const uint8_t *row, int /*rem*/) {
        const uint4 h = *reinterpret_cast<const uint4 *>(row);
        const float d = h2f(h.x), dmin = h2f(h.x >> 16);
        const uint32_t sw[3] = {h.y, h.z, h.w};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            uint32_t sc, m;
            auto byte = [&](int k) { return (sw[k >> 2] >> (8 * (k & 3))) & 0xffu; };
            if (s < 4) {
                sc = byte(s) & 63u;
                m = byte(s + 4) & 63u;
            } else {
                sc = (byte(s + 4) & 15u) | ((byte(s - 4) >> 6) << 4);
                m = (byte(s + 4) >> 4) | ((byte(s) >> 6) << 4);
            }
            dl[s] = __fmul_rn(d, static_cast<float>(sc));
            ml[s] = __fmul_rn(dmin, static_cast<float>(m));
        }
    }
    // Values 64a..64a+63: chunk c < 4 = low nibbles of qs[32a + 8c ..], sub-block 2a;
    // chunk c >= 4 = high nibbles of qs[32a + 8(c-4) ..], sub-block 2a+1.
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *row, int /*rem*/, uint8_t *tile, int r) const {
        const uint4 q0 = *reinterpret_cast<const uint4 *>(row + 16 + 32 * A);
        const uint4 q1 = *reinterpret_cast<const uint4 *>(row + 16 + 32 * A + 16);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            st_chunk(tile, r, c,
                     chunk_affine(w[2 * c] & 0x0F0F0F0Fu, w[2 * c + 1] & 0x0F0F0F0Fu, dl[2 * A], ml[2 * A]));
            st_chunk(tile, r, c + 4,
                     chunk_affine((w[2 * c] >> 4) & 0x0F0F0F0Fu, (w[2 * c + 1] >> 4) & 0x0F0F0F0Fu, dl[2 * A + 1],
                                  ml[2 * A + 1]));
        }
    }
};

template <> struct SbState<kQ2_K> {
    float d, dmin;
    __device__ __forceinline__ void load(const uint8_t *row, int rem) {
        const uint32_t dd = *reinterpret_cast<const uint32_t *>(row + rem + 80);
        d = h2f(dd);
        dmin = h2f(dd >> 16);
    }
    // Values 64a..: q of value 128n + 32j + l is bits 2j..2j+1 of qs[32n + l];
    // sub-block of 16 values s = v/16 with scale byte scales[s] (sc low nibble,
    // m high nibble).  Chunk c: j = 2(a%2) + c/4, l = 8(c%4).., s = 4a + c/2.
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *row, int rem, uint8_t *tile, int r) const {
        const uint32_t *rw = reinterpret_cast<const uint32_t *>(row + rem);
        const uint32_t sw = rw[A];                             // scales[4a .. 4a+3]
        float dl[4], ml[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t b = (sw >> (8 * k)) & 0xffu;
            dl[k] = __fmul_rn(d, static_cast<float>(b & 15u));
            ml[k] = __fmul_rn(dmin, static_cast<float>(b >> 4));
        }
        constexpr int n = A / 2;
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = rw[4 + 8 * n + k];  // qs[32n .. 32n+31]
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int j = 2 * (A % 2) + c / 4;
            const int wl = 2 * (c % 4);
            st_chunk(tile, r, c,
                     chunk_affine((w[wl] >> (2 * j)) & 0x03030303u, (w[wl + 1] >> (2 * j)) & 0x03030303u,
                                  dl[c / 2], ml[c / 2]));
        }
    }
};

template <> struct SbState<kQ6_K> {
    float d;
    __device__ __forceinline__ void load(const uint8_t *row, int rem) {
        const uint32_t *base = reinterpret_cast<const uint32_t *>(row);
        d = h2f(ld_word_at(base, rem, 52));                     // bytes 208..209
    }
    // Value 128n + 32j + l: low 4 bits = nibble (low for j < 2, high for j >= 2)
    // of ql[64n + l + 32(j&1)], high 2 bits = bits 2j..2j+1 of qh[32n + l];
    // sub-block s = v/16 with int8 scale.  Atom a: n = a/2, j = 2(a%2) for
    // chunks 0-3 and 2(a%2)+1 for chunks 4-7.
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *row, int rem, uint8_t *tile, int r) const {
        const uint32_t *base = reinterpret_cast<const uint32_t *>(row);
        constexpr int n = A / 2;
        const uint32_t sw = ld_word_at(base, rem, 48 + A);     // scales[4a .. 4a+3]
        float dl[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            dl[k] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>((sw >> (8 * k)) & 0xffu)));
        uint32_t ql[16], qh[8];
#pragma unroll
        for (int k = 0; k < 16; ++k) ql[k] = ld_word_at(base, rem, 16 * n + k);
#pragma unroll
        for (int k = 0; k < 8; ++k) qh[k] = ld_word_at(base, rem, 32 + 8 * n + k);
        constexpr int nsh = (A % 2) ? 4 : 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int j = 2 * (A % 2) + c / 4;
            const int lw = (c / 4) * 8 + 2 * (c % 4);          // ql word: 32(j&1) + 8(c%4) bytes
            const int hw = 2 * (c % 4);
            const uint32_t u0 = ((ql[lw] >> nsh) & 0x0F0F0F0Fu) | (((qh[hw] >> (2 * j)) & 0x03030303u) << 4);
            const uint32_t u1 =
                ((ql[lw + 1] >> nsh) & 0x0F0F0F0Fu) | (((qh[hw + 1] >> (2 * j)) & 0x03030303u) << 4);
            st_chunk(tile, r, c, chunk_scaled(u0, u1, dl[c / 2], 8388640.0f));  // 2^23 + 32
        }
    }
};

template <> struct SbState<kQ8_0> {
    __device__ __forceinline__ void load(const uint8_t *, int) {}
    // Atom a = blocks 2a and 2a+1 of the eight in the slice: bytes 68a .. 68a+67
    // hold d0, q0[32], d1, q1[32].  q + 128 = byte ^ 0x80.
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *row, int /*rem*/, uint8_t *tile, int r) const {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(row) + 17 * A;
        uint32_t v[17];
#pragma unroll
        for (int k = 0; k < 17; ++k) v[k] = w[k];
        const float d0 = h2f(v[0]), d1 = h2f(v[8] >> 16);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t a0 = __funnelshift_r(v[2 * c], v[2 * c + 1], 16) ^ 0x80808080u;
            const uint32_t a1 = __funnelshift_r(v[2 * c + 1], v[2 * c + 2], 16) ^ 0x80808080u;
            st_chunk(tile, r, c, chunk_scaled(a0, a1, d0, 8388736.0f));          // 2^23 + 128
            st_chunk(tile, r, c + 4,
                     chunk_scaled(v[9 + 2 * c] ^ 0x80808080u, v[10 + 2 * c] ^ 0x80808080u, d1, 8388736.0f));
        }
    }
};

template <> struct SbState<0> {
    __device__ __forceinline__ void load(const uint8_t *, int) {}
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *, int, uint8_t *, int) const {}
};

// ----------------------------------------------------------------- kernel --

template <int TYPE>
__global__ void __launch_bounds__(Cfg<TYPE>::THREADS, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        float *__restrict__ Y, int out_f, int T, int nk, int m_tiles, int num_tiles,
                        uint32_t *err, uint64_t limit_ns, int inject_stall) {
    using C = Cfg<TYPE>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    Shared sh;
    sh.full = bars;
    sh.empty = bars + S;
    sh.qfull = bars + 2 * S;
    sh.qempty = bars + 2 * S + QSTAGES;
    sh.accfull = bars + 2 * S + 2 * QSTAGES;
    sh.accempty = sh.accfull + 2;
    sh.done = sh.accfull + 4;
    sh.tmem_base = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    sh.abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sh.full[s], C::FUSED ? 1 + 4 : 1);  // TMA arrive (+ 4 dequant warps)
            mbar_init(&sh.empty[s], 1);                    // MMA commit
        }
        for (int s = 0; s < QSTAGES; ++s) {
            mbar_init(&sh.qfull[s], 1);
            mbar_init(&sh.qempty[s], 4);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sh.accfull[a], 1);
            mbar_init(&sh.accempty[a], 4);
        }
        mbar_init(sh.done, 1);
        *sh.abort_flag = 0u;
        mbar_fence_init();
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(sh.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sh.tmem_base;

    uint8_t *xs = smem + C::OFF_X;
    uint8_t *ws = smem + C::OFF_W;
    uint8_t *qslots = smem + C::OFF_Q;

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            int stage = 0, qs = 0, loads = 0;
            uint32_t phase = 0, qphase = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                const int m0 = (tile % m_tiles) * BM, n0 = (tile / m_tiles) * BN;
                for (int kb = 0; kb < nk; ++kb) {
                    if constexpr (C::FUSED) {
                        if (!wait_phase(&sh.qempty[qs], qphase ^ 1u, limit_ns, sh.abort_flag, err,
                                        kErrTimeoutProducer))
                            goto producer_done;
                        const int start = kb * QFmt<TYPE>::SB_BYTES;
                        mbar_arrive_expect_tx(&sh.qfull[qs], C::Q_SLOT_BYTES);
                        tma_load_2d(qslots + qs * C::Q_SLOT_BYTES, &tmW, &sh.qfull[qs], (start & ~15) >> 2, m0);
                        advance(qs, qphase, QSTAGES);
                    }
#pragma unroll 1
                    for (int a = 0; a < SB / BK; ++a) {
                        if (!wait_phase(&sh.empty[stage], phase ^ 1u, limit_ns, sh.abort_flag, err,
                                        kErrTimeoutProducer))
                            goto producer_done;
                        const int k0 = kb * SB + a * BK;
                        mbar_arrive_expect_tx(&sh.full[stage],
                                              C::FUSED ? X_STAGE_BYTES : X_STAGE_BYTES + W_STAGE_BYTES);
                        if (loads != inject_stall) {
                            tma_load_2d(xs + stage * X_STAGE_BYTES, &tmX, &sh.full[stage], k0, n0);
                            if constexpr (!C::FUSED)
                                tma_load_2d(ws + stage * W_STAGE_BYTES, &tmW, &sh.full[stage], k0, m0);
                        }
                        ++loads;
                        advance(stage, phase, S);
                    }
                }
            }
        producer_done:;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA --
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                if (!wait_phase(&sh.accempty[acc], acc_phase ^ 1u, limit_ns, sh.abort_flag, err, kErrTimeoutMma))
                    goto mma_done;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < nk; ++kb) {
#pragma unroll 1
                    for (int a = 0; a < SB / BK; ++a) {
                        if (!wait_phase(&sh.full[stage], phase, limit_ns, sh.abort_flag, err, kErrTimeoutMma))
                            goto mma_done;
                        tc_fence_after();
                        const uint64_t adesc = desc_sw128_kmajor(smem_u32(ws + stage * W_STAGE_BYTES));
                        const uint64_t bdesc = desc_sw128_kmajor(smem_u32(xs + stage * X_STAGE_BYTES));
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)  // advance 16 fp16 = 32 B inside the swizzle row
                            mma_f16_ss(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb | a | k) != 0);
                        mma_commit(&sh.empty[stage]);      // frees the stage when these MMAs finish
                        advance(stage, phase, S);
                    }
                }
                mma_commit(&sh.accfull[acc]);              // accumulator ready for the epilogue
                advance(acc, acc_phase, 2);
            }
        mma_done:
            // Everything issued has completed before TMEM is released.
            mma_commit(sh.done);
            wait_phase(sh.done, 0, limit_ns, sh.abort_flag, err, kErrTimeoutMma);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------ epilogue --
        const int quarter = warp & 3;                      // TMEM lanes 32*quarter .. +31
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int m0 = (tile % m_tiles) * BM, n0 = (tile / m_tiles) * BN;
            if (!wait_phase_warp(&sh.accfull[acc], acc_phase, limit_ns, sh.abort_flag, err, kErrTimeoutEpilogue))
                break;
            tc_fence_after();
            const int o = m0 + quarter * 32 + lane;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + c * 32, r);
                tmem_wait_ld();
                const int t0 = n0 + c * 32;
                if (o < out_f) {
                    float *yp = Y + static_cast<int64_t>(t0) * out_f + o;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (t0 + j < T) __stcs(yp + static_cast<int64_t>(j) * out_f, __uint_as_float(r[j]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.accempty[acc]);
            advance(acc, acc_phase, 2);
        }
    } else if constexpr (C::FUSED) {
        // ------------------------------------------------------- dequant --
        const int r = (warp - 6) * 32 + lane;              // weight row within the tile
        int stage = 0, qs = 0;
        uint32_t phase = 0, qphase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            for (int kb = 0; kb < nk; ++kb) {
                if (!wait_phase_warp(&sh.qfull[qs], qphase, limit_ns, sh.abort_flag, err, kErrTimeoutDequant))
                    goto dequant_done;
                const uint8_t *row = qslots + qs * C::Q_SLOT_BYTES + r * QFmt<TYPE>::BOX;
                const int rem = (kb * QFmt<TYPE>::SB_BYTES) & 15;
                SbState<TYPE> st;
                st.load(row, rem);
#define QP_DEQUANT_ATOM(A)                                                                                 \
    {                                                                                                      \
        if (!wait_phase_warp(&sh.empty[stage], phase ^ 1u, limit_ns, sh.abort_flag, err, kErrTimeoutDequant)) \
            goto dequant_done;                                                                             \
        st.template atom<A>(row, rem, ws + stage * W_STAGE_BYTES, r);                                      \
        fence_proxy_async_smem();                                                                          \
        __syncwarp();                                                                                      \
        if (lane == 0) mbar_arrive(&sh.full[stage]);                                                       \
        advance(stage, phase, S);                                                                          \
    }
                QP_DEQUANT_ATOM(0)
                QP_DEQUANT_ATOM(1)
                QP_DEQUANT_ATOM(2)
                QP_DEQUANT_ATOM(3)
#undef QP_DEQUANT_ATOM
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.qempty[qs]);
                advance(qs, qphase, QSTAGES);
            }
        }
    dequant_done:;
    }

    __syncthreads();
    if (*sh.abort_flag) {
        // A role gave up: give TMA copies already issued time to land before
        // this CTA's shared memory is released.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------- host --

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_2d(EncodeFn enc, CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
               uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TYPE>
cudaError_t launch_typed(const GemmArgs &a, EncodeFn enc, cudaStream_t stream) {
    using C = Cfg<TYPE>;
    CUtensorMap tmX, tmW;
    if (!encode_2d(enc, &tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.X, a.in_f, a.T, a.in_f * 2, BK, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if constexpr (C::FUSED) {
        const int64_t row_bytes = (a.in_f / SB) * QFmt<TYPE>::SB_BYTES;
        if (!encode_2d(enc, &tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.W, row_bytes / 4, a.out_f, row_bytes,
                       QFmt<TYPE>::BOX / 4, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        if (!encode_2d(enc, &tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.W, a.in_f, a.out_f, a.in_f * 2, BK, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    const int m_tiles = static_cast<int>((a.out_f + BM - 1) / BM);
    const int n_tiles = static_cast<int>((a.T + BN - 1) / BN);
    const int num_tiles = m_tiles * n_tiles;
    const int grid = num_tiles < a.num_sms ? num_tiles : a.num_sms;
    auto kern = prefill_gemm_kernel<TYPE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tmX, tmW, a.Y, static_cast<int>(a.out_f),
                                                      static_cast<int>(a.T), static_cast<int>(a.in_f / SB),
                                                      m_tiles, num_tiles, a.err, a.wait_limit_ns, a.inject_stall);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_gemm(const GemmArgs &a, void *encode_fn, cudaStream_t stream) {
    const EncodeFn enc = reinterpret_cast<EncodeFn>(encode_fn);
    switch (a.type) {
    case 0: return launch_typed<0>(a, enc, stream);
    case kQ4_K: return launch_typed<kQ4_K>(a, enc, stream);
    case kQ2_K: return launch_typed<kQ2_K>(a, enc, stream);
    case kQ6_K: return launch_typed<kQ6_K>(a, enc, stream);
    case kQ8_0: return launch_typed<kQ8_0>(a, enc, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qp
