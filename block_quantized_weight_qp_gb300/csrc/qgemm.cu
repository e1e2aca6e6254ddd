// qgemm.cu — the batched-prefill projection Y[T x out] = X[T x in] * W16^T
// on the sm_103a tensor cores ("QK-norm models take the FP16 batched prefill
// when it fits", §What changes: one GEMM per projection over a prompt chunk;
// "Qwen3.5 batched prefill has no f32 dequant for IQ2_XXS, IQ3_S, IQ3_XXS,
// Q2_K", §Cause: the weights are the per-type dequantized blocks, and the f16
// mode works from an f16 copy of them).
//
// Two modes:
//   FUSED  W is block-quantized.  TMA stages one superblock-wide slice of 128
//          weight rows (raw bytes) into shared memory; eight dequant warps
//          decode it into fp16, written straight into the 128-byte-swizzled
//          K-major layout the tensor cores read.
//   F16W   W is a dense fp16 weight (the cached mode), staged by TMA.
// Two tilings of each, all persistent and warp-specialized:
//   CTA pairs (default; pair_fused_kernel, pair_gemm_kernel): a cluster of
//          two CTAs on two SMs computes a 256-row x 256-token tile with the
//          paired MMA (tcgen05 cta_group::2, M = 256); each CTA stages (or
//          decodes) its own 128 weight rows and 128 of the tokens, so each
//          SM's shared memory carries half the token operand.  The fused
//          pair kernel's stages hold two 64-value K panels each.
//   one CTA (prefill_gemm_kernel): 128-row x 256-token tiles, M = 128.
// Both run each output through the same K steps and give bitwise equal Y.
// Roles (one-CTA kernel; the pair kernels keep the same warp layout, with
// the MMA issued by the first CTA of the pair; tiles 128 weight rows x 256
// tokens, K step 64):
//   warp 0      TMA producer (X tiles; quantized slices or fp16 W tiles)
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16,
//               M=128 (weight rows) N=256 (tokens) K=16, fp32 accumulators
//               in TMEM, double buffered (2 x 256 columns)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, fp32 stores of Y
//               (each warp owns the 32 TMEM lanes its warp index selects)
//   warps 6-15  dequant (FUSED only; 9 and 13 idle, so no decode work shares
//               the MMA thread's SM sub-partition): unit u = 0..7 decodes
//               weight rows 32(u%4)..+31, values 32(u/4)..+31 of every
//               64-value K step
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
// latches an error bit in the device error word and makes every role stop (in
// a CTA pair, the partner's roles too).  Before shared memory and TMEM are
// released it waits, again with a bound, for what it issued itself: each
// producer for the copies it started, the MMA thread for its MMAs.  Only if
// one of those waits runs out, or where a copy's completion is signalled to
// the other CTA of a pair, does the CTA fall back to a fixed pause.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qp_decode.cuh"
#include "qp_internal.h"
#include "qp_ptx.cuh"
#include "qp_sync.cuh"

namespace qp {
namespace {

constexpr int BM = 128;                       // weight rows per tile (MMA M)
constexpr int BN = 256;                       // tokens per tile (MMA N)
constexpr int BK = 64;                        // K per pipeline stage (one 128-B swizzle row)
constexpr int SB = 256;                       // K per quantized slice (one superblock)
constexpr int X_STAGE_BYTES = BN * BK * 2;    // 32 KiB
constexpr int W_STAGE_BYTES = BM * BK * 2;    // 16 KiB
constexpr int TMEM_COLS = 2 * BN;             // two fp32 accumulators of 256 columns
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);

// Geometry of one quantized slice: SB_BYTES bytes of one row cover 256
// values; the TMA box (BOX bytes wide, an odd multiple of 16 so that 16-byte
// loads from eight consecutive rows never share a bank) starts at the slice
// start rounded down to 16 bytes, so the slice begins REM = start % 16 bytes
// into each smem row.
template <int TYPE> struct QFmt;
template <> struct QFmt<kQ4_K> { static constexpr int SB_BYTES = 144, BOX = 144; };
template <> struct QFmt<kQ5_K> { static constexpr int SB_BYTES = 176, BOX = 176; };
template <> struct QFmt<kQ2_K> { static constexpr int SB_BYTES = 84, BOX = 112; };
template <> struct QFmt<kQ6_K> { static constexpr int SB_BYTES = 210, BOX = 240; };
template <> struct QFmt<kQ8_0> { static constexpr int SB_BYTES = 272, BOX = 272; };  // 8 blocks
template <> struct QFmt<0> { static constexpr int BOX = 0; };                           // fp16 weight

// Pipeline depths.  X tiles (TMA), fp16 W tiles (written by the dequant
// warps in fused mode) and quantized slices (TMA, one superblock = four K
// steps each) have rings of their own, so X can be prefetched deeper than
// the decode runs ahead; the cached mode stages X and W together.
// Shared memory: XST * 32 KiB + WST * 16 KiB + QST slices, <= 227 KiB.
template <int TYPE> struct Depth { static constexpr int XST = 4, WST = 4, QST = 1; };   // Q4_K, Q5_K, Q2_K
template <> struct Depth<kQ6_K> { static constexpr int XST = 4, WST = 3, QST = 1; };
template <> struct Depth<kQ8_0> { static constexpr int XST = 3, WST = 3, QST = 2; };
template <> struct Depth<0> { static constexpr int XST = 4, WST = 4, QST = 0; };

// Decode warps per CTA.  In a CTA that issues MMAs they sit only on SM
// sub-partitions 0, 2 and 3 (warp w runs on sub-partition w % 4):
// sub-partition 1 keeps its issue slots for the single MMA-issuing thread of
// warp 1.  Warps 6..15 minus 9 and 13.
constexpr int kDecodeWarps = 8;

template <int TYPE> struct Cfg {
    static constexpr bool FUSED = TYPE != 0;
    static constexpr int XST = Depth<TYPE>::XST;
    static constexpr int WST = Depth<TYPE>::WST;
    static constexpr int QST = Depth<TYPE>::QST;
    static constexpr int THREADS = FUSED ? 16 * 32 : 6 * 32;
    static constexpr int Q_SLOT_BYTES = FUSED ? BM * QFmt<TYPE>::BOX : 0;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_W = OFF_X + XST * X_STAGE_BYTES;
    static constexpr int OFF_Q = OFF_W + WST * W_STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_Q + QST * Q_SLOT_BYTES;
    // barriers: fullx[XST], emptyx[XST], fullw[WST], emptyw[WST], qfull[Q], qempty[Q],
    //           accfull[2], accempty[2], done
    static constexpr int NBAR = 2 * XST + 2 * WST + 2 * QST + 5;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
    static_assert(OFF_Q % 1024 == 0 && Q_SLOT_BYTES % 16 == 0, "alignment");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
    static_assert(FUSED || XST == WST, "the cached mode stages X and W together");
};

struct Shared {
    uint64_t *fullx, *emptyx, *fullw, *emptyw, *qfull, *qempty, *accfull, *accempty, *done;
    uint32_t *tmem_base;
    Stop stop;
    volatile uint32_t *drain_failed;     // a wait for the CTA's own copies or MMAs ran out
    uint32_t fullw_remote = 0;           // second CTA of a pair: shared::cluster address of the first CTA's fullw
};

// A launch runs up to MAX_GROUPS projections of one weight type over the
// same T tokens ("groups").  Tiles are numbered group after group, in the
// order the host chose (longest K first), weight-row tile fastest within a
// group; CTA b takes tiles b, b + gridDim.x, ...  Every output tile runs the
// same K loop however the tiles are scheduled, so a projection's result does
// not depend on what else shares its launch.
constexpr int MAX_GROUPS = kMaxGroup;
struct GroupParams {
    CUtensorMap tmX[MAX_GROUPS];   // X [T x in] fp16, box 64 x 256, 128-B swizzle
    CUtensorMap tmW[MAX_GROUPS];   // quantized rows (box BOX/4 words x 128 rows) or fp16 W (64 x 128)
    CUtensorMap tmY[MAX_GROUPS];   // Y [T x out] fp32, box 32 x 32 (CTA-pair epilogue stores)
    float *Y[MAX_GROUPS];
    int out_f[MAX_GROUPS];
    int nk[MAX_GROUPS];            // 256-value K slices per weight row (in_f / 256)
    int m_tiles[MAX_GROUPS];       // 128-row weight tiles
    int tile_end[MAX_GROUPS];      // one past the group's last tile
    int n_groups, T, num_tiles;
};

struct TileLoc {
    int g, m0, n0;
};

__device__ __forceinline__ TileLoc locate(const GroupParams &p, int tile) {
    int g = 0, base = 0;
    while (g + 1 < p.n_groups && tile >= p.tile_end[g]) {
        base = p.tile_end[g];
        ++g;
    }
    const int t = tile - base;
    return {g, (t % p.m_tiles[g]) * BM, (t / p.m_tiles[g]) * BN};
}

// --------------------------------------------------------- fused decoding --
//
// Each dequant thread owns one weight row of the tile and one half of every
// 64-value K step ("atom"): half H produces output chunks 4H..4H+3 (values
// 32H..32H+31 of the atom), 8 fp16 values = one 16-byte chunk at a time.
// Quantized bytes are read from the staged slice with 16-byte shared loads
// (row pitches are odd multiples of 16 bytes, so eight consecutive rows hit
// eight different bank groups); misaligned fields are realigned in registers
// with compile-time word offsets (and, for Q6_K, a run-time half-word shift).

// 16-byte shared load through the 32-bit shared address: the staged slices
// are reached through generic pointers derived by integer alignment
// arithmetic, which the compiler would otherwise read with generic loads.
__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// NW consecutive 32-bit words starting at byte OFF (+2 when hs16 == 16) of a
// 16-byte aligned smem row, read with 16-byte loads.  OFF % 4 == 0.
template <int OFF, int NW, bool HALF>
__device__ __forceinline__ void row_words(const uint8_t *row, uint32_t hs16, uint32_t (&w)[NW]) {
    static_assert(OFF % 4 == 0, "word aligned");
    constexpr int LO = OFF & ~15;
    constexpr int HI = (OFF + 4 * NW + (HALF ? 4 : 0) + 15) & ~15;
    constexpr int NC = (HI - LO) / 16;
    uint32_t c[4 * NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const uint4 v = lds128(row + LO + 16 * i);
        c[4 * i] = v.x;
        c[4 * i + 1] = v.y;
        c[4 * i + 2] = v.z;
        c[4 * i + 3] = v.w;
    }
    constexpr int B = (OFF - LO) / 4;
#pragma unroll
    for (int k = 0; k < NW; ++k) {
        if constexpr (HALF) w[k] = __funnelshift_r(c[B + k], c[B + k + 1], hs16);
        else w[k] = c[B + k];
    }
}

// Output chunk addresses of this thread's row and half in a stage's W tile:
// chunk 4h + c (k = 32h + 8c ..) sits at row*128 + (((4h + c) ^ (row & 7)) << 4)
// (128-byte swizzle).
struct ChunkAddr {
    uint32_t off[4];
    __device__ __forceinline__ ChunkAddr(int row, int h) {
#pragma unroll
        for (int c = 0; c < 4; ++c) off[c] = static_cast<uint32_t>(row * 128 + (((4 * h + c) ^ (row & 7)) << 4));
    }
};

// Per-type decoders.  slice(): per-superblock state of this thread's row and
// half h; atom<A>(): writes the thread's four chunks of K step A (values
// 64A + 32h .. 64A + 32h + 31 of the superblock).  WO = (slice start % 16)/4,
// the slice's word offset in the staged row (Q2_K, Q6_K); hs16 = 16 when the
// start is 2 bytes past a word (Q6_K), else 0.
template <int TYPE, int WO> struct Dec;

// Q4_K / Q5_K scales: the 6-bit (sc, m) pairs of sub-blocks 2a + h (a =
// 0..3) from d, dmin and the 12 packed scale bytes (hd = the block's first
// 16 bytes), as dl = d*sc and -ml = -(dmin*m) pairs.
__device__ __forceinline__ void k4_scales(const uint4 &hd, int h, pair_t (&dl2)[4], pair_t (&nml2)[4]) {
    const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        uint32_t sc, m;
        if (a < 2) {                                 // s = 2a + h < 4: bytes s, s + 4
            const int sh = 8 * (2 * a + h);
            sc = (hd.y >> sh) & 63u;
            m = (hd.z >> sh) & 63u;
        } else {                                     // s >= 4, t = s - 4: bytes t + 8, t, t + 4
            const int sh = 8 * (2 * (a - 2) + h);
            const uint32_t lo = hd.w >> sh;
            sc = (lo & 15u) | (((hd.y >> sh) >> 6 & 3u) << 4);
            m = ((lo >> 4) & 15u) | (((hd.z >> sh) >> 6 & 3u) << 4);
        }
        const float dl = __fmul_rn(d, static_cast<float>(sc));
        const float nml = -__fmul_rn(dmin, static_cast<float>(m));
        dl2[a] = pk2(dl, dl);
        nml2[a] = pk2(nml, nml);
    }
}

// Q4_K: sub-block 2A+h holds values 64A+32h..; they are the low (h=0) or
// high (h=1) nibbles of qs[32A .. 32A+31].  The thread keeps its nibbles of
// the whole slice (32 words, one per 4 values) in registers.
template <int WO> struct Dec<kQ4_K, WO> {
    static constexpr bool REGS = true;           // slice() keeps all it needs in registers
    pair_t dl2[4], nml2[4];
    uint32_t qn[32];
    __device__ __forceinline__ void slice(const uint8_t *row, uint32_t, int h) {
        uint32_t w[32];
        row_words<16, 32, false>(row, 0, w);       // qs[0 .. 127]
#pragma unroll
        for (int k = 0; k < 32; ++k) qn[k] = (w[k] >> (4 * h)) & 0x0F0F0F0Fu;
        k4_scales(lds128(row), h, dl2, nml2);
    }
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *, uint32_t, int, uint32_t tile,
                                         const ChunkAddr &ca) const {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint2 lo = word_affine(qn[8 * A + 2 * c], dl2[A], nml2[A]);
            const uint2 hi = word_affine(qn[8 * A + 2 * c + 1], dl2[A], nml2[A]);
            sts128(tile + ca.off[c], lo.x, lo.y, hi.x, hi.y);
        }
    }
};

// Q5_K: Q4_K's sub-blocks, scales and nibbles (qs now at byte 48), plus the
// fifth bit of value 64A + 32h + l in bit 2A + h of qh[l] (bytes 16..47),
// merged into the nibble words once per slice; q <= 31.
template <int WO> struct Dec<kQ5_K, WO> {
    static constexpr bool REGS = true;
    pair_t dl2[4], nml2[4];
    uint32_t qn[32];
    __device__ __forceinline__ void slice(const uint8_t *row, uint32_t, int h) {
        uint32_t qh[8], w[32];
        row_words<16, 8, false>(row, 0, qh);       // qh[0 .. 31]
        row_words<48, 32, false>(row, 0, w);       // qs[0 .. 127]
#pragma unroll
        for (int k = 0; k < 32; ++k)
            qn[k] = ((w[k] >> (4 * h)) & 0x0F0F0F0Fu) | (((qh[k & 7] >> (2 * (k >> 3) + h)) & 0x01010101u) << 4);
        k4_scales(lds128(row), h, dl2, nml2);
    }
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *, uint32_t, int, uint32_t tile,
                                         const ChunkAddr &ca) const {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint2 lo = word_affine(qn[8 * A + 2 * c], dl2[A], nml2[A]);
            const uint2 hi = word_affine(qn[8 * A + 2 * c + 1], dl2[A], nml2[A]);
            sts128(tile + ca.off[c], lo.x, lo.y, hi.x, hi.y);
        }
    }
};

// Q2_K: value 128n + 32j + l takes bits 2j..2j+1 of qs[32n + l]; sub-block
// s = v/16 has scale byte scales[s] (sc low nibble, m high nibble).  A 4-bit
// sc/m pair gives each sub-block only four distinct values, f16(dl*q - ml)
// for q = 0..3: they are computed exactly once per sub-block and then
// selected per value with byte permutes (a lookup stored as a low-byte plane
// and a high-byte plane).  The thread keeps the slice's 64 qs bytes in
// registers: K steps 2n and 2n+1 read the same bytes with different j.
template <int WO> struct Dec<kQ2_K, WO> {
    static constexpr bool REGS = true;           // slice() keeps all it needs in registers
    float d, dmin;
    uint32_t sc[4], qs[16];
    __device__ __forceinline__ void slice(const uint8_t *row, uint32_t, int) {
        uint32_t dd[1];
        row_words<80 + 4 * WO, 1, false>(row, 0, dd);
        d = h2f(dd[0]);
        dmin = h2f(dd[0] >> 16);
        row_words<4 * WO, 4, false>(row, 0, sc);
        row_words<16 + 4 * WO, 16, false>(row, 0, qs);
    }
    // 4 crumb values in the bytes of u -> 2 half2
    __device__ __forceinline__ static uint2 pick(uint32_t u, uint32_t plo, uint32_t phi) {
        // byte q -> nibbles (q, q + 4); the high half's selector (u * 0x11) >> 16
        // + 0x4040 comes from the multiply's high word
        return make_uint2(prmt_sel(plo, phi, u * 0x11u + 0x40404040u), prmt_sel(plo, phi, mad_hi(u, 0x110000u, 0x4040u)));
    }
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *, uint32_t, int h, uint32_t tile,
                                         const ChunkAddr &ca) const {
        constexpr int n = A / 2;
        const int sh = 2 * (2 * (A % 2) + h);            // 2j
        const uint32_t sw = sc[A] >> (16 * h);           // scale bytes of sub-blocks 4A+2h, 4A+2h+1
        uint32_t plo_[2], phi_[2];                       // their value tables
        q2k_tables(sw, d, dmin, plo_, phi_);
#pragma unroll
        for (int half = 0; half < 2; ++half) {           // two sub-blocks of 16 values
            const uint32_t plo = plo_[half], phi = phi_[half];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * half + cc;
                const uint2 lo = pick((qs[8 * n + 2 * c] >> sh) & 0x03030303u, plo, phi);
                const uint2 hi = pick((qs[8 * n + 2 * c + 1] >> sh) & 0x03030303u, plo, phi);
                sts128(tile + ca.off[c], lo.x, lo.y, hi.x, hi.y);
            }
        }
    }
};

// Q6_K: value 128n + 32j + l has low four bits = a nibble (low for j < 2,
// high for j >= 2) of ql[64n + l + 32(j&1)] and high two bits = bits
// 2j..2j+1 of qh[32n + l]; sub-block s = v/16 has an int8 scale.
// y = d*s*(q - 32), an exact product.  Half h of K step A has j = 2(A%2) + h,
// so over a slice the thread reads ql[64n + 32h ..+31] and qh[32n ..+31] for
// n = 0, 1: 32 words, realigned once per slice and kept in registers.
template <int WO> struct Dec<kQ6_K, WO> {
    static constexpr bool REGS = true;
    float d;
    uint32_t sc[4], ql[16], qh[16];
    __device__ __forceinline__ void slice(const uint8_t *row, uint32_t hs16, int h) {
        uint32_t dd[1];
        row_words<208 + 4 * WO, 1, true>(row, hs16, dd);
        d = h2f(dd[0]);
        row_words<192 + 4 * WO, 4, true>(row, hs16, sc);
        uint32_t t[8];
        row_words<4 * WO, 8, true>(row + 32 * h, hs16, t);          // ql[32h ..]
#pragma unroll
        for (int k = 0; k < 8; ++k) ql[k] = t[k];
        row_words<64 + 4 * WO, 8, true>(row + 32 * h, hs16, t);     // ql[64 + 32h ..]
#pragma unroll
        for (int k = 0; k < 8; ++k) ql[8 + k] = t[k];
        row_words<128 + 4 * WO, 16, true>(row, hs16, qh);           // qh[0 .. 63]
        // this half only ever needs crumbs j = h and j = 2 + h of each qh byte:
        // keep them at bits 0..1 and 4..5 and clear the rest, so that each
        // K step merges a word of 6-bit q with one shift and one select
#pragma unroll
        for (int k = 0; k < 16; ++k) qh[k] = (qh[k] >> (2 * h)) & 0x33333333u;
    }
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *, uint32_t, int h, uint32_t tile,
                                         const ChunkAddr &ca) const {
        constexpr int n = A / 2;
        const pair_t nbias2 = pk2(-8388640.0f, -8388640.0f);     // -(2^23 + 32)
        const uint32_t sw = sc[A] >> (16 * h);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int8_t s = static_cast<int8_t>((sw >> (8 * half)) & 0xffu);
            const float dl = __fmul_rn(d, static_cast<float>(s));
            const pair_t dl2 = pk2(dl, dl);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * half + cc;
                uint32_t u[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    // low four bits: the low (j < 2) or high nibble of the ql byte;
                    // bits 4..5: crumb j = 2(A%2) + h of the qh byte (bits 0..1 of the
                    // masked word for A even, bits 4..5 for A odd); bits 6..7 clear
                    const uint32_t qhw = qh[8 * n + 2 * c + k], qlw = ql[8 * n + 2 * c + k];
                    const uint32_t a = (A % 2) ? (qlw >> 4) : qlw;
                    const uint32_t b = (A % 2) ? qhw : (qhw << 4);
                    u[k] = (a & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
                }
                const uint2 lo = word_scaled(u[0], dl2, nbias2);
                const uint2 hi = word_scaled(u[1], dl2, nbias2);
                sts128(tile + ca.off[c], lo.x, lo.y, hi.x, hi.y);
            }
        }
    }
};

// Q8_0: the slice holds eight 34-byte blocks; K step A = blocks 2A (h = 0)
// and 2A+1 (h = 1), i.e. bytes 68A .. 68A+67 = d0, q0[32], d1, q1[32].
// q + 128 = byte XOR 0x80.
template <int WO> struct Dec<kQ8_0, WO> {
    static constexpr bool REGS = false;
    __device__ __forceinline__ void slice(const uint8_t *, uint32_t, int) {}
    template <int A>
    __device__ __forceinline__ void atom(const uint8_t *row, uint32_t, int h, uint32_t tile,
                                         const ChunkAddr &ca) const {
        uint32_t w[17];
        row_words<68 * A, 17, false>(row, 0, w);
        const float dv = h2f(h ? (w[8] >> 16) : w[0]);
        uint32_t q[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = h ? w[k + 9] : __funnelshift_r(w[k], w[k + 1], 16);
        const pair_t d2 = pk2(dv, dv);
        const pair_t nbias2 = pk2(-8388736.0f, -8388736.0f);     // -(2^23 + 128)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint2 lo = word_scaled(q[2 * c] ^ 0x80808080u, d2, nbias2);
            const uint2 hi = word_scaled(q[2 * c + 1] ^ 0x80808080u, d2, nbias2);
            sts128(tile + ca.off[c], lo.x, lo.y, hi.x, hi.y);
        }
    }
};

// One superblock slice of one half-row: four K steps, each waiting for its
// W stage to be free, decoding into it and signalling the MMA.  Decoders
// whose slice() keeps everything the four K steps need in registers (REGS)
// hand the staged slice back to the producer right away, so the next slice's
// copy overlaps these four K steps.
#ifdef QP_NOINLINE_SLICE
#define QP_SLICE_INLINE __noinline__
#else
#define QP_SLICE_INLINE __forceinline__
#endif
// PPS: K panels (64-value K steps) per W16 stage: 1 (single-CTA kernel), or
// 2 (pair kernel: a stage is two 16 KiB panels, one barrier round per
// 128 values of K).
template <int TYPE, int WO, int S, int PPS = 1>
__device__ QP_SLICE_INLINE bool dequant_slice(const Shared &sh, const uint8_t *row, uint32_t hs16, int p,
                                              uint32_t ws_addr, const ChunkAddr &ca, uint64_t *qempty, int lane,
                                              int &stage, uint32_t &phase, uint64_t limit_ns, uint32_t *err) {
    Dec<TYPE, WO> dec;
    dec.slice(row, hs16, p);
    if constexpr (Dec<TYPE, WO>::REGS) {
        __syncwarp();
        if (lane == 0) mbar_arrive(qempty);
    }
    // The atoms go in pairs: both K panels are written, then one proxy fence
    // makes the pair's stores visible to the tensor cores before the arrive
    // (one fence per atom measured 1.2% slower on the Q6_K down projection).
    // With one panel per stage the pair spans two stages, and the second
    // stage's wait needs no arrive of the first: the ring is at least two
    // stages deep.  With two panels per stage the pair is one stage.
#define QP_DEQUANT_STAGE2(A)                                                                                   \
    {                                                                                                          \
        if (!wait_phase_warp(&sh.emptyw[stage], phase ^ 1u, limit_ns, sh.stop, err, kErrTimeoutDequant)) \
            return false;                                                                                      \
        const uint32_t st = ws_addr + static_cast<uint32_t>(stage * 2 * W_STAGE_BYTES);                        \
        dec.template atom<A>(row, hs16, p, st, ca);                                                            \
        dec.template atom<A + 1>(row, hs16, p, st + W_STAGE_BYTES, ca);                                        \
        fence_proxy_async_smem();                                                                              \
        __syncwarp();                                                                                          \
        if (lane == 0) {                                                                                       \
            if (sh.fullw_remote) mbar_arrive_remote(sh.fullw_remote + static_cast<uint32_t>(stage * 8));       \
            else mbar_arrive(&sh.fullw[stage]);                                                                \
        }                                                                                                      \
        advance(stage, phase, S);                                                                              \
    }
#define QP_DEQUANT_PAIR(A)                                                                                     \
    {                                                                                                          \
        const int s0 = stage;                                                                                  \
        if (!wait_phase_warp(&sh.emptyw[stage], phase ^ 1u, limit_ns, sh.stop, err, kErrTimeoutDequant)) \
            return false;                                                                                      \
        dec.template atom<A>(row, hs16, p, ws_addr + static_cast<uint32_t>(stage * W_STAGE_BYTES), ca);         \
        advance(stage, phase, S);                                                                              \
        if (!wait_phase_warp(&sh.emptyw[stage], phase ^ 1u, limit_ns, sh.stop, err, kErrTimeoutDequant)) \
            return false;                                                                                      \
        dec.template atom<A + 1>(row, hs16, p, ws_addr + static_cast<uint32_t>(stage * W_STAGE_BYTES), ca);     \
        fence_proxy_async_smem();                                                                              \
        __syncwarp();                                                                                          \
        if (lane == 0) {                                                                                       \
            if (sh.fullw_remote) {                                                                             \
                mbar_arrive_remote(sh.fullw_remote + static_cast<uint32_t>(s0 * 8));                           \
                mbar_arrive_remote(sh.fullw_remote + static_cast<uint32_t>(stage * 8));                        \
            } else {                                                                                           \
                mbar_arrive(&sh.fullw[s0]);                                                                    \
                mbar_arrive(&sh.fullw[stage]);                                                                 \
            }                                                                                                  \
        }                                                                                                      \
        advance(stage, phase, S);                                                                              \
    }
    if constexpr (PPS == 2) {
        QP_DEQUANT_STAGE2(0)
        QP_DEQUANT_STAGE2(2)
    } else {
        static_assert(PPS == 1 && S >= 2, "a pair of atoms needs two W stages");
        QP_DEQUANT_PAIR(0)
        QP_DEQUANT_PAIR(2)
    }
#undef QP_DEQUANT_PAIR
#undef QP_DEQUANT_STAGE2
    return true;
}

// (first, stride): this CTA's tile sequence.
template <int TYPE, int WST, int QST, int PPS = 1>
__device__ __forceinline__ void dequant_role(const Shared &sh, const GroupParams &gp, int first, int stride,
                                             const uint8_t *qslots, uint32_t ws_addr, int r, int p, int lane,
                                             uint64_t limit_ns, uint32_t *err) {
    constexpr int Q_SLOT_BYTES = BM * QFmt<TYPE>::BOX;
    const ChunkAddr ca(r, p);
    int stage = 0, qs = 0;
    uint32_t phase = 0, qphase = 0;
    for (int tile = first; tile < gp.num_tiles; tile += stride) {
        const int nk = gp.nk[locate(gp, tile).g];
        for (int kb = 0; kb < nk; ++kb) {
            if (!wait_phase_warp(&sh.qfull[qs], qphase, limit_ns, sh.stop, err, kErrTimeoutDequant)) return;
            const uint8_t *row = qslots + qs * Q_SLOT_BYTES + r * QFmt<TYPE>::BOX;
            const int rem = (kb * QFmt<TYPE>::SB_BYTES) & 15;
            const uint32_t hs16 = (rem & 2) ? 16u : 0u;
            bool ok;
            if constexpr (TYPE == kQ2_K || TYPE == kQ6_K) {
                switch (rem >> 2) {
                case 0: ok = dequant_slice<TYPE, 0, WST, PPS>(sh, row, hs16, p, ws_addr, ca, &sh.qempty[qs], lane, stage, phase, limit_ns, err); break;
                case 1: ok = dequant_slice<TYPE, 1, WST, PPS>(sh, row, hs16, p, ws_addr, ca, &sh.qempty[qs], lane, stage, phase, limit_ns, err); break;
                case 2: ok = dequant_slice<TYPE, 2, WST, PPS>(sh, row, hs16, p, ws_addr, ca, &sh.qempty[qs], lane, stage, phase, limit_ns, err); break;
                default: ok = dequant_slice<TYPE, 3, WST, PPS>(sh, row, hs16, p, ws_addr, ca, &sh.qempty[qs], lane, stage, phase, limit_ns, err); break;
                }
            } else {
                ok = dequant_slice<TYPE, 0, WST, PPS>(sh, row, hs16, p, ws_addr, ca, &sh.qempty[qs], lane, stage, phase, limit_ns, err);
            }
            if (!ok) return;
            if constexpr (!Dec<TYPE, 0>::REGS) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.qempty[qs]);
            }
            advance(qs, qphase, QST);
        }
    }
}

// ----------------------------------------------------------------- kernel --

template <int TYPE>
__global__ void __launch_bounds__(Cfg<TYPE>::THREADS, 1)
    prefill_gemm_kernel(const __grid_constant__ GroupParams gp, uint32_t *err, uint64_t limit_ns, int inject_stall) {
    using C = Cfg<TYPE>;
    constexpr int XS = C::XST, WS = C::WST;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    Shared sh;
    sh.fullx = bars;
    sh.emptyx = bars + XS;
    sh.fullw = bars + 2 * XS;
    sh.emptyw = bars + 2 * XS + WS;
    sh.qfull = bars + 2 * XS + 2 * WS;
    sh.qempty = sh.qfull + C::QST;
    sh.accfull = sh.qempty + C::QST;
    sh.accempty = sh.accfull + 2;
    sh.done = sh.accfull + 4;
    sh.tmem_base = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    sh.stop = Stop{reinterpret_cast<volatile uint32_t *>(smem + C::OFF_MISC + 4), 0u};
    sh.drain_failed = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_MISC + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < XS; ++s) {
            mbar_init(&sh.fullx[s], 1);                    // TMA arrive with the byte count
            mbar_init(&sh.emptyx[s], 1);                   // MMA commit
        }
        if constexpr (C::FUSED) {                        // W16 and quantized-slice rings (fused mode only)
            for (int s = 0; s < WS; ++s) {
                mbar_init(&sh.fullw[s], kDecodeWarps);      // each dequant warp
                mbar_init(&sh.emptyw[s], 1);               // MMA commit
            }
            for (int s = 0; s < C::QST; ++s) {
                mbar_init(&sh.qfull[s], 1);
                mbar_init(&sh.qempty[s], kDecodeWarps);
            }
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sh.accfull[a], 1);
            mbar_init(&sh.accempty[a], 4);
        }
        mbar_init(sh.done, 1);
        *sh.stop.flag = 0u;
        *sh.drain_failed = 0u;
        mbar_fence_init();
        for (int g = 0; g < gp.n_groups; ++g) {
            prefetch_tensormap(&gp.tmX[g]);
            prefetch_tensormap(&gp.tmW[g]);
        }
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
            int stage = 0, qs = 0, loads = 0, qloads = 0;
            uint32_t phase = 0, qphase = 0;
            for (int tile = blockIdx.x; tile < gp.num_tiles; tile += gridDim.x) {
                const TileLoc L = locate(gp, tile);
                const int m0 = L.m0, n0 = L.n0, nk = gp.nk[L.g];
                const CUtensorMap *tmX = &gp.tmX[L.g], *tmW = &gp.tmW[L.g];
                for (int kb = 0; kb < nk; ++kb) {
                    if constexpr (C::FUSED) {
                        if (!wait_phase_sleepy(&sh.qempty[qs], qphase ^ 1u, 256, limit_ns, sh.stop, err,
                                               kErrTimeoutProducer))
                            goto producer_done;
                        const int start = kb * QFmt<TYPE>::SB_BYTES;
                        mbar_arrive_expect_tx(&sh.qfull[qs], C::Q_SLOT_BYTES);
                        tma_load_2d(qslots + qs * C::Q_SLOT_BYTES, tmW, &sh.qfull[qs], (start & ~15) >> 2, m0);
                        ++qloads;
                        advance(qs, qphase, C::QST);
                    }
#pragma unroll 1
                    for (int a = 0; a < SB / BK; ++a) {
                        // fused: the decode warps share this sub-partition, so poll gently;
                        // cached: the producer feeds the MMA directly, so poll hot
                        if (!(C::FUSED ? wait_phase_sleepy(&sh.emptyx[stage], phase ^ 1u, 256, limit_ns,
                                                           sh.stop, err, kErrTimeoutProducer)
                                       : wait_phase(&sh.emptyx[stage], phase ^ 1u, limit_ns, sh.stop, err,
                                                    kErrTimeoutProducer)))
                            goto producer_done;
                        const int k0 = kb * SB + a * BK;
                        mbar_arrive_expect_tx(&sh.fullx[stage],
                                              C::FUSED ? X_STAGE_BYTES : X_STAGE_BYTES + W_STAGE_BYTES);
                        if (loads != inject_stall) {
                            tma_load_2d(xs + stage * X_STAGE_BYTES, tmX, &sh.fullx[stage], k0, n0);
                            if constexpr (!C::FUSED)
                                tma_load_2d(ws + stage * W_STAGE_BYTES, tmW, &sh.fullx[stage], k0, m0);
                        }
                        ++loads;
                        advance(stage, phase, XS);
                    }
                }
            }
        producer_done:
            // every copy issued has landed before shared memory can be released
            bool drained = drain_ring(sh.fullx, XS, loads, inject_stall, limit_ns);
            if constexpr (C::FUSED) drained = drain_ring(sh.qfull, C::QST, qloads, -1, limit_ns) && drained;
            if (!drained) {
                *sh.drain_failed = 1u;
                atomicOr(err, kErrTimeoutProducer);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA --
        if (lane == 0) {
            int stage = 0, wstage = 0, acc = 0;
            uint32_t phase = 0, wphase = 0, acc_phase = 0;
            for (int tile = blockIdx.x; tile < gp.num_tiles; tile += gridDim.x) {
                const int nk = gp.nk[locate(gp, tile).g];
                if (!wait_phase(&sh.accempty[acc], acc_phase ^ 1u, limit_ns, sh.stop, err, kErrTimeoutMma))
                    goto mma_done;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < nk; ++kb) {
#pragma unroll 1
                    for (int a = 0; a < SB / BK; ++a) {
                        if (!wait_phase(&sh.fullx[stage], phase, limit_ns, sh.stop, err, kErrTimeoutMma))
                            goto mma_done;
                        if constexpr (C::FUSED) {
                            if (!wait_phase(&sh.fullw[wstage], wphase, limit_ns, sh.stop, err, kErrTimeoutMma))
                                goto mma_done;
                        }
                        tc_fence_after();
                        const int wt = C::FUSED ? wstage : stage;
                        const uint64_t adesc = desc_sw128_kmajor(smem_u32(ws + wt * W_STAGE_BYTES));
                        const uint64_t bdesc = desc_sw128_kmajor(smem_u32(xs + stage * X_STAGE_BYTES));
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)  // advance 16 fp16 = 32 B inside the swizzle row
                            mma_f16_ss(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb | a | k) != 0);
                        mma_commit(&sh.emptyx[stage]);     // frees the stages when these MMAs finish
                        advance(stage, phase, XS);
                        if constexpr (C::FUSED) {
                            mma_commit(&sh.emptyw[wstage]);
                            advance(wstage, wphase, WS);
                        }
                    }
                }
                mma_commit(&sh.accfull[acc]);              // accumulator ready for the epilogue
                advance(acc, acc_phase, 2);
            }
        mma_done:
            // Everything issued has completed before TMEM is released.
            mma_commit(sh.done);
            if (!wait_drain(sh.done, 0, limit_ns)) {
                *sh.drain_failed = 1u;
                atomicOr(err, kErrTimeoutMma);
            }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------ epilogue --
        const int quarter = warp & 3;                      // TMEM lanes 32*quarter .. +31
        int acc = 0;
        uint32_t acc_phase = 0;
        const int T = gp.T;
        for (int tile = blockIdx.x; tile < gp.num_tiles; tile += gridDim.x) {
            const TileLoc L = locate(gp, tile);
            const int m0 = L.m0, n0 = L.n0, out_f = gp.out_f[L.g];
            float *const Y = gp.Y[L.g];
            if (!__all_sync(0xffffffffu, wait_phase_sleepy(&sh.accfull[acc], acc_phase, 512, limit_ns,
                                                           sh.stop, err, kErrTimeoutEpilogue)))
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
        // unit u = 0..7 <- warps 6, 7, 8, 10, 11, 12, 14, 15 (none on sub-partition 1)
        const int u = warp < 9 ? warp - 6 : (warp < 13 ? warp - 7 : warp - 8);
        if (warp != 9 && warp != 13) {
            const int r = (u & 3) * 32 + lane;             // weight row within the tile
            dequant_role<TYPE, C::WST, C::QST>(sh, gp, blockIdx.x, gridDim.x, qslots, smem_u32(ws), r, u >> 2, lane, limit_ns,
                                       err);
        }
    }

    __syncthreads();
    if (*sh.drain_failed) pause_ns(200000ull);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// --------------------------------------------------- CTA-pair cached GEMM --
//
// The cached (fp16 weight) mode as clusters of two CTAs sharing one
// tcgen05.mma.cta_group::2: a pair tile is 256 weight rows x 256 tokens;
// CTA r of the pair stages weight rows m0 + 128r and tokens n0 + 128r (its
// halves of A and B, 16 KiB each per K step) with the pair form of TMA,
// whose bytes complete on the leader's (rank 0) barrier; the leader issues
// M = 256, N = 256 MMAs over both CTAs' shared memory, each CTA's TMEM
// receiving its 128 rows of the accumulator, and multicasts its commits to
// both CTAs; each CTA's epilogue drains its own rows and signals the leader.
// Per SM a K step moves half the token operand of the single-CTA kernel.
// ACC = accumulators in TMEM (256 columns each).
// Drains this warp's share of one accumulator: TMEM lanes = weight rows
// o0 .. o0 + 31 (one per lane), 256 columns = tokens n0 .. n0 + 255, into Y
// [T x out_f], 32 tokens at a time.  Each 32 x 32 block is transposed
// through one of this warp's EPI_BUFS staging buffers (4 KiB, token-major
// rows of 32 weight rows: lanes write consecutive words, so no bank
// conflicts) and written by a TMA bulk store, which leaves out what lies past
// out_f or T; `nst` counts this warp's stores so far.  Against plain stores
// from registers this takes the per-token address and bounds arithmetic and
// the global stores off the SM's load/store path, which the decode warps
// share (measured: +17% on a 1.7B-shaped Q4_K layer at T = 2048, whose
// tiles are short in K; +3% on the 8B-shaped layer at T = 8192).
template <int EPI_BUFS>
__device__ __forceinline__ void drain_acc(uint32_t taddr, const CUtensorMap *tmY, int out_f, int T, int o0, int n0,
                                          uint32_t stage, int lane, uint32_t &nst) {
    if (o0 >= out_f) return;                    // every row of this warp lies past the weight's end
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        const int t0 = n0 + c * 32;
        if (t0 >= T) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_wait_ld();
        const uint32_t buf = stage + (nst % EPI_BUFS) * 4096u;
        if (lane == 0) bulk_wait_group_read<EPI_BUFS - 1>();   // the buffer's last store has read it
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 32; ++j) sts32(buf + static_cast<uint32_t>(j * 128 + lane * 4), r[j]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmY, buf, o0, t0);
            bulk_commit_group();
        }
        ++nst;
    }
}

// A stage holds two 64-value K panels, each this CTA's A half and B half, so
// the MMA thread and the producer meet once per 128 values of K (as in the
// fused pair kernel).
template <int ACC> struct PairCfg {
    static constexpr int ST = 3, EPI = 2;
    static constexpr int HALF_BYTES = 128 * BK * 2;              // 16 KiB
    static constexpr int PANEL_BYTES = 2 * HALF_BYTES;           // A half + B half of one K panel
    static constexpr int STAGE_BYTES = 2 * PANEL_BYTES;          // two K panels
    static constexpr int OFF_EPI = ST * STAGE_BYTES;             // 4 epilogue warps x EPI x 4 KiB
    static constexpr int OFF_BAR = OFF_EPI + 4 * EPI * 4096;
    static constexpr int NBAR = 2 * ST + 5;                      // full, empty, accfull[2], accempty[2], done
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int THREADS = 6 * 32;
    static constexpr uint32_t COLS = 256u * ACC;
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

constexpr uint32_t IDESC_PAIR = idesc_f16_f32(2 * BM, BN);

template <int ACC>
__global__ void __launch_bounds__(PairCfg<ACC>::THREADS, 1)
    pair_gemm_kernel(const __grid_constant__ GroupParams gp, uint32_t *err, uint64_t limit_ns, int inject_stall) {
    using P = PairCfg<ACC>;
    const uint32_t rank = cluster_ctarank();
    const int first = static_cast<int>(blockIdx.x) / 2, stride = static_cast<int>(gridDim.x) / 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::OFF_BAR);
    uint64_t *full = bars, *empty = bars + P::ST, *accfull = bars + 2 * P::ST, *accempty = accfull + 2,
             *done = accfull + 4;
    uint32_t *tmem_base = reinterpret_cast<uint32_t *>(smem + P::OFF_MISC);
    volatile uint32_t *const flag = reinterpret_cast<volatile uint32_t *>(smem + P::OFF_MISC + 4);
    volatile uint32_t *const drain_failed = reinterpret_cast<volatile uint32_t *>(smem + P::OFF_MISC + 8);
    const Stop stop{flag, mapa_shared(smem_u32(const_cast<uint32_t *>(flag)), rank ^ 1u)};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P::ST; ++s) {
            mbar_init(&full[s], 1);         // leader: its producer's arrive with both CTAs' bytes
            mbar_init(&empty[s], 1);        // the leader's multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accfull[a], 1);      // the leader's multicast commit
            mbar_init(&accempty[a], 8);     // leader: four epilogue warps of each CTA
        }
        mbar_init(done, 1);
        *flag = 0u;
        *drain_failed = 0u;
        mbar_fence_init();
        for (int g = 0; g < gp.n_groups; ++g) {
            prefetch_tensormap(&gp.tmX[g]);
            prefetch_tensormap(&gp.tmW[g]);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_base, P::COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();                         // both CTAs' barriers and TMEM exist
    tc_fence_after();
    const uint32_t tmem = *tmem_base;
    const bool alloc_ok = tmem == ld_shared_cluster_u32(mapa_shared(smem_u32(tmem_base), rank ^ 1u));
    if (!alloc_ok && threadIdx.x == 0) atomicOr(err, kErrPairAlloc);

    uint8_t *stages = smem;
    if (alloc_ok && warp == 0) {
        // --------------------------------------------------------- producer --
        if (lane == 0) {
            int stage = 0, loads = 0, skip_arm = -1;   // loads: stages armed
            uint32_t phase = 0;
            for (int tile = first; tile < gp.num_tiles; tile += stride) {
                const TileLoc L = locate(gp, tile);
                const int m0 = 2 * L.m0 + 128 * static_cast<int>(rank), n0 = L.n0 + 128 * static_cast<int>(rank);
                const CUtensorMap *tmX = &gp.tmX[L.g], *tmW = &gp.tmW[L.g];
                for (int k = 0; k < gp.nk[L.g] * (SB / BK); k += 2) {   // K panels k, k + 1
                    if (!wait_phase(&empty[stage], phase ^ 1u, limit_ns, stop, err, kErrTimeoutProducer))
                        goto producer_done;
                    const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0u);
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * P::STAGE_BYTES);
                    uint8_t *st = stages + stage * P::STAGE_BYTES;
                    // test hook: loads counted in panels; the stage holding the
                    // named panel gets no copies at all
                    if (inject_stall == 2 * loads || inject_stall == 2 * loads + 1) {
                        skip_arm = loads;
                    } else {
#pragma unroll
                        for (int pp = 0; pp < 2; ++pp) {
                            tma_load_2d_pair(st + pp * P::PANEL_BYTES, tmW, bar, (k + pp) * BK, m0);
                            tma_load_2d_pair(st + pp * P::PANEL_BYTES + P::HALF_BYTES, tmX, bar, (k + pp) * BK, n0);
                        }
                    }
                    ++loads;
                    advance(stage, phase, P::ST);
                }
            }
        producer_done:
            // The leader's stage barriers count both CTAs' bytes: once every
            // phase it armed has completed, every copy of both has landed.
            if (rank == 0 && !drain_ring(full, P::ST, loads, skip_arm, limit_ns)) {
                *drain_failed = 1u;
                atomicOr(err, kErrTimeoutProducer);
            }
        }
        __syncwarp();
    } else if (alloc_ok && warp == 1) {
        // -------------------------------------------------- MMA (leader only) --
        if (lane == 0 && rank == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int tile = first; tile < gp.num_tiles; tile += stride) {
                const int nks = gp.nk[locate(gp, tile).g] * (SB / BK) / 2;   // stages of two K panels
                if (!wait_phase(&accempty[acc], acc_phase ^ 1u, limit_ns, stop, err, kErrTimeoutMma))
                    goto mma_done;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
                for (int k = 0; k < nks; ++k) {
                    if (!wait_phase(&full[stage], phase, limit_ns, stop, err, kErrTimeoutMma)) goto mma_done;
                    tc_fence_after();
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {            // the K panels in order
                        uint8_t *st = stages + stage * P::STAGE_BYTES + pp * P::PANEL_BYTES;
                        const uint64_t adesc = desc_sw128_kmajor(smem_u32(st));
                        const uint64_t bdesc = desc_sw128_kmajor(smem_u32(st + P::HALF_BYTES));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_f16_ss_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC_PAIR, (k | pp | kk) != 0);
                    }
                    mma_commit_pair_multicast(&empty[stage], 0x3);
                    advance(stage, phase, P::ST);
                }
                mma_commit_pair_multicast(&accfull[acc], 0x3);
                advance(acc, acc_phase, ACC);
            }
        mma_done:
            // both CTAs' TMEM is written by these MMAs: they complete before
            // the cluster barrier that precedes the deallocation
            mma_commit_pair_multicast(done, 0x1);
            if (!wait_drain(done, 0, limit_ns)) {
                *drain_failed = 1u;
                atomicOr(err, kErrTimeoutMma);
            }
        }
        __syncwarp();
    } else if (alloc_ok && warp < 6) {
        // --------------------------------------------------------- epilogue --
        const int quarter = warp & 3;
        const uint32_t accempty_leader = mapa_shared(smem_u32(accempty), 0u);
        const uint32_t epi = smem_u32(smem + P::OFF_EPI) + static_cast<uint32_t>(quarter * P::EPI * 4096);
        int acc = 0;
        uint32_t acc_phase = 0, nst = 0;
        for (int tile = first; tile < gp.num_tiles; tile += stride) {
            const TileLoc L = locate(gp, tile);
            if (!__all_sync(0xffffffffu, wait_phase(&accfull[acc], acc_phase, limit_ns, stop, err,
                                                      kErrTimeoutEpilogue)))
                break;
            tc_fence_after();
            const uint32_t taddr =
                tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
            drain_acc<P::EPI>(taddr, &gp.tmY[L.g], gp.out_f[L.g], gp.T,
                              2 * L.m0 + 128 * static_cast<int>(rank) + quarter * 32, L.n0, epi, lane, nst);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(accempty_leader + static_cast<uint32_t>(acc * 8));
            advance(acc, acc_phase, ACC);
        }
        if (lane == 0) bulk_wait_all();         // Y stores complete before the CTA's shared memory goes
    }

    __syncthreads();
    // The second CTA's copies complete on the leader's barriers, which it
    // cannot poll: after a stop it pauses instead.
    if (*drain_failed || (rank == 1 && stop.raised())) pause_ns(200000ull);
    cluster_sync();                         // nothing of either CTA still in flight
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, P::COLS);
    }
}

// ---------------------------------------------------- CTA-pair fused GEMM --
//
// The fused mode on CTA pairs, as the cached mode above: a pair tile is 256
// weight rows x 256 tokens; CTA r decodes weight rows m0 + 128r (its half of
// A) into its own shared memory exactly as the single-CTA kernel does, and
// stages tokens n0 + 128r (its half of B) with the pair form of TMA.  The
// leader's MMA thread waits for the token halves (TMA bytes on its fullx)
// and for the decoded stage of both CTAs (its fullw counts the leader's eight
// decode warps and the peer's eight, which arrive remotely, each after its
// stores were made visible to the tensor cores), issues the M = 256 MMAs and
// multicasts its commits: the stages' emptyx / emptyw and the accumulators'
// accfull in both CTAs.  (A forwarding thread in the peer that waited on the
// peer's own barrier and passed one arrival on measured 2% slower on the
// Q2_K launch.)
// A stage holds two 64-value K panels of both operands (X: 2 x 16 KiB of
// this CTA's tokens; W16: 2 x 16 KiB), so the MMA thread and the decode warps
// meet once per 128 values of K: measured on the 8B-shaped layer against
// one-panel stages of the same bytes (6 X, 4 W16): Q2_K launch +1.8%, Q6_K
// launch +5.1%.  Ring depths in stages and epilogue staging buffers per warp.
// The token ring is the one that pays for depth (measured with one-panel
// stages on the Q2_K / Q6_K layer: 4 -> 6 -> 8 stages, +5% then +0.5%); more
// fp16 W stages or a second slice slot did not help.
template <int TYPE> struct PairDepth { static constexpr int XST = 3, WST = 2, QST = 1, EPI = 2; };
template <> struct PairDepth<kQ8_0> { static constexpr int XST = 2, WST = 2, QST = 2, EPI = 1; };

template <int TYPE> struct PairFCfg {
    static constexpr int XST = PairDepth<TYPE>::XST, WST = PairDepth<TYPE>::WST, QST = PairDepth<TYPE>::QST;
    static constexpr int EPI = PairDepth<TYPE>::EPI;
    static constexpr int X_HALF = 128 * BK * 2;                  // 16 KiB: this CTA's 128 tokens, one panel
    static constexpr int X_ST = 2 * X_HALF, W_ST = 2 * W_STAGE_BYTES;   // a stage: two K panels
    static constexpr int THREADS = 16 * 32;
    static constexpr int Q_SLOT_BYTES = BM * QFmt<TYPE>::BOX;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_W = OFF_X + XST * X_ST;
    static constexpr int OFF_Q = OFF_W + WST * W_ST;
    static constexpr int OFF_EPI = OFF_Q + QST * Q_SLOT_BYTES;   // 4 epilogue warps x EPI x 4 KiB
    static constexpr int OFF_BAR = OFF_EPI + 4 * EPI * 4096;
    // fullx, emptyx, fullw, emptyw, qfull, qempty, accfull[2], accempty[2], done
    static constexpr int NBAR = 2 * XST + 2 * WST + 2 * QST + 5;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static_assert(OFF_Q % 1024 == 0 && OFF_EPI % 128 == 0 && SMEM_BYTES <= 232448, "shared memory layout");
};

template <int TYPE>
__global__ void __launch_bounds__(PairFCfg<TYPE>::THREADS, 1)
    pair_fused_kernel(const __grid_constant__ GroupParams gp, uint32_t *err, uint64_t limit_ns, int inject_stall) {
    using C = PairFCfg<TYPE>;
    constexpr int XS = C::XST, WS = C::WST, QS = C::QST;
    const uint32_t rank = cluster_ctarank();
    const int first = static_cast<int>(blockIdx.x) / 2, stride = static_cast<int>(gridDim.x) / 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    Shared sh;
    sh.fullx = bars;
    sh.emptyx = bars + XS;
    sh.fullw = bars + 2 * XS;
    sh.emptyw = sh.fullw + WS;
    sh.qfull = sh.emptyw + WS;
    sh.qempty = sh.qfull + QS;
    sh.accfull = sh.qempty + QS;
    sh.accempty = sh.accfull + 2;
    sh.done = sh.accfull + 4;
    sh.tmem_base = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    {
        volatile uint32_t *const flag = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_MISC + 4);
        sh.stop = Stop{flag, mapa_shared(smem_u32(const_cast<uint32_t *>(flag)), rank ^ 1u)};
    }
    sh.drain_failed = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_MISC + 8);
    if (rank == 1) sh.fullw_remote = mapa_shared(smem_u32(sh.fullw), 0u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < XS; ++s) {
            mbar_init(&sh.fullx[s], 1);            // leader: its producer's arrive with both token halves' bytes
            mbar_init(&sh.emptyx[s], 1);           // the leader's multicast commit
        }
        for (int s = 0; s < WS; ++s) {
            mbar_init(&sh.fullw[s], 2 * kDecodeWarps);  // leader: both CTAs' decode warps (the peer's: unused)
            mbar_init(&sh.emptyw[s], 1);           // the leader's multicast commit
        }
        for (int s = 0; s < QS; ++s) {
            mbar_init(&sh.qfull[s], 1);
            mbar_init(&sh.qempty[s], kDecodeWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sh.accfull[a], 1);
            mbar_init(&sh.accempty[a], 8);         // leader: four epilogue warps of each CTA
        }
        mbar_init(sh.done, 1);
        *sh.stop.flag = 0u;
        *sh.drain_failed = 0u;
        mbar_fence_init();
        for (int g = 0; g < gp.n_groups; ++g) {
            prefetch_tensormap(&gp.tmX[g]);
            prefetch_tensormap(&gp.tmW[g]);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(sh.tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *sh.tmem_base;
    const bool alloc_ok = tmem == ld_shared_cluster_u32(mapa_shared(smem_u32(sh.tmem_base), rank ^ 1u));
    if (!alloc_ok && threadIdx.x == 0) atomicOr(err, kErrPairAlloc);

    uint8_t *xs = smem + C::OFF_X;
    uint8_t *ws = smem + C::OFF_W;
    uint8_t *qslots = smem + C::OFF_Q;

    if (alloc_ok && warp == 0) {
        // --------------------------------------------------------- producer --
        if (lane == 0) {
            int stage = 0, qs = 0, loads = 0, qloads = 0, skip_arm = -1;   // loads: token stages armed
            uint32_t phase = 0, qphase = 0;
            for (int tile = first; tile < gp.num_tiles; tile += stride) {
                const TileLoc L = locate(gp, tile);
                const int m0 = 2 * L.m0 + 128 * static_cast<int>(rank), n0 = L.n0 + 128 * static_cast<int>(rank);
                const int nk = gp.nk[L.g];
                const CUtensorMap *tmX = &gp.tmX[L.g], *tmW = &gp.tmW[L.g];
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_phase_sleepy(&sh.qempty[qs], qphase ^ 1u, 256, limit_ns, sh.stop, err,
                                           kErrTimeoutProducer))
                        goto producer_done;
                    const int start = kb * QFmt<TYPE>::SB_BYTES;
                    mbar_arrive_expect_tx(&sh.qfull[qs], C::Q_SLOT_BYTES);
                    tma_load_2d(qslots + qs * C::Q_SLOT_BYTES, tmW, &sh.qfull[qs], (start & ~15) >> 2, m0);
                    ++qloads;
                    advance(qs, qphase, QS);
#pragma unroll 1
                    for (int a = 0; a < SB / BK; a += 2) {   // a stage: K panels a, a + 1
                        if (!wait_phase(&sh.emptyx[stage], phase ^ 1u, limit_ns, sh.stop, err,
                                        kErrTimeoutProducer))
                            goto producer_done;
                        if (rank == 0) mbar_arrive_expect_tx(&sh.fullx[stage], 4 * C::X_HALF);
                        // the test hook counts loads in panels; the stage holding
                        // the named panel gets no copies at all
                        if (inject_stall == 2 * loads || inject_stall == 2 * loads + 1) {
                            skip_arm = loads;
                        } else {
                            const uint32_t fx = mapa_shared(smem_u32(&sh.fullx[stage]), 0u);
                            tma_load_2d_pair(xs + stage * C::X_ST, tmX, fx, kb * SB + a * BK, n0);
                            tma_load_2d_pair(xs + stage * C::X_ST + C::X_HALF, tmX, fx, kb * SB + (a + 1) * BK, n0);
                        }
                        ++loads;
                        advance(stage, phase, XS);
                    }
                }
            }
        producer_done:
            // Each CTA's slice copies complete on its own barriers; the token
            // halves of both CTAs on the leader's.
            bool drained = drain_ring(sh.qfull, QS, qloads, -1, limit_ns);
            if (rank == 0) drained = drain_ring(sh.fullx, XS, loads, skip_arm, limit_ns) && drained;
            if (!drained) {
                *sh.drain_failed = 1u;
                atomicOr(err, kErrTimeoutProducer);
            }
        }
        __syncwarp();
    } else if (alloc_ok && warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA (leader) --
            int stage = 0, wstage = 0, acc = 0;
            uint32_t phase = 0, wphase = 0, acc_phase = 0;
            for (int tile = first; tile < gp.num_tiles; tile += stride) {
                const int nks = gp.nk[locate(gp, tile).g] * (SB / BK) / 2;   // stages of two K panels
                if (!wait_phase(&sh.accempty[acc], acc_phase ^ 1u, limit_ns, sh.stop, err,
                                      kErrTimeoutMma))
                    goto mma_done;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
                for (int k = 0; k < nks; ++k) {
                    if (!wait_phase(&sh.fullx[stage], phase, limit_ns, sh.stop, err, kErrTimeoutMma) ||
                        !wait_phase(&sh.fullw[wstage], wphase, limit_ns, sh.stop, err, kErrTimeoutMma))
                        goto mma_done;
                    tc_fence_after();
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {            // the K panels in order
                        const uint64_t adesc = desc_sw128_kmajor(smem_u32(ws + wstage * C::W_ST + pp * W_STAGE_BYTES));
                        const uint64_t bdesc = desc_sw128_kmajor(smem_u32(xs + stage * C::X_ST + pp * C::X_HALF));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_f16_ss_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC_PAIR, (k | pp | kk) != 0);
                    }
                    mma_commit_pair_multicast(&sh.emptyx[stage], 0x3);
                    mma_commit_pair_multicast(&sh.emptyw[wstage], 0x3);
                    advance(stage, phase, XS);
                    advance(wstage, wphase, WS);
                }
                mma_commit_pair_multicast(&sh.accfull[acc], 0x3);
                advance(acc, acc_phase, 2);
            }
        mma_done:
            // both CTAs' TMEM is written by these MMAs: they complete before
            // the cluster barrier that precedes the deallocation
            mma_commit_pair_multicast(sh.done, 0x1);
            if (!wait_drain(sh.done, 0, limit_ns)) {
                *sh.drain_failed = 1u;
                atomicOr(err, kErrTimeoutMma);
            }
        }
        __syncwarp();
    } else if (alloc_ok && warp < 6) {
        // --------------------------------------------------------- epilogue --
        const int quarter = warp & 3;
        const uint32_t accempty_leader = mapa_shared(smem_u32(sh.accempty), 0u);
        const uint32_t epi = smem_u32(smem + C::OFF_EPI) + static_cast<uint32_t>(quarter * C::EPI * 4096);
        int acc = 0;
        uint32_t acc_phase = 0, nst = 0;
        for (int tile = first; tile < gp.num_tiles; tile += stride) {
            const TileLoc L = locate(gp, tile);
            if (!__all_sync(0xffffffffu, wait_phase_sleepy(&sh.accfull[acc], acc_phase, 512, limit_ns,
                                                                 sh.stop, err, kErrTimeoutEpilogue)))
                break;
            tc_fence_after();
            const uint32_t taddr =
                tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
            drain_acc<C::EPI>(taddr, &gp.tmY[L.g], gp.out_f[L.g], gp.T,
                              2 * L.m0 + 128 * static_cast<int>(rank) + quarter * 32, L.n0, epi, lane, nst);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(accempty_leader + static_cast<uint32_t>(acc * 8));
            advance(acc, acc_phase, 2);
        }
        if (lane == 0) bulk_wait_all();         // Y stores complete before the CTA's shared memory goes
    } else if (alloc_ok) {
        // ------------------------------------------------------------ decode --
        // Unit u = 0..7 decodes rows 32(u%4)..+31, half u/4 of each K step.  In
        // the leader the units sit on warps 6, 7, 8, 10, 11, 12, 14, 15, off the
        // MMA thread's sub-partition 1 (3/3/2 on sub-partitions 2, 3, 0); the
        // peer issues no MMAs, so its units take warps 6..13, two on each
        // sub-partition.  Measured on the 8B-shaped layer: decode warps on
        // sub-partition 1 in both CTAs 1190 TFLOP/s; in neither 1451; in the
        // peer only 1471.
        int u = -1;
        if (rank == 1) {
            if (warp >= 6 && warp < 14) u = warp - 6;
        } else if (warp != 9 && warp != 13) {
            u = warp < 9 ? warp - 6 : (warp < 13 ? warp - 7 : warp - 8);
        }
        if (u >= 0) {
            const int r = (u & 3) * 32 + lane;                 // this CTA's weight row
            dequant_role<TYPE, WS, QS, 2>(sh, gp, first, stride, qslots, smem_u32(ws), r, u >> 2, lane, limit_ns,
                                            err);
        }
    }

    __syncthreads();
    // The second CTA's token copies complete on the leader's barriers, which
    // it cannot poll: after a stop it pauses instead.
    if (*sh.drain_failed || (rank == 1 && sh.stop.raised())) pause_ns(200000ull);
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, TMEM_COLS);
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

// Tensor maps of one projection: X boxes of x_rows tokens (256 for one CTA,
// 128 for a CTA pair) x 64 values; W boxes of 128 rows (quantized slice or
// fp16 K step).
template <int TYPE>
bool encode_group(EncodeFn enc, const GemmArgs &a, CUtensorMap *tmX, CUtensorMap *tmW, uint32_t x_rows) {
    if (!encode_2d(enc, tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.X, a.in_f, a.T, a.in_f * 2, BK, x_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    if constexpr (TYPE != 0) {
        const int64_t row_bytes = (a.in_f / SB) * QFmt<TYPE>::SB_BYTES;
        return encode_2d(enc, tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.W, row_bytes / 4, a.out_f, row_bytes,
                         QFmt<TYPE>::BOX / 4, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
        return encode_2d(enc, tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.W, a.in_f, a.out_f, a.in_f * 2, BK, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    }
}

// The launch's GroupParams over n projections of type TYPE (same T).  Groups
// are ordered by in_f, longest first: their tiles take longest, and dealing
// them out first keeps the CTAs' total work even.  A tile is 128 weight rows
// (one CTA) or 256 (a CTA pair) by 256 tokens.
template <int TYPE>
bool build_group(const GemmArgs *a, int n, EncodeFn enc, bool pair, GroupParams &gp) {
    if (n < 1 || n > MAX_GROUPS) return false;
    int order[MAX_GROUPS];
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order, order + n, [&](int x, int y) { return a[x].in_f > a[y].in_f; });
    std::memset(&gp, 0, sizeof(gp));
    const int64_t rows_per_tile = pair ? 2 * BM : BM;
    const int64_t n_tiles = (a[0].T + BN - 1) / BN;
    int64_t tiles = 0;
    for (int j = 0; j < n; ++j) {
        const GemmArgs &g = a[order[j]];
        if (g.T != a[0].T || !encode_group<TYPE>(enc, g, &gp.tmX[j], &gp.tmW[j], pair ? BN / 2 : BN)) return false;
        const int64_t m_tiles = (g.out_f + rows_per_tile - 1) / rows_per_tile;
        tiles += m_tiles * n_tiles;
        if (tiles > INT32_MAX) return false;
        gp.Y[j] = g.Y;
        // the pair kernels store Y by TMA (the C ABI keeps Y 16-byte aligned, out_f % 4 == 0)
        if (pair && !encode_2d(enc, &gp.tmY[j], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.Y, g.out_f, g.T, g.out_f * 4, 32,
                               32, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
        gp.out_f[j] = static_cast<int>(g.out_f);
        gp.nk[j] = static_cast<int>(g.in_f / SB);
        gp.m_tiles[j] = static_cast<int>(m_tiles);
        gp.tile_end[j] = static_cast<int>(tiles);
    }
    gp.n_groups = n;
    gp.T = static_cast<int>(a[0].T);
    gp.num_tiles = static_cast<int>(tiles);
    return true;
}

// One-CTA kernel: one persistent CTA per SM.
template <int TYPE>
cudaError_t launch_typed(const GemmArgs *a, int n, EncodeFn enc, cudaStream_t stream) {
    using C = Cfg<TYPE>;
    GroupParams gp;
    if (!build_group<TYPE>(a, n, enc, false, gp)) return cudaErrorInvalidValue;
    const int grid = gp.num_tiles < a[0].num_sms ? gp.num_tiles : a[0].num_sms;
    auto kern = prefill_gemm_kernel<TYPE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(gp, a[0].err, a[0].wait_limit_ns, a[0].inject_stall);
    return cudaGetLastError();
}

// CTA-pair kernels: clusters of two, as many as the GPU holds at once.
template <typename Kern, typename... Args>
cudaError_t launch_clusters(Kern kern, int threads, int smem, const GroupParams &gp, int num_sms,
                            std::atomic<int> &max_clusters,
                            cudaStream_t stream, Args... args) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int mc = max_clusters.load();                 // queried once per kernel and device, then cached
    if (mc == 0) {
        cfg.gridDim = dim3(num_sms, 1, 1);
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, kern, &cfg) != cudaSuccess || c < 1) {
            cudaGetLastError();
            c = num_sms / 2;
        }
        mc = c;
        max_clusters.store(c);
    }
    const int clusters = gp.num_tiles < mc ? gp.num_tiles : mc;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    e = cudaLaunchKernelEx(&cfg, kern, gp, args...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int TYPE>
cudaError_t launch_pair_typed(const GemmArgs *a, int n, EncodeFn enc, cudaStream_t stream) {
    GroupParams gp;
    if (!build_group<TYPE>(a, n, enc, true, gp)) return cudaErrorInvalidValue;
    static std::atomic<int> max_clusters[kMaxDevices];
    std::atomic<int> &mc = max_clusters[a[0].device];
    if constexpr (TYPE == 0) {
        using P = PairCfg<2>;
        return launch_clusters(pair_gemm_kernel<2>, P::THREADS, P::SMEM_BYTES, gp, a[0].num_sms, mc,
                               stream, a[0].err, a[0].wait_limit_ns, a[0].inject_stall);
    } else {
        using P = PairFCfg<TYPE>;
        return launch_clusters(pair_fused_kernel<TYPE>, P::THREADS, P::SMEM_BYTES, gp, a[0].num_sms, mc,
                               stream, a[0].err, a[0].wait_limit_ns, a[0].inject_stall);
    }
}

template <int TYPE>
cudaError_t launch_any(const GemmArgs *a, int n, EncodeFn enc, cudaStream_t stream) {
    return a[0].cta_pairs ? launch_pair_typed<TYPE>(a, n, enc, stream) : launch_typed<TYPE>(a, n, enc, stream);
}

}  // namespace

cudaError_t launch_prefill_gemm(const GemmArgs *a, int n, void *encode_fn, cudaStream_t stream) {
    const EncodeFn enc = reinterpret_cast<EncodeFn>(encode_fn);
    if (n < 1) return cudaErrorInvalidValue;
    for (int i = 1; i < n; ++i)
        if (a[i].type != a[0].type) return cudaErrorInvalidValue;
    switch (a[0].type) {
    case 0: return launch_any<0>(a, n, enc, stream);
    case kQ4_K: return launch_any<kQ4_K>(a, n, enc, stream);
    case kQ5_K: return launch_any<kQ5_K>(a, n, enc, stream);
    case kQ2_K: return launch_any<kQ2_K>(a, n, enc, stream);
    case kQ6_K: return launch_any<kQ6_K>(a, n, enc, stream);
    case kQ8_0: return launch_any<kQ8_0>(a, n, enc, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qp
