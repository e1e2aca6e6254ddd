// gemv.cu — the decode-side projection over the same weight blocks:
//   Y[t, o] = sum_k X[t, k] * W16[o, k]      0 <= t < T <= 8
// for a handful of token rows: the serial path one token at a time ("QK-norm
// models take the FP16 batched prefill when it fits", §What changes: the
// serial prefill is one forward per prompt token) and the decode GEMVs that
// run over the same block types ("Qwen3.5 batched prefill has no f32 dequant
// for IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", §Cause).  W16 = the fp16 weights the
// fused prefill GEMM multiplies (the exact f32 dequant rounded to fp16), and
// the products are accumulated in f32, so this is the same projection as
// the prefill GEMM on T <= 8 rows.
//
// Meant to be bound by HBM on W (every weight byte is read once), which puts
// the integer pipe on a budget of about one to two instructions per weight
// value: the lanes only decode, and the dot products run on the tensor cores
// with the warp-level mma.sync m16n8k16, whose cost per value does not depend
// on T.  The MMA's A operand is 16 weight rows x 16 K values in fp16, B is
// the K values of the T token rows (columns >= T zero), D = f32.
//
// Two persistent CTAs per SM take 16-row blocks b, b + gridDim.x, ... of the
// launch.  A producer warp streams each block's rows through a ring of
// shared-memory tiles with 2-D TMA copies: a tile is the 16 rows x S steps
// (S x 256 values) of one K range, as the 16-byte aligned cover of that range
// in every row (up to 2 KB per row, so that the copies are long).  Eight
// consumer warps split the tiles: warp w takes step w % S of every tile its
// team w / S is given (the teams take a block's tiles in turn); every
// consumer warp still waits for and releases every tile.  Measured on
// the 8B-shaped layer's weights at T = 1, two such CTAs per SM stream 13%
// faster than one with twice the warps and ring.  In a step,
// lane (g, c) (g = lane / 4, c = lane % 4) decodes runs 2c and 2c + 1 of
// the step in weight rows g and g + 8 from the tile (the K-quants with
// steps written out per type, Q8_0 and F16 with the exact run decoders of
// qp_runs.cuh), rounds them to fp16 and feeds each run's 32 values to eight
// MMAs, four per MMA.  The MMA's K order is permuted: K slots 2c,
// 2c + 1, 2c + 8, 2c + 9 hold values 4i .. 4i + 3 of lane c's run in MMA i,
// for A and B alike, so the sum over K is unchanged, each lane's A fragment
// is its own decoded values and its B fragment is 4 consecutive values of
// token row g of X.  Steps past the row's end contribute zeros.  At a
// block's end the consumer warps' 16 x 8 partial tiles are summed through
// shared memory in warp order (a named barrier over the consumers only), so
// results are deterministic.
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

// ----------------------------------------------------- Q2_K and Q6_K steps --
// A consumer lane (g, c) decodes, in each step of 256 values, runs 2c and
// 2c + 1 of weight rows g and g + 8.  For the K-quants the step is written
// out per type: a row's fields are read
// from shared memory once for both runs, and each word of quants feeds the
// MMAs of both runs as soon as it is decoded.  The MMA order is the one
// described above: MMA k of run rho takes values 4k .. 4k + 3 of the run.

// Q2_K tables of four sub-blocks whose scale bytes are the bytes of sw:
// t01[s] = entries 0, 1 of sub-block s as a half2, t23[s] = entries 2, 3;
// entry q = RN_f16(fma(d * sc, q, -(dmin * m))), each f32 operation rounded
// once (the value formula of the K-quant page, "Q2_K" section), then fp16.
// A byte-permute selector nibble 2q (2q + 1) then picks entry q's low (high)
// byte from {t01, t23}.
template <int P>
__device__ __forceinline__ void q2k_pair_tables(uint32_t scw, uint32_t mw, pair_t d2, pair_t nd2, uint32_t (&t01)[4],
                                                uint32_t (&t23)[4]) {
    const pair_t nbias = pk2(-8388608.0f, -8388608.0f);
    const pair_t sc = fadd2(pk2(bias_float<2 * P>(scw), bias_float<2 * P + 1>(scw)), nbias);   // exact
    const pair_t m = fadd2(pk2(bias_float<2 * P>(mw), bias_float<2 * P + 1>(mw)), nbias);
    const pair_t dl = fmul2(d2, sc), nml = fmul2(nd2, m);
    float x[4], y[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) unpk2(ffma2(dl, pk2(static_cast<float>(q), static_cast<float>(q)), nml), x[q], y[q]);
    t01[2 * P] = h2_of(x[0], x[1]);
    t23[2 * P] = h2_of(x[2], x[3]);
    t01[2 * P + 1] = h2_of(y[0], y[1]);
    t23[2 * P + 1] = h2_of(y[2], y[3]);
}

__device__ __forceinline__ void q2k_tables4(uint32_t sw, uint32_t dd, uint32_t (&t01)[4], uint32_t (&t23)[4]) {
    const float d = h2f(dd), dmin = h2f(dd >> 16);
    const pair_t d2 = pk2(d, d), nd2 = pk2(-dmin, -dmin);   // -(dmin * m) = (-dmin) * m: rounding is sign-symmetric
    const uint32_t scw = sw & 0x0F0F0F0Fu, mw = (sw >> 4) & 0x0F0F0F0Fu;
    q2k_pair_tables<0>(scw, mw, d2, nd2, t01, t23);
    q2k_pair_tables<1>(scw, mw, d2, nd2, t01, t23);
}

// Four 2-bit quants (bits 0-1 of each byte of v) -> four fp16 weights of
// sub-block s: the selectors 2q | (2q + 1) << 4 per value, for the low and
// the high two bytes of v.
__device__ __forceinline__ void q2k_pick(uint32_t v, uint32_t t01, uint32_t t23, uint32_t &h01, uint32_t &h23) {
    h01 = prmt_sel(t01, t23, v * 0x22u + 0x10101010u);
    h23 = prmt_sel(t01, t23, mad_hi(v, 0x00220000u, 0x1010u));   // (v * 0x22) >> 16, + 0x1010
}

// Q2_K (84-byte superblocks, 4-byte aligned in the stage): run t = 2c + rho
// takes bits 2(t & 3) of qs[32(t >> 2) + l] and scale bytes 2t, 2t + 1; the
// lane's two runs share the quant words and the scale word of bytes 4c .. 4c + 3.
__device__ __forceinline__ void step_q2k(const uint8_t *b0, const uint8_t *b1, int c, const uint4 *xv, bool tok,
                                         float (&d)[4], float (&e)[4]) {
    uint32_t ta0[4], tb0[4], ta1[4], tb1[4];
    q2k_tables4(Smem::u32(b0 + 4 * c), Smem::u32(b0 + 80), ta0, tb0);
    q2k_tables4(Smem::u32(b1 + 4 * c), Smem::u32(b1 + 80), ta1, tb1);
    const uint8_t *q0 = b0 + 16 + 32 * (c >> 1), *q1 = b1 + 16 + 32 * (c >> 1);
    const int sh = 4 * (c & 1);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint4 xa = tok ? __ldg(xv + u) : make_uint4(0u, 0u, 0u, 0u);       // run 2c, values 8u .. 8u + 7
        const uint4 xb = tok ? __ldg(xv + 4 + u) : make_uint4(0u, 0u, 0u, 0u);   // run 2c + 1
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int k = 2 * u + hh, s = k >> 2;
            const uint32_t w0 = Smem::u32(q0 + 4 * k) >> sh, w1 = Smem::u32(q1 + 4 * k) >> sh;
            uint32_t a0, a1, a2, a3;
            q2k_pick(w0 & 0x03030303u, ta0[s], tb0[s], a0, a2);
            q2k_pick(w1 & 0x03030303u, ta1[s], tb1[s], a1, a3);
            mma_16816(d, a0, a1, a2, a3, hh ? xa.z : xa.x, hh ? xa.w : xa.y);
            q2k_pick((w0 >> 2) & 0x03030303u, ta0[s + 2], tb0[s + 2], a0, a2);
            q2k_pick((w1 >> 2) & 0x03030303u, ta1[s + 2], tb1[s + 2], a1, a3);
            mma_16816(e, a0, a1, a2, a3, hh ? xb.z : xb.x, hh ? xb.w : xb.y);
        }
    }
}

// Q6_K (210-byte superblocks, 2-byte aligned in the stage): run t = 2c + rho
// takes the low (c even) or high (c odd) nibbles of ql[64(t >> 2) + 32 rho + l]
// and bits 2(t & 3) of qh[32(t >> 2) + l], int8 scales 2t, 2t + 1; the two
// runs share the qh words and the scale bytes 4c .. 4c + 3.
// MIS: the superblock starts 2 bytes past a 4-byte boundary.  Its fields are
// then read as the aligned words starting 2 bytes early, so assembled word
// k holds values 4k - 2 .. 4k + 1 and a value's byte is taken from word k or
// k + 1 (all reads stay inside the superblock).
template <bool MIS>
struct Q6Row {
    static constexpr int NW = MIS ? 9 : 8;
    uint32_t u0[NW], u1[NW];   // 6-bit quants of runs 2c, 2c + 1, one per byte
    pair_t dl[4];              // d * scale of sub-blocks 4c .. 4c + 3, as pairs

    __device__ __forceinline__ void load(const uint8_t *b, int c) {
        const int o = MIS ? -2 : 0;
        const uint8_t *ql = b + 64 * (c >> 1) + o, *qh = b + 128 + 32 * (c >> 1) + o;
        const int hs = 4 * (c & 1);
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const uint32_t h = Smem::u32(qh + 4 * k) >> hs;
            u0[k] = ((Smem::u32(ql + 4 * k) >> hs) & 0x0F0F0F0Fu) + ((h & 0x03030303u) << 4);
            u1[k] = ((Smem::u32(ql + 32 + 4 * k) >> hs) & 0x0F0F0F0Fu) + ((h & 0x0C0C0C0Cu) << 2);
        }
        const uint32_t sw = MIS ? (Smem::u16(b + 192 + 4 * c) | (Smem::u16(b + 194 + 4 * c) << 16))
                                : Smem::u32(b + 192 + 4 * c);
        const float dd = h2f(Smem::u16(b + 208));
        const pair_t nb = pk2(-8388736.0f, -8388736.0f);   // -(2^23 + 128): int8 = (byte ^ 0x80) - 128
        const uint32_t sx = sw ^ 0x80808080u;
        const pair_t s01 = fadd2(pk2(bias_float<0>(sx), bias_float<1>(sx)), nb);
        const pair_t s23 = fadd2(pk2(bias_float<2>(sx), bias_float<3>(sx)), nb);
        float s[4];
        unpk2(s01, s[0], s[1]);
        unpk2(s23, s[2], s[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float v = __fmul_rn(dd, s[i]);   // exact: 11 x 8 significant bits
            dl[i] = pk2(v, v);
        }
    }
};

// A row read in the 2-byte offset form, brought to the aligned form (word k
// = values 4k .. 4k + 3), for warps whose lanes' rows start differently.
__device__ __forceinline__ void q6k_realign(const Q6Row<true> &a, Q6Row<false> &r) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        r.u0[k] = __funnelshift_r(a.u0[k], a.u0[k + 1], 16);
        r.u1[k] = __funnelshift_r(a.u1[k], a.u1[k + 1], 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) r.dl[i] = a.dl[i];
}

// Values 4k .. 4k + 3 of a run's quant words -> two half2 words.
template <bool MIS>
__device__ __forceinline__ void q6k_word(const uint32_t *u, int k, pair_t dl, uint32_t &h01, uint32_t &h23) {
    const pair_t nb = pk2(-8388640.0f, -8388640.0f);   // -(2^23 + 32)
    pair_t q01, q23;
    if (MIS) {
        q01 = pk2(bias_float<2>(u[k]), bias_float<3>(u[k]));
        q23 = pk2(bias_float<0>(u[k + 1]), bias_float<1>(u[k + 1]));
    } else {
        q01 = pk2(bias_float<0>(u[k]), bias_float<1>(u[k]));
        q23 = pk2(bias_float<2>(u[k]), bias_float<3>(u[k]));
    }
    h01 = f2h2(fmul2(dl, fadd2(q01, nb)));   // d * s * (q - 32): exact product, one rounding to fp16
    h23 = f2h2(fmul2(dl, fadd2(q23, nb)));
}

// The MMAs of a step over two rows already read.  mma.sync needs the whole
// warp: callers reach this with all 32 lanes.
template <bool MIS>
__device__ __forceinline__ void q6k_mma(const Q6Row<MIS> &r0, const Q6Row<MIS> &r1, const uint4 *xv, bool tok,
                                        float (&d)[4], float (&e)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint4 xa = tok ? __ldg(xv + u) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 xb = tok ? __ldg(xv + 4 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int k = 2 * u + hh, s = k >> 2;
            uint32_t a0, a1, a2, a3;
            q6k_word<MIS>(r0.u0, k, r0.dl[s], a0, a2);
            q6k_word<MIS>(r1.u0, k, r1.dl[s], a1, a3);
            mma_16816(d, a0, a1, a2, a3, hh ? xa.z : xa.x, hh ? xa.w : xa.y);
            q6k_word<MIS>(r0.u1, k, r0.dl[s + 2], a0, a2);
            q6k_word<MIS>(r1.u1, k, r1.dl[s + 2], a1, a3);
            mma_16816(e, a0, a1, a2, a3, hh ? xb.z : xb.x, hh ? xb.w : xb.y);
        }
    }
}

// One Q6_K step.  Rows g and g + 8 start alike modulo 4 (8 row pitches
// apart); with TMA tiles every row of a step starts alike too, so a warp's
// lanes agree and the warp takes the form of its rows' offset.  Rows staged
// by one copy each can disagree from lane to lane: then each lane reads its
// rows in its own form, brings them to the aligned one, and the warp's MMAs
// run together afterwards.
__device__ __forceinline__ void step_q6k(const uint8_t *b0, const uint8_t *b1, int c, const uint4 *xv, bool tok,
                                         float (&d)[4], float (&e)[4]) {
    const bool mis = (smem_u32(b0) & 2u) != 0u;
    if (__all_sync(0xffffffffu, mis)) {
        Q6Row<true> r0, r1;
        r0.load(b0, c);
        r1.load(b1, c);
        q6k_mma<true>(r0, r1, xv, tok, d, e);
    } else if (!__any_sync(0xffffffffu, mis)) {
        Q6Row<false> r0, r1;
        r0.load(b0, c);
        r1.load(b1, c);
        q6k_mma<false>(r0, r1, xv, tok, d, e);
    } else {
        Q6Row<false> r0, r1;
        if (mis) {
            Q6Row<true> a;
            a.load(b0, c);
            q6k_realign(a, r0);
            a.load(b1, c);
            q6k_realign(a, r1);
        } else {
            r0.load(b0, c);
            r1.load(b1, c);
        }
        q6k_mma<false>(r0, r1, xv, tok, d, e);
    }
}

// Q4_K / Q5_K (144- / 176-byte superblocks, 16-byte aligned in the stage):
// run t is sub-block t: the low (t even) or high (t odd) nibbles of
// qs[32(t >> 1) + l], Q5_K's fifth bit being bit t of qh[l].  The lane's runs
// 2c and 2c + 1 share the 32 bytes qs[32c ..] (and qh[0 .. 31]).  Scales:
// the 6-bit (sc, m) of sub-block t from the packed scale bytes, dl = d * sc
// and nml = -(dmin * m), each rounded once; a value is fma(dl, q, nml),
// rounded to fp16 (the K-quant page's value formula, as the run decoders).
__device__ __forceinline__ void k4_run_scales(const uint4 &hd, int t, pair_t &dl2, pair_t &nml2) {
    const int sh = 8 * (t & 3);
    const uint32_t ys = hd.y >> sh, zs = hd.z >> sh, ws = hd.w >> sh;
    const uint32_t sc = t < 4 ? (ys & 63u) : ((ws & 15u) | ((ys >> 6 & 3u) << 4));
    const uint32_t m = t < 4 ? (zs & 63u) : (((ws >> 4) & 15u) | ((zs >> 6 & 3u) << 4));
    const float dl = __fmul_rn(h2f(hd.x), u2f_exact(sc));
    const float nml = -__fmul_rn(h2f(hd.x >> 16), u2f_exact(m));
    dl2 = pk2(dl, dl);
    nml2 = pk2(nml, nml);
}

template <bool Q5>
struct K4Row {
    pair_t dla, nmla, dlb, nmlb;   // runs 2c (a) and 2c + 1 (b)
    uint32_t q[8], h[Q5 ? 8 : 1];

    __device__ __forceinline__ void load(const uint8_t *b, int c) {
        const uint4 hd = Smem::u128(b);
        k4_run_scales(hd, 2 * c, dla, nmla);
        k4_run_scales(hd, 2 * c + 1, dlb, nmlb);
        const uint8_t *qs = b + (Q5 ? 48 : 16) + 32 * c;
        const uint4 q0 = Smem::u128(qs), q1 = Smem::u128(qs + 16);
        q[0] = q0.x; q[1] = q0.y; q[2] = q0.z; q[3] = q0.w;
        q[4] = q1.x; q[5] = q1.y; q[6] = q1.z; q[7] = q1.w;
        if constexpr (Q5) {
            const uint4 h0 = Smem::u128(b + 16), h1 = Smem::u128(b + 32);
            h[0] = h0.x; h[1] = h0.y; h[2] = h0.z; h[3] = h0.w;
            h[4] = h1.x; h[5] = h1.y; h[6] = h1.z; h[7] = h1.w;
        }
    }
    // 4-value quant words of word k for runs a and b
    __device__ __forceinline__ void quants(int k, int c, uint32_t &ua, uint32_t &ub) const {
        ua = q[k] & 0x0F0F0F0Fu;
        ub = (q[k] >> 4) & 0x0F0F0F0Fu;
        if constexpr (Q5) {
            ua |= ((h[k] >> (2 * c)) & 0x01010101u) << 4;
            ub |= ((h[k] >> (2 * c + 1)) & 0x01010101u) << 4;
        }
    }
};

template <bool Q5>
__device__ __forceinline__ void step_k4(const uint8_t *b0, const uint8_t *b1, int c, const uint4 *xv, bool tok,
                                        float (&d)[4], float (&e)[4]) {
    K4Row<Q5> r0, r1;
    r0.load(b0, c);
    r1.load(b1, c);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint4 xa = tok ? __ldg(xv + u) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 xb = tok ? __ldg(xv + 4 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int k = 2 * u + hh;
            uint32_t ua0, ub0, ua1, ub1;
            r0.quants(k, c, ua0, ub0);
            r1.quants(k, c, ua1, ub1);
            const uint2 p0 = word_affine(ua0, r0.dla, r0.nmla), p1 = word_affine(ua1, r1.dla, r1.nmla);
            mma_16816(d, p0.x, p1.x, p0.y, p1.y, hh ? xa.z : xa.x, hh ? xa.w : xa.y);
            const uint2 q0 = word_affine(ub0, r0.dlb, r0.nmlb), q1 = word_affine(ub1, r1.dlb, r1.nmlb);
            mma_16816(e, q0.x, q1.x, q0.y, q1.y, hh ? xb.z : xb.x, hh ? xb.w : xb.y);
        }
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
template <> struct Stage<kQ2_K> { static constexpr int STEP = 84, S = 8, PITCH = 688, NST = 8; };
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
};

// Block b of the launch: its projection, first weight row, steps per row
// and tiles.
struct BlockLoc {
    int grp, m0, nsteps, ntiles;
};

template <int TYPE>
__device__ __forceinline__ BlockLoc block_loc(const GemvParams &gp, int b) {
    int k = 0;
    while (k < gp.n - 1 && b >= gp.g[k].blk_end) ++k;
    const int nsteps = (gp.g[k].in_f + STEP_VALUES - 1) / STEP_VALUES;
    return {k, (b - (k ? gp.g[k - 1].blk_end : 0)) * ROWS, nsteps, (nsteps + Stage<TYPE>::S - 1) / Stage<TYPE>::S};
}

template <int TYPE>
__global__ void __launch_bounds__(GEMV_THREADS, 2) gemv_kernel(const __grid_constant__ GemvParams gp) {
    using G = Geom<TYPE>;
    using S = Stage<TYPE>;
    using Raw = typename RawOf<TYPE>::T;
    constexpr int TILE = tile_bytes<TYPE>();
    constexpr int TEAMS = NC / S::S;                      // tiles in work at once
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ float part[NC][ROWS][8];                   // each consumer warp's 16 weight rows x 8 tokens
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
        for (int k = 0; k < gp.n; ++k)
            if (gp.g[k].use_tma) prefetch_tensormap(&gp.tmW[k]);
        mbar_fence_init();
    }
    __syncthreads();
    grid_dependency_wait();                               // the previous grid's memory operations are done
    grid_launch_dependents();                             // the next grid may launch; it still waits for this one
    const int nblk = gp.g[gp.n - 1].blk_end;

    if (warp == NC) {
        // ------------------------------------------------------------ producer --
        // The CTA's tiles in order: block after block, each block's tiles
        // 0 .. ntiles - 1; tile n goes to slot n % NST.
        int n = 0;
        bool ok = true;
        for (int b = blockIdx.x; ok && b < nblk; b += gridDim.x) {
            const BlockLoc L = block_loc<TYPE>(gp, b);
            const GemvGroup &P = gp.g[L.grp];
            for (int j = 0; j < L.ntiles; ++j, ++n) {
                const int s = n % S::NST;
                if (!wait_phase_warp(&empty[s], ((n / S::NST) & 1) ^ 1u, gp.limit_ns, stop, gp.err,
                                     kErrTimeoutGemv)) {
                    ok = false;
                    break;
                }
                uint8_t *const slot = ring + s * TILE;
                const int64_t off = static_cast<int64_t>(j) * S::S * S::STEP;   // the tile's first byte in a row
                if (P.use_tma) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[s], TILE);
                        tma_load_2d(slot, &gp.tmW[L.grp], &full[s], static_cast<int32_t>((off & ~int64_t(15)) >> 3),
                                    L.m0);
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
                    if (bytes) bulk_load(dst, a0, bytes, &full[s]);
                }
                __syncwarp();
            }
        }
        // the copies issued land before the CTA's shared memory goes
        if (lane == 0) {
            bool drained = true;
            for (int m = n - S::NST < 0 ? 0 : n - S::NST; m < n; ++m)
                drained = wait_drain(&full[m % S::NST], static_cast<uint32_t>((m / S::NST) & 1), gp.limit_ns) &&
                          drained;
            if (!drained) {
                drain_failed = 1u;
                atomicOr(gp.err, kErrTimeoutGemv);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers --
        const int g = lane >> 2, c = lane & 3;
        const int team = warp / S::S, sl = warp % S::S;   // this warp's team and step within a tile
        const int T = gp.T;
        const bool tok = g < T;                           // this lane's B column is a token row
        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f}, e[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        bool live = true;
        int n0 = 0;                                       // the block's first tile in the CTA's sequence
        for (int b = blockIdx.x; b < nblk; b += gridDim.x) {
            const BlockLoc L = block_loc<TYPE>(gp, b);
            const GemvGroup &P = gp.g[L.grp];
            // rows g, g + 8: the row's start modulo 16 (0 when staged by TMA)
            const int base0 = P.use_tma ? 0
                                        : static_cast<int>((reinterpret_cast<uintptr_t>(P.W) +
                                                            static_cast<uint64_t>(L.m0 + g) * P.row_bytes) & 15);
            const int base1 = P.use_tma ? 0
                                        : static_cast<int>((reinterpret_cast<uintptr_t>(P.W) +
                                                            static_cast<uint64_t>(L.m0 + g + 8) * P.row_bytes) & 15);
            const uint16_t *xrow = P.X + static_cast<int64_t>(tok ? g : 0) * P.in_f;
            for (int j = 0; j < L.ntiles; ++j) {
                // Every consumer warp waits for every tile and releases it, also
                // the tiles another team reads: a warp that skipped ring rounds
                // could meet a slot's barrier two phases on, where a parity wait
                // no longer tells the phases apart.
                const int n = n0 + j, s = n % S::NST;
                live = live && wait_phase_warp(&full[s], static_cast<uint32_t>((n / S::NST) & 1), gp.limit_ns, stop,
                                               gp.err, kErrTimeoutGemv);
                if (!live) continue;
                const int q = j * S::S + sl;              // this warp's step of the row
                if (j % TEAMS == team && q < L.nsteps) {
                    const int off = j * S::S * S::STEP;
                    const uint8_t *slot = ring + s * TILE;
                    const uint8_t *src0 = slot + g * S::PITCH + ((base0 + off) & 15) + sl * S::STEP;
                    const uint8_t *src1 = slot + (g + 8) * S::PITCH + ((base1 + off) & 15) + sl * S::STEP;
                    if constexpr (TYPE == kQ2_K) {
                        step_q2k(src0, src1, c, reinterpret_cast<const uint4 *>(xrow + 256 * q + 64 * c), tok, d, e);
                    } else if constexpr (TYPE == kQ6_K) {
                        step_q6k(src0, src1, c, reinterpret_cast<const uint4 *>(xrow + 256 * q + 64 * c), tok, d, e);
                    } else if constexpr (TYPE == kQ4_K || TYPE == kQ5_K) {
                        step_k4<TYPE == kQ5_K>(src0, src1, c, reinterpret_cast<const uint4 *>(xrow + 256 * q + 64 * c),
                                               tok, d, e);
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
                            float (&acc)[4] = rho ? e : d;
#pragma unroll
                            for (int u = 0; u < 4; ++u) {     // 8 values of X per 16-byte load: two MMAs
                                const uint4 x = tok && valid ? __ldg(xv + u) : make_uint4(0u, 0u, 0u, 0u);
                                mma_16816(acc, h0[4 * u], h1[4 * u], h0[4 * u + 1], h1[4 * u + 1], x.x, x.y);
                                mma_16816(acc, h0[4 * u + 2], h1[4 * u + 2], h0[4 * u + 3], h1[4 * u + 3], x.z, x.w);
                            }
                        }
                    }
                }
                __syncwarp();                             // the tile is read before it is released
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            n0 += L.ntiles;
            // block end: D rows g, g + 8 (weight rows), columns 2c, 2c + 1 (tokens)
            part[warp][g][2 * c] = d[0] + e[0];
            part[warp][g][2 * c + 1] = d[1] + e[1];
            part[warp][g + 8][2 * c] = d[2] + e[2];
            part[warp][g + 8][2 * c + 1] = d[3] + e[3];
#pragma unroll
            for (int k = 0; k < 4; ++k) d[k] = e[k] = 0.0f;
            named_barrier_sync(1, NC * 32);
            for (int o = threadIdx.x; o < ROWS * 8; o += NC * 32) {
                const int tt = o / ROWS, r = o % ROWS;    // consecutive threads: consecutive rows of Y
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < NC; ++w) v += part[w][r][tt];
                if (tt < T && L.m0 + r < P.out_f) P.Y[static_cast<int64_t>(tt) * P.out_f + L.m0 + r] = v;
            }
            named_barrier_sync(1, NC * 32);
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
template <int TYPE>
cudaError_t launch_typed(const GemvArgs *a, int n, cudaStream_t stream, const LaunchEnv &env) {
    auto kern = gemv_kernel<TYPE>;
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
