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
// the ALUs on a budget of a few instructions per weight value: they only
// decode, and the dot products run on the tensor cores with the warp-level
// mma.sync m16n8k16, whose cost per value does not depend on T.  The MMA's
// A operand is the token rows (16 rows, of which rows >= T and all of rows
// 8..15 are zeros), B is 8 weight rows x 16 K values in fp16, D = f32.
//
// A CTA owns 8 weight rows at a time; its NW warps split the rows' steps of
// 8 runs (one K-quant superblock, or 8 Q8_0 / F16 blocks).  Each warp stages
// its steps' bytes -- 8 rows x one step, copied as the 16-byte aligned span
// that covers it, so that every byte keeps its alignment modulo 16 -- into a
// private ring of NST shared-memory slots with coalesced 16-byte cp.async
// copies issued NST - 1 steps ahead; the ring runs on from one 8-row block
// into the CTA's next.  In a step, lane (g, c) (g = lane / 4, c = lane % 4)
// decodes runs 2c and 2c + 1 of the step in weight row g from the slot with
// the exact run decoders (qp_runs.cuh), rounds them to fp16 and feeds each
// run's 32 values to eight MMAs, four per MMA.  The MMA's K order is
// permuted: K slots 2c, 2c + 1, 2c + 8, 2c + 9 hold values 4i .. 4i + 3 of
// lane c's run in MMA i, for A and B alike, so the sum over K is unchanged,
// each lane's B fragment is its own decoded values and its A fragment is 4
// consecutive values of token row g of X.  Runs past the row's end
// contribute zeros.  The warps' 8 x 8 partial tiles are summed through
// shared memory in warp order, so results are deterministic.
#include <atomic>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qp_decode.cuh"
#include "qp_internal.h"
#include "qp_runs.cuh"

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

// Q2_K straight to fp16: per 16-value sub-block, the four possible fp16
// weights (q2k_tables: the same one-rounding f32 arithmetic, then the same
// fp16 rounding), held byte-planar in two words; each value's 2-bit q then
// selects its two bytes with byte permutes.
template <>
__device__ __forceinline__ void run_f16<kQ2_K>(const RawQ2K &raw, int t, uint32_t (&h)[16]) {
    uint32_t plo[2], phi[2];
    q2k_tables(raw.sb >> (16 * (t & 1)), h2f(raw.dd), h2f(raw.dd >> 16), plo, phi);   // scales[2t], scales[2t+1]
    const int sh = 2 * (t & 3);
#pragma unroll
    for (int i = 0; i < 8; ++i) {                        // values 4i .. 4i + 3, sub-block i / 4
        const uint32_t sel = ((raw.w[i] >> sh) & 0x03030303u) * 0x11u + 0x40404040u;   // q -> nibbles q, q + 4
        h[2 * i] = __byte_perm(plo[i >> 2], phi[i >> 2], sel);
        h[2 * i + 1] = __byte_perm(plo[i >> 2], phi[i >> 2], sel >> 16);
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

#ifndef QP_GEMV_MINB
#define QP_GEMV_MINB 3        // resident CTAs per SM the register budget is cut for
#endif

// A step's bytes per row (STEP), the staged row pitch (an odd multiple of 16
// bytes, at least the widest 16-byte aligned cover of a step, so that the
// eight rows' 16-byte loads of a load phase hit eight bank groups) and the
// ring depth (steps in flight, scaled to keep a few KB per warp in flight).
template <int TYPE> struct Stage;
template <> struct Stage<kQ4_K> { static constexpr int STEP = 144, PITCH = 144, NST = 4; };
template <> struct Stage<kQ5_K> { static constexpr int STEP = 176, PITCH = 176, NST = 4; };
template <> struct Stage<kQ2_K> { static constexpr int STEP = 84, PITCH = 112, NST = 5; };
template <> struct Stage<kQ6_K> { static constexpr int STEP = 210, PITCH = 240, NST = 3; };
template <> struct Stage<kQ8_0> { static constexpr int STEP = 272, PITCH = 304, NST = 3; };
template <> struct Stage<kF16> { static constexpr int STEP = 512, PITCH = 528, NST = 2; };

template <int TYPE, int NW> constexpr int gemv_smem() { return NW * Stage<TYPE>::NST * 8 * Stage<TYPE>::PITCH; }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// A launch runs up to kMaxGroup projections of one type over the same T
// token rows.  Their 8-row blocks are numbered projection after projection;
// CTA b takes blocks b, b + gridDim.x, ...  A block's sums do not depend on
// which CTA computes it or what shares the launch.
struct GemvGroup {
    const uint8_t *W;
    const uint16_t *X;
    float *Y;
    int64_t row_bytes;
    int out_f, in_f, blk_end;      // blk_end: one past the projection's last block
};
struct GemvParams {
    GemvGroup g[kMaxGroup];
    int n, T;
};

template <int TYPE, int NW>
__global__ void __launch_bounds__(NW * 32, QP_GEMV_MINB) gemv_kernel(const __grid_constant__ GemvParams gp) {
    using G = Geom<TYPE>;
    using S = Stage<TYPE>;
    using Raw = typename RawOf<TYPE>::T;
    extern __shared__ __align__(16) uint8_t ring_all[];
    __shared__ float part[NW][8][8];                      // each warp's 8 weight rows x 8 tokens
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    uint8_t *ring = ring_all + warp * (S::NST * 8 * S::PITCH);
    const int T = gp.T, nblk = gp.g[gp.n - 1].blk_end;
    const bool tok = g < T;                               // this lane's A row is a token row
    // A cursor over this warp's items (block, step): the warp takes steps
    // warp, warp + NW, ... of each block's rows, spw of them for every warp
    // (spw = the projection's steps per row / NW, rounded up), in block order.
    struct Cur {
        int b, i;                                         // block, item within the block
        int grp, m0, nsteps, spw;
    };
    auto locate = [&](Cur &u) {
        int k = 0;
        while (k < gp.n - 1 && u.b >= gp.g[k].blk_end) ++k;
        u.grp = k;
        u.m0 = (u.b - (k ? gp.g[k - 1].blk_end : 0)) * 8;
        u.nsteps = (gp.g[k].in_f / 32 + 7) / 8;
        u.spw = (u.nsteps + NW - 1) / NW;
    };
    auto advance = [&](Cur &u) {
        if (++u.i == u.spw) {
            u.i = 0;
            u.b += gridDim.x;
            if (u.b < nblk) locate(u);
        }
    };
    // Stage the producer cursor's item into slot `slot_i`: lane (g, c)
    // copies 16-byte vectors c, c + 4, ... of row g's cover [start & ~15,
    // end) of the step (a copy that would pass the end of W -- only the
    // last row's last step can -- is done 2 bytes at a time instead).
    auto stage = [&](const Cur &u, int slot_i) {
        const int q = u.i * NW + warp;
        if (u.b < nblk && q < u.nsteps) {
            const GemvGroup &P = gp.g[u.grp];
            const int row = min(u.m0 + g, P.out_f - 1);   // rows past out_f: a copy of the last row
            const uint8_t *start = P.W + static_cast<int64_t>(row) * P.row_bytes + static_cast<int64_t>(q) * S::STEP;
            const uint8_t *a0 = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(start) & ~uintptr_t(15));
            const int64_t left = P.row_bytes - static_cast<int64_t>(q) * S::STEP;   // bytes of the row from start
            const int nbytes = static_cast<int>((left < S::STEP ? left : S::STEP) + (start - a0));
            const uint32_t dst0 = static_cast<uint32_t>(__cvta_generic_to_shared(ring)) +
                                  static_cast<uint32_t>((slot_i * 8 + g) * S::PITCH);
            const bool last_row = row == P.out_f - 1;
#pragma unroll
            for (int k = c; k < S::PITCH / 16; k += 4) {
                if (16 * k >= nbytes) break;
                const uint8_t *src = a0 + 16 * k;
                const uint32_t dst = dst0 + static_cast<uint32_t>(16 * k);
                if (!last_row || 16 * (k + 1) <= nbytes) {
                    cp_async16(dst, src);
                } else {                                  // the tail of W: whole 2-byte units only
                    for (int o = 0; 16 * k + o < nbytes; o += 2)
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(dst + static_cast<uint32_t>(o)),
                                     "h"(__ldg(reinterpret_cast<const unsigned short *>(src + o))));
                }
            }
        }
        cp_async_commit();
    };
    Cur cons{static_cast<int>(blockIdx.x), 0, 0, 0, 0, 0};
    if (cons.b >= nblk) return;
    locate(cons);
    Cur prod = cons;
#pragma unroll 1
    for (int p = 0; p < S::NST - 1; ++p) {
        stage(prod, p);
        advance(prod);
    }
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int n = 0; cons.b < nblk; ++n) {
        stage(prod, (n + S::NST - 1) % S::NST);           // refills the slot read in the previous item
        advance(prod);
        cp_async_wait<S::NST - 1>();                      // this lane's copies of item n have landed
        __syncwarp();                                     // ... and every lane's
        const GemvGroup &P = gp.g[cons.grp];
        const int q = cons.i * NW + warp;
        const int nruns = P.in_f / 32;
        const int row = min(cons.m0 + g, P.out_f - 1);
        const uint8_t *start = P.W + static_cast<int64_t>(row) * P.row_bytes + static_cast<int64_t>(q) * S::STEP;
        const uint8_t *srow = ring + (n % S::NST) * 8 * S::PITCH + g * S::PITCH +
                              (reinterpret_cast<uintptr_t>(start) & 15);
        const uint16_t *xrow = P.X + static_cast<int64_t>(tok ? g : 0) * P.in_f;
#pragma unroll
        for (int rho = 0; rho < 2; ++rho) {
            const int j = 8 * q + 2 * c + rho;            // this lane's run of the row
            const bool valid = q < cons.nsteps && j < nruns;
            uint32_t h[16];
            if (valid) {
                Raw raw;
                raw.template load<Smem>(srow + ((2 * c + rho) / G::RPB) * G::BB, j % G::RPB);
                run_f16<TYPE>(raw, j % G::RPB, h);
            } else {
#pragma unroll
                for (int p = 0; p < 16; ++p) h[p] = 0u;
            }
            const uint4 *xv = reinterpret_cast<const uint4 *>(xrow + 32 * j);
#pragma unroll
            for (int u = 0; u < 4; ++u) {                 // 8 values of X per 16-byte load: two MMAs
                const uint4 x = tok && valid ? __ldg(xv + u) : make_uint4(0u, 0u, 0u, 0u);
                mma_16816(d, x.x, 0u, x.y, 0u, h[4 * u], h[4 * u + 1]);
                mma_16816(d, x.z, 0u, x.w, 0u, h[4 * u + 2], h[4 * u + 3]);
            }
        }
        __syncwarp();                                     // the slot is read before it is refilled
        if (cons.i == cons.spw - 1) {                     // the block's last item (the same n in every warp)
            // D rows 0..7 = tokens g, columns 2c, 2c + 1 = weight rows; rows 8..15 are zero
            part[warp][2 * c][g] = d[0];
            part[warp][2 * c + 1][g] = d[1];
            d[0] = d[1] = d[2] = d[3] = 0.0f;
            __syncthreads();
            for (int o = threadIdx.x; o < 64; o += NW * 32) {
                const int t = o >> 3, r = o & 7;          // consecutive threads: consecutive rows of Y
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < NW; ++w) v += part[w][r][t];
                if (t < T && cons.m0 + r < P.out_f) P.Y[static_cast<int64_t>(t) * P.out_f + cons.m0 + r] = v;
            }
            __syncthreads();
        }
        advance(cons);
    }
    cp_async_wait<0>();                                   // no copy outlives the kernel
}

#ifndef QP_GEMV_NW
#define QP_GEMV_NW 8          // warps per CTA (split of each 8-row block's steps)
#endif

// Persistent grid: as many CTAs as fit at once (queried once per
// instantiation: the decode GEMVs are microsecond kernels), at most one per
// 8-row block; each CTA's ring runs on from one block into its next, across
// the projections of the launch.
template <int TYPE, int NW>
cudaError_t launch_nw(const GemvArgs *a, int n, cudaStream_t stream, int device, int num_sms) {
    auto kern = gemv_kernel<TYPE, NW>;
    constexpr int smem = gemv_smem<TYPE, NW>();
    // the shared-memory opt-in and the occupancy query hold for one device:
    // done once per device and instantiation
    static std::atomic<int> per_sm[kMaxDevices];
    int k = per_sm[device].load();
    if (k == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, kern, NW * 32, smem) != cudaSuccess || k < 1) {
            cudaGetLastError();
            k = 1;
        }
        per_sm[device].store(k);
    }
    GemvParams gp;
    int64_t blocks = 0;
    for (int i = 0; i < n; ++i) {
        blocks += (a[i].out_f + 7) / 8;
        if (blocks > INT32_MAX) return cudaErrorInvalidValue;
        gp.g[i] = GemvGroup{static_cast<const uint8_t *>(a[i].W), a[i].X, a[i].Y, a[i].row_bytes,
                            static_cast<int>(a[i].out_f), static_cast<int>(a[i].in_f), static_cast<int>(blocks)};
    }
    gp.n = n;
    gp.T = static_cast<int>(a[0].T);
    const int64_t cap = static_cast<int64_t>(num_sms) * k;
    kern<<<static_cast<unsigned>(blocks < cap ? blocks : cap), NW * 32, smem, stream>>>(gp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_gemv(int type, const GemvArgs *a, int n, cudaStream_t stream, int device, int num_sms) {
    if (n < 1 || n > kMaxGroup) return cudaErrorInvalidValue;
    switch (type) {
    case kQ8_0: return launch_nw<kQ8_0, QP_GEMV_NW>(a, n, stream, device, num_sms);
    case kQ2_K: return launch_nw<kQ2_K, QP_GEMV_NW>(a, n, stream, device, num_sms);
    case kQ4_K: return launch_nw<kQ4_K, QP_GEMV_NW>(a, n, stream, device, num_sms);
    case kQ5_K: return launch_nw<kQ5_K, QP_GEMV_NW>(a, n, stream, device, num_sms);
    case kQ6_K: return launch_nw<kQ6_K, QP_GEMV_NW>(a, n, stream, device, num_sms);
    case kF16: return launch_nw<kF16, QP_GEMV_NW>(a, n, stream, device, num_sms);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qp
