// dequant.cu — block-quantized weight -> dense f32 / f16 (the per-type
// dequantize-to-f32 step of "Qwen3.5 batched prefill has no f32 dequant for
// IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", §Cause; the f16 copy built from it).
//
// HBM-bound.  Each lane decodes one run of 32 consecutive values per step of
// a grid-stride loop: a whole 32-value sub-block of Q4_K, two 16-value
// sub-blocks of Q2_K / Q6_K, or one Q8_0 block, so the per-run work (scale
// unpacking, addresses, loop control) is paid once per 32 values.  A warp
// covers four K-quant superblocks (or 32 Q8_0 blocks) per step and writes each
// lane's run with 16-byte stores.  Block fields are read straight from
// global memory with loads no wider than the block's alignment (Q4_K blocks
// are 16-byte aligned, Q2_K 4-byte, Q6_K and Q8_0 2-byte; 2-byte aligned runs
// are assembled from aligned words).  The (row, block) position of a lane's
// run is divided out once and then stepped.
//
// Arithmetic (qp_decode.cuh): every field is widened exactly and each value
// is one fma / mul with an exact product, i.e. one f32 rounding — the same
// bits as the value formula evaluated with separately rounded f32 operations
// (the CPU oracle).  f16 output is round-to-nearest-even of that f32.
//
// Stores: where the output is a whole number of 32-value runs per row (cols
// a multiple of the block size), a warp step's 32 runs are one contiguous
// stretch of the output; the warp writes them into a shared-memory tile in
// the 128-byte (f32) / 64-byte (f16) swizzled layout of a TMA box of 32 runs
// and one lane stores the tile with a single TMA tensor store.  Otherwise
// the runs go through padded shared memory and leave as 16-byte stores.
//
// Tail guard: a lane writes only columns < cols; the padding values of a
// partial last block are decoded but never stored.
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

namespace qp {
namespace {

using namespace runs;


// ----------------------------------------------------------------- kernel --

// Position of a lane's run: block index, its (row, block-in-row), stepped by
// a grid stride whose (rows, blocks) split was divided out on the host.
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

// Blocks a warp covers per grid-stride step: four superblocks (8 runs each),
// or 32 Q8_0 blocks (one run each) -- 1024 values either way.
template <int TYPE> __host__ __device__ constexpr int blocks_per_warp() { return TYPE == kQ8_0 ? 32 : 4; }

constexpr int WARPS = 8;                                       // per 256-thread block

// Per-warp staging area: 32 runs, each run's bytes padded by 16 so that 16-byte
// accesses of eight consecutive runs fall in eight different bank groups.
template <typename OutT> struct Stage {
    static constexpr int RUN = 32 * static_cast<int>(sizeof(OutT));   // bytes per run
    static constexpr int PITCH = RUN + 16;
    static constexpr int CHUNKS = 32 * RUN / 16;                      // 16-byte chunks per warp step
    static constexpr int PER_RUN = RUN / 16;
};

template <typename OutT>
__device__ __forceinline__ void put_run(uint8_t *stage, int lane, const pair_t (&y)[16]);

// The lane's run as row `lane` of a swizzled TMA box tile: 16-byte chunk k
// of the row at chunk position k ^ (lane % 8) (f32: 128-byte rows) or
// k ^ ((lane / 2) % 4) (f16: 64-byte rows), so the 8 lanes of a store phase
// hit 8 different bank groups.
template <typename OutT>
__device__ __forceinline__ void put_run_swz(uint32_t tile, int lane, const pair_t (&y)[16]);

template <>
__device__ __forceinline__ void put_run_swz<float>(uint32_t tile, int lane, const pair_t (&y)[16]) {
    const uint32_t row = tile + static_cast<uint32_t>(lane * 128);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float a, b, c, d;
        unpk2(y[2 * k], a, b);
        unpk2(y[2 * k + 1], c, d);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(row + static_cast<uint32_t>((k ^ (lane & 7)) << 4)),
                     "f"(a), "f"(b), "f"(c), "f"(d)
                     : "memory");
    }
}

template <>
__device__ __forceinline__ void put_run_swz<uint16_t>(uint32_t tile, int lane, const pair_t (&y)[16]) {
    const uint32_t row = tile + static_cast<uint32_t>(lane * 64);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         row + static_cast<uint32_t>((k ^ ((lane >> 1) & 3)) << 4)),
                     "r"(f2h2(y[4 * k])), "r"(f2h2(y[4 * k + 1])), "r"(f2h2(y[4 * k + 2])), "r"(f2h2(y[4 * k + 3]))
                     : "memory");
}

template <>
__device__ __forceinline__ void put_run<float>(uint8_t *stage, int lane, const pair_t (&y)[16]) {
    uint8_t *p = stage + lane * Stage<float>::PITCH;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float a, b, c, d;
        unpk2(y[2 * k], a, b);
        unpk2(y[2 * k + 1], c, d);
        *reinterpret_cast<float4 *>(p + 16 * k) = make_float4(a, b, c, d);
    }
}

template <>
__device__ __forceinline__ void put_run<uint16_t>(uint8_t *stage, int lane, const pair_t (&y)[16]) {
    uint8_t *p = stage + lane * Stage<uint16_t>::PITCH;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        *reinterpret_cast<uint4 *>(p + 16 * k) =
            make_uint4(f2h2(y[4 * k]), f2h2(y[4 * k + 1]), f2h2(y[4 * k + 2]), f2h2(y[4 * k + 3]));
}

// tmo: the output as [rows * cols / 32 runs x 32 values], box 32 x 32,
// used when use_tma (every run of every row whole: cols a multiple of the
// block size).
// Resident 256-thread CTAs per SM the register budget is cut for: three
// (80 registers a thread) keeps the most bytes in flight -- measured against
// two (the register use left alone) and four (heavy spills): Q4_K 4096^2 ->
// f32 69% -> 73% of HBM.  Q5_K and Q6_K, whose runs carry the most raw
// bytes, spill at 80 registers and keep two (Q6_K 4096 x 12288 -> f32: 84%
// at two, 75% at three).
template <int TYPE> struct MinBlocks { static constexpr int N = 3; };
template <> struct MinBlocks<kQ5_K> { static constexpr int N = 2; };
template <> struct MinBlocks<kQ6_K> { static constexpr int N = 2; };

template <int TYPE, typename OutT>
__global__ void __launch_bounds__(256, MinBlocks<TYPE>::N) dequant_kernel(const uint8_t *__restrict__ blocks, int64_t cols, int64_t nb,
                                                      int64_t nblocks, int64_t drow, int64_t dkb,
                                                      OutT *__restrict__ out, const __grid_constant__ CUtensorMap tmo,
                                                      int use_tma) {
    using S = Stage<OutT>;
    using Raw = typename RawOf<TYPE>::T;
    constexpr int QK = TYPE == kQ8_0 ? 32 : 256;
    constexpr int BB =
        TYPE == kQ8_0 ? 34 : (TYPE == kQ4_K ? 144 : (TYPE == kQ5_K ? 176 : (TYPE == kQ2_K ? 84 : 210)));
    constexpr int BPW = blocks_per_warp<TYPE>();
    constexpr int RUNS_PER_BLOCK = 32 / BPW;                  // 8 (K-quants) or 1 (Q8_0)
    // padded staging (32 runs x PITCH per warp), or two TMA box tiles per warp
    constexpr int STAGE_BYTES = WARPS * 32 * S::PITCH > WARPS * 64 * S::RUN ? WARPS * 32 * S::PITCH : WARPS * 64 * S::RUN;
    __shared__ __align__(16) uint8_t stage_all[STAGE_BYTES + 1024];
    const int lane = threadIdx.x & 31;
    uint8_t *const base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(stage_all) + 1023) & ~uintptr_t(1023));
    uint8_t *stage = base + (threadIdx.x >> 5) * 32 * S::PITCH;
    // TMA box tiles of this warp: 2 x 32 runs x RUN bytes, aligned to the swizzle span
    const uint32_t tiles = smem_u32(base) + static_cast<uint32_t>((threadIdx.x >> 5) * 64 * S::RUN);
    uint32_t nst = 0;                                     // TMA stores this warp has issued
    const int64_t warps = static_cast<int64_t>(gridDim.x) * WARPS;
    const int64_t w0 = static_cast<int64_t>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
    const int t = TYPE == kQ8_0 ? 0 : (lane & 7);             // run within the superblock
    Cursor c;
    c.blk = w0 * BPW + lane / RUNS_PER_BLOCK;
    c.row = c.blk / nb;
    c.kb = c.blk - c.row * nb;
    const int64_t dblk = warps * BPW;
    const bool vec_ok = (cols & (16 / sizeof(OutT) - 1)) == 0;  // output rows keep 16-byte alignment
    Raw raw;
    if (c.blk < nblocks) raw.load(blocks + c.blk * BB, t);
    while (__any_sync(0xffffffffu, c.blk < nblocks)) {
        Cursor n = c;
        n.step(dblk, drow, dkb, nb);
        Raw next;
        if (n.blk < nblocks) next.load(blocks + n.blk * BB, t);   // in flight while this step decodes
        const bool valid = c.blk < nblocks;
        pair_t y[16];
        if (valid) raw.decode(t, y);
        const int64_t col0 = c.kb * QK + 32 * t;
        // Coalesced path: every run of the warp is whole and inside its row, and
        // the runs of each 512-byte output piece are contiguous in memory.
        bool whole = valid && vec_ok && col0 + 32 <= cols;
        if constexpr (TYPE == kQ8_0) {
            // every lane takes part in the shuffle (it must not sit behind a
            // short-circuit): all 32 blocks in one row, consecutive
            const int64_t kb_first = __shfl_sync(0xffffffffu, c.kb, 0);
            whole = whole && (c.kb - lane == kb_first);
        }
        if (use_tma && __all_sync(0xffffffffu, whole)) {
            // the warp's 32 runs are runs first .. first + 31 of the output
            const int64_t first = __shfl_sync(0xffffffffu, c.blk, 0) * RUNS_PER_BLOCK;
            const uint32_t tile = tiles + (nst & 1u) * 32u * S::RUN;
            if (lane == 0) bulk_wait_group_read<1>();     // the tile's previous store has read it
            __syncwarp();
            put_run_swz<OutT>(tile, lane, y);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&tmo, tile, 0, static_cast<int32_t>(first));
                bulk_commit_group();
            }
            ++nst;
        } else if (__all_sync(0xffffffffu, whole)) {
            put_run<OutT>(stage, lane, y);
            __syncwarp();
            // piece k of the warp step: 32 chunks = 512 bytes, all from one block
            // run group (K-quants: superblock (k*32)/(8*PER_RUN); Q8_0: one row)
#pragma unroll
            for (int k = 0; k < S::CHUNKS / 32; ++k) {
                const int chunk = 32 * k + lane;
                const int run = chunk / S::PER_RUN;
                const int within = chunk % S::PER_RUN;
                const uint4 v = *reinterpret_cast<const uint4 *>(stage + run * S::PITCH + 16 * within);
                const int src = TYPE == kQ8_0 ? 0 : (run & ~7);    // a lane holding that run's block cursor
                const int64_t row = __shfl_sync(0xffffffffu, c.row, src);
                const int64_t kb0 = __shfl_sync(0xffffffffu, c.kb, src);
                const int64_t col = kb0 * QK + (TYPE == kQ8_0 ? 32 * run : 32 * (run & 7));
                __stcs(reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(out + row * cols + col) + 16 * within),
                       v);
            }
            __syncwarp();
        } else if (valid && col0 < cols) {
            // Guarded per-lane path (partial blocks, unaligned rows, row ends).
            OutT *p = out + c.row * cols + col0;
            if constexpr (sizeof(OutT) == 4) {
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float a, b;
                    unpk2(y[k], a, b);
                    if (col0 + 2 * k < cols) p[2 * k] = a;
                    if (col0 + 2 * k + 1 < cols) p[2 * k + 1] = b;
                }
            } else {
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const uint32_t h = f2h2(y[k]);
                    if (col0 + 2 * k < cols) p[2 * k] = static_cast<uint16_t>(h);
                    if (col0 + 2 * k + 1 < cols) p[2 * k + 1] = static_cast<uint16_t>(h >> 16);
                }
            }
        }
        raw = next;
        c = n;
    }
    if (use_tma && lane == 0) bulk_wait_all();            // the stores are complete before the CTA exits
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The output as [rows * cols / 32 runs x 32 values] for TMA stores of 32-run
// boxes, when every row is a whole number of blocks (so that a warp step's
// runs are contiguous) and the run index fits the 32-bit coordinate.
template <int TYPE, typename OutT>
bool encode_out(void *encode_fn, int64_t rows, int64_t cols, OutT *out, CUtensorMap *map) {
    const int64_t qk = TYPE == kQ8_0 ? 32 : 256;
    if (!encode_fn || cols % qk != 0 || (reinterpret_cast<uintptr_t>(out) & 15u) != 0) return false;
    const int64_t runs = rows * cols / 32;
    if (runs > INT32_MAX) return false;
    const cuuint64_t dims[2] = {32, static_cast<cuuint64_t>(runs)};
    const cuuint64_t strides[1] = {32 * sizeof(OutT)};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    const bool f32 = sizeof(OutT) == 4;
    return reinterpret_cast<EncodeFn>(encode_fn)(
               map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, out, dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TYPE, typename OutT>
cudaError_t launch(const void *blocks, int64_t rows, int64_t cols, OutT *out, cudaStream_t stream, int num_sms,
                   void *encode_fn) {
    const int64_t qk = TYPE == kQ8_0 ? 32 : 256;
    const int64_t nb = (cols + qk - 1) / qk;
    const int64_t nblocks = rows * nb;
    const int64_t nwarps = (nblocks + blocks_per_warp<TYPE>() - 1) / blocks_per_warp<TYPE>();
    // one resident wave of 256-thread blocks at most
    static std::atomic<int> cached{0};                 // queried once per kernel, then cached
    int per_sm = cached.load();
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dequant_kernel<TYPE, OutT>, 256, 0) !=
                cudaSuccess ||
            per_sm < 1) {
            cudaGetLastError();
            per_sm = 1;
        }
        cached.store(per_sm);
    }
    const int64_t want = (nwarps + WARPS - 1) / WARPS;
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
    const int64_t dblk = static_cast<int64_t>(grid) * WARPS * blocks_per_warp<TYPE>();
    CUtensorMap tmo;
    const bool use_tma = encode_out<TYPE, OutT>(encode_fn, rows, cols, out, &tmo);
    if (!use_tma) memset(&tmo, 0, sizeof(tmo));
    dequant_kernel<TYPE, OutT><<<grid, 256, 0, stream>>>(static_cast<const uint8_t *>(blocks), cols, nb, nblocks,
                                                         dblk / nb, dblk % nb, out, tmo, use_tma ? 1 : 0);
    return cudaGetLastError();
}

// F16 weights: each "block" is one fp16 value and rows carry no padding, so
// the input and the output hold the same n values in the same order: a flat
// conversion (exact widening to f32) or copy (f16), 8 values = one 16-byte
// load per thread and step; a last partial group of 8 is done value by value.
template <typename OutT>
__global__ void __launch_bounds__(256) f16_weights_kernel(const uint16_t *__restrict__ in, int64_t n,
                                                          OutT *__restrict__ out) {
    const int64_t n8 = n / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(in) + i);
        if constexpr (sizeof(OutT) == 4) {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            float f[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                f[2 * k] = h2f(w[k]);
                f[2 * k + 1] = h2f(w[k] >> 16);
            }
            float4 *o = reinterpret_cast<float4 *>(out) + 2 * i;
            __stcs(o, make_float4(f[0], f[1], f[2], f[3]));
            __stcs(o + 1, make_float4(f[4], f[5], f[6], f[7]));
        } else {
            __stcs(reinterpret_cast<uint4 *>(out) + i, v);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < n - 8 * n8) {
        const int64_t j = 8 * n8 + threadIdx.x;
        if constexpr (sizeof(OutT) == 4) out[j] = h2f(in[j]);
        else out[j] = in[j];
    }
}

template <typename OutT>
cudaError_t launch_f16(const uint16_t *in, int64_t n, OutT *out, cudaStream_t stream, int num_sms) {
    const int64_t want = (n / 8 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
    f16_weights_kernel<OutT><<<grid, 256, 0, stream>>>(in, n, out);
    return cudaGetLastError();
}

template <typename OutT>
cudaError_t dispatch(int type, const void *blocks, int64_t rows, int64_t cols, OutT *out, cudaStream_t stream,
                     int num_sms, void *enc) {
    switch (type) {
    case kQ8_0: return launch<kQ8_0>(blocks, rows, cols, out, stream, num_sms, enc);
    case kQ2_K: return launch<kQ2_K>(blocks, rows, cols, out, stream, num_sms, enc);
    case kQ4_K: return launch<kQ4_K>(blocks, rows, cols, out, stream, num_sms, enc);
    case kQ5_K: return launch<kQ5_K>(blocks, rows, cols, out, stream, num_sms, enc);
    case kQ6_K: return launch<kQ6_K>(blocks, rows, cols, out, stream, num_sms, enc);
    case kF16: return launch_f16(static_cast<const uint16_t *>(blocks), rows * cols, out, stream, num_sms);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_dequant_f32(int type, const void *blocks, int64_t rows, int64_t cols, float *out,
                               cudaStream_t stream, int num_sms, void *encode_fn) {
    return dispatch(type, blocks, rows, cols, out, stream, num_sms, encode_fn);
}

cudaError_t launch_dequant_f16(int type, const void *blocks, int64_t rows, int64_t cols, uint16_t *out,
                               cudaStream_t stream, int num_sms, void *encode_fn) {
    return dispatch(type, blocks, rows, cols, out, stream, num_sms, encode_fn);
}

}  // namespace qp
