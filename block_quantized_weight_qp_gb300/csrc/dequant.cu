// dequant.cu — block-quantized weight -> dense f32 / f16 (the per-type
// dequantize-to-f32 step of "Qwen3.5 batched prefill has no f32 dequant for
// IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", §Cause; the f16 copy built from it).
//
// HBM-bound, and short: a 4096 x 4096 weight is read in a few microseconds,
// so what limits it is how many bytes are in flight, not the decode.  One
// persistent CTA per SM takes one contiguous stretch of the block array (the
// stretches differ by at most one alignment unit of 1024 values, so the SMs
// finish together).  A producer warp streams the stretch into a ring of
// shared-memory stages with bulk copies (cp.async.bulk, completing on the
// stage's mbarrier) as far ahead as the ring allows (90-160 KB of stages per
// SM), so that HBM sees the whole stretch requested from the first
// microsecond on.  Sixteen decode warps each take one
// "warp step" of every stage: 32 runs of 32 consecutive values (four K-quant
// superblocks, 32 Q8_0 blocks, or 1024 F16 values), one run per lane, decoded
// from shared memory by the exact run decoders of qp_runs.cuh.
//
// Arithmetic (qp_decode.cuh): every field is widened exactly and each value
// is one fma / mul with an exact product, i.e. one f32 rounding -- the same
// bits as the value formula evaluated with separately rounded f32 operations
// (the CPU oracle).  f16 output is round-to-nearest-even of that f32.
//
// Stores: where every output row is a whole number of blocks, a warp step's
// 32 runs are one contiguous stretch of the output; the warp writes them into
// a shared-memory tile in the 128-byte (f32) / 64-byte (f16) swizzled layout
// of a 32-run TMA box and one lane stores the tile with a TMA tensor store
// (two tiles per warp, recycled once their store has read them).  Rows with a
// partial last block take a guarded per-lane store path.
//
// Tail guard: a lane writes only columns < cols; the padding values of a
// partial last block are decoded but never stored.
//
// Launched with programmatic stream serialization: the CTAs of a launch may
// be scheduled while the previous kernel in the stream drains, and wait for
// it (griddepcontrol.wait) before they touch global memory.
//
// Every wait is bounded; on expiry the kernel records an error bit, stops,
// waits for the copies it issued, and returns.
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

// Per type: bytes per block (BB), 32-value runs per block (RPB), values per
// block (QK) and warp steps per unit of the split between CTAs (ALIGN: the
// smallest number of steps whose bytes are a multiple of 16, so that every
// stretch and stage starts 16-byte aligned).  F16 weights are taken as
// blocks of one run of 32 fp16 values.
template <int TYPE> struct RFmt;
template <> struct RFmt<kQ4_K> { static constexpr int BB = 144, RPB = 8, QK = 256, ALIGN = 1; };
template <> struct RFmt<kQ5_K> { static constexpr int BB = 176, RPB = 8, QK = 256, ALIGN = 1; };
template <> struct RFmt<kQ2_K> { static constexpr int BB = 84, RPB = 8, QK = 256, ALIGN = 1; };
template <> struct RFmt<kQ6_K> { static constexpr int BB = 210, RPB = 8, QK = 256, ALIGN = 2; };
template <> struct RFmt<kQ8_0> { static constexpr int BB = 34, RPB = 1, QK = 32, ALIGN = 1; };
template <> struct RFmt<kF16> { static constexpr int BB = 64, RPB = 1, ALIGN = 1; };

constexpr int RD_WARPS = 16;                        // decode warps per CTA
constexpr int RD_THREADS = (RD_WARPS + 1) * 32;     // + the producer warp
constexpr int SMEM_CAP = 232448;                    // shared memory a CTA may opt in to

// Shared memory: the decode warps' output tiles (two 32-run boxes each,
// 1024-byte aligned for the swizzle), the ring of ST stages of one chunk
// (RD_WARPS warp steps) each, the stage barriers and two flags.  The ring
// takes what the tiles leave (at most 16 stages): 90-100 KB per SM with f32
// output, up to 160 KB with f16, so that a 4096 x 4096 weight's share of an
// SM is in flight at once.
template <int TYPE, typename OutT> struct RLayout {
    using F = RFmt<TYPE>;
    static constexpr int BPS = 32 / F::RPB;                     // blocks per warp step
    static constexpr int STEP_BYTES = BPS * F::BB;
    static constexpr int CHUNK_BYTES = RD_WARPS * STEP_BYTES;
    static constexpr int RUN = 32 * static_cast<int>(sizeof(OutT));
    static constexpr int TILE = 32 * RUN;
    static constexpr int OFF_RING = RD_WARPS * 2 * TILE;
    static constexpr int ST_FIT = (SMEM_CAP - 1024 - 16 - OFF_RING) / (CHUNK_BYTES + 16);
    static constexpr int ST = ST_FIT < 16 ? ST_FIT : 16;
    static constexpr int OFF_BAR = OFF_RING + ST * CHUNK_BYTES;
    static constexpr int OFF_FLAG = OFF_BAR + 2 * ST * 8;
    static constexpr int SMEM = OFF_FLAG + 16 + 1024;
    static_assert(ST >= 2, "at least two ring stages");
    static_assert((F::ALIGN * STEP_BYTES) % 16 == 0 && CHUNK_BYTES % 16 == 0, "stages start 16-byte aligned");
    static_assert(SMEM <= SMEM_CAP, "shared memory per CTA");
};

struct RingArgs {
    const uint8_t *blocks;
    int64_t nblocks;      // blocks of the tensor (F16: runs of 32 values, the last maybe partial)
    int64_t in_bytes;     // bytes of the block array
    int64_t steps;        // warp steps, ceil(nblocks / BPS)
    int64_t units;        // split units, ceil(steps / ALIGN)
    int64_t cols, nb;     // output row length, blocks per row (guarded path)
    int64_t nvals;        // rows * cols
    void *out;
    uint32_t *err;
    uint64_t limit_ns;
    int use_tma;          // a warp step's 32 runs are one contiguous box of the output
};

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

// Values p0 .. p0 + n - 1 (n <= 32) of a decoded run to out[i0 ..].
template <typename OutT>
__device__ __forceinline__ void put_run_guarded(OutT *out, int64_t i0, int n, const pair_t (&y)[16]) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        if constexpr (sizeof(OutT) == 4) {
            float a, b;
            unpk2(y[k], a, b);
            if (2 * k < n) out[i0 + 2 * k] = a;
            if (2 * k + 1 < n) out[i0 + 2 * k + 1] = b;
        } else {
            const uint32_t h = f2h2(y[k]);
            if (2 * k < n) out[i0 + 2 * k] = static_cast<uint16_t>(h);
            if (2 * k + 1 < n) out[i0 + 2 * k + 1] = static_cast<uint16_t>(h >> 16);
        }
    }
}

template <int TYPE, typename OutT>
__global__ void __launch_bounds__(RD_THREADS, 1)
    ring_dequant_kernel(const __grid_constant__ RingArgs a, const __grid_constant__ CUtensorMap tmo) {
    using F = RFmt<TYPE>;
    using L = RLayout<TYPE, OutT>;
    using Raw = typename RawOf<TYPE>::T;
    constexpr int BPS = L::BPS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR), *empty = full + L::ST;
    const Stop stop{reinterpret_cast<volatile uint32_t *>(smem + L::OFF_FLAG), 0u};
    volatile uint32_t *const drain_failed = reinterpret_cast<volatile uint32_t *>(smem + L::OFF_FLAG + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::ST; ++s) {
            mbar_init(&full[s], 1);           // the producer's arrive + the copy's bytes
            mbar_init(&empty[s], RD_WARPS);   // every decode warp
        }
        *stop.flag = 0u;
        *drain_failed = 0u;
        mbar_fence_init();
        if (a.use_tma) prefetch_tensormap(&tmo);
    }
    __syncthreads();
    grid_dependency_wait();                   // the previous grid's memory operations are done

    // this CTA's warp steps [s0, s1), in chunks of RD_WARPS steps
    const int64_t u0 = static_cast<int64_t>(blockIdx.x) * a.units / gridDim.x;
    const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * a.units / gridDim.x;
    const int64_t s0 = u0 * F::ALIGN;
    const int64_t s1 = u1 * F::ALIGN < a.steps ? u1 * F::ALIGN : a.steps;
    const int nchunks = s1 > s0 ? static_cast<int>((s1 - s0 + RD_WARPS - 1) / RD_WARPS) : 0;
    uint8_t *const ring = smem + L::OFF_RING;

    if (warp == RD_WARPS) {
        // ------------------------------------------------------------ producer --
        if (lane == 0) {
            int stage = 0, armed = 0;
            uint32_t phase = 0;
            for (int i = 0; i < nchunks; ++i) {
                if (!wait_phase_sleepy(&empty[stage], phase ^ 1u, 256, a.limit_ns, stop, a.err, kErrTimeoutRing))
                    break;
                const int64_t c0 = s0 + static_cast<int64_t>(i) * RD_WARPS;
                const int64_t c1 = c0 + RD_WARPS < s1 ? c0 + RD_WARPS : s1;
                const int64_t off = c0 * BPS * F::BB;
                const int64_t end = c1 * BPS * F::BB < a.in_bytes ? c1 * BPS * F::BB : a.in_bytes;
                const uint32_t bytes = static_cast<uint32_t>(end - off), b16 = bytes & ~15u;
                uint8_t *dst = ring + stage * L::CHUNK_BYTES;
                // the block array's last bytes past a multiple of 16 (only the
                // tensor's last chunk has them): plain loads, published by the
                // arrive below
                for (uint32_t k = b16; k < bytes; ++k) dst[k] = a.blocks[off + k];
                mbar_arrive_expect_tx(&full[stage], b16);
                if (b16) bulk_load(dst, a.blocks + off, b16, &full[stage]);
                ++armed;
                advance(stage, phase, L::ST);
            }
            grid_launch_dependents();
            if (!drain_ring(full, L::ST, armed, -1, a.limit_ns)) {
                *drain_failed = 1u;
                atomicOr(a.err, kErrTimeoutRing);
            }
        }
    } else {
        // -------------------------------------------------------------- decode --
        OutT *const out = static_cast<OutT *>(a.out);
        const uint32_t tiles = smem_u32(smem) + static_cast<uint32_t>(warp * 2 * L::TILE);
        const int j = lane / F::RPB;                            // block of the warp step
        const int t = F::RPB == 1 ? 0 : (lane % F::RPB);         // run within the block
        int stage = 0;
        uint32_t phase = 0, nst = 0;
        for (int i = 0; i < nchunks; ++i) {
            if (!wait_phase_warp(&full[stage], phase, a.limit_ns, stop, a.err, kErrTimeoutRing)) break;
            const int64_t step = s0 + static_cast<int64_t>(i) * RD_WARPS + warp;
            if (step < s1) {
                const int64_t blk = step * BPS + j;
                const bool valid = blk < a.nblocks;
                const uint8_t *src = ring + stage * L::CHUNK_BYTES + (warp * BPS + j) * F::BB;
                constexpr bool kRawCopy = TYPE == kF16 && sizeof(OutT) == 2;
                if (kRawCopy && a.use_tma) {
                    // fp16 weights to fp16: the run's 64 bytes move as they are
                    const uint32_t tile = tiles + (nst & 1u) * static_cast<uint32_t>(L::TILE);
                    if (lane == 0) bulk_wait_group_read<1>();   // the tile's previous store has read it
                    __syncwarp();
                    const uint32_t row = tile + static_cast<uint32_t>(lane * 64);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 v = valid ? Smem::u128(src + 16 * k) : make_uint4(0u, 0u, 0u, 0u);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         row + static_cast<uint32_t>((k ^ ((lane >> 1) & 3)) << 4)),
                                     "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmo, tile, 0, static_cast<int32_t>(step * 32));
                        bulk_commit_group();
                    }
                    ++nst;
                    if (valid && blk * 32 + 32 > a.nvals) {      // a last run of fewer than 32 values
                        OutT *o = out + blk * 32;
                        for (int64_t k = 0; k < a.nvals - blk * 32; ++k)
                            o[k] = static_cast<OutT>(Smem::u16(src + 2 * k));
                    }
                } else {
                    pair_t y[16];
                    if (valid) {
                        Raw raw;
                        raw.template load<Smem>(src, t);
                        raw.decode(t, y);
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) y[k] = pk2(0.0f, 0.0f);
                    }
                    if (a.use_tma) {
                        // box rows past the end of the output view are not written
                        const uint32_t tile = tiles + (nst & 1u) * static_cast<uint32_t>(L::TILE);
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
                        put_run_swz<OutT>(tile, lane, y);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmo, tile, 0, static_cast<int32_t>(step * 32));
                            bulk_commit_group();
                        }
                        ++nst;
                        if constexpr (TYPE == kF16) {
                            // a last run of fewer than 32 values lies outside the view
                            if (valid && blk * 32 + 32 > a.nvals)
                                put_run_guarded<OutT>(out, blk * 32, static_cast<int>(a.nvals - blk * 32), y);
                        }
                    } else if (valid) {
                        if constexpr (TYPE == kF16) {
                            const int64_t left = a.nvals - blk * 32;
                            put_run_guarded<OutT>(out, blk * 32, left < 32 ? static_cast<int>(left) : 32, y);
                        } else {
                            const int64_t row = blk / a.nb;
                            const int64_t col0 = (blk - row * a.nb) * F::QK + 32 * t;
                            if (col0 < a.cols) {
                                const int64_t left = a.cols - col0;
                                put_run_guarded<OutT>(out, row * a.cols + col0,
                                                      left < 32 ? static_cast<int>(left) : 32, y);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            advance(stage, phase, L::ST);
        }
        if (lane == 0) bulk_wait_all();                       // the stores have completed
    }
    __syncthreads();
    if (*drain_failed) pause_ns(200000ull);
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The output as [runs x 32 values] for TMA stores of 32-run boxes.
template <typename OutT>
bool encode_out(void *encode_fn, int64_t runs, OutT *out, CUtensorMap *map) {
    if (!encode_fn || runs < 1 || runs > INT32_MAX || (reinterpret_cast<uintptr_t>(out) & 15u) != 0) return false;
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
cudaError_t launch(const void *blocks, int64_t rows, int64_t cols, OutT *out, cudaStream_t stream,
                   const LaunchEnv &env) {
    using F = RFmt<TYPE>;
    using L = RLayout<TYPE, OutT>;
    RingArgs a;
    a.blocks = static_cast<const uint8_t *>(blocks);
    a.cols = cols;
    a.nvals = rows * cols;
    int64_t view_runs;                                    // whole runs the TMA view holds (0: no TMA)
    if constexpr (TYPE == kF16) {
        a.nb = cols;
        a.nblocks = (a.nvals + 31) / 32;
        a.in_bytes = 2 * a.nvals;
        view_runs = a.nvals / 32;                         // a partial last run is stored by its lane
    } else {
        a.nb = (cols + F::QK - 1) / F::QK;
        a.nblocks = rows * a.nb;
        a.in_bytes = a.nblocks * F::BB;
        view_runs = cols % F::QK == 0 ? a.nblocks * F::RPB : 0;
    }
    a.steps = (a.nblocks + L::BPS - 1) / L::BPS;
    a.units = (a.steps + F::ALIGN - 1) / F::ALIGN;
    a.out = out;
    a.err = env.err;
    a.limit_ns = env.wait_limit_ns;
    CUtensorMap tmo;
    a.use_tma = view_runs > 0 && encode_out<OutT>(env.encode_fn, view_runs, out, &tmo) ? 1 : 0;
    if (!a.use_tma) memset(&tmo, 0, sizeof(tmo));

    auto kern = ring_dequant_kernel<TYPE, OutT>;
    static std::atomic<int> smem_set[kMaxDevices];        // the opt-in holds per device
    if (!smem_set[env.device].load()) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
        if (e != cudaSuccess) return e;
        smem_set[env.device].store(1);
    }
    const int64_t grid = a.units < env.num_sms ? a.units : env.num_sms;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(RD_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, tmo);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename OutT>
cudaError_t dispatch(int type, const void *blocks, int64_t rows, int64_t cols, OutT *out, cudaStream_t stream,
                     const LaunchEnv &env) {
    switch (type) {
    case kQ8_0: return launch<kQ8_0>(blocks, rows, cols, out, stream, env);
    case kQ2_K: return launch<kQ2_K>(blocks, rows, cols, out, stream, env);
    case kQ4_K: return launch<kQ4_K>(blocks, rows, cols, out, stream, env);
    case kQ5_K: return launch<kQ5_K>(blocks, rows, cols, out, stream, env);
    case kQ6_K: return launch<kQ6_K>(blocks, rows, cols, out, stream, env);
    case kF16: return launch<kF16>(blocks, rows, cols, out, stream, env);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_dequant_f32(int type, const void *blocks, int64_t rows, int64_t cols, float *out,
                               cudaStream_t stream, const LaunchEnv &env) {
    return dispatch(type, blocks, rows, cols, out, stream, env);
}

cudaError_t launch_dequant_f16(int type, const void *blocks, int64_t rows, int64_t cols, uint16_t *out,
                               cudaStream_t stream, const LaunchEnv &env) {
    return dispatch(type, blocks, rows, cols, out, stream, env);
}

}  // namespace qp
