// qp_internal.h — declarations shared by the library's translation units
// (kernel launchers called from the C-ABI layer in api.cu).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qp {

// GGUF type ids.
constexpr int kF16 = 1;
constexpr int kQ8_0 = 8;
constexpr int kQ2_K = 10;
constexpr int kQ4_K = 12;
constexpr int kQ5_K = 13;
constexpr int kQ6_K = 14;

// Device error word bits (OR-ed by kernels, read and cleared by qp_check).
constexpr uint32_t kErrTimeoutProducer = 1u << 0;
constexpr uint32_t kErrTimeoutMma = 1u << 1;
constexpr uint32_t kErrTimeoutEpilogue = 1u << 2;
constexpr uint32_t kErrTimeoutDequant = 1u << 3;
constexpr uint32_t kErrPairAlloc = 1u << 4;  // the CTA pair got different TMEM addresses
constexpr uint32_t kErrTimeoutRing = 1u << 5;    // standalone dequant: a wait on its copy ring
constexpr uint32_t kErrTimeoutGemv = 1u << 6;    // decode GEMV: a wait on a warp's copy ring

// Devices a process may drive; launchers keep per-device caches of their
// occupancy queries, indexed by the device ordinal (0 <= device < this).
constexpr int kMaxDevices = 64;

// `encode_fn` is cuTensorMapEncodeTiled (the output's tensor map for the
// kernels' TMA stores).
// Per-device facts and settings a launch needs, prepared by api.cu.
struct LaunchEnv {
    int device;            // the current device's ordinal
    int num_sms;
    uint32_t *err;         // device error word
    uint64_t wait_limit_ns;
    void *encode_fn;       // cuTensorMapEncodeTiled
    int inject_stall;      // test hook (decode GEMV): >= 0 makes each CTA's producer drop that ring tile's copy
};

cudaError_t launch_dequant_f32(int type, const void *blocks, int64_t rows, int64_t cols, float *out,
                               cudaStream_t stream, const LaunchEnv &env);
cudaError_t launch_dequant_f16(int type, const void *blocks, int64_t rows, int64_t cols, uint16_t *out,
                               cudaStream_t stream, const LaunchEnv &env);

// Everything a GEMM launch needs, prepared on the host by api.cu.
struct GemmArgs {
    int type;              // block type, or 0 for the cached f16 weight
    int64_t out_f, in_f, T;
    const void *W;         // quantized blocks or fp16 weight
    const uint16_t *X;
    float *Y;
    int device;            // the current device's ordinal
    int num_sms;
    uint32_t *err;         // device error word
    uint64_t wait_limit_ns;
    int inject_stall;      // test hook: >= 0 makes the producer drop that load
    bool cta_pairs;        // two-CTA (M = 256) tiles, else one CTA (M = 128)
};

// Most projections one launch takes (qp_prefill_gemm_group).
constexpr int kMaxGroup = 8;

// Builds the tensor maps and launches one persistent kernel over n (1..8)
// projections of one type and one T; `encode` is cuTensorMapEncodeTiled.
cudaError_t launch_prefill_gemm(const GemmArgs *a, int n, void *encode_fn, cudaStream_t stream);

// Decode GEMV (T = 1..8 token rows) over block-quantized or F16 weights:
// one launch over n <= kMaxGroup projections of one type and one T, checked
// by api.cu; row_bytes = qp_row_bytes(type, in_f).
struct GemvArgs {
    const void *W;
    int64_t row_bytes, out_f, in_f, T;
    const uint16_t *X;
    float *Y;
};
cudaError_t launch_decode_gemv(int type, const GemvArgs *a, int n, cudaStream_t stream, const LaunchEnv &env);

}  // namespace qp
