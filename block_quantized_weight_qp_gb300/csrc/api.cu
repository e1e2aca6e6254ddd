// api.cu — the C ABI declared in include/qp.h: argument checks, per-device
// setup, the device error word, and the chunked prefill driver.  Every
// argument error is returned before anything is launched; there is no CPU
// path (a GPU run that falls back to the CPU is a failure, "Qwen3.5 batched
// prefill has no f32 dequant for IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", first
// paragraph).
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "qp.h"
#include "qp_internal.h"

namespace {

// Latched device-side errors (bit flags, see qp_internal.h).
__device__ uint32_t g_qp_error;

using qp::kMaxDevices;

struct DeviceInfo {
    bool ready = false;
    int dev = 0;
    int num_sms = 0;
    uint32_t *err = nullptr;  // device address of g_qp_error on this device
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
void *g_encode = nullptr;
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_inject_stall{-1};
std::atomic<int> g_cta_pairs{1};

bool valid_type(int t) {
    return t == qp::kF16 || t == qp::kQ8_0 || t == qp::kQ2_K || t == qp::kQ4_K || t == qp::kQ5_K ||
           t == qp::kQ6_K;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device setup on the current device: SM count, compute capability check,
// the error word's device address, the tensor-map encoder.
qp_status device_info(DeviceInfo **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return QP_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return QP_ERR_NO_DEVICE;
        }
        if (major != 10 || minor != 3) return QP_ERR_NO_DEVICE;  // built for sm_103a only
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_qp_error) != cudaSuccess) {
            cudaGetLastError();
            return QP_ERR_CUDA;
        }
        if (cudaMemset(addr, 0, sizeof(uint32_t)) != cudaSuccess) return QP_ERR_CUDA;
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn) {
                cudaGetLastError();
                return QP_ERR_CUDA;
            }
            g_encode = fn;
        }
        d.dev = dev;
        d.num_sms = sms;
        d.err = static_cast<uint32_t *>(addr);
        d.ready = true;
    }
    *out = &d;
    return QP_OK;
}

qp::LaunchEnv env_of(const DeviceInfo *d) {
    return qp::LaunchEnv{d->dev, d->num_sms, d->err, g_wait_limit_ns.load(), g_encode, -1};
}

int64_t qk_of(int t) { return t == qp::kF16 ? 1 : (t == qp::kQ8_0 ? 32 : 256); }
int64_t bytes_of(int t) {
    switch (t) {
    case qp::kQ8_0: return 34;
    case qp::kQ2_K: return 84;
    case qp::kQ4_K: return 144;
    case qp::kQ5_K: return 176;
    case qp::kQ6_K: return 210;
    case qp::kF16: return 2;
    default: return -1;
    }
}

qp_status gemm_shape_ok(int64_t out_f, int64_t in_f, int64_t T) {
    if (out_f <= 0 || in_f <= 0 || T <= 0) return QP_ERR_INVALID_PARAMETER;
    if (in_f % 256 != 0 || out_f % 4 != 0) return QP_ERR_UNSUPPORTED_SHAPE;
    // coordinates and loop bounds in the kernel are 32-bit
    if (T > (int64_t(1) << 30) || out_f > (int64_t(1) << 30) || in_f > (int64_t(1) << 24))
        return QP_ERR_UNSUPPORTED_SHAPE;
    return QP_OK;
}

static_assert(QP_MAX_GROUP == qp::kMaxGroup, "group limit of the C ABI and the kernel");

// One launch over n already-validated projections of one type.
qp_status run_gemms(int type, const qp_gemm_desc *descs, int n, int64_t T, void *stream) {
    DeviceInfo *d = nullptr;
    qp_status s = device_info(&d);
    if (s != QP_OK) return s;
    qp::GemmArgs a[qp::kMaxGroup];
    const int inject = g_inject_stall.exchange(-1);
    for (int i = 0; i < n; ++i) {
        a[i].type = type == qp::kF16 ? 0 : type;   // F16 weights are the cached mode's dense fp16 W
        a[i].out_f = descs[i].out_f;
        a[i].in_f = descs[i].in_f;
        a[i].T = T;
        a[i].W = descs[i].W;
        a[i].X = descs[i].X;
        a[i].Y = descs[i].Y;
        a[i].device = d->dev;
        a[i].num_sms = d->num_sms;
        a[i].err = d->err;
        a[i].wait_limit_ns = g_wait_limit_ns.load();
        a[i].inject_stall = inject;
        a[i].cta_pairs = g_cta_pairs.load() != 0;
    }
    const cudaError_t e = qp::launch_prefill_gemm(a, n, g_encode, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return QP_ERR_CUDA;
    }
    return QP_OK;
}

qp_status run_gemm(int type, const void *W, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T, float *Y,
                   void *stream) {
    const qp_gemm_desc d = {W, out_f, in_f, X, Y};
    return run_gemms(type, &d, 1, T, stream);
}

qp_status check_quant_gemm(int type, const void *W, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                           const float *Y) {
    if (!W || !X || !Y) return QP_ERR_INVALID_PARAMETER;
    if (!valid_type(type)) return QP_ERR_UNSUPPORTED_TYPE;
    const qp_status s = gemm_shape_ok(out_f, in_f, T);
    if (s != QP_OK) return s;
    if (qp_row_bytes(type, in_f) % 16 != 0) return QP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(W) || !aligned16(X) || !aligned16(Y)) return QP_ERR_MISALIGNED;
    return QP_OK;
}

qp_status check_f16w_gemm(const uint16_t *W16, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                          const float *Y) {
    if (!W16 || !X || !Y) return QP_ERR_INVALID_PARAMETER;
    const qp_status s = gemm_shape_ok(out_f, in_f, T);
    if (s != QP_OK) return s;
    if (!aligned16(W16) || !aligned16(X) || !aligned16(Y)) return QP_ERR_MISALIGNED;
    return QP_OK;
}

qp_status check_group(int type, const qp_gemm_desc *descs, int n, int64_t T) {
    if (!descs || n < 1 || n > QP_MAX_GROUP) return QP_ERR_INVALID_PARAMETER;
    if (type != 0 && !valid_type(type)) return QP_ERR_UNSUPPORTED_TYPE;
    for (int i = 0; i < n; ++i) {
        const qp_gemm_desc &g = descs[i];
        const qp_status s =
            type == 0 ? check_f16w_gemm(static_cast<const uint16_t *>(g.W), g.out_f, g.in_f, g.X, T, g.Y)
                      : check_quant_gemm(type, g.W, g.out_f, g.in_f, g.X, T, g.Y);
        if (s != QP_OK) return s;
    }
    return QP_OK;
}

}  // namespace

extern "C" {

const char *qp_status_str(qp_status s) {
    switch (s) {
    case QP_OK: return "ok";
    case QP_ERR_INVALID_PARAMETER: return "invalid parameter";
    case QP_ERR_UNSUPPORTED_TYPE: return "no kernel for this block type";
    case QP_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case QP_ERR_CUDA: return "CUDA error";
    case QP_ERR_TIMEOUT: return "device-side wait timed out";
    case QP_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case QP_ERR_NO_DEVICE: return "no usable sm_103 CUDA device";
    case QP_ERR_PAIR_ALLOC: return "the two CTAs of a pair got different tensor-memory allocations";
    default: return "unknown status";
    }
}

qp_status qp_block_info(int type, int64_t *qk, int64_t *block_bytes) {
    if (!valid_type(type)) return QP_ERR_UNSUPPORTED_TYPE;
    if (qk) *qk = qk_of(type);
    if (block_bytes) *block_bytes = bytes_of(type);
    return QP_OK;
}

int64_t qp_row_bytes(int type, int64_t cols) {
    if (!valid_type(type) || cols <= 0) return -1;
    return (cols + qk_of(type) - 1) / qk_of(type) * bytes_of(type);
}

qp_status qp_dequant_f32(int type, const void *blocks, int64_t rows, int64_t cols, float *out, void *stream) {
    if (!blocks || !out || rows <= 0 || cols <= 0) return QP_ERR_INVALID_PARAMETER;
    if (!valid_type(type)) return QP_ERR_UNSUPPORTED_TYPE;
    if (!aligned16(blocks) || !aligned16(out)) return QP_ERR_MISALIGNED;
    DeviceInfo *d = nullptr;
    const qp_status s = device_info(&d);
    if (s != QP_OK) return s;
    if (qp::launch_dequant_f32(type, blocks, rows, cols, out, static_cast<cudaStream_t>(stream), env_of(d)) !=
        cudaSuccess) {
        cudaGetLastError();
        return QP_ERR_CUDA;
    }
    return QP_OK;
}

qp_status qp_dequant_f16(int type, const void *blocks, int64_t rows, int64_t cols, uint16_t *out, void *stream) {
    if (!blocks || !out || rows <= 0 || cols <= 0) return QP_ERR_INVALID_PARAMETER;
    if (!valid_type(type)) return QP_ERR_UNSUPPORTED_TYPE;
    if (!aligned16(blocks) || !aligned16(out)) return QP_ERR_MISALIGNED;
    DeviceInfo *d = nullptr;
    const qp_status s = device_info(&d);
    if (s != QP_OK) return s;
    if (qp::launch_dequant_f16(type, blocks, rows, cols, out, static_cast<cudaStream_t>(stream), env_of(d)) !=
        cudaSuccess) {
        cudaGetLastError();
        return QP_ERR_CUDA;
    }
    return QP_OK;
}

qp_status qp_prefill_gemm(int type, const void *W, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                          float *Y, void *stream) {
    const qp_status s = check_quant_gemm(type, W, out_f, in_f, X, T, Y);
    if (s != QP_OK) return s;
    return run_gemm(type, W, out_f, in_f, X, T, Y, stream);
}

qp_status qp_prefill_gemm_f16w(const uint16_t *W16, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                               float *Y, void *stream) {
    const qp_status s = check_f16w_gemm(W16, out_f, in_f, X, T, Y);
    if (s != QP_OK) return s;
    return run_gemm(0, W16, out_f, in_f, X, T, Y, stream);
}

qp_status qp_prefill_gemm_group(int type, const qp_gemm_desc *descs, int n, int64_t T, void *stream) {
    const qp_status s = check_group(type, descs, n, T);
    if (s != QP_OK) return s;
    return run_gemms(type, descs, n, T, stream);
}

qp_status qp_prefill_chunked_group(int type, const qp_gemm_desc *descs, int n, int64_t T, int64_t chunk,
                                   void *stream) {
    if (chunk <= 0) return QP_ERR_INVALID_PARAMETER;
    qp_status s = check_group(type, descs, n, T);
    if (s != QP_OK) return s;
    // Row c of X starts at byte 2*c*in_f, of Y at 4*c*out_f: both stay
    // 16-byte aligned because in_f % 256 == 0 and out_f % 4 == 0.
    qp_gemm_desc part[QP_MAX_GROUP];
    for (int64_t c0 = 0; c0 < T; c0 += chunk) {
        const int64_t rows = T - c0 < chunk ? T - c0 : chunk;
        for (int i = 0; i < n; ++i) {
            part[i] = descs[i];
            part[i].X = descs[i].X + c0 * descs[i].in_f;
            part[i].Y = descs[i].Y + c0 * descs[i].out_f;
        }
        s = run_gemms(type, part, n, rows, stream);
        if (s != QP_OK) return s;
    }
    return QP_OK;
}

qp_status qp_prefill_chunked(int type, const void *W, const uint16_t *W16, int64_t out_f, int64_t in_f,
                             const uint16_t *X, int64_t T, float *Y, int64_t chunk, int mode, void *stream) {
    if (chunk <= 0 || (mode != 0 && mode != 1)) return QP_ERR_INVALID_PARAMETER;
    qp_status s = mode == 0 ? check_quant_gemm(type, W, out_f, in_f, X, T, Y)
                            : check_f16w_gemm(W16, out_f, in_f, X, T, Y);
    if (s != QP_OK) return s;
    // Row c of X starts at byte 2*c*in_f, of Y at 4*c*out_f: both stay
    // 16-byte aligned because in_f % 256 == 0 and out_f % 4 == 0.
    for (int64_t c0 = 0; c0 < T; c0 += chunk) {
        const int64_t rows = T - c0 < chunk ? T - c0 : chunk;
        s = run_gemm(mode == 0 ? type : 0, mode == 0 ? W : static_cast<const void *>(W16), out_f, in_f,
                     X + c0 * in_f, rows, Y + c0 * out_f, stream);
        if (s != QP_OK) return s;
    }
    return QP_OK;
}

qp_status check_gemv(int type, const void *W, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                     const float *Y) {
    if (!W || !X || !Y || out_f < 1 || in_f < 1 || T < 1) return QP_ERR_INVALID_PARAMETER;
    if (!valid_type(type)) return QP_ERR_UNSUPPORTED_TYPE;
    if (T > QP_GEMV_MAX_T || in_f % 32 != 0 || in_f % qk_of(type) != 0 || out_f > (int64_t(1) << 30) ||
        in_f > (int64_t(1) << 24))
        return QP_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(W) || !aligned16(X) || (reinterpret_cast<uintptr_t>(Y) & 3u) != 0) return QP_ERR_MISALIGNED;
    return QP_OK;
}

qp_status run_gemv(int type, const qp_gemm_desc *descs, int n, int64_t T, void *stream) {
    DeviceInfo *d = nullptr;
    const qp_status s = device_info(&d);
    if (s != QP_OK) return s;
    qp::GemvArgs a[qp::kMaxGroup];
    for (int i = 0; i < n; ++i)
        a[i] = qp::GemvArgs{descs[i].W, qp_row_bytes(type, descs[i].in_f), descs[i].out_f, descs[i].in_f, T,
                            descs[i].X, descs[i].Y};
    qp::LaunchEnv env = env_of(d);
    env.inject_stall = g_inject_stall.exchange(-1);
    if (qp::launch_decode_gemv(type, a, n, static_cast<cudaStream_t>(stream), env) != cudaSuccess) {
        cudaGetLastError();
        return QP_ERR_CUDA;
    }
    return QP_OK;
}

qp_status qp_decode_gemv(int type, const void *W, int64_t out_f, int64_t in_f, const uint16_t *X, int64_t T,
                         float *Y, void *stream) {
    const qp_status s = check_gemv(type, W, out_f, in_f, X, T, Y);
    if (s != QP_OK) return s;
    const qp_gemm_desc d = {W, out_f, in_f, X, Y};
    return run_gemv(type, &d, 1, T, stream);
}

qp_status qp_decode_gemv_group(int type, const qp_gemm_desc *descs, int n, int64_t T, void *stream) {
    if (!descs || n < 1 || n > QP_MAX_GROUP) return QP_ERR_INVALID_PARAMETER;
    for (int i = 0; i < n; ++i) {
        const qp_status s = check_gemv(type, descs[i].W, descs[i].out_f, descs[i].in_f, descs[i].X, T, descs[i].Y);
        if (s != QP_OK) return s;
    }
    int64_t blocks = 0;
    for (int i = 0; i < n; ++i) blocks += (descs[i].out_f + 15) / 16;
    if (blocks > INT32_MAX) return QP_ERR_UNSUPPORTED_SHAPE;
    return run_gemv(type, descs, n, T, stream);
}

qp_status qp_plan_prefill(const qp_proj_shape *proj, int n, int64_t T, int64_t free_bytes, int64_t kv_bytes,
                          int64_t reserve_bytes, int64_t max_chunk, qp_prefill_plan *out) {
    if (!proj || !out || n < 1 || T < 1 || free_bytes < 0 || kv_bytes < 0 || reserve_bytes < 0)
        return QP_ERR_INVALID_PARAMETER;
    int64_t wb = 0, cache = 0, act = 0;
    for (int i = 0; i < n; ++i) {
        const qp_proj_shape &p = proj[i];
        if (p.out_f < 1 || p.in_f < 1) return QP_ERR_INVALID_PARAMETER;
        if (!valid_type(p.type)) return QP_ERR_UNSUPPORTED_TYPE;
        wb += p.out_f * qp_row_bytes(p.type, p.in_f);
        if (p.type != qp::kF16) cache += p.out_f * p.in_f * 2;
        act += 2 * p.in_f + 4 * p.out_f;
    }
    const int64_t cap = max_chunk > 0 && max_chunk < T ? max_chunk : T;
    // largest chunk <= cap with fixed + chunk * act <= free; 0 if none
    auto fit = [&](int64_t fixed) -> int64_t {
        if (fixed > free_bytes) return 0;
        int64_t rows = (free_bytes - fixed) / act;
        if (rows > cap) rows = cap;
        if (rows >= 256) rows -= rows % 256;
        return rows;
    };
    out->weight_bytes = wb;
    out->f16_cache_bytes = cache;
    out->act_bytes_per_row = act;
    const int64_t base = wb + kv_bytes + reserve_bytes;
    int64_t c = fit(base + cache);
    if (c >= 1) {
        out->mode = 1;
        out->chunk = c;
        out->total_bytes = base + cache + c * act;
        return QP_OK;
    }
    c = fit(base);
    out->mode = c >= 1 ? 0 : -1;
    out->chunk = c;
    out->total_bytes = c >= 1 ? base + c * act : 0;
    return QP_OK;
}

qp_status qp_check(void *stream) {
    DeviceInfo *d = nullptr;
    const qp_status s = device_info(&d);
    if (s != QP_OK) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return QP_ERR_CUDA;
    }
    uint32_t word = 0;
    if (cudaMemcpy(&word, d->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return QP_ERR_CUDA;
    if (word != 0) {
        if (cudaMemset(d->err, 0, sizeof(word)) != cudaSuccess) return QP_ERR_CUDA;
        // a pairing failure is the cause, not a consequence: the launch that
        // met it ran none of its roles, so no wait of it could run out
        return (word & qp::kErrPairAlloc) ? QP_ERR_PAIR_ALLOC : QP_ERR_TIMEOUT;
    }
    return QP_OK;
}

void qp_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 2000000000ull); }

void qp_debug_inject_stall(int load_index) { g_inject_stall.store(load_index); }

void qp_set_gemm_cta_pairs(int on) { g_cta_pairs.store(on != 0); }

}  // extern "C"
