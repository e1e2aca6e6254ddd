/*
 * qp.h — C ABI of libqp: block-quantized weight dequantization and the
 * batched-prefill projection over those weights, on one NVIDIA GB300
 * (sm_103a).
 *
 * Sources of each operation (page title, section):
 *  - "Qwen3.5 batched prefill has no f32 dequant for IQ2_XXS, IQ3_S, IQ3_XXS,
 *    Q2_K" (aprender issue #4952), §Cause: the batched prefill expands every
 *    projection weight from its quantized blocks to f32, per block type, before
 *    its GEMM; the f16 GEMM mode caches an f16 copy built from that f32
 *    result; a type with no kernel fails with an invalid-parameter error.
 *    §Acceptance: bit-exact against a CPU oracle, including rows whose last
 *    block is partial, with no out-of-bounds writes.  §Rows adds Q2_K.
 *  - "QK-norm models take the FP16 batched prefill when it fits" (aprender PR
 *    #4624), §What changes: the prefill runs one GEMM per projection over a
 *    whole prompt chunk, and the prompt is chunked to bound memory.
 *  - same issue, first paragraph: a GPU run that falls back to the CPU is a
 *    failure.  This library has no CPU path at all.
 *
 * Conventions for every call:
 *  - All data pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing per call (it keeps one small device error word and a
 *    per-device attribute cache).
 *  - `stream` is a cudaStream_t handle passed as void* (NULL = the legacy
 *    default stream).  Calls are asynchronous on that stream.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns an error status and launches nothing.
 *  - Device-side failures (a bounded wait that ran out) are latched in the
 *    device error word and reported by qp_check().
 *  - fp16 data is passed as uint16_t bit patterns (IEEE binary16).
 *
 * Block formats (values per block / bytes per block), row-major: row r of a
 * [rows x cols] weight is ceil(cols/QK) whole blocks, back to back, with no
 * padding between rows; values at columns >= cols in a partial last block are
 * never written anywhere.
 *   QP_Q8_0  32 / 34:  d:f16, q:int8[32];                value = d*q
 *   QP_Q4_K 256 / 144: d:f16, dmin:f16, scales:u8[12] (eight packed 6-bit
 *                      scale/min pairs), qs:u8[128] (4-bit q);
 *                                                        value = d*sc*q - dmin*m
 *   QP_Q2_K 256 / 84:  scales:u8[16] (4-bit scale | 4-bit min per 16 values),
 *                      qs:u8[64] (2-bit q), d:f16, dmin:f16;
 *                                                        value = d*sc*q - dmin*m
 *   QP_Q6_K 256 / 210: ql:u8[128] (low 4 bits), qh:u8[64] (high 2 bits),
 *                      scales:int8[16], d:f16;           value = d*s*(q-32)
 *   QP_Q5_K 256 / 176: d:f16, dmin:f16, scales:u8[12] (as Q4_K), qh:u8[32]
 *                      (fifth bit of each q), qs:u8[128] (low 4 bits);
 *                                                        value = d*sc*q - dmin*m
 *   QP_F16    1 / 2:   one fp16 weight;                  value = that number
 * The byte layout within a block is the GGUF one.  (Q5_K and F16 are in the
 * list of types the f32 dequant has device kernels for, issue #4952
 * §Cause.)  For F16 the GEMM entry points run the cached-f16 kernel on W
 * itself: qp_prefill_gemm(QP_F16, W16, ...) equals qp_prefill_gemm_f16w.
 */
#ifndef QP_H
#define QP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Block types; the values are the GGUF type ids. */
typedef enum {
    QP_F16 = 1,
    QP_Q8_0 = 8,
    QP_Q2_K = 10,
    QP_Q4_K = 12,
    QP_Q5_K = 13,
    QP_Q6_K = 14
} qp_type;

typedef enum {
    QP_OK = 0,
    QP_ERR_INVALID_PARAMETER = 1, /* null pointer, non-positive size, bad mode */
    QP_ERR_UNSUPPORTED_TYPE = 2,  /* no kernel for this block type */
    QP_ERR_UNSUPPORTED_SHAPE = 3, /* shape the GEMM cannot tile (see qp_prefill_gemm) */
    QP_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
    QP_ERR_TIMEOUT = 5,           /* a bounded device-side wait ran out (from qp_check) */
    QP_ERR_MISALIGNED = 6,        /* a pointer is not aligned as required */
    QP_ERR_NO_DEVICE = 7,         /* no usable sm_103 CUDA device */
    QP_ERR_PAIR_ALLOC = 8         /* the two CTAs of a GEMM pair got different tensor-memory
                                     allocations; that launch computed nothing (from qp_check) */
} qp_status;

/* Static description of the status code. */
const char *qp_status_str(qp_status s);

/* Values per block (*qk) and bytes per block (*block_bytes) of `type`.
 * Returns QP_OK or QP_ERR_UNSUPPORTED_TYPE.  Host only; needs no device. */
qp_status qp_block_info(int type, int64_t *qk, int64_t *block_bytes);

/* Bytes of one row of `cols` values: ceil(cols/QK) * block_bytes; -1 for an
 * unsupported type or cols <= 0.  Host only. */
int64_t qp_row_bytes(int type, int64_t cols);

/*
 * Dequantize a [rows x cols] block-quantized weight to dense row-major f32.
 * (issue #4952 §Cause: the per-type dequantize-to-f32 step.)
 *   type    one of qp_type
 *   blocks  device pointer, rows * qp_row_bytes(type, cols) bytes, 16-byte aligned
 *   out     device pointer, rows * cols floats, 16-byte aligned
 * Every value equals the CPU oracle's bit for bit: each block field is widened
 * exactly and the value formula is evaluated in f32 with one rounding (the
 * products are exact for these formats).  Exactly rows*cols floats are written.
 * Errors: QP_ERR_INVALID_PARAMETER (null pointer, rows or cols <= 0),
 * QP_ERR_UNSUPPORTED_TYPE, QP_ERR_MISALIGNED, QP_ERR_CUDA.
 */
qp_status qp_dequant_f32(int type, const void *blocks, int64_t rows, int64_t cols,
                         float *out, void *stream);

/*
 * As qp_dequant_f32 but writes fp16 bit patterns: round-to-nearest-even of
 * the f32 value (issue #4952 §Cause: the f16 weight copy is built from the f32
 * dequant).  `out` holds rows * cols uint16_t, 16-byte aligned.
 */
qp_status qp_dequant_f16(int type, const void *blocks, int64_t rows, int64_t cols,
                         uint16_t *out, void *stream);

/*
 * Batched-prefill projection with the dequantization fused into the GEMM
 * (PR #4624 §What changes; issue #4952 §Cause):
 *   Y[t, o] = sum_k X[t, k] * W16[o, k]      0 <= t < T, 0 <= o < out_f
 * where W16 = the f16 dequantized weight (exactly what qp_dequant_f16 writes),
 * decoded tile by tile inside the kernel, never written to memory; products
 * on the tensor cores with fp32 accumulation.
 *   W      device pointer, out_f * qp_row_bytes(type, in_f) bytes, 16-byte aligned
 *   X      device pointer, [T x in_f] fp16 row-major, 16-byte aligned
 *   Y      device pointer, [T x out_f] f32 row-major, 16-byte aligned
 * Requirements (else QP_ERR_UNSUPPORTED_SHAPE): in_f % 256 == 0 and
 * qp_row_bytes(type, in_f) % 16 == 0 (Q2_K: in_f % 1024 == 0; Q6_K:
 * in_f % 2048 == 0), out_f % 4 == 0.  Any T >= 1.
 * The result does not depend on T or on where a row sits in X: each output
 * element is accumulated in the same order, so a chunked run is bitwise equal
 * to an unchunked one.  Deterministic run to run.
 */
qp_status qp_prefill_gemm(int type, const void *W, int64_t out_f, int64_t in_f,
                          const uint16_t *X, int64_t T, float *Y, void *stream);

/*
 * The cached-f16-weight mode (issue #4952 §Cause, the f16 GEMM mode): the same
 * GEMM over a dense fp16 weight W16 [out_f x in_f] row-major, e.g. one made
 * once by qp_dequant_f16.  Same requirements on in_f (a multiple of 256) and
 * out_f; bitwise equal to qp_prefill_gemm when W16 = qp_dequant_f16(W).
 */
qp_status qp_prefill_gemm_f16w(const uint16_t *W16, int64_t out_f, int64_t in_f,
                               const uint16_t *X, int64_t T, float *Y, void *stream);

/*
 * One projection of a grouped call: Y[T x out_f] = X[T x in_f] * W^T, with
 * the same meaning, layouts and requirements as the arguments of
 * qp_prefill_gemm (W block-quantized) or qp_prefill_gemm_f16w (W a dense
 * fp16 [out_f x in_f] weight).  Caller-owned device memory.
 */
typedef struct {
    const void *W;
    int64_t out_f, in_f;
    const uint16_t *X;
    float *Y;
} qp_gemm_desc;

#define QP_MAX_GROUP 8

/*
 * Several projections over the same prompt chunk in one launch
 * (PR #4624 §What changes: the batched prefill runs one GEMM per projection
 * over the chunk; a layer's projections are independent GEMMs): the n
 * (1..QP_MAX_GROUP) descriptors share `type` and T and are computed by one
 * persistent kernel whose CTAs deal out the tiles of all of them, so small
 * projections do not each leave SMs idle.  type = QP_Q8_0 ... QP_Q6_K runs
 * the fused mode on block-quantized W; type = 0 runs the cached mode on fp16
 * W.  Each Y is bitwise what the single-projection call gives.  Descriptors
 * are validated as those calls validate their arguments (the first failure
 * is returned and nothing is launched); outputs must not overlap inputs or
 * each other.  Asynchronous on `stream`.
 */
qp_status qp_prefill_gemm_group(int type, const qp_gemm_desc *descs, int n, int64_t T, void *stream);

/*
 * qp_prefill_gemm_group over consecutive row chunks of every X and Y,
 * [c, min(c + chunk, T)) for c = 0, chunk, 2*chunk, ... (PR #4624 §What
 * changes: the batched prefill is chunked to bound memory): one launch per
 * chunk.  Bitwise equal to one unchunked call.  chunk >= 1.
 */
qp_status qp_prefill_chunked_group(int type, const qp_gemm_desc *descs, int n, int64_t T, int64_t chunk,
                                   void *stream);

/*
 * Chunked prefill (PR #4624 §What changes: the batched prefill is chunked to
 * bound memory): runs the projection on consecutive row chunks of X and Y,
 * [c, min(c + chunk, T)) for c = 0, chunk, 2*chunk, ...; a short last chunk
 * is normal.  mode 0 = fused (W block-quantized, W16 ignored, may be NULL);
 * mode 1 = cached f16 (W16 required, W ignored).  Bitwise equal to one
 * unchunked call.  chunk >= 1.
 */
qp_status qp_prefill_chunked(int type, const void *W, const uint16_t *W16, int64_t out_f,
                             int64_t in_f, const uint16_t *X, int64_t T, float *Y,
                             int64_t chunk, int mode, void *stream);

#define QP_GEMV_MAX_T 8

/*
 * Decode-side projection over the same weights (PR #4624 §What changes: the
 * serial prefill is one forward per prompt token; issue #4952 §Cause: the
 * decode GEMVs run over the same block types):
 *   Y[t, o] = sum_k X[t, k] * Wd[o, k]      0 <= t < T <= QP_GEMV_MAX_T
 * with Wd = the f32 weights qp_dequant_f32 gives for the K-quants (Q2_K,
 * Q4_K, Q5_K, Q6_K: the quantized codes are multiplied exactly on the
 * tensor cores and each sub-block's scale and min applied in f32) and the
 * fp16 weights qp_dequant_f16 gives for Q8_0 and F16; f32 accumulation, W
 * read once.  A one-hot X row returns a column of Wd bit for bit.
 * Deterministic run to run; within the GEMM tolerance of the fp64
 * reference (not bitwise equal to qp_prefill_gemm, which multiplies the
 * fp16 weights and sums in another order).  The launch may start before an
 * earlier kernel on the stream has finished when that kernel allows it (this
 * library's kernels do); block-quantized W is then read right away, so it
 * must not be the output of such a kernel (F16 weights, which
 * qp_dequant_f16 may just have written, are read only after it).
 *   W   device, out_f * qp_row_bytes(type, in_f) bytes, 16-byte aligned
 *   X   device, [T x in_f] fp16 row-major, 16-byte aligned
 *   Y   device, [T x out_f] f32 row-major, 4-byte aligned
 * Any type of qp_type.  Requirements (else QP_ERR_UNSUPPORTED_SHAPE): whole
 * blocks (in_f a multiple of 256 for the K-quants, of 32 for Q8_0 and F16),
 * 1 <= T <= QP_GEMV_MAX_T, out_f <= 2^30, in_f <= 2^24.
 * Errors also: QP_ERR_INVALID_PARAMETER (null pointer, non-positive size),
 * QP_ERR_UNSUPPORTED_TYPE, QP_ERR_MISALIGNED, QP_ERR_CUDA.
 */
qp_status qp_decode_gemv(int type, const void *W, int64_t out_f, int64_t in_f, const uint16_t *X,
                         int64_t T, float *Y, void *stream);

/*
 * The decode GEMV of up to QP_MAX_GROUP projections of one type over the
 * same T token rows in one launch (each desc: W blocks, out_f, in_f, its own
 * X [T x in_f] and Y [T x out_f], as for qp_decode_gemv).  A layer's
 * projections are microsecond GEMVs each; one launch streams their weights
 * back to back instead of paying a pipeline fill and tail per projection.
 * Every Y is bitwise the qp_decode_gemv result.  Requirements and errors are
 * those of qp_decode_gemv for every desc, plus QP_ERR_INVALID_PARAMETER for a
 * NULL descs or n outside 1..QP_MAX_GROUP, and QP_ERR_UNSUPPORTED_SHAPE when
 * the descs hold more than 2^31 - 1 blocks of 16 weight rows in all.
 */
qp_status qp_decode_gemv_group(int type, const qp_gemm_desc *descs, int n, int64_t T, void *stream);

/*
 * Prefill fit planner (PR #4624 §What changes: the FP16 batched prefill is
 * taken only when weights + FP16 cache + KV + prefill reserve fit in free
 * VRAM, and the resident estimate is read from the projection tensors'
 * own bytes; CUDA prefill VRAM loans PR, §Individual feature evidence: free
 * memory sets the prompt chunk).  Host only; needs no device.
 *
 * For the n projections `proj` (block type, out_f, in_f) of a prompt of T
 * rows it computes
 *   weight_bytes      = sum out_f * qp_row_bytes(type, in_f)
 *   f16_cache_bytes   = sum out_f * in_f * 2       (the cached mode's copies)
 *   act_bytes_per_row = sum (2 * in_f + 4 * out_f) (each projection's X and
 *                       Y row; an upper bound when projections share X)
 * and picks, in this order:
 *   mode 1 (cached f16) if weights + f16 cache + kv_bytes + reserve_bytes
 *          + chunk * act_bytes_per_row <= free_bytes for some chunk >= 1,
 *   mode 0 (fused, no f16 copies) if the same holds without the f16 cache,
 *   mode -1 otherwise (does not fit: the caller keeps its serial path).
 * chunk = the largest number of rows <= min(T, max_chunk) that fits,
 * rounded down to a multiple of 256 (the GEMM's token tile) when it is at
 * least 256; max_chunk <= 0 means no cap.  With mode -1, chunk = 0.
 * total_bytes = the memory the chosen plan needs.  Type F16 counts its
 * weight bytes once (it is its own f16 copy).
 * Errors: QP_ERR_INVALID_PARAMETER (null pointer, n < 1, T < 1, a negative
 * byte count, out_f or in_f < 1), QP_ERR_UNSUPPORTED_TYPE.
 */
typedef struct {
    int type;
    int64_t out_f, in_f;
} qp_proj_shape;

typedef struct {
    int mode;
    int64_t chunk;
    int64_t weight_bytes, f16_cache_bytes, act_bytes_per_row, total_bytes;
} qp_prefill_plan;

qp_status qp_plan_prefill(const qp_proj_shape *proj, int n, int64_t T, int64_t free_bytes,
                          int64_t kv_bytes, int64_t reserve_bytes, int64_t max_chunk,
                          qp_prefill_plan *out);

/*
 * Synchronize `stream`, then read and clear the device error word.
 * Returns QP_OK, QP_ERR_TIMEOUT (a bounded wait inside a GEMM ran out; its
 * output is incomplete), QP_ERR_PAIR_ALLOC (a CTA pair of a GEMM launch was
 * given two different tensor-memory allocations and skipped its tiles; its
 * output is incomplete) or QP_ERR_CUDA (the stream reported an error).
 */
qp_status qp_check(void *stream);

/*
 * Upper bound, in nanoseconds, on any single device-side wait inside the GEMM
 * kernels; after it a kernel records QP_ERR_TIMEOUT, releases what it holds
 * and returns.  Default 2e9 (2 s).  0 restores the default.  Host only.
 */
void qp_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook for the bounded-wait path.  The next GEMM or decode GEMV launch
 * made by this process arms the barrier of its `load_index`-th pipeline stage
 * (GEMM: the load_index-th 64-value K panel a CTA loads; GEMV: the
 * load_index-th weight tile of each CTA's ring) but never issues the copy
 * that would complete it, so the consumers' wait on that stage runs out
 * after the wait limit: the launch records QP_ERR_TIMEOUT (read by
 * qp_check), stops, frees its tensor memory and returns; its output is
 * incomplete.  Applies to one launch only; -1 disarms.  Host only.
 */
void qp_debug_inject_stall(int load_index);

/*
 * Tiling of the prefill GEMM kernels (qp_prefill_gemm*, qp_prefill_chunked*).
 * 1 (the default): a tile is 256 weight rows x 256 tokens computed by a
 * cluster of two CTAs on two SMs with the paired tensor-core MMA
 * (tcgen05 cta_group::2, M = 256); each CTA decodes and stages its own 128
 * weight rows and 128 of the tokens.  0: a tile is 128 weight rows x 256
 * tokens on one CTA (M = 128).  Both compute every output with the same
 * sequence of K steps.  Applies to launches made after the call; host only.
 */
void qp_set_gemm_cta_pairs(int on);

#ifdef __cplusplus
}
#endif
#endif /* QP_H */
