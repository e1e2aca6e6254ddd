/*
 * qpo.h — scalar CPU oracle for block-quantized weight dequantization and the
 * batched-prefill projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this code; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the CUDA
 * path.
 *
 * What it follows:
 *  - "Qwen3.5 batched prefill has no f32 dequant for IQ2_XXS, IQ3_S, IQ3_XXS,
 *    Q2_K" (aprender issue #4952), §Cause: every projection weight is expanded
 *    from its quantized blocks to f32 before the prefill GEMM, per block type
 *    (Q4_K, Q6_K, Q8_0 named there; Q2_K is one of its §Rows); the f16 weight
 *    copy is built from that same f32 result.
 *  - same page, §Acceptance: bit-exact against a CPU oracle, rows whose last
 *    block is partial, NaN-prefilled outputs checked for stray writes.
 *  - "QK-norm models take the FP16 batched prefill when it fits" (aprender PR
 *    #4624), §What changes: the batched prefill is a GEMM over a whole
 *    (chunked) prompt with the dequantized weights.
 *
 * Readings taken where the pages are silent (each one is listed in the
 * repository's design notes):
 *  - block byte layouts are the GGUF Q8_0 / K-quant layouts (see qpo.c);
 *  - arithmetic is f32 with every operation rounded separately, no FMA;
 *  - the f16 output is round-to-nearest-even of the f32 value;
 *  - a row holds ceil(cols/QK) whole blocks; values past `cols` are never
 *    written;
 *  - the GEMM reference is Y[t,o] = sum_k X[t,k]*W[o,k] in fp64, X fp16 and W
 *    the f32 dequantized weight; A[t,o] = sum_k |X[t,k]|*|W[o,k]| bounds it.
 *
 * Parity pins: see the tests (hand-worked blocks, closed forms, bit-flip
 * bijection, brute-force round trip, numpy fp16 rounding, numpy fp64 matmul).
 * Compatibility of the byte layout with real GGUF files is parity unpinned:
 * no such file is available to check against.
 */
#ifndef QPO_H
#define QPO_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* GGUF type ids. */
enum { QPO_F16 = 1, QPO_Q8_0 = 8, QPO_Q2_K = 10, QPO_Q4_K = 12, QPO_Q5_K = 13, QPO_Q6_K = 14 };

/* Values per block and bytes per block; returns 0 on success, -1 if the type
 * is not one of the six. */
int qpo_block_info(int type, int64_t *qk, int64_t *block_bytes);

/* Exact binary16 -> binary32. */
float qpo_f16_to_f32(uint16_t h);
/* binary32 -> binary16, round to nearest, ties to even; overflow to +-inf;
 * NaN maps to a quiet NaN of the same sign. */
uint16_t qpo_f32_to_f16(float f);

/* Element-wise array forms of the two conversions above. */
void qpo_f16_to_f32_array(const uint16_t *h, int64_t n, float *out);
void qpo_f32_to_f16_array(const float *f, int64_t n, uint16_t *out);

/* Value v (0 <= v < QK) of one block. */
float qpo_decode_value(int type, const uint8_t *block, int v);

/* Dequantize a row-major [rows x ceil(cols/QK)] array of blocks to a dense
 * row-major [rows x cols] output.  Returns 0, or -1 on a bad type. */
int qpo_dequant_f32(int type, const void *blocks, int64_t rows, int64_t cols, float *out);
int qpo_dequant_f16(int type, const void *blocks, int64_t rows, int64_t cols, uint16_t *out);

/* fp64 reference of the projection for a subset of token rows.
 *   X    [T x in]   fp16 bits, row-major
 *   W    [out x in] f32, row-major (the f32 dequantized weight)
 *   rows [nrows]    token indices t to evaluate (NULL: all T rows, nrows=T)
 *   Y, A [nrows x out] fp64 outputs: Y = sum x*w, A = sum |x|*|w|.
 * Parallel over (row, output) pairs with OpenMP when compiled with it. */
void qpo_gemm_f64(const uint16_t *X, const float *W, int64_t T, int64_t out, int64_t in,
                  const int64_t *rows, int64_t nrows, double *Y, double *A);

/* Number of threads an OpenMP region of this library runs with. */
int qpo_num_threads(void);
/* Sets that number (n >= 1); the results do not depend on it: every output
 * value is computed by one thread in a fixed order. */
void qpo_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
