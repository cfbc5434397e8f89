/*
 * bq_oracle.h — plain CPU oracle for block-quantized weight rows.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path
 * (the CUDA library and its Python binding) never links, imports or calls it.
 *
 * This header is the oracle's own statement of the block layouts; it shares
 * nothing with the CUDA library's headers.
 *
 * Block layouts (sizes fixed by the pages; byte order and nibble order are
 * this project's reading, documented in the design notes):
 *   Q4_0: 18 bytes = { fp16 scale d (little endian, bytes 0-1),
 *                      16 bytes qs: qs[j] = (q[j]+8) | ((q[j+16]+8) << 4) }
 *         "32 weights per block, one FP16 scale, each weight a 4-bit
 *         integer, 18 bytes, 4.5 bits per weight"
 *         (llama.cpp 原理：如何在普通硬件跑本地大模型, §量化：内存真正去哪了).
 *   Q8_0: 34 bytes = { fp16 scale d (LE), int8 qs[32] }
 *         "every 32 weights one FP16 scale; Q8_0 about 8.5 bits"
 *         (05. llama.cpp：从 GGUF 文件到本地推理服务, §量化类型, format table).
 *
 * Parity status of each function is listed in the implementation file.
 */
#ifndef BQ_ORACLE_H
#define BQ_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_TYPE_Q4_0 2
#define ORACLE_TYPE_Q8_0 8
/* legacy types with a 5th bit and/or a minimum ("_1 adds a minimum";
 * 05. llama.cpp…, §量化类型). Layouts, this project's reading:
 *   Q4_1: 20 bytes = { fp16 d, fp16 m, 16 nibble bytes }
 *   Q5_0: 22 bytes = { fp16 d, uint32 qh, 16 nibble bytes }
 *   Q5_1: 24 bytes = { fp16 d, fp16 m, uint32 qh, 16 nibble bytes }
 * nibbles as Q4_0 (element j: low nibble of byte j for j < 16, high nibble of
 * byte j - 16), bit 4 of element j = bit j of qh; codes unsigned u, value
 * d * u + m (Q4_1, Q5_1) or d * (u - 16) (Q5_0). */
#define ORACLE_TYPE_Q4_1 3
#define ORACLE_TYPE_Q5_0 6
#define ORACLE_TYPE_Q5_1 7
/* k-quants: super-blocks of 256 weights (05. llama.cpp…, §量化类型); layouts
 * in bq_oracle.c (R20-R23); rows must hold a multiple of 256 values. Taken
 * by quantize/dequantize and the GEMV/GEMM dots only. */
#define ORACLE_TYPE_Q4_K 12
#define ORACLE_TYPE_Q6_K 14

/* bases of a K cache: plain, or Hadamard-rotated per 64 channels */
#define ORACLE_BASIS_PLAIN 0
#define ORACLE_BASIS_HADAMARD64 1

/* bytes of one block of the given type, 0 for an unknown type; a block is
 * oracle_block_values(type) values: 32, or 256 for the k-quants */
int64_t oracle_block_bytes(int type);
int64_t oracle_block_values(int type);

/* IEEE binary16 <-> binary32 (round to nearest, ties to even). */
uint16_t oracle_f32_to_f16(float f);
float oracle_f16_to_f32(uint16_t h);

/* ties-to-even rounding to the nearest integer, as a float */
float oracle_round_half_even(float v);

/* src: n_rows x n_cols fp32, row-major. dst: n_rows x (n_cols/32) blocks.
 * Returns 0, or -1 for an unknown type / n_cols % 32 != 0. */
int oracle_quantize_rows(int type, const float *src, uint8_t *dst,
                         int64_t n_rows, int64_t n_cols);

/* inverse map: x_hat = d * q, exact in fp32 */
int oracle_dequantize_rows(int type, const uint8_t *blocks, float *dst,
                           int64_t n_rows, int64_t n_cols);

/* out[m][b] = sum_{j<32} qw[m][b][j] * qx[b][j] (int32, exact).
 * w_type is Q4_0 or Q8_0; xq is K/32 Q8_0 blocks. */
int oracle_block_dots(int w_type, const uint8_t *w_blocks, const uint8_t *xq_blocks,
                      int32_t *out, int64_t M, int64_t K);

/* Decode GEMV. x (fp32, K) is quantized to Q8_0 first; then
 * y[m] = fp32( sum_b dw[m][b] * dx[b] * sumi[m][b] ) with the sum in fp64.
 * mag[m] (nullable) = sum_b |dw dx sumi| in fp64, for normwise tolerances. */
int oracle_gemv(int w_type, const uint8_t *w_blocks, const float *x, float *y,
                double *mag, int64_t M, int64_t K);

/* Prefill GEMM. X is N x K fp32 (row-major), each row quantized to Q8_0;
 * Y is N x M fp32: Y[n][m] = fp32( sum_b dx[n][b] dw[m][b] sumi ) (fp64 sum).
 * mag (nullable) is N x M. */
int oracle_gemm(int w_type, const uint8_t *w_blocks, const float *X, float *Y,
                double *mag, int64_t M, int64_t N, int64_t K);

/* KV-cache write. rows: n_tokens x n_kv_heads x head_dim fp32.
 * bias (nullable): n_kv_heads x head_dim fp32, subtracted before quantization.
 * A bias with a type other than Q4_0 is rejected (returns -2).
 * dst: n_tokens x n_kv_heads x (head_dim/32) blocks. */
int oracle_kv_quantize(int type, const float *rows, const float *bias, uint8_t *dst,
                       int64_t n_tokens, int64_t n_kv_heads, int64_t head_dim);

/* In place, every group of 64 consecutive values of x (n % 64 == 0):
 * x <- H64 x / 8, H64[i][j] = (-1)^popcount(i & j), by fp32 butterflies of
 * span 1, 2, 4, 8, 16, 32 ((a, b) -> (a + b, a - b)) then * 0.125.
 * Returns 0, -1 when n % 64 != 0. */
int oracle_hadamard64(float *x, int64_t n);

/* KV write in a basis: with basis ORACLE_BASIS_HADAMARD64 (head_dim % 64 ==
 * 0) each head's row is rotated by oracle_hadamard64 first; then the bias
 * (nullable, Q4_0 only) is subtracted, then the row is quantized. A bias
 * calibrated in another basis (bias_basis != basis) returns -4. */
int oracle_kv_quantize_basis(int type, const float *rows, const float *bias, int bias_basis, int basis,
                             uint8_t *dst, int64_t n_tokens, int64_t n_kv_heads, int64_t head_dim);

/* Bias calibration: bias[h][c] = fp32( sum_t r_t[h][c] / n_tokens ), the sum
 * in fp64 in token order, r_t the row in `basis` (rotated as above or not).
 * rows: n_tokens x n_kv_heads x head_dim fp32; bias: n_kv_heads x head_dim. */
int oracle_kv_bias(const float *rows, int basis, float *bias, int64_t n_tokens, int64_t n_kv_heads,
                   int64_t head_dim);

/* Decode attention over a K cache in k_basis: with ORACLE_BASIS_HADAMARD64,
 * q is rotated like K (oracle_hadamard64 per head) before everything else. */
int oracle_attn_decode_basis(int k_type, int v_type, int k_basis, const float *q, const uint8_t *K,
                             const uint8_t *V, float *o, double *mag, double *smax, int64_t n_tokens,
                             int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, float scale);

/* Decode attention of one token over a block-quantized KV cache.
 * q: n_heads x head_dim fp32. K, V: n_tokens x n_kv_heads x (head_dim/32)
 * blocks of k_type / v_type (the layout oracle_kv_quantize writes).
 * Query head h reads kv head h / (n_heads / n_kv_heads). Each head of q is
 * quantized to Q8_0; score s_t = scale * sum_b dk dq sumi (fp64);
 * w = softmax_t(s) (fp64); o[h][d] = fp32( sum_t w_t * v_hat[t][d] ).
 * mag (nullable, n_heads x head_dim) = sum_t w_t |v_hat[t][d]|;
 * smax (nullable, n_heads) = max_t |s_t|. Returns 0, -1 on bad arguments. */
int oracle_attn_decode(int k_type, int v_type, const float *q, const uint8_t *K, const uint8_t *V,
                       float *o, double *mag, double *smax, int64_t n_tokens, int64_t n_heads,
                       int64_t n_kv_heads, int64_t head_dim, float scale);

#ifdef __cplusplus
}
#endif

#endif /* BQ_ORACLE_H */
