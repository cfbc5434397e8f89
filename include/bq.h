/*
 * bq.h — C ABI of libbq.so: block-quantized weight rows on one GB300 GPU.
 *
 * Formats (sizes fixed by the pages; byte and nibble order are this
 * library's stated layout):
 *   Q4_0 block, 18 bytes: 32 weights share one FP16 scale, each weight is a
 *     4-bit integer, 4.5 bits per weight ("llama.cpp 原理：如何在普通硬件跑本地
 *     大模型", §量化：内存真正去哪了); symmetric, value = scale * q with no zero
 *     point (lpnh.cn KV-cache article, §kv-mean-center 进阶技巧 / §问题).
 *     Layout: bytes 0-1 the scale (IEEE binary16, little endian), bytes 2-17
 *     qs[j] = (q[j] + 8) | ((q[j + 16] + 8) << 4), q in [-8, 7].
 *   Q8_0 block, 34 bytes: one FP16 scale per 32 weights, about 8.5 bits per
 *     weight ("05. llama.cpp：从 GGUF 文件到本地推理服务", §量化类型, format
 *     table). Layout: bytes 0-1 the scale, bytes 2-33 int8 q[j] in [-127, 127].
 *   Quantization of a 32-value block: amax = max |x|; d = amax / 7 (Q4_0) or
 *     amax / 127 (Q8_0) in fp32 IEEE division; the stored scale is d rounded
 *     to binary16 (ties to even); q = clamp(round_half_even(x / scale), ...)
 *     with an IEEE division by the stored scale; a zero scale gives q = 0.
 *
 * Conventions for every entry point:
 *   - Status: 0 (BQ_OK) on success, a negative BQ_ERR_* code otherwise; the
 *     message for the last failure on the calling thread is bq_last_error().
 *     ("nonzero means failure", as the quantize tool's library entry reports
 *     it: "采样、量化与部署 — 代码走读", §tools/quantize/.)
 *   - Data pointers are DEVICE pointers owned by the caller. Inputs and
 *     outputs must not alias. Nothing is allocated by the library: entry
 *     points that need scratch use the caller-provided workspace.
 *   - Calls are asynchronous on the calling thread's current stream
 *     (bq_set_stream; NULL = the legacy default stream). Argument errors and
 *     launch errors are returned at once; faults inside a kernel surface at
 *     the caller's next synchronization. Bounded waits inside kernels that run
 *     out set a device error word that bq_device_status() reports.
 *   - A call whose sizes make the output empty is a successful no-op.
 *   - Block pointers (weights, quantized outputs) must be 16-byte aligned and
 *     fp32 pointers 16-byte aligned, else BQ_ERR_ALIGN.
 *   - Sizes are int64; a row length (n_cols, K, head_dim) must be a multiple
 *     of 32, else BQ_ERR_SHAPE.
 */
#ifndef BQ_H
#define BQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BQ_TYPE_Q4_0 2
#define BQ_TYPE_Q8_0 8
/* Legacy types with a fifth bit and/or a minimum: one FP16 scale per 32
 * weights, and "_1" adds a minimum ("05. llama.cpp…", §量化类型; q4_1, q5_0
 * and q5_1 are also K/V cache types, §KV Cache 类型与 Flash Attention). The
 * pages give no layout; this library's reading (little endian):
 *   Q4_1: 20 bytes = { fp16 d, fp16 m, 16 nibble bytes }        5.0 bits/weight
 *   Q5_0: 22 bytes = { fp16 d, u32 qh, 16 nibble bytes }        5.5
 *   Q5_1: 24 bytes = { fp16 d, fp16 m, u32 qh, 16 nibble bytes } 6.0
 * The low 4 bits of code j sit as in Q4_0 (low nibble of byte j for j < 16,
 * high nibble of byte j - 16), bit 4 of code j is bit j of qh; codes are
 * unsigned u. Q5_0: d = amax / 15, u = clamp(rn(x / d), -16, 15) + 16, value
 * d * (u - 16). Q4_1 / Q5_1: m = min x, d = (max x - m) / (2^bits - 1),
 * u = clamp(rn((x - m) / d), 0, 2^bits - 1) with the stored fp16 d and m,
 * value d * u + m (fp32 product, then fp32 sum); a block whose scale or
 * minimum overflows binary16 is outside the supported range. Taken by bq_quantize_rows,
 * bq_dequantize_rows, bq_gemv / bq_gemv_multi (the minimum adds
 * m_w * d_x * sum(qx) per block) and bq_kv_quantize (without a bias or a
 * rotation); the other entry points answer BQ_ERR_UNSUPPORTED. */
#define BQ_TYPE_Q4_1 3
#define BQ_TYPE_Q5_0 6
#define BQ_TYPE_Q5_1 7
/* k-quants: super-blocks of 256 weights with 8 sub-blocks of 32 whose scales
 * are themselves quantized to 6 bits ("05. llama.cpp…", §量化类型). The pages
 * give no bit layout or quantization search; this library's reading
 * (little endian):
 *   Q4_K, 144 bytes per 256: fp16 d, fp16 dmin, 12 bytes = 6-bit sub-block
 *     scales sc[0..7] then minimums mn[0..7] as one 96-bit stream (value k
 *     at bits 6k..6k+5), 128 bytes: sub-block j's codes in bytes 16j.., low
 *     nibble code i, high nibble code i + 16; value fp32(d sc_j) u -
 *     fp32(dmin mn_j). Quantizer: m_j = max(0, -min), s_j = (max + m_j)/15,
 *     d = max s_j / 63, dmin = max m_j / 63 (fp16), sc/mn = rn(s_j / d),
 *     rn(m_j / dmin) in 0..63, u = clamp(rn((x + M_j) / S_j), 0, 15).
 *   Q6_K, 210 bytes per 256 (the size the pages' Llama-3-8B file sizes
 *     imply): 128 bytes ql (byte i: low 4 bits of code i, then code i + 128),
 *     64 bytes qh (byte i: top 2 bits of codes i, i+64, i+128, i+192), 16 int8
 *     scales of the sub-blocks of 16, fp16 d; value fp32(d sc_k) (u - 32).
 *     Quantizer: s_k = amax / 31, d = max s_k / 127, sc_k = rn(s_k / d),
 *     u = clamp(rn(x / S_k), -32, 31) + 32.
 * Rows hold a multiple of 256 values (else BQ_ERR_SHAPE). Taken by
 * bq_quantize_rows, bq_dequantize_rows and bq_gemv / bq_gemv_multi; every
 * other entry point answers BQ_ERR_UNSUPPORTED. bq_block_bytes gives the
 * bytes of one super-block, bq_block_values 256. */
#define BQ_TYPE_Q4_K 12
#define BQ_TYPE_Q6_K 14

#define BQ_OK 0
#define BQ_ERR_INVALID_ARG (-1) /* null pointer, negative size, aliasing */
#define BQ_ERR_SHAPE (-2)       /* row length not a multiple of 32, or above a stated limit */
#define BQ_ERR_UNSUPPORTED (-3) /* unknown type, or a type this entry point does not take */
#define BQ_ERR_ALIGN (-4)       /* pointer alignment */
#define BQ_ERR_CUDA (-5)        /* a CUDA runtime call failed (message has the CUDA error) */
#define BQ_ERR_TIMEOUT (-6)     /* a bounded in-kernel wait ran out (see bq_device_status) */
#define BQ_ERR_WORKSPACE (-7)   /* workspace missing or smaller than bq_workspace_size() */
#define BQ_ERR_BASIS (-8)       /* a mean-centering bias calibrated in another basis than the K cache */

/* Largest K taken by bq_gemv (the quantized activation lives in shared memory). */
#define BQ_GEMV_MAX_K 65536

/* Quantize rows (row quantize for Q4_0 and Q8_0).
 * Pages: Q4_0 and Q8_0 block rules above ("llama.cpp 原理…", §量化：内存真正去哪了;
 * "05. llama.cpp…", §量化类型).
 * src: n_rows x n_cols fp32, row-major, 16-byte aligned.
 * dst_blocks: n_rows x (n_cols/32) blocks of `type`, contiguous, 16-byte aligned,
 *   n_rows * n_cols / 32 * bq_block_bytes(type) bytes.
 * Errors: BQ_ERR_UNSUPPORTED (type), BQ_ERR_SHAPE (n_cols % 32), BQ_ERR_ALIGN,
 *   BQ_ERR_INVALID_ARG (null pointers with a nonzero size, negative sizes). */
int bq_quantize_rows(int type, const float *src_f32, void *dst_blocks, int64_t n_rows,
                     int64_t n_cols);

/* Dequantize rows: x_hat = scale * q, exact in fp32 (the pages name
 * dequantize_row_q4_0: xdnf.cn/news/348240, §2.2).
 * blocks: n_rows x (n_cols/32) blocks; dst: n_rows x n_cols fp32. */
int bq_dequantize_rows(int type, const void *blocks, float *dst, int64_t n_rows, int64_t n_cols);

/* Decode GEMV: y = W . x for one token. Decode reads every weight once per
 * token, so it is bound by memory bandwidth ("05. llama.cpp…", §性能直觉：带宽决定
 * Decode，算力决定 Prefill).
 * W_blocks: M rows of K/32 blocks of `type` (Q4_0 or Q8_0), row-major, 16-byte aligned.
 * x: K fp32 (quantized to Q8_0 inside the kernel with the block rule above).
 * y: M fp32. y[m] = sum_b scale_w[m][b] * scale_x[b] * sumi[m][b] where sumi is
 *   the exact int32 dot of the block codes; accumulated in fp32 (partial sums
 *   per lane, then a tree), relative error well under 1e-5 of sum_b |term|.
 * Limits: K <= BQ_GEMV_MAX_K. A workspace is optional (bq_gemv_workspace_size). */
int bq_gemv(int type, const void *W_blocks, const float *x, float *y, int64_t M, int64_t K);

/* Largest number of matrices one bq_gemv_multi call takes. */
#define BQ_GEMV_MAX_MATS 8

/* Decode GEMV over n matrices that read the same input x (e.g. the q, k and
 * v projections, or gate and up): y_i = W_i . x for i < n, in one launch, with
 * x quantized once. Same per-element result as n calls of bq_gemv.
 * W_blocks, y and M are HOST arrays of n entries; W_blocks[i] (16-byte
 * aligned) and y[i] are device pointers, M[i] >= 0 rows; all share type and K.
 * n in 1..BQ_GEMV_MAX_MATS and sum(M) < 2^31, else BQ_ERR_SHAPE. No y[i] may
 * overlap x, a weight matrix or another y[j]. */
int bq_gemv_multi(int type, int n, const void *const *W_blocks, float *const *y, const int64_t *M,
                  const float *x, int64_t K);

/* Largest K taken by bq_gemv_sequence. */
#define BQ_GEMV_SEQ_MAX_K 16384

/* A sequence of decode GEMV batches in one persistent launch (a decode step's
 * matrix products, "05. llama.cpp…", §性能直觉：带宽决定 Decode: every weight is
 * read once per token). Batch g has n_mats[g] matrices that read the input
 * x[g] and the same K[g]; its matrices are entries mat0 .. mat0 + n_mats[g] - 1
 * of the flattened arrays W_blocks, y and M, mat0 being the sum of the earlier
 * n_mats. The result is that of one bq_gemv_multi call per batch, issued in
 * order, bit for bit: x[g] may be (part of) an output of an earlier batch, and
 * an output of batch g may overwrite the input of an earlier batch. Inside the
 * launch the weights stream without a pause from batch to batch; a batch waits
 * for other CTAs only where memory orders it after an earlier batch (its x
 * overlaps that batch's outputs, or its outputs overlap that batch's x), and
 * then until every CTA has finished that batch (bounded waits). Batches that
 * share no memory run without any wait.
 * All arrays are HOST arrays; their entries are device pointers. W_blocks
 * (16-byte aligned): M rows of K/32 blocks of `type`; x[g] (16-byte aligned):
 * K[g] fp32; y (4-byte aligned): M fp32. Runs of more than 256 batches or 512
 * matrices take several launches, ordered by the stream.
 * Errors: BQ_ERR_SHAPE (K[g] not a positive multiple of 256 or above
 * BQ_GEMV_SEQ_MAX_K, a batch of 2^31 rows or more), BQ_ERR_ALIGN,
 * BQ_ERR_INVALID_ARG (null pointers, negative sizes, an output overlapping
 * another output, any weight matrix or its own batch's x), BQ_ERR_WORKSPACE
 * (no workspace of bq_gemv_sequence_workspace_size() bytes set: the launch
 * keeps its per-batch counters there, so calls sharing a workspace must not
 * run concurrently). The pages have no persistent launch; llama.cpp launches
 * one kernel per matrix product. */
int bq_gemv_sequence(int type, int n_groups, const int *n_mats, const void *const *W_blocks, float *const *y,
                     const int64_t *M, const float *const *x, const int64_t *K);
size_t bq_gemv_sequence_workspace_size(void);

/* Decode attention of one token over a block-quantized KV cache (flash
 * decoding): a quantized V cache is read by flash attention ("05.
 * llama.cpp…", §KV Cache 类型与 Flash Attention; lpnh.cn KV-cache article,
 * §量化 KV Cache 的一键配置方法).
 * q: n_heads x head_dim fp32 (16-byte aligned). K_cache / V_cache: n_tokens x
 * n_kv_heads x (head_dim/32) blocks of k_type / v_type (Q4_0 or Q8_0; the
 * layout bq_kv_quantize writes), 16-byte aligned. o: n_heads x head_dim fp32.
 * Query head h reads kv head h / G, G = n_heads / n_kv_heads. Each head of q
 * is quantized to Q8_0 per 32 channels; s_t = scale * sum_b dk dq sumi (the
 * GEMV's block dot); o_h = sum_t softmax_t(s) * v_hat_t (dequantized V).
 * A mean-centered K cache needs no correction: softmax ignores the constant
 * q . k_bar (lpnh.cn KV-cache article, §解法).
 * Limits: 1 <= n_tokens <= 2^21; head_dim a multiple of 32; G in {1, 2, 4, 8};
 * n_heads * head_dim <= 4096. Needs a workspace of bq_attn_workspace_size(...)
 * bytes (bq_set_workspace). Errors: BQ_ERR_UNSUPPORTED (types, G),
 * BQ_ERR_SHAPE (limits), BQ_ERR_ALIGN, BQ_ERR_INVALID_ARG (null pointers, o
 * overlapping an input), BQ_ERR_WORKSPACE. */
/* As bq_attn_decode over a K cache written in k_basis (bq_kv_quantize_basis):
 * with BQ_BASIS_HADAMARD64 each head of q is rotated like K before it is
 * quantized, so that the scores are unchanged ((Hq).(Hk) = q.k); head_dim
 * must then be a multiple of 64 (else BQ_ERR_SHAPE). */
int bq_attn_decode_basis(int k_type, int v_type, int k_basis, const float *q, const void *K_cache,
                         const void *V_cache, float *o, int64_t n_tokens, int64_t n_heads, int64_t n_kv_heads,
                         int64_t head_dim, float scale);
int bq_attn_decode(int k_type, int v_type, const float *q, const void *K_cache, const void *V_cache, float *o,
                   int64_t n_tokens, int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, float scale);
size_t bq_attn_workspace_size(int k_type, int v_type, int64_t n_tokens, int64_t n_heads, int64_t n_kv_heads,
                              int64_t head_dim);

/* Prefill GEMM: Y = X . W^T for N tokens; prefill reuses each weight across
 * many tokens and is compute-bound ("05. llama.cpp…", §性能直觉).
 * type: Q8_0 weights. W_blocks: M x K/32 blocks. X: N x K fp32 (each row
 *   quantized to Q8_0 into the workspace first). Y: N x M fp32 (row-major,
 *   Y[n][m]), same per-element sum as bq_gemv, fp32 accumulation.
 * Needs a workspace of bq_workspace_size(type, M, N, K) bytes set with
 *   bq_set_workspace, else BQ_ERR_WORKSPACE. */
int bq_gemm(int type, const void *W_blocks, const float *X, float *Y, int64_t M, int64_t N,
            int64_t K);

/* KV-cache write, one tensor per call (K or V). rows: n_tokens x n_kv_heads x
 * head_dim fp32. bias: NULL or n_kv_heads x head_dim fp32; when given, each row
 * of head h becomes rows - bias[h] (one fp32 subtraction) before quantization
 * ("kv-mean-center": lpnh.cn KV-cache article, §解法; the bias is one fp32 tensor
 * per layer indexed by (kv-head, channel), §适用边界).
 * A bias with a type other than Q4_0 is rejected with BQ_ERR_UNSUPPORTED (the
 * article: mean-centering requires a q4_0 K cache and errors out otherwise,
 * §三步上手). dst: n_tokens x n_kv_heads x head_dim/32 blocks of `type`. */
int bq_kv_quantize(int type, const float *K_rows, const float *bias, void *dst, int64_t n_tokens,
                   int64_t n_kv_heads, int64_t head_dim);

/* Bases of a K cache. A quantized K cache whose head dimension is a multiple
 * of 64 may be Hadamard-rotated; the mean-centering bias must then be measured
 * in the rotated basis, the calibration records its basis, and a mismatch
 * fails fast (lpnh.cn KV-cache article, §三步上手, third step). The pages name
 * neither the size nor the scaling of the rotation; here it is orthonormal and
 * block diagonal: every 64 channels of a head become H64 x / 8, H64[i][j] =
 * (-1)^popcount(i & j), computed by fp32 butterflies of span 1, 2, 4, ..., 32
 * ((a, b) -> (a + b, a - b)) followed by the exact scaling by 1/8. */
#define BQ_BASIS_PLAIN 0
#define BQ_BASIS_HADAMARD64 1

/* KV-cache write in a basis: with basis BQ_BASIS_HADAMARD64 each head's row is
 * rotated first (head_dim % 64 == 0, else BQ_ERR_SHAPE), then the bias (NULL
 * or Q4_0 only, as in bq_kv_quantize) is subtracted, then the row quantized.
 * bias_basis: the basis the bias was calibrated in (bq_kv_bias); a bias from
 * another basis is rejected with BQ_ERR_BASIS before anything runs. Other
 * arguments, layouts and errors as bq_kv_quantize; an unknown basis gives
 * BQ_ERR_UNSUPPORTED. */
int bq_kv_quantize_basis(int type, const float *K_rows, const float *bias, int bias_basis, int basis, void *dst,
                         int64_t n_tokens, int64_t n_kv_heads, int64_t head_dim);

/* KV-cache write of one layer in one call: K_rows to k_type in k_basis
 * (rotation and bias as bq_kv_quantize_basis: the bias NULL or with a Q4_0 K
 * only, calibrated in bias_basis == k_basis) and V_rows to v_type (plain
 * basis, no bias), both n_tokens x n_kv_heads x head_dim fp32 (16-byte
 * aligned); K_dst / V_dst: n_tokens x n_kv_heads x head_dim/32 blocks
 * (16-byte aligned). The bytes written are those of bq_kv_quantize_basis on K
 * and bq_kv_quantize on V. As the two tensors share no memory, the second
 * tensor's launch follows the first's as a programmatic dependent that does
 * not wait for it: its blocks start on the SMs that the first launch's
 * finishing blocks leave, instead of after its last one (K first for a plain
 * K, V first for a rotated one; the pages write the cache one tensor per
 * kernel; this is a schedule, not a different result). Ordered after all earlier work on the
 * stream; later work is ordered after both. Types: Q4_0 or Q8_0 for each
 * (else BQ_ERR_UNSUPPORTED). Errors as bq_kv_quantize_basis, and
 * BQ_ERR_INVALID_ARG when an output overlaps an input or the other output. */
int bq_kv_write(int k_type, const float *K_rows, const float *bias, int bias_basis, int k_basis, void *K_dst,
                int v_type, const float *V_rows, void *V_dst, int64_t n_tokens, int64_t n_kv_heads,
                int64_t head_dim);

/* Mean-centering bias calibration (lpnh.cn KV-cache article, §三步上手: the
 * channel mean of K over a calibration run): bias[h][c] = fp32(sum_t
 * r_t[h][c] / n_tokens), the sum in fp64 in token order, r_t the token's row
 * in `basis`. K_rows: n_tokens x n_kv_heads x head_dim fp32 (16-byte
 * aligned); bias: n_kv_heads x head_dim fp32 (4-byte aligned), written.
 * Errors: BQ_ERR_SHAPE (head_dim not a multiple of 32, or of 64 for the
 * rotated basis), BQ_ERR_UNSUPPORTED (basis), BQ_ERR_INVALID_ARG (null
 * pointers, n_tokens < 1, bias overlapping K_rows), BQ_ERR_ALIGN. */
int bq_kv_bias(const float *K_rows, int basis, float *bias, int64_t n_tokens, int64_t n_kv_heads,
               int64_t head_dim);

/* Test export: out[m][b] = int32 dot of W block (m, b) (type Q4_0 or Q8_0)
 * with the Q8_0 block b of xq, computed by the same device code as bq_gemv's
 * inner loop. out: M x K/32 int32. */
int bq_block_dots(int type, const void *W_blocks, const void *xq_blocks, int32_t *out, int64_t M,
                  int64_t K);

/* Bytes of the static scratch array that bq_gemm_noalloc uses (8 MiB). */
#define BQ_GEMM_NOALLOC_SCRATCH_BYTES (8 << 20)

/* Prefill GEMM that allocates nothing and needs no workspace. The pages have
 * no counterpart: this entry point exists for callers that cannot allocate
 * device memory when they call (a plugin hook that must not call cudaMalloc
 * while it runs, a process whose device memory is fixed after start-up) and
 * have no workspace of their own to lend.
 * Same arguments, layouts and result as bq_gemm (Q8_0 weights only). The
 * quantized activations go to a file-scope device array of
 * BQ_GEMM_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits: bq_gemm's tensor-core path when its activations (2.125
 * bytes per value, tokens rounded up to 128) fit, else the mma.sync path over
 * Q8_0 activations; N * (K/32) * 34 bytes beyond the array are rejected with
 * BQ_ERR_WORKSPACE. The call makes no cudaMalloc, cudaFree or other allocating
 * call. Its first call on a device looks up the array's device address with
 * that device current and keeps it for the life of the process; make that
 * first call before any stream capture, and make no call on a device after
 * cudaDeviceReset on it (the reset unloads the array the kept address
 * points to). All
 * calls share the one array (every call overwrites the part it uses before
 * reading it), so calls that overlap on the GPU race: issue them on one
 * stream, or order them. */
int bq_gemm_noalloc(int type, const void *W_blocks, const float *X, float *Y, int64_t M, int64_t N,
                    int64_t K);

/* Stream used by the calling thread's subsequent calls (a cudaStream_t);
 * NULL selects the legacy default stream. */
int bq_set_stream(void *cuda_stream);
void *bq_get_stream(void);

/* Weight prefetch across kernel boundaries for the calling thread's bq_gemv
 * calls (default off). When enabled, a GEMV is launched with programmatic
 * dependent launch: it may start, and stream W_blocks into shared memory,
 * while the previous kernel on the stream is still running; it reads x and
 * writes y only after that kernel has completed. Enable it only when no
 * kernel that may still be running on the stream writes W_blocks (model
 * weights loaded ahead of time); x and y carry no such restriction. */
int bq_set_weight_prefetch(int enable);

/* Caller-owned device workspace for the calling thread (NULL, 0 clears it). */
int bq_set_workspace(void *dev_ptr, size_t bytes);
/* Bytes of workspace an entry point needs for these sizes (0 if none). */
size_t bq_workspace_size(int type, int64_t M, int64_t N, int64_t K);

/* Workspace bytes that let bq_gemv / bq_gemv_multi quantize x once per call
 * (0 when K is not a positive multiple of 32). With a workspace of at least
 * this size set by bq_set_workspace, a call launches a small prep kernel,
 * which (on the bulk-copy path, with weight prefetch enabled and at most
 * 64 MB of weights in the call) first asks L2 to fetch the call's weights and
 * then writes x's Q8_0 codes, scales and code sums to the workspace, and then
 * the GEMV kernel, which copies them; shapes off the bulk-copy path (K % 256
 * != 0, Q6_K with K % 2048 != 0) take a generic kernel that reads the same
 * codes from the workspace. Without one, every GEMV CTA quantizes x itself.
 * Both give bit-identical results. The workspace must not be in use by
 * another call that may run concurrently. */
size_t bq_gemv_workspace_size(int type, int64_t K);

/* Thread-local message of the last failure (never NULL). */
const char *bq_last_error(void);

/* Bytes per block: 18 (Q4_0), 34 (Q8_0), 20 (Q4_1), 22 (Q5_0), 24 (Q5_1),
 * 144 (Q4_K) and 210 (Q6_K) per super-block; 0 for an unknown type. */
int bq_block_bytes(int type);
/* Values per block: 32, or 256 for the k-quant super-blocks; 0 for an
 * unknown type. */
int bq_block_values(int type);

/* Synchronize the calling thread's stream, then read and clear the device
 * error word: BQ_OK, BQ_ERR_TIMEOUT if a bounded wait ran out, BQ_ERR_CUDA if
 * the synchronization itself failed. */
int bq_device_status(void);

/* Poll budget of the bounded waits inside kernels (each poll of an mbarrier
 * may suspend for a short, hardware-chosen time). polls < 0 restores the
 * default (2^22); 0 makes every bounded wait give up at once, so that the
 * timeout path can be exercised: the kernel then drains its own copies in
 * flight, returns, and bq_device_status() reports BQ_ERR_TIMEOUT. Global to
 * the process. */
int bq_set_spin_limit(int64_t polls);

/* Library version, (major << 16) | minor. */
int bq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BQ_H */
