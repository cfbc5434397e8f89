// bq_internal.h — host-side interfaces between the C-ABI layer (bq_api.cu)
// and the kernel translation units. Not installed; not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "bq.h"

namespace bq {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int max_smem_optin = 0;      // bytes of dynamic shared memory a CTA may opt into
  int smem_per_sm = 0;         // bytes of shared memory per SM
  unsigned *err_word = nullptr;  // device address of the error word (bit kErrTimeout, ...)
};

// Info of the current device (cached after the first call on each device).
// Returns nullptr and sets *err on failure.
const DeviceInfo *device_info(cudaError_t *err);

// Poll budget of the bounded mbarrier waits inside kernels.
uint32_t spin_limit();

// Whether bq_gemv may stream weights before the previous kernel on the stream
// has completed (calling thread's setting, see bq_set_weight_prefetch).
bool weight_prefetch();

// Integer launch-tuning override from the environment (0 when unset); read
// once per name. Used to compare launch shapes, never to skip work.
int tuning_value(const char *name);

// Raise the dynamic shared memory limit of `func` on the current device to
// `bytes` unless an earlier call already did (so that launches recorded in a
// stream capture make no attribute calls after the first, uncaptured one).
cudaError_t ensure_smem(const void *func, int bytes);

// Record a failure message for bq_last_error() on the calling thread and
// return `status`; report_ok() records "no error" and returns BQ_OK.
int report_error(int status, const char *fmt, ...);
int report_ok();

// Launchers; each returns the launch status. Sizes were validated by the ABI layer.
// rotate: each group of 64 values (blocks 2m, 2m+1) is Hadamard-rotated
// before the bias is subtracted; n_blocks must then be even.
cudaError_t launch_quantize_rows(int type, const float *src, uint8_t *dst, int64_t n_blocks,
                                 int64_t blocks_per_row, const float *bias, int64_t bias_period,
                                 cudaStream_t stream, bool rotate = false);
// K (k_type, rotated when k_rot, the bias subtracted when given) and V
// (v_type, plain), n_blocks blocks each: the same launches as
// launch_quantize_rows on each tensor, the second a programmatic dependent
// of the first that does not wait for it (the tensors share no memory).
cudaError_t launch_kv_write(int k_type, int v_type, bool k_rot, const float *k_src, uint8_t *k_dst,
                            const float *v_src, uint8_t *v_dst, int64_t n_blocks, const float *bias,
                            int64_t bias_period, cudaStream_t stream);
// bias[c] = fp32(sum_t rows[t][c] / n_tokens) (fp64 sum in token order), in the
// Hadamard basis when rotate (row_len % 64 == 0).
cudaError_t launch_kv_bias(const float *rows, float *bias, int64_t n_tokens, int64_t row_len, bool rotate,
                           cudaStream_t stream);
cudaError_t launch_dequantize_rows(int type, const uint8_t *blocks, float *dst, int64_t n_blocks,
                                   cudaStream_t stream);
// n matrices (n <= BQ_GEMV_MAX_MATS) sharing one input x; matrix i has M[i] rows.
// rec_ws: optional workspace of gemv_workspace_bytes(K) for x's quantized
// records (then a prep kernel quantizes x once and prefetches the weights
// into L2); null: every GEMV CTA quantizes x itself.
cudaError_t launch_gemv(int type, int n, const uint8_t *const *W, float *const *y, const int64_t *M,
                        const float *x, int64_t K, uint32_t *rec_ws, cudaStream_t stream);
size_t gemv_workspace_bytes(int64_t K);
// A sequence of GEMV batches in one launch per at most 256 batches: batch g
// (n_mats[g] matrices from the flattened W / y / M arrays, input x[g], K[g] a
// multiple of 256) behaves as a launch_gemv issued after those of batches
// 0..g-1. ws: gemv_seq_workspace_bytes() of scratch (counters, zeroed before
// each launch, then x's quantized records).
size_t gemv_seq_workspace_bytes();
cudaError_t launch_gemv_seq(int type, int n_groups, const int *n_mats, const uint8_t *const *W, float *const *y,
                            const int64_t *M, const float *const *x, const int64_t *K, unsigned *sync,
                            cudaStream_t stream);
// Decode attention of one token over a block-quantized KV cache (attn.cu):
// chunks of tokens in parallel, then a combine; `ws` holds
// attn_workspace_bytes(...) bytes of partial results.
size_t attn_workspace_bytes(int kt, int vt, int64_t T, int64_t H, int64_t n_kv, int64_t D);
size_t attn_smem_bytes(int kt, int vt, int64_t T, int64_t H, int64_t n_kv, int64_t D);
// The compile-time-shaped decode-attention warp kernel (head_dim 128) for a
// Q4_0 / Q8_0 K cache, V type vt, G query heads per kv head and n_kv kv heads;
// nullptr where none is built.
const void *attn_warp_fixed_fn_q4k(int vt, int G, int n_kv);
const void *attn_warp_fixed_fn_q8k(int vt, int G, int n_kv);
cudaError_t launch_attn_decode(int kt, int vt, const float *q, const uint8_t *K, const uint8_t *V, float *o,
                               int64_t T, int64_t H, int64_t n_kv, int64_t D, float scale, void *ws,
                               cudaStream_t stream, bool k_rot = false);
cudaError_t launch_gemm(int type, const uint8_t *W, const uint8_t *Xq, float *Y, int64_t M,
                        int64_t N, int64_t K, cudaStream_t stream);
// Prefill GEMM on the tcgen05 tensor cores (K a multiple of 256): quantizes X
// into `ws` (gemm_tc_workspace_bytes(N, K) bytes) and runs the GEMM.
bool gemm_tc_supported(int64_t M, int64_t N, int64_t K);
size_t gemm_tc_workspace_bytes(int64_t N, int64_t K);
cudaError_t launch_gemm_tc(const uint8_t *W, const float *X, float *Y, int64_t M, int64_t N, int64_t K, void *ws,
                           cudaStream_t stream);
// The prefill path bq_gemm and bq_gemm_noalloc take for these sizes, given
// `ws_limit` bytes of scratch (SIZE_MAX: any): the tcgen05 kernel where it
// applies and its workspace fits, else the mma.sync kernel over Q8_0
// activations. *ws_bytes receives the scratch the chosen path needs.
enum class PrefillPath { kTc, kMmaSync };
PrefillPath prefill_path(int64_t M, int64_t N, int64_t K, size_t ws_limit, size_t *ws_bytes);
cudaError_t launch_prefill(PrefillPath path, const uint8_t *W, const float *X, float *Y, int64_t M, int64_t N,
                           int64_t K, void *ws, cudaStream_t stream);
cudaError_t launch_block_dots(int type, const uint8_t *W, const uint8_t *xq, int32_t *out,
                              int64_t M, int64_t K, cudaStream_t stream);

}  // namespace bq
