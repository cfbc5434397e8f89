// bq_api.cu — the C ABI of libbq.so (declared in include/bq.h): argument
// validation, per-thread stream / workspace / error state, per-device info,
// and the device error word that bounded in-kernel waits report through.
#include <algorithm>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "bq.h"
#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {

// Set by kernels whose bounded waits ran out; read and cleared by bq_device_status.
static __device__ unsigned int g_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint32_t kDefaultSpinLimit = 1u << 22;

thread_local cudaStream_t t_stream = nullptr;
thread_local bool t_weight_prefetch = false;
thread_local void *t_ws = nullptr;
thread_local size_t t_ws_bytes = 0;
thread_local std::string t_error = "no error";

std::mutex g_info_mutex;
DeviceInfo g_info[kMaxDevices];
bool g_info_ready[kMaxDevices] = {};
uint32_t g_spin_limit = kDefaultSpinLimit;

int fail(int status, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char *where) {
  return fail(BQ_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

int block_bytes(int type) {
  if (type == BQ_TYPE_Q4_0) return Fmt<kTypeQ4_0>::kBytes;
  if (type == BQ_TYPE_Q8_0) return Fmt<kTypeQ8_0>::kBytes;
  if (type == BQ_TYPE_Q4_1) return Fmt<kTypeQ4_1>::kBytes;
  if (type == BQ_TYPE_Q5_0) return Fmt<kTypeQ5_0>::kBytes;
  if (type == BQ_TYPE_Q5_1) return Fmt<kTypeQ5_1>::kBytes;
  if (type == BQ_TYPE_Q4_K) return Fmt<kTypeQ4_K>::kBytes;
  if (type == BQ_TYPE_Q6_K) return Fmt<kTypeQ6_K>::kBytes;
  return 0;
}

// values per block: 256 for the k-quant super-blocks, else 32
int block_values(int type) { return (type == BQ_TYPE_Q4_K || type == BQ_TYPE_Q6_K) ? kQK_K : kQK; }

// Q4_0 / Q8_0: the types every entry point takes
bool core_type(int type) { return type == BQ_TYPE_Q4_0 || type == BQ_TYPE_Q8_0; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// n_rows * n_cols within int64 and both non-negative
bool sizes_ok(int64_t a, int64_t b) {
  if (a < 0 || b < 0) return false;
  return b == 0 || a <= (int64_t(1) << 62) / b;
}

int ok() {
  t_error = "no error";
  return BQ_OK;
}

}  // namespace

const DeviceInfo *device_info(cudaError_t *err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_info_mutex);
  if (!g_info_ready[dev]) {
    DeviceInfo d;
    d.device = dev;
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess ||
        (e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err_word), g_error_word)) != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    g_info[dev] = d;
    g_info_ready[dev] = true;
  }
  *err = cudaSuccess;
  return &g_info[dev];
}

uint32_t spin_limit() { return g_spin_limit; }

bool weight_prefetch() { return t_weight_prefetch; }

int tuning_value(const char *name) {
  const char *v = getenv(name);
  return v ? atoi(v) : 0;
}

int report_error(int status, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_error = buf;
  return status;
}

int report_ok() { return ok(); }

namespace {
struct SmemEntry {
  int device;
  const void *func;
  int bytes;
};
std::mutex g_smem_mutex;
SmemEntry g_smem[256];
int g_smem_n = 0;
}  // namespace

cudaError_t ensure_smem(const void *func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_smem_mutex);
  for (int i = 0; i < g_smem_n; ++i)
    if (g_smem[i].device == dev && g_smem[i].func == func) {
      if (g_smem[i].bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) g_smem[i].bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && g_smem_n < 256) g_smem[g_smem_n++] = SmemEntry{dev, func, bytes};
  return e;
}

}  // namespace bq

using namespace bq;

extern "C" {

int bq_version(void) { return (0 << 16) | 1; }

int bq_block_bytes(int type) { return block_bytes(type); }
int bq_block_values(int type) { return block_bytes(type) ? block_values(type) : 0; }

const char *bq_last_error(void) { return t_error.c_str(); }

int bq_set_stream(void *cuda_stream) {
  t_stream = static_cast<cudaStream_t>(cuda_stream);
  return ok();
}

void *bq_get_stream(void) { return t_stream; }

int bq_set_weight_prefetch(int enable) {
  t_weight_prefetch = enable != 0;
  return ok();
}

int bq_set_workspace(void *dev_ptr, size_t bytes) {
  if ((dev_ptr == nullptr) != (bytes == 0))
    return fail(BQ_ERR_INVALID_ARG, "bq_set_workspace: pointer and size must be both set or both empty");
  if (dev_ptr && !aligned(dev_ptr, 256)) return fail(BQ_ERR_ALIGN, "bq_set_workspace: pointer must be 256-byte aligned");
  t_ws = dev_ptr;
  t_ws_bytes = bytes;
  return ok();
}

size_t bq_workspace_size(int type, int64_t M, int64_t N, int64_t K) {
  if (type != BQ_TYPE_Q8_0 || M <= 0 || N <= 0 || K <= 0 || K % kQK) return 0;
  if (!sizes_ok(N, K) || M > 0x7fffffffll || N > 0x7fffffffll) return 0;
  size_t bytes = 0;
  prefill_path(M, N, K, SIZE_MAX, &bytes);
  return bytes;
}

size_t bq_gemv_workspace_size(int type, int64_t K) {
  if (!block_bytes(type)) return 0;
  return gemv_workspace_bytes(K);
}

int bq_set_spin_limit(int64_t polls) {
  g_spin_limit = polls < 0 ? kDefaultSpinLimit : uint32_t(polls > 0xffffffffll ? 0xffffffffll : polls);
  return ok();
}

int bq_device_status(void) {
  cudaError_t e = cudaStreamSynchronize(t_stream);
  if (e != cudaSuccess) return cuda_fail(e, "bq_device_status: stream synchronize");
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof word);
  if (e != cudaSuccess) return cuda_fail(e, "bq_device_status: read error word");
  if (word) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "bq_device_status: clear error word");
    if (word & kErrTimeout) return fail(BQ_ERR_TIMEOUT, "a bounded in-kernel wait ran out (error word 0x%x)", word);
  }
  return ok();
}

int bq_quantize_rows(int type, const float *src, void *dst, int64_t n_rows, int64_t n_cols) {
  const int bb = block_bytes(type);
  if (!bb) return fail(BQ_ERR_UNSUPPORTED, "bq_quantize_rows: unknown type %d", type);
  if (!sizes_ok(n_rows, n_cols)) return fail(BQ_ERR_INVALID_ARG, "bq_quantize_rows: bad sizes %lld x %lld", (long long)n_rows, (long long)n_cols);
  const int bv = block_values(type);
  if (n_cols % bv) return fail(BQ_ERR_SHAPE, "bq_quantize_rows: n_cols %lld is not a multiple of %d", (long long)n_cols, bv);
  const int64_t n_blocks = n_rows * (n_cols / bv);
  if (n_blocks == 0) return ok();
  if (!src || !dst) return fail(BQ_ERR_INVALID_ARG, "bq_quantize_rows: null pointer");
  if (!aligned(src, 16) || !aligned(dst, 16)) return fail(BQ_ERR_ALIGN, "bq_quantize_rows: src and dst must be 16-byte aligned");
  if (overlap(src, size_t(n_blocks) * bv * 4, dst, size_t(n_blocks) * bb))
    return fail(BQ_ERR_INVALID_ARG, "bq_quantize_rows: src and dst overlap");
  cudaError_t e = launch_quantize_rows(type, src, static_cast<uint8_t *>(dst), n_blocks, n_cols / bv, nullptr, 1, t_stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_quantize_rows launch");
}

int bq_dequantize_rows(int type, const void *blocks, float *dst, int64_t n_rows, int64_t n_cols) {
  const int bb = block_bytes(type);
  if (!bb) return fail(BQ_ERR_UNSUPPORTED, "bq_dequantize_rows: unknown type %d", type);
  if (!sizes_ok(n_rows, n_cols)) return fail(BQ_ERR_INVALID_ARG, "bq_dequantize_rows: bad sizes");
  const int bv = block_values(type);
  if (n_cols % bv) return fail(BQ_ERR_SHAPE, "bq_dequantize_rows: n_cols %lld is not a multiple of %d", (long long)n_cols, bv);
  const int64_t n_blocks = n_rows * (n_cols / bv);
  if (n_blocks == 0) return ok();
  if (!blocks || !dst) return fail(BQ_ERR_INVALID_ARG, "bq_dequantize_rows: null pointer");
  if (!aligned(blocks, 16) || !aligned(dst, 16)) return fail(BQ_ERR_ALIGN, "bq_dequantize_rows: pointers must be 16-byte aligned");
  if (overlap(blocks, size_t(n_blocks) * bb, dst, size_t(n_blocks) * bv * 4))
    return fail(BQ_ERR_INVALID_ARG, "bq_dequantize_rows: blocks and dst overlap");
  cudaError_t e = launch_dequantize_rows(type, static_cast<const uint8_t *>(blocks), dst, n_blocks, t_stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_dequantize_rows launch");
}

int bq_gemv_multi(int type, int n, const void *const *W, float *const *y, const int64_t *M, const float *x,
                  int64_t K) {
  const int bb = block_bytes(type);
  if (!bb) return fail(BQ_ERR_UNSUPPORTED, "bq_gemv: unknown type %d", type);
  if (n < 1 || n > BQ_GEMV_MAX_MATS) return fail(BQ_ERR_SHAPE, "bq_gemv_multi: n %d not in 1..%d", n, BQ_GEMV_MAX_MATS);
  if (!W || !y || !M) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_multi: null array");
  if (K < 0) return fail(BQ_ERR_INVALID_ARG, "bq_gemv: negative K");
  const int bv = block_values(type);
  if (K % bv) return fail(BQ_ERR_SHAPE, "bq_gemv: K %lld is not a multiple of %d", (long long)K, bv);
  if (K > BQ_GEMV_MAX_K) return fail(BQ_ERR_SHAPE, "bq_gemv: K %lld exceeds %d", (long long)K, BQ_GEMV_MAX_K);
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    if (M[i] < 0) return fail(BQ_ERR_INVALID_ARG, "bq_gemv: negative M");
    total += M[i];
    if (total > 0x7fffffffll) return fail(BQ_ERR_SHAPE, "bq_gemv: rows exceed 2^31-1");
  }
  if (total == 0) return ok();
  for (int i = 0; i < n; ++i) {
    if (M[i] == 0) continue;
    if (!y[i] || (K > 0 && (!W[i] || !x))) return fail(BQ_ERR_INVALID_ARG, "bq_gemv: null pointer");
    if (!aligned(y[i], 4) || (K > 0 && (!aligned(W[i], 16) || !aligned(x, 16))))
      return fail(BQ_ERR_ALIGN, "bq_gemv: W and x must be 16-byte aligned, y 4-byte aligned");
    const size_t ybytes = size_t(M[i]) * 4;
    if (overlap(y[i], ybytes, x, size_t(K) * 4)) return fail(BQ_ERR_INVALID_ARG, "bq_gemv: y overlaps x");
    for (int j = 0; j < n; ++j) {
      if (M[j] == 0) continue;
      if (overlap(y[i], ybytes, W[j], size_t(M[j]) * size_t(K / bv) * bb))
        return fail(BQ_ERR_INVALID_ARG, "bq_gemv: y overlaps a weight matrix");
      if (j != i && overlap(y[i], ybytes, y[j], size_t(M[j]) * 4))
        return fail(BQ_ERR_INVALID_ARG, "bq_gemv_multi: outputs overlap");
    }
  }
  cudaError_t e = cudaSuccess;
  if (K == 0) {
    for (int i = 0; i < n && e == cudaSuccess; ++i)
      if (M[i] > 0) e = cudaMemsetAsync(y[i], 0, size_t(M[i]) * 4, t_stream);
  } else {
    // with a large enough workspace, x is quantized once by a prep kernel that
    // also prefetches the weights into L2; otherwise every CTA quantizes x
    const size_t need = gemv_workspace_bytes(K);
    uint32_t *rec = (need && t_ws && t_ws_bytes >= need) ? static_cast<uint32_t *>(t_ws) : nullptr;
    if (rec && overlap(rec, need, x, size_t(K) * 4)) return fail(BQ_ERR_INVALID_ARG, "bq_gemv: workspace overlaps x");
    for (int i = 0; rec && i < n; ++i)
      if (M[i] > 0 && overlap(rec, need, y[i], size_t(M[i]) * 4))
        return fail(BQ_ERR_INVALID_ARG, "bq_gemv: workspace overlaps y");
    e = launch_gemv(type, n, reinterpret_cast<const uint8_t *const *>(W), y, M, x, K, rec, t_stream);
  }
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_gemv launch");
}

int bq_gemv(int type, const void *W, const float *x, float *y, int64_t M, int64_t K) {
  return bq_gemv_multi(type, 1, &W, &y, &M, x, K);
}

size_t bq_gemv_sequence_workspace_size(void) { return (gemv_seq_workspace_bytes() + 255) / 256 * 256; }

int bq_gemv_sequence(int type, int n_groups, const int *n_mats, const void *const *W, float *const *y,
                     const int64_t *M, const float *const *x, const int64_t *K) {
  const int bb = block_bytes(type);
  if (!bb) return fail(BQ_ERR_UNSUPPORTED, "bq_gemv_sequence: unknown type %d", type);
  if (!core_type(type)) return fail(BQ_ERR_UNSUPPORTED, "bq_gemv_sequence: Q4_0 or Q8_0 weights only");
  if (n_groups < 0) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: negative batch count");
  if (n_groups == 0) return ok();
  if (!n_mats || !x || !K) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: null array");
  int64_t total = 0;
  for (int g = 0; g < n_groups; ++g) {
    if (n_mats[g] < 0) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: batch %d has a negative matrix count", g);
    total += n_mats[g];
  }
  if (total > (int64_t(1) << 30)) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: too many matrices");
  if (total > 0 && (!W || !y || !M)) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: null array");
  struct Span {
    uintptr_t lo, hi;
    int g;
  };
  std::vector<Span> outs;
  outs.reserve(size_t(total));
  int64_t mi = 0;
  for (int g = 0; g < n_groups; ++g) {
    const int64_t Kg = K[g];
    if (Kg <= 0 || Kg % 256 || Kg > BQ_GEMV_SEQ_MAX_K)
      return fail(BQ_ERR_SHAPE, "bq_gemv_sequence: batch %d: K %lld is not a multiple of 256 in 256..%d", g,
                  (long long)Kg, BQ_GEMV_SEQ_MAX_K);
    int64_t rows = 0;
    for (int k = 0; k < n_mats[g]; ++k, ++mi) {
      if (M[mi] < 0) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: negative M");
      rows += M[mi];
      if (M[mi] == 0) continue;
      if (!W[mi] || !y[mi]) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: null matrix or output");
      if (!aligned(W[mi], 16) || !aligned(y[mi], 4))
        return fail(BQ_ERR_ALIGN, "bq_gemv_sequence: W must be 16-byte and y 4-byte aligned");
      const uintptr_t lo = reinterpret_cast<uintptr_t>(y[mi]);
      outs.push_back({lo, lo + uintptr_t(M[mi]) * 4, g});
    }
    if (rows >= (int64_t(1) << 31)) return fail(BQ_ERR_SHAPE, "bq_gemv_sequence: batch %d has 2^31 rows or more", g);
    if (rows > 0 && (!x[g] || !aligned(x[g], 16)))
      return fail(x[g] ? BQ_ERR_ALIGN : BQ_ERR_INVALID_ARG, "bq_gemv_sequence: x of batch %d null or not 16-byte aligned", g);
  }
  // outputs are pairwise disjoint; no weight matrix overlaps an output; no
  // output overlaps its own batch's input
  std::sort(outs.begin(), outs.end(), [](const Span &a, const Span &b) { return a.lo < b.lo; });
  for (size_t i = 1; i < outs.size(); ++i)
    if (outs[i].lo < outs[i - 1].hi) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: two outputs overlap");
  auto hits = [&](uintptr_t lo, uintptr_t hi, int only_g) {
    // the last output starting below hi is the only one that can overlap [lo, hi)
    auto it = std::lower_bound(outs.begin(), outs.end(), hi, [](const Span &a, uintptr_t v) { return a.lo < v; });
    while (it != outs.begin()) {
      --it;
      if (it->hi <= lo) return false;
      if (only_g < 0 || it->g == only_g) return true;
    }
    return false;
  };
  mi = 0;
  for (int g = 0; g < n_groups; ++g) {
    for (int k = 0; k < n_mats[g]; ++k, ++mi) {
      if (M[mi] == 0) continue;
      const uintptr_t lo = reinterpret_cast<uintptr_t>(W[mi]);
      if (hits(lo, lo + uintptr_t(M[mi]) * uintptr_t(K[g] / kQK) * uintptr_t(bb), -1))
        return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: an output overlaps a weight matrix");
    }
    if (x[g]) {
      const uintptr_t lo = reinterpret_cast<uintptr_t>(x[g]);
      if (hits(lo, lo + uintptr_t(K[g]) * 4, g))
        return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: an output of batch %d overlaps its x", g);
    }
  }
  if (outs.empty()) return ok();
  const size_t need = bq_gemv_sequence_workspace_size();
  if (!t_ws || t_ws_bytes < need)
    return fail(BQ_ERR_WORKSPACE, "bq_gemv_sequence: needs %zu workspace bytes, %zu set", need, t_ws_bytes);
  const uintptr_t ws0 = reinterpret_cast<uintptr_t>(t_ws), ws1 = ws0 + need;
  if (hits(ws0, ws1, -1)) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: the workspace overlaps an output");
  mi = 0;
  for (int g = 0; g < n_groups; ++g) {  // the launch writes the workspace while it reads x and W
    const uintptr_t xl = reinterpret_cast<uintptr_t>(x[g]);
    bool bad = x[g] && xl < ws1 && ws0 < xl + uintptr_t(K[g]) * 4;
    for (int k = 0; k < n_mats[g]; ++k, ++mi) {
      const uintptr_t wl = reinterpret_cast<uintptr_t>(W[mi]);
      bad = bad || (M[mi] > 0 && wl < ws1 && ws0 < wl + uintptr_t(M[mi]) * uintptr_t(K[g] / kQK) * uintptr_t(bb));
    }
    if (bad) return fail(BQ_ERR_INVALID_ARG, "bq_gemv_sequence: the workspace overlaps an input of batch %d", g);
  }
  cudaError_t e = launch_gemv_seq(type, n_groups, n_mats, reinterpret_cast<const uint8_t *const *>(W), y, M, x, K,
                                  static_cast<unsigned *>(t_ws), t_stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_gemv_sequence launch");
}

namespace {
int attn_check(int k_type, int v_type, int64_t T, int64_t H, int64_t n_kv, int64_t D, const char *who) {
  if (!core_type(k_type) || !core_type(v_type)) return fail(BQ_ERR_UNSUPPORTED, "%s: caches are Q4_0 or Q8_0", who);
  if (T < 1 || H < 1 || n_kv < 1 || D < kQK || D % kQK || H % n_kv)
    return fail(BQ_ERR_SHAPE, "%s: needs n_tokens >= 1, head_dim a multiple of 32, n_heads a multiple of n_kv_heads", who);
  const int64_t G = H / n_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return fail(BQ_ERR_UNSUPPORTED, "%s: %lld query heads per kv head", who, (long long)G);
  if (H * D > 4096) return fail(BQ_ERR_SHAPE, "%s: n_heads * head_dim above 4096", who);
  if (T > (int64_t(1) << 21)) return fail(BQ_ERR_SHAPE, "%s: n_tokens above 2^21", who);
  return BQ_OK;
}
}  // namespace

size_t bq_attn_workspace_size(int k_type, int v_type, int64_t n_tokens, int64_t n_heads, int64_t n_kv_heads,
                              int64_t head_dim) {
  if (attn_check(k_type, v_type, n_tokens, n_heads, n_kv_heads, head_dim, "bq_attn_workspace_size") != BQ_OK) return 0;
  return attn_workspace_bytes(k_type, v_type, n_tokens, n_heads, n_kv_heads, head_dim);
}

int bq_attn_decode(int k_type, int v_type, const float *q, const void *K, const void *V, float *o, int64_t n_tokens,
                   int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, float scale) {
  return bq_attn_decode_basis(k_type, v_type, BQ_BASIS_PLAIN, q, K, V, o, n_tokens, n_heads, n_kv_heads, head_dim,
                              scale);
}

int bq_attn_decode_basis(int k_type, int v_type, int k_basis, const float *q, const void *K, const void *V, float *o,
                         int64_t n_tokens, int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, float scale) {
  const int st = attn_check(k_type, v_type, n_tokens, n_heads, n_kv_heads, head_dim, "bq_attn_decode");
  if (st != BQ_OK) return st;
  if (k_basis != BQ_BASIS_PLAIN && k_basis != BQ_BASIS_HADAMARD64)
    return fail(BQ_ERR_UNSUPPORTED, "bq_attn_decode: unknown basis %d", k_basis);
  if (k_basis == BQ_BASIS_HADAMARD64 && head_dim % 64)
    return fail(BQ_ERR_SHAPE, "bq_attn_decode: a rotated K cache needs head_dim %% 64 == 0");
  if (!q || !K || !V || !o) return fail(BQ_ERR_INVALID_ARG, "bq_attn_decode: null pointer");
  if (!aligned(q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(o, 4))
    return fail(BQ_ERR_ALIGN, "bq_attn_decode: q, K and V must be 16-byte aligned, o 4-byte aligned");
  const size_t nb = size_t(head_dim / kQK);
  const size_t kbytes = size_t(n_tokens) * size_t(n_kv_heads) * nb * block_bytes(k_type);
  const size_t vbytes = size_t(n_tokens) * size_t(n_kv_heads) * nb * block_bytes(v_type);
  const size_t qbytes = size_t(n_heads) * size_t(head_dim) * 4;
  if (overlap(o, qbytes, q, qbytes) || overlap(o, qbytes, K, kbytes) || overlap(o, qbytes, V, vbytes))
    return fail(BQ_ERR_INVALID_ARG, "bq_attn_decode: o overlaps an input");
  const size_t need = attn_workspace_bytes(k_type, v_type, n_tokens, n_heads, n_kv_heads, head_dim);
  if (!t_ws || t_ws_bytes < need)
    return fail(BQ_ERR_WORKSPACE, "bq_attn_decode: needs %zu workspace bytes, %zu set", need, t_ws_bytes);
  if (overlap(t_ws, need, o, qbytes) || overlap(t_ws, need, q, qbytes) || overlap(t_ws, need, K, kbytes) ||
      overlap(t_ws, need, V, vbytes))
    return fail(BQ_ERR_INVALID_ARG, "bq_attn_decode: the workspace overlaps an argument");
  cudaError_t e = launch_attn_decode(k_type, v_type, q, static_cast<const uint8_t *>(K), static_cast<const uint8_t *>(V),
                                     o, n_tokens, n_heads, n_kv_heads, head_dim, scale, t_ws, t_stream,
                                     k_basis == BQ_BASIS_HADAMARD64);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_attn_decode launch");
}

int bq_gemm(int type, const void *W, const float *X, float *Y, int64_t M, int64_t N, int64_t K) {
  const int bb = block_bytes(type);
  if (!bb) return fail(BQ_ERR_UNSUPPORTED, "bq_gemm: unknown type %d", type);
  if (type != BQ_TYPE_Q8_0) return fail(BQ_ERR_UNSUPPORTED, "bq_gemm: only Q8_0 weights are supported");
  if (!sizes_ok(M, K) || !sizes_ok(N, K) || !sizes_ok(M, N)) return fail(BQ_ERR_INVALID_ARG, "bq_gemm: bad sizes");
  if (K % kQK) return fail(BQ_ERR_SHAPE, "bq_gemm: K %lld is not a multiple of 32", (long long)K);
  if (M > 0x7fffffffll || N > 0x7fffffffll) return fail(BQ_ERR_SHAPE, "bq_gemm: M and N must be below 2^31");
  if (M == 0 || N == 0) return ok();
  if (!Y || (K > 0 && (!W || !X))) return fail(BQ_ERR_INVALID_ARG, "bq_gemm: null pointer");
  if (!aligned(Y, 4) || (K > 0 && (!aligned(W, 16) || !aligned(X, 16))))
    return fail(BQ_ERR_ALIGN, "bq_gemm: W and X must be 16-byte aligned, Y 4-byte aligned");
  const size_t ybytes = size_t(M) * size_t(N) * 4;
  if (overlap(Y, ybytes, W, size_t(M) * size_t(K / kQK) * bb) || overlap(Y, ybytes, X, size_t(N) * size_t(K) * 4))
    return fail(BQ_ERR_INVALID_ARG, "bq_gemm: Y overlaps an input");
  if (K == 0) {
    cudaError_t e = cudaMemsetAsync(Y, 0, ybytes, t_stream);
    return e == cudaSuccess ? ok() : cuda_fail(e, "bq_gemm memset");
  }
  size_t need = 0;
  const PrefillPath path = prefill_path(M, N, K, SIZE_MAX, &need);
  if (!t_ws || t_ws_bytes < need)
    return fail(BQ_ERR_WORKSPACE, "bq_gemm: needs %zu workspace bytes, %zu set", need, t_ws_bytes);
  if (overlap(t_ws, need, Y, ybytes) || overlap(t_ws, need, X, size_t(N) * size_t(K) * 4) ||
      overlap(t_ws, need, W, size_t(M) * size_t(K / kQK) * bb))
    return fail(BQ_ERR_INVALID_ARG, "bq_gemm: workspace overlaps an argument");
  cudaError_t e = launch_prefill(path, static_cast<const uint8_t *>(W), X, Y, M, N, K, t_ws, t_stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_gemm launch");
}

int bq_kv_quantize(int type, const float *rows, const float *bias, void *dst, int64_t n_tokens,
                   int64_t n_kv_heads, int64_t head_dim) {
  return bq_kv_quantize_basis(type, rows, bias, BQ_BASIS_PLAIN, BQ_BASIS_PLAIN, dst, n_tokens, n_kv_heads, head_dim);
}

int bq_kv_quantize_basis(int type, const float *rows, const float *bias, int bias_basis, int basis, void *dst,
                         int64_t n_tokens, int64_t n_kv_heads, int64_t head_dim) {
  const int bb = block_bytes(type);
  if (!bb) return fail(BQ_ERR_UNSUPPORTED, "bq_kv_quantize: unknown type %d", type);
  if (basis != BQ_BASIS_PLAIN && basis != BQ_BASIS_HADAMARD64)
    return fail(BQ_ERR_UNSUPPORTED, "bq_kv_quantize: unknown basis %d", basis);
  if (bias && type != BQ_TYPE_Q4_0)
    return fail(BQ_ERR_UNSUPPORTED, "bq_kv_quantize: a mean-centering bias requires the Q4_0 type");
  if (bias && bias_basis != basis)
    return fail(BQ_ERR_BASIS, "bq_kv_quantize: the bias was calibrated in basis %d, the cache is in basis %d",
                bias_basis, basis);
  if (!sizes_ok(n_tokens, n_kv_heads) || !sizes_ok(n_tokens * n_kv_heads, head_dim))
    return fail(BQ_ERR_INVALID_ARG, "bq_kv_quantize: bad sizes");
  if (head_dim % kQK) return fail(BQ_ERR_SHAPE, "bq_kv_quantize: head_dim %lld is not a multiple of 32", (long long)head_dim);
  if (basis == BQ_BASIS_HADAMARD64 && head_dim % 64)
    return fail(BQ_ERR_SHAPE, "bq_kv_quantize: the rotated basis needs head_dim %% 64 == 0, got %lld",
                (long long)head_dim);
  if (basis == BQ_BASIS_HADAMARD64 && !core_type(type))
    return fail(BQ_ERR_UNSUPPORTED, "bq_kv_quantize: the rotated basis takes Q4_0 or Q8_0");
  if (block_values(type) != kQK)
    return fail(BQ_ERR_UNSUPPORTED, "bq_kv_quantize: k-quants are weight types, not cache types");
  const int64_t n_blocks = n_tokens * n_kv_heads * (head_dim / kQK);
  if (n_blocks == 0) return ok();
  if (!rows || !dst) return fail(BQ_ERR_INVALID_ARG, "bq_kv_quantize: null pointer");
  if (!aligned(rows, 16) || !aligned(dst, 16) || (bias && !aligned(bias, 16)))
    return fail(BQ_ERR_ALIGN, "bq_kv_quantize: rows, bias and dst must be 16-byte aligned");
  if (overlap(rows, size_t(n_blocks) * 128, dst, size_t(n_blocks) * bb) ||
      overlap(bias, size_t(n_kv_heads * head_dim) * 4, dst, size_t(n_blocks) * bb))
    return fail(BQ_ERR_INVALID_ARG, "bq_kv_quantize: dst overlaps an input");
  cudaError_t e = launch_quantize_rows(type, rows, static_cast<uint8_t *>(dst), n_blocks, head_dim / kQK, bias,
                                       n_kv_heads * (head_dim / kQK), t_stream, basis == BQ_BASIS_HADAMARD64);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_kv_quantize launch");
}

int bq_kv_write(int k_type, const float *K_rows, const float *bias, int bias_basis, int k_basis, void *K_dst,
                int v_type, const float *V_rows, void *V_dst, int64_t n_tokens, int64_t n_kv_heads,
                int64_t head_dim) {
  if (!core_type(k_type) || !core_type(v_type))
    return fail(BQ_ERR_UNSUPPORTED, "bq_kv_write: K and V types must be Q4_0 or Q8_0 (got %d, %d)", k_type, v_type);
  if (k_basis != BQ_BASIS_PLAIN && k_basis != BQ_BASIS_HADAMARD64)
    return fail(BQ_ERR_UNSUPPORTED, "bq_kv_write: unknown basis %d", k_basis);
  if (bias && k_type != BQ_TYPE_Q4_0)
    return fail(BQ_ERR_UNSUPPORTED, "bq_kv_write: a mean-centering bias requires a Q4_0 K cache");
  if (bias && bias_basis != k_basis)
    return fail(BQ_ERR_BASIS, "bq_kv_write: the bias was calibrated in basis %d, the K cache is in basis %d",
                bias_basis, k_basis);
  if (!sizes_ok(n_tokens, n_kv_heads) || !sizes_ok(n_tokens * n_kv_heads, head_dim))
    return fail(BQ_ERR_INVALID_ARG, "bq_kv_write: bad sizes");
  if (head_dim % kQK) return fail(BQ_ERR_SHAPE, "bq_kv_write: head_dim %lld is not a multiple of 32", (long long)head_dim);
  if (k_basis == BQ_BASIS_HADAMARD64 && head_dim % 64)
    return fail(BQ_ERR_SHAPE, "bq_kv_write: the rotated basis needs head_dim %% 64 == 0, got %lld", (long long)head_dim);
  const int64_t n_blocks = n_tokens * n_kv_heads * (head_dim / kQK);
  if (n_blocks == 0) return ok();
  if (!K_rows || !K_dst || !V_rows || !V_dst) return fail(BQ_ERR_INVALID_ARG, "bq_kv_write: null pointer");
  if (!aligned(K_rows, 16) || !aligned(K_dst, 16) || !aligned(V_rows, 16) || !aligned(V_dst, 16) ||
      (bias && !aligned(bias, 16)))
    return fail(BQ_ERR_ALIGN, "bq_kv_write: rows, bias and outputs must be 16-byte aligned");
  const size_t in_bytes = size_t(n_blocks) * 128, bias_bytes = size_t(n_kv_heads * head_dim) * 4;
  const size_t kb = size_t(n_blocks) * size_t(block_bytes(k_type)), vb = size_t(n_blocks) * size_t(block_bytes(v_type));
  if (overlap(K_dst, kb, K_rows, in_bytes) || overlap(K_dst, kb, V_rows, in_bytes) || overlap(K_dst, kb, bias, bias_bytes) ||
      overlap(V_dst, vb, K_rows, in_bytes) || overlap(V_dst, vb, V_rows, in_bytes) || overlap(V_dst, vb, bias, bias_bytes) ||
      overlap(K_dst, kb, V_dst, vb))
    return fail(BQ_ERR_INVALID_ARG, "bq_kv_write: an output overlaps an input or the other output");
  cudaError_t e = launch_kv_write(k_type, v_type, k_basis == BQ_BASIS_HADAMARD64, K_rows, static_cast<uint8_t *>(K_dst),
                                  V_rows, static_cast<uint8_t *>(V_dst), n_blocks, bias, n_kv_heads * (head_dim / kQK),
                                  t_stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_kv_write launch");
}

int bq_kv_bias(const float *rows, int basis, float *bias, int64_t n_tokens, int64_t n_kv_heads, int64_t head_dim) {
  if (basis != BQ_BASIS_PLAIN && basis != BQ_BASIS_HADAMARD64)
    return fail(BQ_ERR_UNSUPPORTED, "bq_kv_bias: unknown basis %d", basis);
  if (!sizes_ok(n_tokens, n_kv_heads) || !sizes_ok(n_tokens * n_kv_heads, head_dim) || n_tokens < 1)
    return fail(BQ_ERR_INVALID_ARG, "bq_kv_bias: bad sizes (n_tokens must be at least 1)");
  if (head_dim % kQK) return fail(BQ_ERR_SHAPE, "bq_kv_bias: head_dim %lld is not a multiple of 32", (long long)head_dim);
  if (basis == BQ_BASIS_HADAMARD64 && head_dim % 64)
    return fail(BQ_ERR_SHAPE, "bq_kv_bias: the rotated basis needs head_dim %% 64 == 0");
  const int64_t row_len = n_kv_heads * head_dim;
  if (row_len == 0) return ok();
  if (!rows || !bias) return fail(BQ_ERR_INVALID_ARG, "bq_kv_bias: null pointer");
  if (!aligned(rows, 16) || !aligned(bias, 4)) return fail(BQ_ERR_ALIGN, "bq_kv_bias: rows 16-byte, bias 4-byte aligned");
  if (overlap(bias, size_t(row_len) * 4, rows, size_t(n_tokens) * size_t(row_len) * 4))
    return fail(BQ_ERR_INVALID_ARG, "bq_kv_bias: bias overlaps the rows");
  cudaError_t e = launch_kv_bias(rows, bias, n_tokens, row_len, basis == BQ_BASIS_HADAMARD64, t_stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_kv_bias launch");
}

int bq_block_dots(int type, const void *W, const void *xq, int32_t *out, int64_t M, int64_t K) {
  const int bb = block_bytes(type);
  if (!bb) return fail(BQ_ERR_UNSUPPORTED, "bq_block_dots: unknown type %d", type);
  if (!core_type(type)) return fail(BQ_ERR_UNSUPPORTED, "bq_block_dots: Q4_0 or Q8_0 weights only");
  if (!sizes_ok(M, K)) return fail(BQ_ERR_INVALID_ARG, "bq_block_dots: bad sizes");
  if (K % kQK) return fail(BQ_ERR_SHAPE, "bq_block_dots: K %lld is not a multiple of 32", (long long)K);
  if (M == 0 || K == 0) return ok();
  if (!W || !xq || !out) return fail(BQ_ERR_INVALID_ARG, "bq_block_dots: null pointer");
  if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(out, 4)) return fail(BQ_ERR_ALIGN, "bq_block_dots: alignment");
  cudaError_t e = launch_block_dots(type, static_cast<const uint8_t *>(W), static_cast<const uint8_t *>(xq), out, M, K,
                                    t_stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "bq_block_dots launch");
}

}  // extern "C"
