// gemm_noalloc.cu — bq_gemm_noalloc: the prefill GEMM for callers that
// cannot allocate device memory at call time and have no workspace to lend
// (for example a plugin hook that must not call cudaMalloc while it runs, or
// a process whose device memory is fixed once it has started).
//
// The quantized activations, which bq_gemm keeps in the caller's workspace,
// live here in a file-scope device array of fixed size instead. Every GPU
// that loads the library holds that array until the process exits. The
// kernels are the ones bq_gemm launches, except that the tcgen05 path, whose
// binary16 activation codes take twice the bytes of Q8_0 blocks, is used only
// where its activations fit the array; otherwise the mma.sync path runs.
#include <mutex>

#include "bq.h"
#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {
namespace {

// One shared scratch array per device. Host code must not pass the symbol's
// name to a kernel: on the host it is only a stand-in, not a device address.
static __device__ __align__(256) uint8_t g_noalloc_scratch[BQ_GEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does this, with that device current).
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace bq

extern "C" int bq_gemm_noalloc(int type, const void *W, const float *X, float *Y, int64_t M, int64_t N,
                               int64_t K) {
  using namespace bq;
  if (type != BQ_TYPE_Q8_0 && type != BQ_TYPE_Q4_0)
    return report_error(BQ_ERR_UNSUPPORTED, "bq_gemm_noalloc: unknown type %d", type);
  if (type != BQ_TYPE_Q8_0)
    return report_error(BQ_ERR_UNSUPPORTED, "bq_gemm_noalloc: only Q8_0 weights are supported");
  if (M < 0 || N < 0 || K < 0)
    return report_error(BQ_ERR_INVALID_ARG, "bq_gemm_noalloc: negative size");
  if (K % kQK)
    return report_error(BQ_ERR_SHAPE, "bq_gemm_noalloc: K %lld is not a multiple of 32", (long long)K);
  if (M > 0x7fffffffll || N > 0x7fffffffll || K > 0x7fffffffll)
    return report_error(BQ_ERR_SHAPE, "bq_gemm_noalloc: M, N and K must be below 2^31");
  if (M == 0 || N == 0) return report_ok();
  size_t need = 0;
  const PrefillPath path = prefill_path(M, N, K, size_t(BQ_GEMM_NOALLOC_SCRATCH_BYTES), &need);
  if (need > size_t(BQ_GEMM_NOALLOC_SCRATCH_BYTES))
    return report_error(BQ_ERR_WORKSPACE, "bq_gemm_noalloc: N x K/32 x 34 = %zu bytes of quantized activations exceed the "
             "%d-byte static scratch; use bq_gemm with a workspace",
             need, BQ_GEMM_NOALLOC_SCRATCH_BYTES);
  if (!Y || (K > 0 && (!W || !X)))
    return report_error(BQ_ERR_INVALID_ARG, "bq_gemm_noalloc: null pointer");
  const uintptr_t w = reinterpret_cast<uintptr_t>(W), x = reinterpret_cast<uintptr_t>(X),
                  y = reinterpret_cast<uintptr_t>(Y);
  if ((y & 3) || (K > 0 && ((w & 15) || (x & 15))))
    return report_error(BQ_ERR_ALIGN, "bq_gemm_noalloc: W and X must be 16-byte aligned, Y 4-byte aligned");
  const size_t ybytes = size_t(M) * size_t(N) * 4;
  const size_t wbytes = size_t(M) * size_t(K / kQK) * Fmt<kTypeQ8_0>::kBytes;
  const size_t xbytes = size_t(N) * size_t(K) * 4;
  if ((y < w + wbytes && w < y + ybytes) || (y < x + xbytes && x < y + ybytes))
    return report_error(BQ_ERR_INVALID_ARG, "bq_gemm_noalloc: Y overlaps an input");
  cudaStream_t stream = static_cast<cudaStream_t>(bq_get_stream());
  cudaError_t e;
  if (K == 0) {
    e = cudaMemsetAsync(Y, 0, ybytes, stream);
  } else {
    void *scratch = nullptr;
    e = scratch_address(&scratch);
    if (e == cudaSuccess) e = launch_prefill(path, static_cast<const uint8_t *>(W), X, Y, M, N, K, scratch, stream);
  }
  if (e != cudaSuccess)
    return report_error(BQ_ERR_CUDA, "bq_gemm_noalloc: %s (%s)", cudaGetErrorName(e), cudaGetErrorString(e));
  return report_ok();
}
