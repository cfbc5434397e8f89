// probe_mma.cu — measurement probes (libbq_probe.so, not part of the libbq
// ABI): the issue rate of the legacy warp-level tensor-core instructions on
// this GPU, the denominator the prefill GEMM's int8 target is stated against
// (sm_103a has no int8 form of tcgen05.mma, so the int8 tensor path left is
// mma.sync with s8 operands; its f16 form is measured beside it); the issue
// rate of dp4a; and the read rate of 1-D bulk copies by copy size, which
// sets the GEMV's stage size.
//
// Every warp issues long runs of independent mma.sync instructions on
// register operands (no memory traffic); the accumulators are summed and
// stored at the end so that no instruction is dead. Timed with CUDA events
// on the legacy default stream.
#include <cstdint>
#include <cuda_runtime.h>

#include "bq_device.cuh"

namespace {

constexpr int kChains = 8;  // independent accumulators per warp: covers the pipeline latency

__global__ void __launch_bounds__(256) k_mma_s8(int iters, int *out) {
  const uint32_t t = threadIdx.x + 1;
  const uint32_t a0 = t * 0x01010101u, a1 = t * 0x02020202u, a2 = t * 0x03030303u, a3 = t * 0x05050505u;
  const uint32_t b0 = t * 0x07070707u, b1 = t * 0x0b0b0b0bu;
  int c[kChains][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < kChains; ++k)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+r"(c[k][0]), "+r"(c[k][1]), "+r"(c[k][2]), "+r"(c[k][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s += c[k][0] ^ c[k][1] ^ c[k][2] ^ c[k][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(256) k_mma_f16(int iters, int *out) {
  const uint32_t t = threadIdx.x & 7;
  // small exact binary16 pairs (1.0 + t/8), so the sums stay finite
  const uint32_t h = 0x3c00u + (t << 7);
  const uint32_t a = h | (h << 16);
  float c[kChains][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < kChains; ++k)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+f"(c[k][0]), "+f"(c[k][1]), "+f"(c[k][2]), "+f"(c[k][3])
          : "r"(a), "r"(a), "r"(a), "r"(a), "r"(a), "r"(a));
  }
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s += c[k][0] + c[k][1] + c[k][2] + c[k][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = __float_as_int(s);
}

// Integer dot-product issue rate: every thread runs kChains independent
// dp4a.u32.s32 chains (kind 2) or, for comparison, 32-bit integer
// multiply-add chains (kind 3).
__global__ void __launch_bounds__(256) k_dp4a(int iters, int kind, int *out) {
  const uint32_t t = threadIdx.x * 0x01010101u + 0x03050709u;
  int c[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k) c[k] = int(t) + k;
  if (kind == 2) {
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int k = 0; k < kChains; ++k)
        asm volatile("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(c[k]) : "r"(t + uint32_t(k)), "r"(t ^ 0x5a5a5a5au));
    }
  } else {
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int k = 0; k < kChains; ++k)
        asm volatile("mad.lo.s32 %0, %1, %2, %0;" : "+r"(c[k]) : "r"(int(t) + k), "r"(int(t ^ 0x5a5a5a5au)));
    }
  }
  int s = 0;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s ^= c[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// One CTA per SM, one thread streams the CTA's contiguous range of `src`
// with 1-D bulk copies of `sz` bytes into a ring of `depth` shared-memory
// slots (one mbarrier each), issuing a slot's next copy as soon as its
// previous one landed. Waits are bounded; `err` gets 1 if one ran out.
__global__ void __launch_bounds__(32, 1) k_bulk_stream(const uint8_t *src, size_t per_cta, int sz, int depth,
                                                      unsigned *err) {
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + size_t(depth) * sz);
  if (threadIdx.x != 0) return;
  for (int s = 0; s < depth; ++s) bq::mbar_init(&bar[s], 1);
  bq::fence_mbar_init();
  const uint8_t *base = src + per_cta * blockIdx.x;
  const int64_t n = int64_t(per_cta / sz);
  const uint64_t pol = bq::l2_evict_first_policy();
  int64_t issued = 0;
  for (int64_t j = 0; j < n; ++j) {
    const int s = int(j % depth);
    if (j >= depth && !bq::mbar_wait_bounded(&bar[s], uint32_t(((j / depth) - 1) & 1), 1u << 24)) {
      atomicOr(err, 1u);
      break;
    }
    bq::mbar_arrive_expect_tx(&bar[s], uint32_t(sz));
    bq::bulk_g2s_hint(sm + size_t(s) * sz, base + j * sz, uint32_t(sz), &bar[s], pol);
    issued = j + 1;
  }
  for (int s = 0; s < depth && s < issued; ++s) {
    const int64_t last = s + depth * ((issued - 1 - s) / depth);
    if (!bq::mbar_wait_bounded(&bar[s], uint32_t((last / depth) & 1), 1u << 24)) atomicOr(err, 1u);
  }
}

}  // namespace

// Read rate (GB/s) of 1-D bulk copies of `copy_bytes` (a multiple of 16,
// depth * copy_bytes <= 200 KB) over `total_bytes` of device memory
// allocated here, one CTA per SM and `depth` copies in flight per SM; best of
// three runs. Returns 0, -1 on a bad argument, -5 when a CUDA call fails or a
// wait ran out.
extern "C" int bq_probe_bulk_rate(int copy_bytes, int depth, size_t total_bytes, double *gbs) {
  if (copy_bytes < 16 || copy_bytes % 16 || depth < 1 || size_t(depth) * copy_bytes > (200u << 10) || !gbs)
    return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -5;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -5;
  const size_t per_cta = total_bytes / size_t(sms) / size_t(copy_bytes) * size_t(copy_bytes);
  if (per_cta == 0) return -1;
  uint8_t *buf = nullptr;
  unsigned *err = nullptr;
  if (cudaMalloc(&buf, per_cta * sms) != cudaSuccess) return -5;
  if (cudaMalloc(&err, sizeof(unsigned)) != cudaSuccess) {
    cudaFree(buf);
    return -5;
  }
  cudaMemset(buf, 1, per_cta * sms);
  cudaMemset(err, 0, sizeof(unsigned));
  const int smem = depth * copy_bytes + 8 * depth;
  cudaError_t e = cudaFuncSetAttribute(k_bulk_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  float best = 0.0f;
  for (int rep = 0; rep < 3 && e == cudaSuccess; ++rep) {
    cudaEventRecord(e0);
    k_bulk_stream<<<sms, 32, smem>>>(buf, per_cta, copy_bytes, depth, err);
    cudaEventRecord(e1);
    e = cudaEventSynchronize(e1);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess && (best == 0.0f || ms < best)) best = ms;
  }
  unsigned herr = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&herr, err, sizeof(unsigned), cudaMemcpyDeviceToHost);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(buf);
  cudaFree(err);
  if (e != cudaSuccess || herr || best <= 0.0f) return -5;
  *gbs = double(per_cta) * sms / (double(best) * 1e-3) / 1e9;
  return 0;
}

// Thread-instruction rate (tera-instructions per second) of kind 2 = dp4a,
// kind 3 = 32-bit integer multiply-add, each as independent chains.
extern "C" int bq_probe_int_rate(int kind, int iters, int ctas_per_sm, double *tinst) {
  if ((kind != 2 && kind != 3) || iters < 1 || ctas_per_sm < 1 || !tinst) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -5;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -5;
  const int grid = sms * ctas_per_sm, block = 256;
  int *out = nullptr;
  if (cudaMalloc(&out, size_t(grid) * block * sizeof(int)) != cudaSuccess) return -5;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  k_dp4a<<<grid, block>>>(iters / 8 + 1, kind, out);
  cudaEventRecord(e0);
  k_dp4a<<<grid, block>>>(iters, kind, out);
  cudaEventRecord(e1);
  cudaError_t err = cudaEventSynchronize(e1);
  float ms = 0.0f;
  if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
  if (err == cudaSuccess) err = cudaGetLastError();
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(out);
  if (err != cudaSuccess || ms <= 0.0f) return -5;
  *tinst = double(grid) * block * double(iters) * kChains / (double(ms) * 1e-3) / 1e12;
  return 0;
}

// Tensor-op rate of mma.sync on the current device in tera-ops per second
// (2 * m * n * k per instruction): kind 0 = m16n8k32 s8 x s8 -> s32, kind 1
// = m16n8k16 f16 x f16 -> f32. Grid: ctas_per_sm x SMs of 8 warps. Returns 0
// on success, -1 on a bad argument, -5 when a CUDA call fails.
extern "C" int bq_probe_mma_rate(int kind, int iters, int ctas_per_sm, double *tops) {
  if ((kind != 0 && kind != 1) || iters < 1 || ctas_per_sm < 1 || !tops) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -5;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -5;
  const int grid = sms * ctas_per_sm, block = 256;
  int *out = nullptr;
  if (cudaMalloc(&out, size_t(grid) * block * sizeof(int)) != cudaSuccess) return -5;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  auto launch = [&](int it) {
    if (kind == 0)
      k_mma_s8<<<grid, block>>>(it, out);
    else
      k_mma_f16<<<grid, block>>>(it, out);
  };
  launch(iters / 8 + 1);  // warm-up
  cudaEventRecord(e0);
  launch(iters);
  cudaEventRecord(e1);
  cudaError_t err = cudaEventSynchronize(e1);
  float ms = 0.0f;
  if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
  if (err == cudaSuccess) err = cudaGetLastError();
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(out);
  if (err != cudaSuccess || ms <= 0.0f) return -5;
  const double ops_per_mma = kind == 0 ? 2.0 * 16 * 8 * 32 : 2.0 * 16 * 8 * 16;
  const double mmas = double(grid) * (block / 32) * double(iters) * kChains;
  *tops = mmas * ops_per_mma / (double(ms) * 1e-3) / 1e12;
  return 0;
}
