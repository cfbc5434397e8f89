// bq_device.cuh — device helpers shared by the libbq kernels (sm_103a).
//
// Block rules (Q4_0 / Q8_0): 32 values share one binary16 scale; Q4_0 stores
// 4-bit codes in 18 bytes ("llama.cpp 原理：如何在普通硬件跑本地大模型",
// §量化：内存真正去哪了), Q8_0 int8 codes in 34 bytes ("05. llama.cpp：从 GGUF
// 文件到本地推理服务", §量化类型); symmetric, value = scale * q, no zero point
// (lpnh.cn KV-cache article, §问题).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace bq {

constexpr int kQK = 32;
constexpr int kTypeQ4_0 = 2;
constexpr int kTypeQ8_0 = 8;
constexpr unsigned kFull = 0xffffffffu;

// error bits of the device error word
constexpr unsigned kErrTimeout = 1u;

template <int TYPE> struct Fmt;
template <> struct Fmt<kTypeQ4_0> {
  static constexpr int kBytes = 18;   // 2-byte scale + 16 bytes of nibbles
  static constexpr int kQmax = 7;
  static constexpr int kQmin = -8;
};
template <> struct Fmt<kTypeQ8_0> {
  static constexpr int kBytes = 34;   // 2-byte scale + 32 int8
  static constexpr int kQmax = 127;
  static constexpr int kQmin = -127;
};

// ---------------------------------------------------------------- quantize --

// max over the 8 lanes (aligned groups of 8) that hold one 32-value block
__device__ __forceinline__ float group8_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 1));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 2));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 4));
  return v;
}

__device__ __forceinline__ int group8_sum(int v) {
  v += __shfl_xor_sync(kFull, v, 1);
  v += __shfl_xor_sync(kFull, v, 2);
  v += __shfl_xor_sync(kFull, v, 4);
  return v;
}

// scale of a block: d = amax / qmax (IEEE fp32 division), stored as binary16
// rounded to nearest even; `ds` is the stored scale read back as fp32.
template <int TYPE>
__device__ __forceinline__ void block_scale(float amax, uint16_t &bits, float &ds) {
  const float d = __fdiv_rn(amax, static_cast<float>(Fmt<TYPE>::kQmax));
  const __half h = __float2half_rn(d);
  bits = __half_as_ushort(h);
  ds = __half2float(h);
}

// code of one value: round-half-even of the IEEE fp32 quotient x / ds, clamped.
//
// The quotient is formed as r = x * rn(1/ds) (one correctly rounded
// reciprocal per block, one multiply per value). r is within 2 ulp of the
// correctly rounded quotient q = rn(x / ds), so rint(r) == rint(q) unless a
// half-integer lies within that distance of r; values whose distance to the
// nearest integer is that close to 0.5 (a band of 4e-5 * max(|r|, 1), far
// wider than 2 ulp) take the exact IEEE division instead. The result is
// bit-identical to rint(rn(x / ds)) for every input; only the cost differs.
template <int TYPE>
__device__ __forceinline__ int code_of(float x, float ds, float inv) {
  float r = __fmul_rn(x, inv);
  float n = rintf(r);
  if (fabsf(__fsub_rn(r, n)) > 0.5f - 4e-5f * fmaxf(fabsf(r), 1.0f)) n = rintf(__fdiv_rn(x, ds));
  const int q = __float2int_rz(n);  // n is integral
  return min(max(q, Fmt<TYPE>::kQmin), Fmt<TYPE>::kQmax);
}

__device__ __forceinline__ float amax4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// One block held by 8 lanes (lane j of the group holds elements 4j..4j+3).
// Produces, for lane j, the 4 code bytes of elements 4j..4j+3 packed
// little-endian as int8 (Q8_0) or as unsigned nibbles q + 8 (Q4_0, one nibble
// per byte), the scale bits, and the code sum of the whole block.
template <int TYPE>
struct BlockCodes {
  uint32_t bytes4;   // 4 codes, one per byte
  uint16_t scale;    // binary16 bits of the stored scale
  int sum;           // sum of the 32 signed codes (over the 8-lane group)
};

template <int TYPE>
__device__ __forceinline__ BlockCodes<TYPE> quantize_block8(float4 v) {
  BlockCodes<TYPE> r;
  float ds;
  block_scale<TYPE>(group8_max(amax4(v)), r.scale, ds);
  int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
  if (ds != 0.0f) {  // a zero scale (all-zero or underflowing block) gives all codes 0
    const float inv = __frcp_rn(ds);
    q0 = code_of<TYPE>(v.x, ds, inv);
    q1 = code_of<TYPE>(v.y, ds, inv);
    q2 = code_of<TYPE>(v.z, ds, inv);
    q3 = code_of<TYPE>(v.w, ds, inv);
  }
  if (TYPE == kTypeQ4_0) {
    r.bytes4 = uint32_t(q0 + 8) | (uint32_t(q1 + 8) << 8) | (uint32_t(q2 + 8) << 16) |
               (uint32_t(q3 + 8) << 24);
  } else {
    r.bytes4 = (uint32_t(q0) & 0xffu) | ((uint32_t(q1) & 0xffu) << 8) |
               ((uint32_t(q2) & 0xffu) << 16) | ((uint32_t(q3) & 0xffu) << 24);
  }
  r.sum = group8_sum(q0 + q1 + q2 + q3);
  return r;
}

// Q4_0 packing across the 8-lane group: byte i of qs holds element i in its
// low nibble and element i+16 in its high nibble. Lane j < 4 returns qs bytes
// 4j..4j+3 (lanes 4..7 hold the high-nibble halves and return garbage).
__device__ __forceinline__ uint32_t pack_q4_nibbles(uint32_t nib4) {
  const uint32_t hi = __shfl_down_sync(kFull, nib4, 4);
  return nib4 | (hi << 4);
}

// ------------------------------------------------------------- block dots --

// a: 4 unsigned bytes, b: 4 signed bytes
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Integer dot of one Q4_0 block (qs as 4 words) with one Q8_0 block (codes as
// 8 words, xsum = sum of its 32 codes): sum_j (nib_j - 8) * qx_j, computed as
// sum_j nib_j * qx_j - 8 * xsum. The high nibbles are used in place (bytes
// 16 * nib, no shift): their dot is 16 times the wanted one, so it is shifted
// right by 4 at the end, which is exact because every term is a multiple of
// 16. All of it is exact in int32.
__device__ __forceinline__ int sumi_q4_q8(const uint32_t qs[4], const uint32_t xw[8], int xsum) {
  int lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lo = dp4a_us(qs[i] & 0x0f0f0f0fu, xw[i], lo);      // elements 4i..4i+3
    hi = dp4a_us(qs[i] & 0xf0f0f0f0u, xw[4 + i], hi);  // 16 x elements 16+4i..
  }
  return lo + (hi >> 4) - 8 * xsum;
}

// Integer dot of one Q8_0 block with another.
__device__ __forceinline__ int sumi_q8_q8(const uint32_t qw[8], const uint32_t xw[8]) {
  int s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) s = dp4a_ss(qw[i], xw[i], s);
  return s;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xffffu)));
}

// ------------------------------------------------------------------ memory --

__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
  return __ldcs(reinterpret_cast<const float4 *>(p));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------- mbarrier + TMA ----

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete, at most `limit` polls (each
// poll may suspend the thread for a bounded, hardware-chosen time). Returns
// false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream start, and
// wait until the previous one has completed and its writes are visible. Both
// are no-ops when the launch did not opt in.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Ask L2 to fetch [src, src + bytes) from memory; no completion, no data
// returned (src and bytes multiples of 16).
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace bq
