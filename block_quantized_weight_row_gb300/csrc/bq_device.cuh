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
// legacy types with a fifth bit and/or a minimum (below)
constexpr int kTypeQ4_1 = 3;
constexpr int kTypeQ5_0 = 6;
constexpr int kTypeQ5_1 = 7;
// k-quants: super-blocks of 256 weights (below)
constexpr int kTypeQ4_K = 12;
constexpr int kTypeQ6_K = 14;
constexpr int kQK_K = 256;
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
template <> struct Fmt<kTypeQ4_1> { static constexpr int kBytes = 20; };  // d, m, 16 nibble bytes
template <> struct Fmt<kTypeQ5_0> { static constexpr int kBytes = 22; };  // d, qh, 16 nibble bytes
template <> struct Fmt<kTypeQ5_1> { static constexpr int kBytes = 24; };  // d, m, qh, 16 nibble bytes
template <> struct Fmt<kTypeQ4_K> { static constexpr int kBytes = 144; };  // per 256: d, dmin, 12 scale bytes, 128 code bytes
template <> struct Fmt<kTypeQ6_K> { static constexpr int kBytes = 210; };  // per 256: ql 128, qh 64, 16 int8 scales, d
template <int TYPE> struct IsKQuant { static constexpr bool kV = false; };
template <> struct IsKQuant<kTypeQ4_K> { static constexpr bool kV = true; };
template <> struct IsKQuant<kTypeQ6_K> { static constexpr bool kV = true; };

// Legacy types ("05. llama.cpp：从 GGUF 文件到本地推理服务", §量化类型: legacy
// formats keep one FP16 scale per 32 weights, and "_1" adds a minimum). The
// layouts are this library's reading: scale first, then the minimum (_1),
// then bit 4 of every code as one little-endian 32-bit word (5-bit types),
// then the low 4 bits in Q4_0's nibble order. Codes are unsigned u; the value
// is d * u + m (_1) or d * (u - 16) (Q5_0).
template <int TYPE> struct Legacy { static constexpr bool kIs = false; };
template <> struct Legacy<kTypeQ4_1> {
  static constexpr bool kIs = true, kAffine = true;
  static constexpr int kUmax = 15, kQh = -1, kQs = 4;  // byte offsets of qh and the nibbles
};
template <> struct Legacy<kTypeQ5_0> {
  static constexpr bool kIs = true, kAffine = false;
  static constexpr int kUmax = 31, kQh = 2, kQs = 6;
};
template <> struct Legacy<kTypeQ5_1> {
  static constexpr bool kIs = true, kAffine = true;
  static constexpr int kUmax = 31, kQh = 4, kQs = 8;
};

// ---------------------------------------------------------------- quantize --

// scale of a block: d = amax / qmax (IEEE fp32 division), stored as binary16
// rounded to nearest even; `ds` is the stored scale read back as fp32.
template <int TYPE>
__device__ __forceinline__ void block_scale(float amax, uint16_t &bits, float &ds) {
  const float d = __fdiv_rn(amax, static_cast<float>(Fmt<TYPE>::kQmax));
  const __half h = __float2half_rn(d);
  bits = __half_as_ushort(h);
  ds = __half2float(h);
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Code of one value: round-half-even of the IEEE fp32 quotient x / ds,
// clamped to the type's range. ds > 0 with inv ~ 1/ds, or ds = 0 with
// inv = 0, which gives code 0 (the exact path is never taken then).
//
// r = x * inv with inv within 1 ulp of 1/ds is within 3 ulp of the correctly
// rounded quotient q = rn(x / ds); |r| < 256 for every block (|x| <= amax and
// ds ~ amax / qmax), so 3 ulp < 1e-4. Adding 1.5 * 2^23 rounds r to an integer
// (ties to even, the add is correctly rounded) and leaves that integer in the
// low bits of the sum. When r is farther than 0.4999 from its integer (a tie
// may lie between r and q), the value takes the exact division instead; in all
// other cases rint(r) == rint(q). The result is bit-identical to
// clamp(rint(rn(x / ds))) for every input; only the cost differs.
template <int TYPE>
__device__ __forceinline__ int code_of(float x, float ds, float inv) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  const float r = __fmul_rn(x, inv);
  const float t = __fadd_rn(r, kMagic);
  int q = __float_as_int(t) - 0x4B400000;
  if (fabsf(__fsub_rn(r, __fsub_rn(t, kMagic))) > 0.4999f) q = __float2int_rn(__fdiv_rn(x, ds));
  return min(max(q, Fmt<TYPE>::kQmin), Fmt<TYPE>::kQmax);
}

__device__ __forceinline__ uint32_t pack_bytes(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  // byte 0 of each argument, in order (two's complement low byte for codes)
  return __byte_perm(__byte_perm(b0, b1, 0x3340), __byte_perm(b2, b3, 0x3340), 0x5410);
}

// One lane quantizes one whole 32-value block v[0..31]: the scale bits, the
// block's code bytes as words (Q4_0: 4 words, byte i = (q[i]+8) | (q[i+16]+8)
// << 4; Q8_0: 8 words of int8 codes) and, when asked, the sum of the codes.
//
// Common path, per value: r = x * inv, t = r + M with M = 1.5 * 2^23 (+ 8 for
// Q4_0, the code bias): t is rint(r) + M exactly (ties to even; 8 is even, so
// the bias does not change a tie's parity), and the low byte of t's bits is
// already the stored code byte (q + 8 for Q4_0, q mod 256 for Q8_0). The
// block's largest |r - rint(r)| decides, once per block, whether any value may
// lie near a tie (> 0.4999, see code_of); then, and when the stored scale is a
// subnormal binary16 (whose rounding can put |x / ds| above the code range),
// the whole block takes code_of's exact, clamped path instead. With a normal
// scale, |x / ds| <= qmax * (1 + 2^-11) + 3 ulp < qmax + 0.5, so no clamp is
// needed. Every path gives bit-identical codes.
// Code bytes of a block as words from the per-value bits t (low byte = the
// stored code byte, see quantize_block_lane).
template <int TYPE>
__device__ __forceinline__ void pack_code_words(const uint32_t (&tb)[32], uint32_t *words) {
  if (TYPE == kTypeQ4_0) {
    // low byte of each t is q + 8 in 0..15: low nibbles from elements 4i..4i+3,
    // high nibbles from elements 16+4i..16+4i+3
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = pack_bytes(tb[4 * i], tb[4 * i + 1], tb[4 * i + 2], tb[4 * i + 3]);
      const uint32_t hi = pack_bytes(tb[16 + 4 * i], tb[16 + 4 * i + 1], tb[16 + 4 * i + 2], tb[16 + 4 * i + 3]);
      words[i] = lo + (hi << 4);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) words[i] = pack_bytes(tb[4 * i], tb[4 * i + 1], tb[4 * i + 2], tb[4 * i + 3]);
  }
}

template <int TYPE>
__device__ __forceinline__ float block_amax(const float (&v)[32]) {
  // max of |v| as a 5-level tree (exact in any order)
  float m[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) m[j] = fmaxf(fabsf(v[j]), fabsf(v[j + 16]));
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
  return m[0];
}

// The common path of quantize_block_lane alone: false when the block needs the
// exact path (a value near a tie, or a subnormal scale), and then `words` is
// not written. Lets a caller that can fetch the block again drop v early.
template <int TYPE>
__device__ __forceinline__ bool quantize_block_lane_fast(const float (&v)[32], uint16_t &scale, uint32_t *words) {
  float ds;
  block_scale<TYPE>(block_amax<TYPE>(v), scale, ds);
  const float inv = ds > 0.0f ? rcp_approx(ds) : 0.0f;
  constexpr float kMagic = 12582912.0f + float(TYPE == kTypeQ4_0 ? 8 : 0);
  uint32_t tb[32];
  float dmax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float r = __fmul_rn(v[j], inv);
    const float t = __fadd_rn(r, kMagic);
    tb[j] = __float_as_uint(t);
    dmax = fmaxf(dmax, fabsf(__fsub_rn(r, __fsub_rn(t, kMagic))));
  }
  if (dmax > 0.4999f || (ds > 0.0f && ds < 6.103515625e-05f)) return false;
  pack_code_words<TYPE>(tb, words);
  return true;
}

// The exact path of quantize_block_lane alone (any block).
template <int TYPE>
__device__ __forceinline__ void quantize_block_lane_exact(const float (&v)[32], uint16_t &scale, uint32_t *words) {
  float ds;
  block_scale<TYPE>(block_amax<TYPE>(v), scale, ds);
  const float inv = ds > 0.0f ? rcp_approx(ds) : 0.0f;
  constexpr uint32_t kMagicBits = 0x4B400000u + uint32_t(TYPE == kTypeQ4_0 ? 8 : 0);
  uint32_t tb[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) tb[j] = kMagicBits + uint32_t(code_of<TYPE>(v[j], ds, inv));
  pack_code_words<TYPE>(tb, words);
}

template <int TYPE, bool SUM>
__device__ __forceinline__ void quantize_block_lane(const float (&v)[32], uint16_t &scale, uint32_t *words,
                                                    int &sum) {
  float ds;
  block_scale<TYPE>(block_amax<TYPE>(v), scale, ds);
  // a zero scale (all-zero block, or a scale that underflows binary16) gives
  // inv = 0 and so every code 0, without a branch
  const float inv = ds > 0.0f ? rcp_approx(ds) : 0.0f;
  constexpr int kBias = (TYPE == kTypeQ4_0) ? 8 : 0;
  constexpr float kMagic = 12582912.0f + float(kBias);
  constexpr uint32_t kMagicBits = 0x4B400000u + uint32_t(kBias);
  uint32_t tb[32];
  float dmax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float r = __fmul_rn(v[j], inv);
    const float t = __fadd_rn(r, kMagic);
    tb[j] = __float_as_uint(t);
    dmax = fmaxf(dmax, fabsf(__fsub_rn(r, __fsub_rn(t, kMagic))));
  }
  if (dmax > 0.4999f || (ds > 0.0f && ds < 6.103515625e-05f)) {  // rare: near a tie, or a subnormal scale
#pragma unroll
    for (int j = 0; j < 32; ++j) tb[j] = kMagicBits + uint32_t(code_of<TYPE>(v[j], ds, inv));
  }
  if (SUM) {  // sum of the codes: sum of the bits minus 32 magic words (exact modulo 2^32)
    uint32_t t2[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) t2[j] = tb[j] + tb[j + 16];
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
      for (int j = 0; j < w; ++j) t2[j] += t2[j + w];
    sum = int(t2[0] - 32u * kMagicBits);
  }
  pack_code_words<TYPE>(tb, words);
}

// One Q8_0 block held by 8 lanes (lane j of an aligned group of 8 holds
// elements 4j..4j+3): the scale bits, the lane's 4 codes as one word of int8
// and the block's code sum, every lane of the group getting scale and sum.
// Straight-line code apart from the rare exact-division path of code_of.
__device__ __forceinline__ void quantize_block_8lanes(float4 v, uint16_t &scale, uint32_t &word, int &sum) {
  float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
  m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
  m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
  float ds;
  block_scale<kTypeQ8_0>(m, scale, ds);
  // a zero scale (all-zero block, or a scale that underflows binary16) gives
  // inv = 0 and so every code 0, without a branch
  const float inv = ds > 0.0f ? rcp_approx(ds) : 0.0f;
  const int q0 = code_of<kTypeQ8_0>(v.x, ds, inv), q1 = code_of<kTypeQ8_0>(v.y, ds, inv);
  const int q2 = code_of<kTypeQ8_0>(v.z, ds, inv), q3 = code_of<kTypeQ8_0>(v.w, ds, inv);
  word = pack_bytes(uint32_t(q0), uint32_t(q1), uint32_t(q2), uint32_t(q3));
  int s = q0 + q1 + q2 + q3;
  s += __shfl_xor_sync(kFull, s, 1);
  s += __shfl_xor_sync(kFull, s, 2);
  s += __shfl_xor_sync(kFull, s, 4);
  sum = s;
}

// Four int8 codes (one word, code 0 in the low byte) as two words of two
// binary16 values each, exactly: the biased byte q + 128 is the low mantissa
// byte of the binary16 number 1024 + (q + 128) (exponent byte 0x64), and
// subtracting 1152 leaves q. Every step is exact for q in [-128, 127].
__device__ __forceinline__ uint2 codes_to_f16x2(uint32_t w) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
  uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
  return make_uint2(lo, hi);
}

// Load one 32-value fp32 block (16-byte aligned) as 8 vectors.
template <bool STREAM>
__device__ __forceinline__ void load_block(const float *p, float (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 f = STREAM ? __ldcs(reinterpret_cast<const float4 *>(p) + c)
                            : __ldcg(reinterpret_cast<const float4 *>(p) + c);
    v[4 * c] = f.x;
    v[4 * c + 1] = f.y;
    v[4 * c + 2] = f.z;
    v[4 * c + 3] = f.w;
  }
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

// ---------------------------------------------------------- legacy types --

// One block of a legacy type, by a single lane, exactly: symmetric Q5_0
// d = amax / 15, u = clamp(rn(x / d16), -16, 15) + 16; affine "_1" types
// m = min x, d = (max x - m) / umax, u = clamp(rn((x - m16) / d16), 0, umax),
// every step one IEEE fp32 operation on the stored binary16 values. `out` is
// the block, 2-byte aligned.
template <int TYPE>
__device__ __forceinline__ void legacy_quantize_block(const float (&v)[32], uint16_t *out) {
  using L = Legacy<TYPE>;
  uint32_t u[32];
  uint16_t d16, m16 = 0;
  if (L::kAffine) {
    float mn = v[0], mx = v[0];
#pragma unroll
    for (int j = 1; j < 32; ++j) {  // strict comparisons: the first of equal extremes is kept
      if (v[j] < mn) mn = v[j];
      if (v[j] > mx) mx = v[j];
    }
    const __half hd = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), float(L::kUmax)));
    const __half hm = __float2half_rn(mn);
    d16 = __half_as_ushort(hd);
    m16 = __half_as_ushort(hm);
    const float ds = __half2float(hd), ms = __half2float(hm);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      int q = 0;
      if (ds != 0.0f) q = int(rintf(__fdiv_rn(__fsub_rn(v[j], ms), ds)));
      u[j] = uint32_t(min(max(q, 0), L::kUmax));
    }
  } else {
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
    const __half hd = __float2half_rn(__fdiv_rn(amax, 15.0f));
    d16 = __half_as_ushort(hd);
    const float ds = __half2float(hd);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      int q = 0;
      if (ds != 0.0f) q = int(rintf(__fdiv_rn(v[j], ds)));
      u[j] = uint32_t(min(max(q, -16), 15) + 16);
    }
  }
  int o = 0;
  out[o++] = d16;
  if (L::kAffine) out[o++] = m16;
  if (L::kQh >= 0) {
    uint32_t qh = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) qh |= ((u[j] >> 4) & 1u) << j;
    out[o++] = uint16_t(qh & 0xffffu);
    out[o++] = uint16_t(qh >> 16);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t b0 = (u[2 * k] & 15u) | ((u[2 * k + 16] & 15u) << 4);
    const uint32_t b1 = (u[2 * k + 1] & 15u) | ((u[2 * k + 17] & 15u) << 4);
    out[o + k] = uint16_t(b0 | (b1 << 8));
  }
}

// Bit 4 of codes 4i..4i+3 (bits 4i.. of qh) moved to bit 4 of each byte.
__device__ __forceinline__ uint32_t qh_nibble_bits(uint32_t qh, int i) {
  return (((qh >> (4 * i)) & 0xfu) * 0x00204081u & 0x01010101u) << 4;
}

// Integer dot of a legacy block's unsigned codes u with a Q8_0 block's
// codes: sum_j u_j * qx_j. qs: the 4 nibble words (bytes 4i..4i+3 each);
// qh: the high-bit word (0 for Q4_1).
template <int TYPE>
__device__ __forceinline__ int legacy_sumu(const uint32_t (&qs)[4], uint32_t qh, const uint32_t *xw) {
  int lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t a = qs[i] & 0x0f0f0f0fu, b = (qs[i] >> 4) & 0x0f0f0f0fu;
    if (Legacy<TYPE>::kQh >= 0) {
      a |= qh_nibble_bits(qh, i);
      b |= qh_nibble_bits(qh, 4 + i);
    }
    lo = dp4a_us(a, xw[i], lo);      // codes 4i..4i+3
    hi = dp4a_us(b, xw[4 + i], hi);  // codes 16+4i..
  }
  return lo + hi;
}

// --------------------------------------------------------------- k-quants --
// Super-blocks of 256 weights with 8 sub-blocks of 32 whose scales are
// quantized to 6 bits ("05. llama.cpp：从 GGUF 文件到本地推理服务", §量化类型).
// Layouts (this library's reading):
//   Q4_K, 144 bytes: fp16 d, fp16 dmin, 12 bytes = sub-block scales sc[0..7]
//     then minimums mn[0..7] as 6-bit values of a little-endian 96-bit
//     stream (value k at bits 6k..6k+5), then 128 bytes: sub-block j's 32
//     4-bit codes in bytes 16j..16j+15 (low nibble code i, high nibble
//     code i + 16); value fp32(d sc_j) * u - fp32(dmin mn_j).
//   Q6_K, 210 bytes: 128 bytes ql (byte i: low 4 bits of code i, then of
//     code i + 128), 64 bytes qh (byte i: top 2 bits of codes i, i+64,
//     i+128, i+192 at bits 0-1, 2-3, 4-5, 6-7), 16 int8 scales of the
//     sub-blocks of 16, fp16 d; value fp32(d sc_k) * (u - 32).

// 6-bit value k (0..15) of the Q4_K scale stream held in words w1..w3
// (stream bits 0..95 = w1 | w2 << 32 | w3 << 64).
__device__ __forceinline__ int q4k_stream(uint32_t w1, uint32_t w2, uint32_t w3, int k) {
  const int bit = 6 * k;
  const uint64_t lo = uint64_t(w1) | (uint64_t(w2) << 32);
  if (bit + 6 <= 64) return int((lo >> bit) & 63u);
  if (bit >= 64) return int((w3 >> (bit - 64)) & 63u);
  return int(((lo >> bit) | (uint64_t(w3) << (64 - bit))) & 63u);
}

// ------------------------------------------------------ packed fp32 pairs --

// Two fp32 values in one 64-bit register pair (lo = first); the f32x2
// operations round each half like the scalar IEEE operation.
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
  return uint64_t(lo) | (uint64_t(hi) << 32);
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}


// quantize_block_lane_fast on fp32 pairs: per value the same IEEE operations
// (the product by the reciprocal, the rounding add of the magic number, the
// subtraction back, and the distance r - (t - M) as the fused -1 * d + r,
// which rounds once like the subtraction), two values per instruction. The
// codes and the exact-path decision are bit-identical.
template <int TYPE>
__device__ __forceinline__ bool quantize_block_lane_fast_pairs(const float (&v)[32], uint16_t &scale,
                                                               uint32_t *words) {
  float ds;
  block_scale<TYPE>(block_amax<TYPE>(v), scale, ds);
  const float inv = ds > 0.0f ? rcp_approx(ds) : 0.0f;
  constexpr float kMagic = 12582912.0f + float(TYPE == kTypeQ4_0 ? 8 : 0);
  const uint64_t inv2 = pack2(__float_as_uint(inv), __float_as_uint(inv));
  const uint64_t mg2 = pack2(__float_as_uint(kMagic), __float_as_uint(kMagic));
  const uint64_t nmg2 = pack2(__float_as_uint(-kMagic), __float_as_uint(-kMagic));
  const uint64_t m1 = pack2(__float_as_uint(-1.0f), __float_as_uint(-1.0f));
  uint32_t tb[32];
  float dmax = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint64_t r = fmul2(pack2(__float_as_uint(v[2 * k]), __float_as_uint(v[2 * k + 1])), inv2);
    const uint64_t t = fadd2(r, mg2);
    const uint64_t e = ffma2(m1, fadd2(t, nmg2), r);
    tb[2 * k] = uint32_t(t);
    tb[2 * k + 1] = uint32_t(t >> 32);
    dmax = fmaxf(dmax, fmaxf(fabsf(__uint_as_float(uint32_t(e))), fabsf(__uint_as_float(uint32_t(e >> 32)))));
  }
  if (dmax > 0.4999f || (ds > 0.0f && ds < 6.103515625e-05f)) return false;
  pack_code_words<TYPE>(tb, words);
  return true;
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

// As mbar_try_wait, but the thread may stay suspended for up to `hint_ns`
// nanoseconds while the phase is incomplete (it resumes as soon as the phase
// completes): a waiting warp then issues almost nothing, leaving the issue
// slots to the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
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

// L2 policy for data read once (streamed weights): evicted before other lines,
// so the stream does not push activations or prefetched lines out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace bq
