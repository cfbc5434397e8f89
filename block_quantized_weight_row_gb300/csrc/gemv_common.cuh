// gemv_common.cuh — device code shared by the decode GEMV kernels (one
// launch per batch of matrices in gemv.cu, a whole sequence of batches in
// gemv_seq.cu): x's Q8_0 records and the dot product of one group of 8
// weight blocks with them. See gemv.cu for the data layout.
#pragma once

#include "bq_device.cuh"

namespace bq {
namespace gemv {

constexpr int kXRecWords = 84;  // per group of 8 blocks: 64 code words, 8 scales, 8 sums, 4 pad
constexpr int kXRecBytes = kXRecWords * 4;

// Quantize x (K fp32, 16-byte aligned) into the per-group records: words
// [g*84 + 8*jb + i] = codes 4i..4i+3 of block b = 8g+jb, [g*84 + 64 + jb] =
// the scale as fp32, [g*84 + 72 + jb] = the code sum. 8 lanes per block
// (coalesced loads, short dependency chains); `nthreads` (a multiple of 32)
// threads cover nthreads/8 blocks per pass. The loads of up to 12 passes are
// issued before any arithmetic and passes are quantized 4 at a time in
// straight-line code. Every thread runs every pass (the guards are uniform),
// keeping the 8-lane shuffles converged. Passes start at block `rot` so that
// CTAs reading the same x spread their requests over L2.
__device__ __forceinline__ void quantize_x_records(const float *__restrict__ x, int nb, uint32_t *rec, int tid,
                                                   int nthreads, int rot) {
  constexpr int kBatch = 12;
  const int j = tid & 7;
  const int stride = nthreads >> 3;
  const int passes = (nb + stride - 1) / stride;
  const int span = passes * stride;
  for (int p0 = 0; p0 < passes; p0 += kBatch) {
    float4 v[kBatch];
    int b[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      b[u] = (p0 + u < passes) ? ((p0 + u) * stride + (tid >> 3) + rot) % span : nb;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (b[u] < nb) v[u] = __ldcg(reinterpret_cast<const float4 *>(x + b[u] * kQK + j * 4));  // past L1
    }
#pragma unroll
    for (int u0 = 0; u0 < kBatch; u0 += 4) {
      if (p0 + u0 < passes) {  // uniform across the CTA
        uint16_t sc[4];
        uint32_t wd[4];
        int sm[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) quantize_block_8lanes(v[u0 + k], sc[k], wd[k], sm[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (b[u0 + k] < nb) {
            uint32_t *r = rec + (b[u0 + k] >> 3) * kXRecWords;
            const int jb = b[u0 + k] & 7;
            r[8 * jb + j] = wd[k];
            if (j == 0) {
              r[64 + jb] = __float_as_uint(half_bits_to_float(sc[k]));
              r[72 + jb] = uint32_t(sm[k]);
            }
          }
        }
      }
    }
  }
}

// One block of x quantized by a lane pair: the lane with h = 0 holds values
// 0-15, the lane with h = 1 values 16-31 (f). Both lanes of every pair of the
// warp must call it (it exchanges with the pair's other lane); `store` says
// whether this pair writes its block: codes to words 8 jb .. 8 jb + 7 of the
// group record rg, the scale (fp32) to word 64 + jb, the code sum to 72 + jb.
// Each lane decides the exact path for its own 16 values (the rule is exact
// per value), so the record is bit-identical to quantize_x_records'.
__device__ __forceinline__ void quantize_block_pair(const float (&f)[16], int h, uint32_t *rg, int jb, bool store) {
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(f[j]));
  m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
  uint16_t scale;
  float ds;
  block_scale<kTypeQ8_0>(m, scale, ds);
  const float inv = ds > 0.0f ? rcp_approx(ds) : 0.0f;
  constexpr float kMagic = 12582912.0f;
  uint32_t t[16];
  float dmax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float r = __fmul_rn(f[j], inv);
    const float tt = __fadd_rn(r, kMagic);
    t[j] = __float_as_uint(tt);
    dmax = fmaxf(dmax, fabsf(__fsub_rn(r, __fsub_rn(tt, kMagic))));
  }
  if (dmax > 0.4999f || (ds > 0.0f && ds < 6.103515625e-05f)) {
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = 0x4B400000u + uint32_t(code_of<kTypeQ8_0>(f[j], ds, inv));
  }
  uint32_t w[4];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[i] = pack_bytes(t[4 * i], t[4 * i + 1], t[4 * i + 2], t[4 * i + 3]);
#pragma unroll
    for (int k = 0; k < 4; ++k) sum += int(t[4 * i + k] - 0x4B400000u);
  }
  sum += __shfl_xor_sync(kFull, sum, 1);
  if (store) {
    *reinterpret_cast<uint4 *>(rg + 8 * jb + 4 * h) = make_uint4(w[0], w[1], w[2], w[3]);
    if (h == 0) {
      rg[64 + jb] = __float_as_uint(half_bits_to_float(scale));
      rg[72 + jb] = uint32_t(sum);
    }
  }
}

// The same records, two lanes per block (the lanes of a pair hold values
// 0-15 and 16-31 of one block), nthreads / 2 blocks per pass and the loads of
// two passes issued before any arithmetic: one pass for K = 4096 and three
// for K = 11008 with 256 threads, against 4 and 11 dependent 8-lane passes.
// x is quantized after the previous kernel completes, on the critical path of
// every launch without a workspace (measured 1.28 -> 1.19 ms per 7B decode
// step). Bit-identical to quantize_x_records.
__device__ __forceinline__ void quantize_x_records_2lane(const float *__restrict__ x, int nb, uint32_t *rec, int tid,
                                                         int nthreads) {
  const int h = tid & 1;
  const int per_pass = nthreads >> 1;
  for (int b0 = 0; b0 < nb; b0 += 2 * per_pass) {
    float4 v[2][4];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int b = b0 + p * per_pass + (tid >> 1);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        v[p][c] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b < nb) v[p][c] = __ldcg(reinterpret_cast<const float4 *>(x + int64_t(b) * kQK + 16 * h) + c);
      }
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int b = b0 + p * per_pass + (tid >> 1);
      if (b0 + p * per_pass >= nb) break;  // uniform: no block of this pass
      float f[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        f[4 * c] = v[p][c].x;
        f[4 * c + 1] = v[p][c].y;
        f[4 * c + 2] = v[p][c].z;
        f[4 * c + 3] = v[p][c].w;
      }
      quantize_block_pair(f, h, rec + (b >> 3) * kXRecWords, b & 7, b < nb);
    }
  }
}

template <int TYPE>
struct GroupWords;
template <>
struct GroupWords<kTypeQ4_0> {
  static constexpr int kWords = 36;  // 144 bytes
};
template <>
struct GroupWords<kTypeQ8_0> {
  static constexpr int kWords = 68;  // 272 bytes
};
template <>
struct GroupWords<kTypeQ4_K> {
  static constexpr int kWords = 36;  // one 144-byte super-block
};
template <>
struct GroupWords<kTypeQ6_K> {
  static constexpr int kWords = 4;  // unused: Q6_K groups are read by q6k_group_terms
};
template <>
struct GroupWords<kTypeQ4_1> {
  static constexpr int kWords = 40;  // 160 bytes
};
template <>
struct GroupWords<kTypeQ5_0> {
  static constexpr int kWords = 44;  // 176 bytes
};
template <>
struct GroupWords<kTypeQ5_1> {
  static constexpr int kWords = 48;  // 192 bytes
};

// One legacy block's term, block jb of a group (its bytes start at 4-byte
// word w0, plus 2 bytes when `odd`): d_w d_x sum_j u_j qx_j (minus 16 d_w d_x
// sum qx for Q5_0) plus, for the "_1" types, m_w d_x sum qx.
template <int TYPE>
__device__ __forceinline__ float legacy_group_block(const uint32_t *w, int w0, bool odd, const uint32_t *xw,
                                                    float dx, int xsum, float acc) {
  using L = Legacy<TYPE>;
  uint32_t dbits, mbits = 0, qh = 0, qs[4];
  if (!odd) {
    // Q4_1 / Q5_1: d, m in word w0, then qh (Q5_1) and the nibbles word aligned;
    // Q5_0: d in the low half of w0, qh and the nibbles 2 bytes off
    dbits = w[w0] & 0xffffu;
    if (L::kAffine) {
      mbits = w[w0] >> 16;
      const int q0 = w0 + (L::kQh >= 0 ? 2 : 1);
      if (L::kQh >= 0) qh = w[w0 + 1];
#pragma unroll
      for (int i = 0; i < 4; ++i) qs[i] = w[q0 + i];
    } else {
      qh = __funnelshift_r(w[w0], w[w0 + 1], 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) qs[i] = __funnelshift_r(w[w0 + 1 + i], w[w0 + 2 + i], 16);
    }
  } else {
    // Q5_0 at 2 mod 4: d in the high half of w0, qh and the nibbles word aligned
    dbits = w[w0] >> 16;
    qh = w[w0 + 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) qs[i] = w[w0 + 2 + i];
  }
  int sumi = legacy_sumu<TYPE>(qs, qh, xw);
  if (!L::kAffine) sumi -= 16 * xsum;
  acc = __fmaf_rn(__fmul_rn(half_bits_to_float(dbits), dx), float(sumi), acc);
  if (L::kAffine) acc = __fmaf_rn(__fmul_rn(half_bits_to_float(mbits), dx), float(xsum), acc);
  return acc;
}

// 8 words of a shared-memory byte range starting at an even address.
__device__ __forceinline__ void lds_8words_even(const uint8_t *p, uint32_t (&w)[8]) {
  const uint32_t *a = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(3));
  const uint32_t sh = (reinterpret_cast<uintptr_t>(p) & 2) * 8;
  uint32_t r[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) r[i] = a[i];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = __funnelshift_rc(r[i], r[i + 1], sh);
}

// One Q6_K super-block (2-byte aligned in shared memory) against its 8 x
// blocks: x block j holds codes 32j..32j+31 = sub-blocks 2j, 2j+1. The low
// bits of codes 32j' .. (j' < 4) and 128 + 32j' .. share ql bytes 32j'..;
// their top bits sit in qh bytes 32 (j' & 1).. at bit pairs j >> 1.
__device__ __forceinline__ float q6k_group_terms(const uint8_t *sb, const uint32_t *xr, float acc) {
  const float d = half_bits_to_float(uint32_t(*reinterpret_cast<const uint16_t *>(sb + 208)));
#pragma unroll
  for (int jp = 0; jp < 4; ++jp) {
    uint32_t ql[8], qh[8];
    lds_8words_even(sb + 32 * jp, ql);
    lds_8words_even(sb + 128 + 32 * (jp & 1), qh);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int j = jp + 4 * half;
      const uint32_t *xw = xr + 8 * j;
      const float dx = __uint_as_float(xr[64 + j]);
      const uint32_t lsh = 4u * uint32_t(half), hsh = 2u * uint32_t(j >> 1);
      int su[2] = {0, 0}, sx[2] = {0, 0};
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const uint32_t u = ((ql[w] >> lsh) & 0x0f0f0f0fu) | (((qh[w] >> hsh) & 0x03030303u) << 4);
        su[w >> 2] = dp4a_us(u, xw[w], su[w >> 2]);
        sx[w >> 2] = dp4a_ss(0x01010101u, xw[w], sx[w >> 2]);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float S = __fmul_rn(d, float(int8_t(sb[192 + 2 * j + h])));
        acc = __fmaf_rn(__fmul_rn(S, dx), float(su[h] - 32 * sx[h]), acc);
      }
    }
  }
  return acc;
}

// Sum of the 8 block terms of one group. w: the group's bytes as words (the
// group starts 16-byte aligned, block jb starts at byte BB*jb).
template <int TYPE>
__device__ __forceinline__ float group_terms(const uint32_t *w, const uint32_t *xr, float acc) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  const uint4 dx0 = *reinterpret_cast<const uint4 *>(xr + 64);
  const uint4 dx1 = *reinterpret_cast<const uint4 *>(xr + 68);
  const uint32_t dxs[8] = {dx0.x, dx0.y, dx0.z, dx0.w, dx1.x, dx1.y, dx1.z, dx1.w};
  uint32_t sxs[8];
  if (TYPE == kTypeQ4_0 || TYPE == kTypeQ4_K || Legacy<TYPE>::kIs) {
    const uint4 s0 = *reinterpret_cast<const uint4 *>(xr + 72);
    const uint4 s1 = *reinterpret_cast<const uint4 *>(xr + 76);
    sxs[0] = s0.x; sxs[1] = s0.y; sxs[2] = s0.z; sxs[3] = s0.w;
    sxs[4] = s1.x; sxs[5] = s1.y; sxs[6] = s1.z; sxs[7] = s1.w;
  }
  if constexpr (TYPE == kTypeQ4_K) {
    // the group is one super-block: w[0] = d | dmin, w[1..3] the 6-bit
    // scale/minimum stream, sub-block j's codes in w[4 + 4j .. 7 + 4j]
    const float d = half_bits_to_float(w[0] & 0xffffu), dm = half_bits_to_float(w[0] >> 16);
#pragma unroll
    for (int jb = 0; jb < 8; ++jb) {
      const uint4 xa = *reinterpret_cast<const uint4 *>(xr + 8 * jb);
      const uint4 xb = *reinterpret_cast<const uint4 *>(xr + 8 * jb + 4);
      const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      int su = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        su = dp4a_us(w[4 + 4 * jb + i] & 0x0f0f0f0fu, xw[i], su);
        su = dp4a_us((w[4 + 4 * jb + i] >> 4) & 0x0f0f0f0fu, xw[4 + i], su);
      }
      const float dx = __uint_as_float(dxs[jb]);
      const float S = __fmul_rn(d, float(q4k_stream(w[1], w[2], w[3], jb)));
      const float Mn = __fmul_rn(dm, float(q4k_stream(w[1], w[2], w[3], 8 + jb)));
      acc = __fmaf_rn(__fmul_rn(S, dx), float(su), acc);
      acc = __fmaf_rn(__fmul_rn(Mn, dx), float(-int(sxs[jb])), acc);
    }
  } else {
#pragma unroll
  for (int jb = 0; jb < 8; ++jb) {
    if constexpr (Legacy<TYPE>::kIs) {
      const uint4 xa = *reinterpret_cast<const uint4 *>(xr + 8 * jb);
      const uint4 xb = *reinterpret_cast<const uint4 *>(xr + 8 * jb + 4);
      const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      const int byte0 = BB * jb;
      acc = legacy_group_block<TYPE>(w, byte0 >> 2, (byte0 & 3) != 0, xw, __uint_as_float(dxs[jb]), int(sxs[jb]),
                                     acc);
      continue;
    }
    constexpr int kQW = (TYPE == kTypeQ4_0) ? 4 : 8;  // code words per block
    uint32_t q[kQW];
    uint32_t dbits;
    const int byte0 = BB * jb;
    if ((byte0 & 3) == 0) {
      // scale in the low half of word byte0/4; codes start 2 bytes later
      const int w0 = byte0 >> 2;
      dbits = w[w0] & 0xffffu;
#pragma unroll
      for (int i = 0; i < kQW; ++i) q[i] = __funnelshift_r(w[w0 + i], w[w0 + i + 1], 16);
    } else {
      // scale in the high half of word (byte0-2)/4; codes are word aligned
      const int w0 = (byte0 - 2) >> 2;
      dbits = w[w0] >> 16;
#pragma unroll
      for (int i = 0; i < kQW; ++i) q[i] = w[w0 + 1 + i];
    }
    const uint4 xa = *reinterpret_cast<const uint4 *>(xr + 8 * jb);
    const uint4 xb = *reinterpret_cast<const uint4 *>(xr + 8 * jb + 4);
    const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    int sumi;
    if (TYPE == kTypeQ4_0)
      sumi = sumi_q4_q8(q, xw, int(sxs[jb]));
    else
      sumi = sumi_q8_q8(q, xw);
    const float s = __fmul_rn(half_bits_to_float(dbits), __uint_as_float(dxs[jb]));
    acc = __fmaf_rn(s, float(sumi), acc);
  }
  }
  return acc;
}

}  // namespace gemv
}  // namespace bq
