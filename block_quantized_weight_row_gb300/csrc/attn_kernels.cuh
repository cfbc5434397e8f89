// attn_kernels.cuh — the decode-attention kernels (chunk kernels over the
// quantized KV cache and the combine of their partial results), shared by
// the translation units that instantiate them: attn.cu (plans, launches, the
// kernels for any shape) and attn_fixed_*.cu (the compile-time-shaped warp
// kernels, split over files so that they compile in parallel).
#pragma once
#include <algorithm>
#include <type_traits>

#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {
namespace {


constexpr int kAttnThreads = 256;

// Partial results of chunk c (= blockIdx.x of the chunk kernels, gridDim.x
// chunks): o_part[h][d / 32][c][d % 32] and ml[h][c] = (m, l). The chunks of
// one head and 32-channel slice are contiguous (chunks x 128 bytes), so that
// the combine moves them into shared memory with plain 16-byte async copies.
__device__ __forceinline__ size_t part_offset(int h, int d, int D) {
  return ((size_t(h) * (D / 32) + d / 32) * gridDim.x + blockIdx.x) * 32 + d % 32;
}

// q in the basis of a Hadamard-rotated K cache (lpnh.cn KV-cache article,
// §三步上手, third step): every 64 channels of a head become H64 q / 8, so
// (Hq).(Hk) = q.k. Lanes hold 4 channels each, 8 lanes per block of 32, two
// blocks (lanes 16g .. 16g + 15) per group of 64: element 32 * ((lane >> 3) & 1)
// + 4 * (lane & 7) + c. Butterflies (a, b) -> (a + b, a - b) of span 1 and 2
// inside the lane, 4, 8, 16, 32 with lane ^ 1, 2, 4, 8, then * 0.125: the same
// steps, in the same order, as the K cache's rotation.
__device__ __forceinline__ float4 hadamard64_8lanes(float4 v, int lane) {
  float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int h = 1; h < 4; h <<= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = __fadd_rn(a, b);
        x[i + h] = __fsub_rn(a, b);
      }
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float p = __shfl_xor_sync(kFull, x[i], m);
      x[i] = up ? __fsub_rn(p, x[i]) : __fadd_rn(x[i], p);
    }
  }
  return make_float4(__fmul_rn(x[0], 0.125f), __fmul_rn(x[1], 0.125f), __fmul_rn(x[2], 0.125f),
                     __fmul_rn(x[3], 0.125f));
}

// 2^x (hardware approximation, relative error about 2^-22; 0 for -inf)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// per (block, head): 8 code words, scale (fp32), code sum, 3 pad; stored
// block-major with an odd stride, so that the lanes of a warp, which read
// different heads' records of the same block, hit different banks
constexpr int kQRecWords = 13;
constexpr int kMaxStages = 4;

// Words covering `bytes` bytes that start at an even shared-memory offset:
// word i = bytes 4i .. 4i+3 of the block, taken from aligned words by a funnel
// shift of 0 or 16 bits.
template <int NW>
__device__ __forceinline__ void lds_block_words(const uint8_t *p, uint32_t (&w)[NW]) {
  const uint32_t *a = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(3));
  const uint32_t sh = (reinterpret_cast<uintptr_t>(p) & 2) * 8;
  uint32_t r[NW + 1];
#pragma unroll
  for (int i = 0; i <= NW; ++i) r[i] = a[i];
#pragma unroll
  for (int i = 0; i < NW; ++i) w[i] = __funnelshift_rc(r[i], r[i + 1], sh);
}

// score contribution of one K block against q's record: dk * dq * sumi
template <int KT>
__device__ __forceinline__ float k_block_term(const uint8_t *kb, const uint32_t *qr) {
  constexpr int NW = KT == kTypeQ4_0 ? 5 : 9;  // 18 or 34 bytes, rounded up to words
  uint32_t w[NW];
  lds_block_words<NW>(kb, w);
  const float dk = half_bits_to_float(w[0] & 0xffffu);
  uint32_t xw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) xw[i] = qr[i];
  const float dq = __uint_as_float(qr[8]);
  int sumi;
  if (KT == kTypeQ4_0) {
    uint32_t qs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) qs[i] = __funnelshift_rc(w[i], w[i + 1], 16);
    sumi = sumi_q4_q8(qs, xw, int(qr[9]));
  } else {
    uint32_t qs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) qs[i] = __funnelshift_rc(w[i], w[i + 1], 16);
    sumi = sumi_q8_q8(qs, xw);
  }
  return __fmul_rn(__fmul_rn(dk, dq), float(sumi));
}

// DPU dequantized codes of one V block starting at channel c0 (c0 % DPU ==
// 0), as DPU/2 packed pairs. A code byte u (biased to 0..255 for Q8_0, the
// nibble for Q4_0) is put in the low mantissa byte of 2^23 and the bias is
// subtracted, two values per instruction: exact, and without integer-to-float
// conversion instructions.
template <int VT, int DPU>
__device__ __forceinline__ void v_code_pairs(const uint8_t *vb, int c0, uint64_t (&v)[DPU / 2]) {
  uint32_t bits[DPU];
  float bias;
  if (VT == kTypeQ8_0) {
    constexpr int NW = DPU >= 4 ? DPU / 4 : 1;
    uint32_t w[NW];
    lds_block_words<NW>(vb + 2 + (c0 & ~3), w);  // 2 + (c0 & ~3) is even
#pragma unroll
    for (int k = 0; k < DPU; ++k) {
      const int kk = (c0 & 3) + k;  // c0 & 3 != 0 only for DPU = 2
      bits[k] = __byte_perm(w[kk >> 2] ^ 0x80808080u, 0x4B000000u, 0x7540u + uint32_t(kk & 3));
    }
    bias = -8388736.0f;  // 2^23 + 128
  } else {
    // channel c: nibble c (low) of byte c, or nibble c - 16 (high) of byte c - 16
    const int byte0 = c0 & 15;
    constexpr int NW = DPU >= 4 ? DPU / 4 : 1;
    uint32_t w[NW];
    lds_block_words<NW>(vb + 2 + (byte0 & ~3), w);
    const uint32_t sh = c0 >= 16 ? 4u : 0u;
#pragma unroll
    for (int k = 0; k < DPU; ++k) {
      const int kk = (byte0 & 3) + k;
      bits[k] = 0x4B000000u | (((w[kk >> 2] >> (8 * (kk & 3))) >> sh) & 0x0fu);
    }
    bias = -8388616.0f;  // 2^23 + 8
  }
  const uint64_t b2 = pack2(__float_as_uint(bias), __float_as_uint(bias));
#pragma unroll
  for (int k = 0; k < DPU / 2; ++k) v[k] = fadd2(pack2(bits[2 * k], bits[2 * k + 1]), b2);
}

struct AttnArgs {
  const float *q;
  const uint8_t *K, *V;
  float *o_part;  // [chunks][heads][D]: sum_t p v, unnormalized
  float *ml;      // [chunks][heads][2]: m, l
  float scale;
  int n_tokens, n_heads, n_kv, D, nb;
  int k_tok, v_tok;  // bytes of one token's row over all kv heads
  int chunk_tokens;  // tokens per chunk (a multiple of sub)
  int sub;           // tokens per ring stage (8, 16 or 32)
  int stage_bytes;   // sub * max(k_tok, v_tok), a multiple of 16
  int ring_bytes;    // >= the stages and >= the split reduction, a multiple of 16
  int stages;        // ring stages, 2..4
  int k_rot;         // K cache Hadamard-rotated: rotate q alike
  unsigned *err;
  uint32_t spin_limit;
};

// Block-wide chunk kernel: tiles of `sub` tokens (8-32) arrive in a 2-4 stage
// ring, all K tiles of the chunk first, then all V tiles.
//   pass 1: scores s[h][t] of the chunk (thread per (token, head) pair);
//   softmax: per head, m = max_t s, p = 2^(s - m), l = sum_t p;
//   pass 2: o[h][d] = sum_t p[h][t] * dv * qv; a thread owns one kv head's G
//           query heads x 16/G channels (16 outputs), with partial sums per
//           sub-tile of at most 32 tokens.
template <int KT, int VT, int G>
__global__ void __launch_bounds__(kAttnThreads, 2) k_attn_chunk(const AttnArgs a) {
  constexpr int DPU = 16 / G;  // channels per thread unit; G heads x DPU channels = 16 outputs
  constexpr int BBk = Fmt<KT>::kBytes, BBv = Fmt<VT>::kBytes;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = a.nb, H = a.n_heads, CT = a.chunk_tokens;
  const int SP = CT + 1;  // row stride of the scores: odd, so that 16 heads of one token hit 16 banks
  // ring (stages, later the split reduction) | 32 B pad | q records | scores [H][CT] | (m, l) [H] | barriers
  uint8_t *ring = smem;
  uint32_t *qrec = reinterpret_cast<uint32_t *>(smem + size_t(a.ring_bytes) + 32);
  float *S = reinterpret_cast<float *>(qrec + H * nb * kQRecWords);
  float *ML = S + size_t(H) * SP;
  uint64_t *bar = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(ML + 2 * H) + 15) & ~uintptr_t(15));

  const int t0 = blockIdx.x * CT;
  const int tn = min(CT, a.n_tokens - t0);
  const int ns = (tn + a.sub - 1) / a.sub;  // sub-tiles per pass

  const int NS = a.stages;
  if (tid == 0) {
    for (int st = 0; st < NS; ++st) mbar_init(&bar[st], 1);
    fence_mbar_init();
  }
  // q quantized to Q8_0 records, 8 lanes per block (every thread takes every
  // pass: the 8-lane shuffles stay converged)
  for (int base = 0; base < H * nb; base += kAttnThreads / 8) {
    const int blk = base + (tid >> 3), j = tid & 7;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (blk < H * nb) v = __ldg(reinterpret_cast<const float4 *>(a.q + size_t(blk) * kQK) + j);
    if (a.k_rot) v = hadamard64_8lanes(v, lane);  // uniform
    uint16_t sc;
    uint32_t word;
    int sum;
    quantize_block_8lanes(v, sc, word, sum);
    if (blk < H * nb) {
      uint32_t *r = qrec + ((blk % nb) * H + blk / nb) * kQRecWords;  // head blk / nb, block blk % nb
      r[j] = word;
      if (j == 0) {
        r[8] = __float_as_uint(half_bits_to_float(sc));
        r[9] = uint32_t(sum);
      }
    }
  }
  __syncthreads();

  auto tile_tokens = [&](int i) { return min(a.sub, tn - (i < ns ? i : i - ns) * a.sub); };
  auto tile_src = [&](int i) {
    const bool isk = i < ns;
    const int tt = (isk ? i : i - ns) * a.sub;
    return (isk ? a.K : a.V) + int64_t(t0 + tt) * (isk ? a.k_tok : a.v_tok);
  };
  // full sub-tiles arrive by bulk copy (a multiple of 16 bytes); a partial one
  // (only the chunk's last) is copied by all threads when it is consumed
  int issued[kMaxStages] = {0, 0, 0, 0};  // copies armed per stage (thread 0)
  auto issue = [&](int i) {
    if (i >= 2 * ns || tile_tokens(i) != a.sub) return;
    const int st = i % NS;
    ++issued[st];
    const uint32_t bytes = uint32_t(a.sub) * uint32_t(i < ns ? a.k_tok : a.v_tok);
    mbar_arrive_expect_tx(&bar[st], bytes);
    bulk_g2s(ring + size_t(st) * a.stage_bytes, tile_src(i), bytes, &bar[st]);
  };

  // pass-2 thread unit: kv head, DPU channels from d0, G query heads; S_split
  // threads share a unit and take every S_split-th token
  const int units = H * a.D / 16;
  const int splits = kAttnThreads / units;
  const int u = tid % units, split = tid / units;
  const bool has_unit = split < splits;
  const int kvh = u / (a.D / DPU), d0 = (u % (a.D / DPU)) * DPU;
  const int vb_off = (kvh * nb + d0 / kQK) * BBv, c0 = d0 % kQK;
  uint64_t acc[G][DPU / 2], part[G][DPU / 2];  // channel pairs (d0 + 2k, d0 + 2k + 1)
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int k = 0; k < DPU / 2; ++k) acc[g][k] = part[g][k] = 0;

  int armed[kMaxStages] = {0, 0, 0, 0};
  bool ok = true;
  if (tid == 0)
    for (int i = 0; i + 1 < NS; ++i) issue(i);
  for (int i = 0; i < 2 * ns && ok; ++i) {
    // the stage of tile i + NS - 1 held tile i - 1, released by the barrier closing iteration i - 1
    if (tid == 0) issue(i + NS - 1);
    const int n = tile_tokens(i);
    const int st = i % NS;
    const uint8_t *stage = ring + size_t(st) * a.stage_bytes;
    if (n == a.sub) {
      ok = mbar_wait_bounded(&bar[st], uint32_t(armed[st] & 1), a.spin_limit);
      if (ok)
        ++armed[st];
      else
        atomicOr(a.err, kErrTimeout);
      ok = __syncthreads_and(ok);
      if (!ok) break;
    } else {
      const int bytes = n * (i < ns ? a.k_tok : a.v_tok);  // even
      const uint16_t *src = reinterpret_cast<const uint16_t *>(tile_src(i));
      uint16_t *dst = reinterpret_cast<uint16_t *>(ring + size_t(st) * a.stage_bytes);
      for (int k = tid; k < bytes / 2; k += kAttnThreads) dst[k] = src[k];
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the stage is a bulk-copy target later
      __syncthreads();
    }
    if (i < ns) {
      // ---- scores of the sub-tile's tokens for every head ----
      const int tt = i * a.sub;
      for (int p = tid; p < n * H; p += kAttnThreads) {
        const int t = p / H, h = p % H;
        const uint8_t *krow = stage + size_t(t) * a.k_tok + size_t(h / G) * nb * BBk;
        float s = 0.0f;
        for (int b = 0; b < nb; ++b) s = __fadd_rn(s, k_block_term<KT>(krow + b * BBk, qrec + (b * H + h) * kQRecWords));
        S[h * SP + tt + t] = __fmul_rn(s, a.scale);
      }
      if (i == ns - 1) {
        __syncthreads();
        // ---- softmax over the chunk, one warp per head ----
        for (int h = warp; h < H; h += kAttnThreads / 32) {
          float m = -INFINITY;
          for (int t = lane; t < tn; t += 32) m = fmaxf(m, S[h * SP + t]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
          float l = 0.0f;
          for (int t = lane; t < tn; t += 32) {
            const float e = ex2(__fsub_rn(S[h * SP + t], m));
            S[h * SP + t] = e;
            l = __fadd_rn(l, e);
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(kFull, l, off);
          if (lane == 0) {
            ML[2 * h] = m;
            ML[2 * h + 1] = l;
          }
        }
      }
    } else if (has_unit) {
      // ---- values: part[g][k] += p[h_g][t] * dv * qv ----
      const int tt = (i - ns) * a.sub;
      for (int t = split; t < n; t += splits) {
        const uint8_t *vb = stage + size_t(t) * a.v_tok + vb_off;
        const float dv = half_bits_to_float(*reinterpret_cast<const uint16_t *>(vb));
        uint64_t vals[DPU / 2];
        v_code_pairs<VT, DPU>(vb, c0, vals);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint32_t pdv = __float_as_uint(__fmul_rn(S[(kvh * G + g) * SP + tt + t], dv));
          const uint64_t pdv2 = pack2(pdv, pdv);
#pragma unroll
          for (int k = 0; k < DPU / 2; ++k) part[g][k] = ffma2(pdv2, vals[k], part[g][k]);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < DPU / 2; ++k) {
          acc[g][k] = fadd2(acc[g][k], part[g][k]);
          part[g][k] = 0;
        }
    }
    __syncthreads();
  }
  if (!ok) {
    // a wait ran out: let the copies still in flight land before leaving
    if (tid == 0)
      for (int st = 0; st < NS; ++st)
        for (; armed[st] < issued[st]; ++armed[st])
          if (!mbar_wait_bounded(&bar[st], uint32_t(armed[st] & 1), 1u << 26)) break;
    return;
  }
  // ---- the splits of a unit add up (through the ring), split 0 writes ----
  float *red = reinterpret_cast<float *>(ring);
  if (has_unit && split > 0) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int k = 0; k < DPU / 2; ++k)
        reinterpret_cast<uint64_t *>(red)[((split - 1) * units + u) * 8 + g * (DPU / 2) + k] = acc[g][k];
  }
  __syncthreads();
  if (has_unit && split == 0) {
    for (int sp = 1; sp < splits; ++sp)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < DPU / 2; ++k)
          acc[g][k] = fadd2(acc[g][k], reinterpret_cast<const uint64_t *>(red)[((sp - 1) * units + u) * 8 + g * (DPU / 2) + k]);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int k = 0; k < DPU / 2; ++k) {
        float *dst = a.o_part + part_offset(kvh * G + g, d0 + 2 * k, a.D);
        dst[0] = __uint_as_float(uint32_t(acc[g][k]));
        dst[1] = __uint_as_float(uint32_t(acc[g][k] >> 32));
      }
  }
  for (int h = tid; h < H; h += kAttnThreads)
    *reinterpret_cast<float2 *>(a.ml + (size_t(h) * gridDim.x + blockIdx.x) * 2) = make_float2(ML[2 * h], ML[2 * h + 1]);
}

// ---------------------------------------------------------------------------
// Warp-per-kv-head chunk kernel (n_kv in {1, 2, 4, 8}, D * G <= 1024).
//
// The 8 warps of a CTA are (kv head j, token slice ws): warp w takes kv head
// w % n_kv and tokens [ws * tw, ws * tw + tw) of every tile, so each warp
// owns its query heads' softmax state and runs without block-wide barriers:
// tiles of `sub` tokens (K and V rows of the same tokens) arrive by bulk copy
// into an NS-stage ring with a barrier per stage that completes on arrival, and the
// warp keeps a running maximum m, sum l and output o per query head (online
// softmax: when the maximum grows from m to m', l and o are multiplied by
// e^(m - m')). The warps of a CTA merge the same way at the end.
// Ring protocol: all NS stages are filled at the start; the last warp to
// release a stage (a shared counter per stage) issues the copy of the tile NS
// ahead into it, so no thread ever blocks waiting for a free stage. Waits on a
// stage poll without suspending the thread (a suspended thread woke up
// hundreds of cycles after the phase completed).
//   scores:  lanes are (token, block b); the lane's Q8_0 q records for block b
//            of its G heads stay in registers; block terms dk * dq * sumi are
//            summed over the blocks of a token by a butterfly over its lanes;
//   values:  lanes are (token, 32/G channels); each lane converts its codes
//            once and adds p * dv * v for all G heads (fp32 pairs).
constexpr int kWarpAttnWarps = 8;
constexpr int kWarpAttnThreads = 32 * kWarpAttnWarps;
constexpr int kQRecWords2 = 12;  // 8 code words, scale, code sum, 2 pad: 48 bytes
constexpr int kMaxQBlocks = 128;  // H * D <= 4096

struct AttnWArgs {
  const float *q;
  const uint8_t *K, *V;
  float *o_part, *ml;
  float scale;
  int n_tokens, n_heads, n_kv, D, nb;
  int k_tok, v_tok;
  int lb;            // lanes per token in the score step: nb rounded up to a power of two (<= 32)
  int chunk_tokens;  // a multiple of sub
  int tw;            // tokens per warp and tile (<= 32)
  int sub;           // tokens per tile: tw * 8 / n_kv, a multiple of 8
  int stage_bytes;   // sub * (k_tok + v_tok): K rows, then V rows
  int stages;        // 2..4
  int ring_bytes;    // >= stages * stage_bytes and >= the merge buffer
  int k_rot;         // K cache Hadamard-rotated: rotate q alike
  unsigned *err;
  uint32_t spin_limit;
  uint32_t poll_ns;  // 0: stage waits may suspend in the barrier unit; else poll, sleeping poll_ns between polls
  int prefetch_tokens;  // tokens of the chunk asked into L2 before the previous kernel has completed
};

// CPL codes of one V block from channel o (o % CPL == 0), as CPL/2 exact fp32
// pairs (the byte in the low mantissa byte of 2^23, minus the bias).
template <int VT, int CPL>
__device__ __forceinline__ void v_pairs(const uint8_t *vb, int o, uint64_t (&v)[CPL / 2]) {
  uint32_t bits[CPL];
  float bias;
  if constexpr (VT == kTypeQ8_0) {
    uint32_t w[CPL / 4];
    lds_block_words<CPL / 4>(vb + 2 + o, w);
#pragma unroll
    for (int i = 0; i < CPL / 4; ++i) w[i] ^= 0x80808080u;
#pragma unroll
    for (int k = 0; k < CPL; ++k) bits[k] = __byte_perm(w[k >> 2], 0x4B000000u, 0x7540u + uint32_t(k & 3));
    bias = -8388736.0f;  // 2^23 + 128
  } else if constexpr (CPL == 32) {
    // channel c < 16: low nibble of byte c; c >= 16: high nibble of byte c - 16
    uint32_t w[4];
    lds_block_words<4>(vb + 2, w);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      bits[k] = __byte_perm(w[k >> 2] & 0x0f0f0f0fu, 0x4B000000u, 0x7540u + uint32_t(k & 3));
      bits[k + 16] = __byte_perm((w[k >> 2] >> 4) & 0x0f0f0f0fu, 0x4B000000u,
                                                     0x7540u + uint32_t(k & 3));
    }
    bias = -8388616.0f;  // 2^23 + 8
  } else {
    constexpr int NW = CPL / 4;
    uint32_t w[NW];
    lds_block_words<NW>(vb + 2 + (o & 15), w);
    const uint32_t sh = o >= 16 ? 4u : 0u;
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = (w[i] >> sh) & 0x0f0f0f0fu;
#pragma unroll
    for (int k = 0; k < CPL; ++k) bits[k] = __byte_perm(w[k >> 2], 0x4B000000u, 0x7540u + uint32_t(k & 3));
    bias = -8388616.0f;
  }
  const uint64_t b2 = pack2(__float_as_uint(bias), __float_as_uint(bias));
#pragma unroll
  for (int k = 0; k < CPL / 2; ++k) v[k] = fadd2(pack2(bits[2 * k], bits[2 * k + 1]), b2);
}

// NBT > 0: the head size (NBT blocks of 32), the kv-head count NKVT and the
// warp tile (kFixedTW tokens) are compile-time constants, so that the lane
// roles, the row strides and the tile loops unroll, shared-memory offsets
// become immediates and a full tile runs without per-token guards; NBT = 0
// takes every shape from the arguments.
constexpr int kFixedTW = 16;

constexpr int pow2_at_least(int n) { return n <= 1 ? 1 : 2 * pow2_at_least((n + 1) / 2); }

// NWD words starting `sh` / 8 bytes (0 or 2) after the aligned word p[0]:
// word i = bytes 4i .. 4i+3 of that run.
template <int NWD>
__device__ __forceinline__ void lds_words_sh(const uint32_t *p, uint32_t sh, uint32_t (&w)[NWD]) {
  uint32_t r[NWD + 1];
#pragma unroll
  for (int i = 0; i <= NWD; ++i) r[i] = p[i];
#pragma unroll
  for (int i = 0; i < NWD; ++i) w[i] = __funnelshift_rc(r[i], r[i + 1], sh);
}

// CPL/2 exact fp32 pairs of a lane's V codes from the code bytes already in
// words (as v_pairs): Q8_0 w = the CPL code bytes; Q4_0 w = the 16 code bytes
// (CPL = 32) or the CPL bytes holding the lane's nibbles, nsh = 4 for the
// high nibbles.
template <int VT, int CPL>
__device__ __forceinline__ void v_pairs_words(const uint32_t *w, uint32_t nsh, uint64_t (&v)[CPL / 2]) {
  uint32_t bits[CPL];
  float bias;
  if constexpr (VT == kTypeQ8_0) {
#pragma unroll
    for (int k = 0; k < CPL; ++k) bits[k] = __byte_perm(w[k >> 2] ^ 0x80808080u, 0x4B000000u, 0x7540u + uint32_t(k & 3));
    bias = -8388736.0f;  // 2^23 + 128
  } else if constexpr (CPL == 32) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      bits[k] = __byte_perm(w[k >> 2] & 0x0f0f0f0fu, 0x4B000000u, 0x7540u + uint32_t(k & 3));
      bits[k + 16] = __byte_perm((w[k >> 2] >> 4) & 0x0f0f0f0fu, 0x4B000000u, 0x7540u + uint32_t(k & 3));
    }
    bias = -8388616.0f;  // 2^23 + 8
  } else {
#pragma unroll
    for (int k = 0; k < CPL; ++k)
      bits[k] = __byte_perm((w[k >> 2] >> nsh) & 0x0f0f0f0fu, 0x4B000000u, 0x7540u + uint32_t(k & 3));
    bias = -8388616.0f;
  }
  const uint64_t b2 = pack2(__float_as_uint(bias), __float_as_uint(bias));
#pragma unroll
  for (int k = 0; k < CPL / 2; ++k) v[k] = fadd2(pack2(bits[2 * k], bits[2 * k + 1]), b2);
}

template <int KT, int VT, int G, int NBT, int NKVT>
__global__ void __launch_bounds__(kWarpAttnThreads, 2) k_attn_warp(const AttnWArgs a) {
  constexpr int CPL = 32 / G;  // channels per lane in the value step
  constexpr int NP = CPL / 2;
  constexpr int BBk = Fmt<KT>::kBytes, BBv = Fmt<VT>::kBytes;
  constexpr bool kFix = NBT > 0;
  static_assert(!kFix || NKVT > 0, "a fixed shape fixes the kv-head count too");
  constexpr int kKTok = kFix ? NKVT * NBT * BBk : 0;  // bytes of a token's K row (fixed shapes)
  constexpr int kVTok = kFix ? NKVT * NBT * BBv : 0;
  constexpr int kSub = kFix ? kFixedTW * (kWarpAttnWarps / (kFix ? NKVT : 1)) : 0;  // tokens per tile
  constexpr int kStageBytes = kSub * (kKTok + kVTok);
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = kFix ? NBT : a.nb, H = a.n_heads, n_kv = a.n_kv, D = kFix ? NBT * kQK : a.D;
  // ring | q records [H][nb][12] | scores [8 warps][32][G] | (m, l) [8][G][2] |
  // control words (abort flag, tiles issued, release count per stage) | barriers
  uint8_t *ring = smem;
  uint32_t *qrec = reinterpret_cast<uint32_t *>(smem + size_t(a.ring_bytes));
  float *P = reinterpret_cast<float *>(qrec + size_t(H) * nb * kQRecWords2);
  float *WML = P + kWarpAttnWarps * 32 * G;
  int *ctl = reinterpret_cast<int *>(WML + kWarpAttnWarps * G * 2);
  volatile int *abort_flag = ctl;
  int *n_issued = ctl + 1, *released = ctl + 2;
  uint64_t *full = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(ctl + 2 + kMaxStages) + 15) & ~uintptr_t(15));

  const int t0 = blockIdx.x * a.chunk_tokens;
  const int tn = min(a.chunk_tokens, a.n_tokens - t0);
  const int nt = (tn + a.sub - 1) / a.sub;
  const int NS = a.stages;
  const int vpart = kFix ? kSub * kKTok : a.sub * a.k_tok;  // offset of the V rows in a stage (a multiple of 16)

  // Launched as a programmatic dependent of the previous kernel on the
  // stream: q and the K and V rows of the chunk's first prefetch_tokens
  // tokens are asked into L2 at once (always safe: L2 is where writes become
  // visible, so a line the previous kernel writes later is updated there),
  // everything else waits until that kernel has completed. The combine may then be
  // scheduled.
  if (tid == 0) {
    const uint32_t n = uint32_t(min(tn, a.prefetch_tokens));
    prefetch_l2(a.q, uint32_t(H * D) * 4u);  // every CTA reads all of q first
    prefetch_l2(a.K + int64_t(t0) * a.k_tok, (n * uint32_t(a.k_tok)) & ~15u);
    prefetch_l2(a.V + int64_t(t0) * a.v_tok, (n * uint32_t(a.v_tok)) & ~15u);
  }

  // tile i -> stage i % NS: full 16-byte multiples by bulk copy; the tail of
  // a partial tile (under 16 bytes per tensor) by plain copies of this thread
  auto issue = [&](int i) {
    if (i >= nt) return;
    atomicMax(n_issued, i + 1);  // tiles are issued without gaps: 0 .. n_issued - 1
    const int st = i % NS;
    const int n = min(a.sub, tn - i * a.sub);
    uint8_t *dst = ring + size_t(st) * a.stage_bytes;
    const uint8_t *ks = a.K + int64_t(t0 + i * a.sub) * a.k_tok;
    const uint8_t *vs = a.V + int64_t(t0 + i * a.sub) * a.v_tok;
    const uint32_t kb = uint32_t(n) * uint32_t(a.k_tok), vb = uint32_t(n) * uint32_t(a.v_tok);
    const uint32_t kb16 = kb & ~15u, vb16 = vb & ~15u;
    if (kb16 != kb || vb16 != vb) {
      for (uint32_t k = kb16; k < kb; k += 2)
        *reinterpret_cast<uint16_t *>(dst + k) = *reinterpret_cast<const uint16_t *>(ks + k);
      for (uint32_t k = vb16; k < vb; k += 2)
        *reinterpret_cast<uint16_t *>(dst + vpart + k) = *reinterpret_cast<const uint16_t *>(vs + k);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    mbar_arrive_expect_tx(&full[st], kb16 + vb16);
    if (kb16) bulk_g2s(dst, ks, kb16, &full[st]);
    if (vb16) bulk_g2s(dst + vpart, vs, vb16, &full[st]);
  };

  if (tid == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(&full[st], 1);
      released[st] = 0;
    }
    *abort_flag = 0;
    *n_issued = 0;
    fence_mbar_init();
  }
  pdl_wait();
  pdl_launch_dependents();
  // q quantized to Q8_0 records, 8 lanes per block. Every load of q is
  // issued first (one round trip, ahead of the cache tiles in the memory
  // queues), then the first tiles' copies, then the blocks are quantized.
  {
    constexpr int kRounds = kMaxQBlocks * 8 / kWarpAttnThreads;
    float4 v[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int blk = r * (kWarpAttnThreads / 8) + (tid >> 3);
      v[r] = blk < H * nb ? __ldg(reinterpret_cast<const float4 *>(a.q + size_t(blk) * kQK) + (tid & 7))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid == 0)
      for (int i = 0; i < NS; ++i) issue(i);
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int blk = r * (kWarpAttnThreads / 8) + (tid >> 3), jj = tid & 7;
      if (r * (kWarpAttnThreads / 8) >= H * nb) break;  // uniform
      uint16_t sc;
      uint32_t word;
      int sum;
      if (a.k_rot) v[r] = hadamard64_8lanes(v[r], lane);  // uniform
      quantize_block_8lanes(v[r], sc, word, sum);
      if (blk < H * nb) {
        uint32_t *rec = qrec + size_t(blk) * kQRecWords2;  // head blk / nb, block blk % nb
        rec[jj] = word;
        if (jj == 0) {
          rec[8] = __float_as_uint(half_bits_to_float(sc));
          rec[9] = uint32_t(sum);
        }
      }
    }
  }
  __syncthreads();

  const int j = warp % n_kv, ws = warp / n_kv;
  // score step: lane = (token tt1, block b1)
  const int LB = kFix ? pow2_at_least(NBT) : a.lb, b1 = lane % LB, tt1 = lane / LB, tpp1 = 32 / LB;
  const bool b1ok = b1 < nb;
  // the lane's q records (block b1 of its G heads): in registers for G <= 4,
  // else read from shared memory where they are used
  constexpr bool kQRegs = G <= 4;
  const uint32_t *qr0 = qrec + (size_t(j * G) * nb + (b1ok ? b1 : 0)) * kQRecWords2;
  const size_t qstride = size_t(nb) * kQRecWords2;  // next head
  uint32_t qw[G][8];
  float qd[G];
  int qs[G];
  auto load_q = [&](int g) {
    const uint32_t *r = qr0 + g * qstride;
    const uint4 r0 = *reinterpret_cast<const uint4 *>(r), r1 = *reinterpret_cast<const uint4 *>(r + 4);
    const uint2 r2 = *reinterpret_cast<const uint2 *>(r + 8);
    qw[g][0] = r0.x; qw[g][1] = r0.y; qw[g][2] = r0.z; qw[g][3] = r0.w;
    qw[g][4] = r1.x; qw[g][5] = r1.y; qw[g][6] = r1.z; qw[g][7] = r1.w;
    qd[g] = __uint_as_float(r2.x);
    qs[g] = int(r2.y);
  };
  if (kQRegs)
#pragma unroll
    for (int g = 0; g < G; ++g) load_q(g);
  const int kb_off = (j * nb + b1) * BBk;
  // value step: lane = (token tt2, channel group cg)
  const int R = D / CPL, tpp2 = 32 / R, cg = lane % R, tt2 = lane / R;
  const bool p2 = tt2 < tpp2;
  const int c0 = cg * CPL;
  const int vb_off = (j * nb + c0 / kQK) * BBv, o2 = c0 % kQK;
  uint64_t acc[G][NP];
  float m_run[G], l_run[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_run[g] = -INFINITY;
    l_run[g] = 0.0f;
#pragma unroll
    for (int k = 0; k < NP; ++k) acc[g][k] = 0;
  }
  float *Pw = P + warp * 32 * G;  // [token][G]: scores, then weights p
  // online softmax over the warp's tokens of a tile (base 2): scores in Pw
  // become weights p, the running maximum, sum and outputs are updated
  auto online_softmax = [&](int wn) {
    // two heads at a time: lanes 0-15 take head g0, lanes 16-31 head g0 + 1
    // (token = lane & 15; a warp tile has at most 16 tokens)
#pragma unroll
    for (int g0 = 0; g0 < G; g0 += 2) {
      const int hi = lane >> 4, t = lane & 15;
      const bool live = t < wn && (G > 1 || hi == 0);
      const float mo = (G > 1 && hi) ? m_run[G > 1 ? g0 + 1 : 0] : m_run[g0];
      const float sc = live ? Pw[t * G + (G > 1 ? g0 + hi : 0)] : -INFINITY;
      float mt = sc;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, off));
      const float mn = fmaxf(mo, mt);
      const float p = live ? ex2(__fsub_rn(sc, mn)) : 0.0f;
      float ls = p;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) ls += __shfl_xor_sync(kFull, ls, off);
      if (live) Pw[t * G + (G > 1 ? g0 + hi : 0)] = p;
#pragma unroll
      for (int u = 0; u < (G > 1 ? 2 : 1); ++u) {
        const int g = g0 + u;
        const float mg = __shfl_sync(kFull, mn, 16 * u), lg = __shfl_sync(kFull, ls, 16 * u);
        const float alpha = ex2(__fsub_rn(m_run[g], mg));  // 0 on the first tile (m_run = -inf)
        l_run[g] = __fmaf_rn(l_run[g], alpha, lg);
        m_run[g] = mg;
        if (alpha != 1.0f) {  // the same in every lane
          const uint64_t a2 = pack2(__float_as_uint(alpha), __float_as_uint(alpha));
#pragma unroll
          for (int k = 0; k < NP; ++k) acc[g][k] = fmul2(acc[g][k], a2);
        }
      }
    }
  };
  // ---- fixed shapes: one warp tile of kFixedTW tokens (FULL: every token present) ----
  // The lane's K block and V codes sit at lane-constant offsets within a
  // token's rows, so their alignment (and the shifts that realign them) is
  // known once; every row offset below is a compile-time constant.
  const int vw_byte = vb_off + 2 + (VT == kTypeQ8_0 ? o2 : (CPL == 32 ? 0 : (o2 & 15)));
  const uint32_t vsh = (vw_byte & 2) ? 16u : 0u, vnsh = (VT == kTypeQ4_0 && CPL < 32 && o2 >= 16) ? 4u : 0u;
  const uint32_t ksh_c = (kb_off & 2) ? 32u : 16u, ksh_d = (kb_off & 2) ? 16u : 0u;
  auto fixed_tile = [&](auto FULL, const uint8_t *Kw, const uint8_t *Vw, int wn) {
    constexpr bool full = decltype(FULL)::value;
    constexpr int LBf = pow2_at_least(NBT > 0 ? NBT : 1), TPP1 = 32 / LBf;
    constexpr int NWk = KT == kTypeQ4_0 ? 5 : 9;  // words from the block's aligned start
    constexpr int NCk = KT == kTypeQ4_0 ? 4 : 8;  // code words
    const uint32_t *kw = reinterpret_cast<const uint32_t *>(Kw + tt1 * kKTok + (kb_off & ~3));
#pragma unroll
    for (int ps = 0; ps < kFixedTW / TPP1; ++ps) {
      const int t = ps * TPP1 + tt1;
      float part[G];
#pragma unroll
      for (int g = 0; g < G; ++g) part[g] = 0.0f;
      if (full || t < wn) {
        uint32_t r[NWk];
#pragma unroll
        for (int k = 0; k < NWk; ++k) r[k] = kw[ps * TPP1 * (kKTok / 4) + k];
        const float dk = half_bits_to_float(r[0] >> ksh_d);
        uint32_t c[NCk];
#pragma unroll
        for (int k = 0; k < NCk; ++k) c[k] = __funnelshift_rc(r[k], r[k + 1], ksh_c);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (!kQRegs) load_q(g);
          int sumi;
          if constexpr (KT == kTypeQ4_0)
            sumi = sumi_q4_q8(c, qw[g], qs[g]);
          else
            sumi = sumi_q8_q8(c, qw[g]);
          part[g] = __fmul_rn(__fmul_rn(dk, qd[g]), float(sumi));
        }
      }
#pragma unroll
      for (int off = 1; off < LBf; off <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] = __fadd_rn(part[g], __shfl_xor_sync(kFull, part[g], off));
      if (b1 == 0 && (full || t < wn))
#pragma unroll
        for (int g = 0; g < G; ++g) Pw[t * G + g] = __fmul_rn(part[g], a.scale);
    }
    __syncwarp();
    online_softmax(wn);
    __syncwarp();
    // values: o[g][c] += p[g][t] * dv * v[c]
    constexpr int Rf = (NBT > 0 ? NBT : 1) * kQK / CPL, TPP2 = 32 / Rf;
    constexpr int NWv = VT == kTypeQ8_0 ? CPL / 4 : (CPL == 32 ? 4 : (CPL + 3) / 4);
    const uint8_t *vrow = Vw + tt2 * kVTok;
    const uint32_t *vw = reinterpret_cast<const uint32_t *>(vrow + (vw_byte & ~3));
    const float *pw = Pw + tt2 * G;
#pragma unroll
    for (int ps = 0; ps < kFixedTW / TPP2; ++ps) {
      const int t = ps * TPP2 + tt2;
      if (full || t < wn) {
        const float dv = half_bits_to_float(*reinterpret_cast<const uint16_t *>(vrow + ps * TPP2 * kVTok + vb_off));
        uint32_t w[NWv];
        lds_words_sh<NWv>(vw + ps * TPP2 * (kVTok / 4), vsh, w);
        uint64_t vals[NP];
        v_pairs_words<VT, CPL>(w, vnsh, vals);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint32_t pd = __float_as_uint(__fmul_rn(pw[ps * TPP2 * G + g], dv));
          const uint64_t pd2 = pack2(pd, pd);
#pragma unroll
          for (int k = 0; k < NP; ++k) acc[g][k] = ffma2(pd2, vals[k], acc[g][k]);
        }
      }
    }
  };

  for (int i = 0; i < nt; ++i) {
    const int st = i % NS;
    // the decision to go on is the same for every lane of the warp (the
    // shuffles below need all 32 lanes)
    const uint32_t par = uint32_t((i / NS) & 1);
    // a tile that has already landed answers the non-blocking test at once
    // (a limit of 0 polls gives up without looking)
    bool ok = a.spin_limit > 0 && mbar_test_wait(&full[st], par);
    if (ok) {
    } else if (a.poll_ns == 0) {
      for (uint32_t k = 0; k < a.spin_limit; ++k) {
        if (mbar_try_wait(&full[st], par)) {
          ok = true;
          break;
        }
        if ((k & 15) == 15 && *abort_flag) break;
      }
    } else {
      for (uint32_t k = 0; k < a.spin_limit; ++k) {
        if (mbar_test_wait(&full[st], par)) {
          ok = true;
          break;
        }
        if ((k & 63) == 63 && *abort_flag) break;
        __nanosleep(k < 64 ? 20 : a.poll_ns);
      }
    }
    if (!__all_sync(kFull, ok)) {
      if (lane == 0) {
        *abort_flag = 1;
        atomicOr(a.err, kErrTimeout);
      }
      break;
    }
    const uint8_t *Ks = ring + size_t(st) * (kFix ? kStageBytes : a.stage_bytes), *Vs = Ks + vpart;
    const int n = min(a.sub, tn - i * a.sub);
    const int w0 = ws * a.tw, wn = min(a.tw, n - w0);
    if constexpr (kFix) {
      if (wn == kFixedTW)
        fixed_tile(std::true_type{}, Ks + w0 * kKTok, Vs + w0 * kVTok, wn);
      else if (wn > 0)
        fixed_tile(std::false_type{}, Ks + w0 * kKTok, Vs + w0 * kVTok, wn);
    } else if (wn > 0) {
      // ---- scores s = scale * sum_b dk * dq * sumi ----
      const uint8_t *krow = Ks + size_t(w0 + tt1) * a.k_tok + kb_off;  // the lane's block of its token
      const size_t kstep = size_t(tpp1) * a.k_tok;
#pragma unroll
      for (int tb = 0; tb < (kFix ? kFixedTW : wn); tb += tpp1, krow += kstep) {
        const int t = tb + tt1;
        float part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] = 0.0f;
        if (t < wn && b1ok) {
          constexpr int NW = KT == kTypeQ4_0 ? 5 : 9;
          uint32_t w[NW];
          lds_block_words<NW>(krow, w);
          const float dk = half_bits_to_float(w[0] & 0xffffu);
          if (KT == kTypeQ4_0) {
            uint32_t c[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) c[k] = __funnelshift_rc(w[k], w[k + 1], 16);
#pragma unroll
            for (int g = 0; g < G; ++g) {
              if (!kQRegs) load_q(g);
              part[g] = __fmul_rn(__fmul_rn(dk, qd[g]), float(sumi_q4_q8(c, qw[g], qs[g])));
            }
          } else {
            uint32_t c[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) c[k] = __funnelshift_rc(w[k], w[k + 1], 16);
#pragma unroll
            for (int g = 0; g < G; ++g) {
              if (!kQRegs) load_q(g);
              part[g] = __fmul_rn(__fmul_rn(dk, qd[g]), float(sumi_q8_q8(c, qw[g])));
            }
          }
        }
        for (int off = 1; off < LB; off <<= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) part[g] = __fadd_rn(part[g], __shfl_xor_sync(kFull, part[g], off));
        if (b1 == 0 && t < wn)
#pragma unroll
          for (int g = 0; g < G; ++g) Pw[t * G + g] = __fmul_rn(part[g], a.scale);
      }
      __syncwarp();
      online_softmax(wn);
      __syncwarp();
      // ---- values: o[g][c] += p[g][t] * dv * v[c] ----
      if (p2) {
        const uint8_t *vb = Vs + size_t(w0 + tt2) * a.v_tok + vb_off;  // the lane's block of its token
        const size_t vstep = size_t(tpp2) * a.v_tok;
        const float *pw = Pw + tt2 * G;
#pragma unroll
        for (int tb = 0; tb < (kFix ? kFixedTW : wn); tb += tpp2, vb += vstep, pw += tpp2 * G) {
          if (tb + tt2 >= wn) break;  // tokens past the tile's end (the chunk's last tile)
          const float dv = half_bits_to_float(*reinterpret_cast<const uint16_t *>(vb));
          uint64_t vals[NP];
          v_pairs<VT, CPL>(vb, o2, vals);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const uint32_t pd = __float_as_uint(__fmul_rn(pw[g], dv));
            const uint64_t pd2 = pack2(pd, pd);
#pragma unroll
            for (int k = 0; k < NP; ++k) acc[g][k] = ffma2(pd2, vals[k], acc[g][k]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      // release the stage; the last warp to do so refills it with tile i + NS
      __threadfence_block();
      if (atomicAdd(&released[st], 1) == kWarpAttnWarps - 1) {
        released[st] = 0;
        __threadfence_block();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // reads above, bulk writes below
        issue(i + NS);
      }
    }
  }
  __syncthreads();
  if (*abort_flag) {
    // a wait ran out: let every copy still in flight land before leaving
    // (the last tile issued to a stage completes after the earlier ones)
    if (tid == 0)
      for (int k = max(0, *n_issued - NS); k < *n_issued; ++k)
        if (!mbar_wait_bounded(&full[k % NS], uint32_t((k / NS) & 1), 1u << 26)) break;
    return;
  }
  if constexpr (kFix && kWarpAttnWarps == NKVT) {
    // one warp per kv head: its heads' softmax state is already whole, and
    // only the token lanes of each channel group add up (butterflies over
    // the lane bits above the channel groups); the first token lane of each
    // group writes its channels
    constexpr int Rf = NBT * kQK / CPL, TPP2 = 32 / Rf;
#pragma unroll
    for (int off = Rf; off < Rf * TPP2; off <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const uint64_t o = __shfl_xor_sync(kFull, acc[g][k], off);
          acc[g][k] = fadd2(acc[g][k], o);
        }
    if (tt2 == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float *dst = a.o_part + part_offset(j * G + g, c0, D);  // c0 .. c0 + CPL - 1: one 32-channel slice
#pragma unroll
        for (int k = 0; k + 1 < NP; k += 2)
          *reinterpret_cast<float4 *>(dst + 2 * k) =
              make_float4(__uint_as_float(uint32_t(acc[g][k])), __uint_as_float(uint32_t(acc[g][k] >> 32)),
                          __uint_as_float(uint32_t(acc[g][k + 1])), __uint_as_float(uint32_t(acc[g][k + 1] >> 32)));
        if constexpr (NP % 2 == 1)
          *reinterpret_cast<float2 *>(dst + 2 * (NP - 1)) =
              make_float2(__uint_as_float(uint32_t(acc[g][NP - 1])), __uint_as_float(uint32_t(acc[g][NP - 1] >> 32)));
      }
    }
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < G; ++g)
        *reinterpret_cast<float2 *>(a.ml + (size_t(j * G + g) * gridDim.x + blockIdx.x) * 2) = make_float2(m_run[g], l_run[g]);
    return;
  }
  // ---- merge: warps of a kv head and lanes of a channel group ----
  // MB[((w * G + g) * tpp2 + tt2) * R * (CPL + 1) + cg * (CPL + 1) + c]: one
  // padding word per channel group, so that both the writes (lanes differ in
  // tt2 and cg) and the reads (lanes differ in the channel) hit 32 banks
  float *MB = reinterpret_cast<float *>(ring);
  const int RS = R * (CPL + 1);
  if (p2) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float *dst = MB + ((warp * G + g) * tpp2 + tt2) * RS + cg * (CPL + 1);
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        dst[2 * k] = __uint_as_float(uint32_t(acc[g][k]));
        dst[2 * k + 1] = __uint_as_float(uint32_t(acc[g][k] >> 32));
      }
    }
  }
  if (lane == 0)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      WML[(warp * G + g) * 2] = m_run[g];
      WML[(warp * G + g) * 2 + 1] = l_run[g];
    }
  __syncthreads();
  const int WS = kWarpAttnWarps / n_kv;
  for (int h = warp; h < H; h += kWarpAttnWarps) {
    const int jj = h / G, g = h % G;
    float M = -INFINITY;
    for (int s2 = 0; s2 < WS; ++s2) M = fmaxf(M, WML[((jj + s2 * n_kv) * G + g) * 2]);
    float L = 0.0f;
    for (int s2 = 0; s2 < WS; ++s2) {
      const int w = jj + s2 * n_kv;
      L = __fmaf_rn(ex2(__fsub_rn(WML[(w * G + g) * 2], M)), WML[(w * G + g) * 2 + 1], L);
    }
    for (int d = lane; d < D; d += 32) {
      const int off = (d / CPL) * (CPL + 1) + d % CPL;
      float O = 0.0f;
      for (int s2 = 0; s2 < WS; ++s2) {
        const int w = jj + s2 * n_kv;
        const float f = ex2(__fsub_rn(WML[(w * G + g) * 2], M));  // 0 for a warp that saw no token
        const float *src = MB + (w * G + g) * tpp2 * RS + off;
        float Ow = 0.0f;
        for (int q2 = 0; q2 < tpp2; ++q2) Ow = __fadd_rn(Ow, src[q2 * RS]);
        O = __fmaf_rn(f, Ow, O);
      }
      a.o_part[part_offset(h, d, D)] = O;
    }
    if (lane == 0) *reinterpret_cast<float2 *>(a.ml + (size_t(h) * gridDim.x + blockIdx.x) * 2) = make_float2(M, L);
  }
}

// o[h][d] = sum_c e^(m_c - M) o_c[h][d] / sum_c e^(m_c - M) l_c[h]. One CTA
// per head and 32-channel slice: its chunks' partials (contiguous, chunks x
// 128 bytes, and the head's (m, l) pairs) come into shared memory by 16- and
// 8-byte async copies, every thread's copies in flight at once, up to
// kCombineCap chunks per round. Per round: the block's maximum M of the m_c
// (a running maximum over rounds, the sums so far rescaled by 2^(M_old - M)),
// each chunk's weight w_c = 2^(m_c - M) computed once, then 32 slices of the
// chunks add w_c o_c (one lane per channel) and w_c l_c; the slices' sums are
// added at the end. fp32 throughout. Launched as a programmatic dependent of
// the chunk kernel: it lets the next kernel start at once and waits for the
// chunk kernel's writes before reading them.
constexpr int kCombineThreads = 1024;
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kCombineCap = 1024;  // chunks per round: 136 KB of shared memory

__host__ __device__ constexpr int combine_smem_bytes(int chunks) {
  return (chunks < kCombineCap ? chunks : kCombineCap) * (32 * 4 + 8);
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__global__ void __launch_bounds__(kCombineThreads) k_attn_combine(const float *__restrict__ o_part,
                                                                  const float *__restrict__ ml,
                                                                  float *__restrict__ o, int chunks, int H, int D) {
  extern __shared__ __align__(16) uint8_t csm[];
  const int cap = chunks < kCombineCap ? chunks : kCombineCap;
  float *sP = reinterpret_cast<float *>(csm);                         // [cap][32]: o_c of the slice
  float2 *sW = reinterpret_cast<float2 *>(csm + size_t(cap) * 128);  // [cap]: (m_c, l_c), then (w_c, w_c l_c)
  __shared__ float sO[kCombineWarps][33];
  __shared__ float sRed[kCombineWarps], sL[kCombineWarps];
  const int h = blockIdx.x, db = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float4 *src = reinterpret_cast<const float4 *>(o_part + (size_t(h) * (D / 32) + db) * size_t(chunks) * 32);
  const float2 *msrc = reinterpret_cast<const float2 *>(ml) + size_t(h) * chunks;
  pdl_launch_dependents();
  pdl_wait();
  float M = -INFINITY;  // block-uniform running maximum
  float O = 0.0f, L = 0.0f;  // this warp's sums (channel lane; L in every lane)
  for (int base = 0; base < chunks; base += cap) {
    const int n = min(cap, chunks - base);
    for (int i = threadIdx.x; i < n * 8; i += kCombineThreads)
      cp_async16(reinterpret_cast<float4 *>(sP) + i, src + size_t(base) * 8 + i);
    for (int i = threadIdx.x; i < n; i += kCombineThreads) cp_async8(sW + i, msrc + base + i);
    cp_async_wait_all();
    __syncthreads();
    // the round's maximum
    float mx = -INFINITY;
    for (int c = threadIdx.x; c < n; c += kCombineThreads) mx = fmaxf(mx, sW[c].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) sRed[warp] = mx;
    __syncthreads();
    mx = sRed[lane];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float Mn = fmaxf(M, mx);
    if (Mn != -INFINITY) {  // else no chunk so far saw a token: nothing to add
      if (M != Mn && M != -INFINITY) {  // an earlier round's sums, rescaled
        const float f = ex2(__fsub_rn(M, Mn));
        O = __fmul_rn(O, f);
        L = __fmul_rn(L, f);
      }
      M = Mn;
      // chunk weights, each computed once (read after the barrier below)
      for (int c = threadIdx.x; c < n; c += kCombineThreads) {
        const float2 p = sW[c];
        const float w = ex2(__fsub_rn(p.x, M));  // 0 for a chunk that saw no token
        sW[c] = make_float2(w, __fmul_rn(w, p.y));
      }
    }
    __syncthreads();
    if (M != -INFINITY) {
      int c = warp;
      for (; c + 3 * kCombineWarps < n; c += 4 * kCombineWarps) {
        const float2 w0 = sW[c], w1 = sW[c + kCombineWarps], w2 = sW[c + 2 * kCombineWarps],
                     w3 = sW[c + 3 * kCombineWarps];
        const float p0 = sP[c * 32 + lane], p1 = sP[(c + kCombineWarps) * 32 + lane],
                    p2 = sP[(c + 2 * kCombineWarps) * 32 + lane], p3 = sP[(c + 3 * kCombineWarps) * 32 + lane];
        O = __fmaf_rn(w0.x, p0, O);
        L = __fadd_rn(L, w0.y);
        O = __fmaf_rn(w1.x, p1, O);
        L = __fadd_rn(L, w1.y);
        O = __fmaf_rn(w2.x, p2, O);
        L = __fadd_rn(L, w2.y);
        O = __fmaf_rn(w3.x, p3, O);
        L = __fadd_rn(L, w3.y);
      }
      for (; c < n; c += kCombineWarps) {
        const float2 w = sW[c];
        O = __fmaf_rn(w.x, sP[c * 32 + lane], O);
        L = __fadd_rn(L, w.y);
      }
    }
    __syncthreads();  // the round's shared memory is read before the next round's copies
  }
  sO[warp][lane] = O;
  if (lane == 0) sL[warp] = L;
  __syncthreads();
  if (warp == 0) {
    float sum = 0.0f, Lt = 0.0f;
#pragma unroll 8
    for (int k = 0; k < kCombineWarps; ++k) {
      sum = __fadd_rn(sum, sO[k][lane]);
      Lt = __fadd_rn(Lt, sL[k]);
    }
    o[size_t(h) * D + db * 32 + lane] = __fdiv_rn(sum, Lt);
  }
}

template <int KT, int VT, int NBT, int NKVT>
const void *attn_warp_fn_g(int G) {
  switch (G) {
    case 1: return reinterpret_cast<const void *>(k_attn_warp<KT, VT, 1, NBT, NKVT>);
    case 2: return reinterpret_cast<const void *>(k_attn_warp<KT, VT, 2, NBT, NKVT>);
    case 4: return reinterpret_cast<const void *>(k_attn_warp<KT, VT, 4, NBT, NKVT>);
    case 8: return reinterpret_cast<const void *>(k_attn_warp<KT, VT, 8, NBT, NKVT>);
    default: return nullptr;
  }
}

}  // namespace
}  // namespace bq
