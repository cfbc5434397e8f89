// attn.cu — decode attention of one token over a block-quantized KV cache.
//
// A quantized V cache is read by flash attention, which computes attention in
// one pass without materializing the score matrix ("05. llama.cpp：从 GGUF 文件到
// 本地推理服务", §KV Cache 类型与 Flash Attention; lpnh.cn KV-cache article,
// §量化 KV Cache 的一键配置方法). Query head h reads kv head h / G (G = heads per
// kv head); q is quantized to Q8_0 per block of 32 channels and q·k is the
// block dot of the decode GEMV (dp4a on the codes, times dk·dq), scaled by the
// caller's softmax scale; the softmax weights multiply the dequantized V.
// A mean-centered K cache needs nothing here: q·(k - k̄) differs from q·k by
// the same constant for every key of a query row, and softmax ignores it
// (lpnh.cn KV-cache article, §解法).
//
// Split over tokens (flash decoding): the tokens are cut into chunks, about
// two per SM; one CTA takes a chunk and every head, so each token's K and V
// rows (contiguous over the kv heads in the cache layout) arrive with 1-D bulk
// copies of 8-32 tokens into a two-stage shared-memory ring.
//   pass 1: scores s[h][t] of the chunk (thread per (token, head) pair);
//   softmax: per head, m = max_t s, p = exp(s - m), l = sum_t p;
//   pass 2: o[h][d] = sum_t p[h][t] * dv * qv; a thread owns one kv head's G
//           query heads x 16/G channels (16 outputs), with partial sums per
//           sub-tile of at most 32 tokens;
//   the chunk writes (m, l, o) per head; k_attn_combine merges the chunks:
//   o = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c (fp32, two levels).
#include <algorithm>

#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {
namespace {

constexpr int kAttnThreads = 256;
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
  unsigned *err;
  uint32_t spin_limit;
};

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
            const float e = expf(__fsub_rn(S[h * SP + t], m));
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
        float *dst = a.o_part + (size_t(blockIdx.x) * H + kvh * G + g) * a.D + d0 + 2 * k;
        dst[0] = __uint_as_float(uint32_t(acc[g][k]));
        dst[1] = __uint_as_float(uint32_t(acc[g][k] >> 32));
      }
  }
  for (int h = tid; h < H; h += kAttnThreads) {
    a.ml[(size_t(blockIdx.x) * H + h) * 2] = ML[2 * h];
    a.ml[(size_t(blockIdx.x) * H + h) * 2 + 1] = ML[2 * h + 1];
  }
}

// o[h][d] = sum_c e^(m_c - M) o_c[h][d] / sum_c e^(m_c - M) l_c[h]. One CTA
// per head and 32 channels; 8 slices of the chunks per channel, each summed in
// fp32 and then added together (two levels: at most chunks/8 + 8 roundings).
constexpr int kCombineSlices = 8;
__global__ void __launch_bounds__(256) k_attn_combine(const float *__restrict__ o_part, const float *__restrict__ ml,
                                                      float *__restrict__ o, int chunks, int H, int D) {
  extern __shared__ float e[];  // [chunks]
  __shared__ float red[kCombineSlices][33];
  const int h = blockIdx.x, d = blockIdx.y * 32 + (threadIdx.x & 31), slice = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // M = max_c m_c (slices of 32 lanes, then over the slices)
  float m = -INFINITY;
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) m = fmaxf(m, ml[(size_t(c) * H + h) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  if (lane == 0) red[slice][32] = m;
  __syncthreads();
  float M = red[0][32];
#pragma unroll
  for (int k = 1; k < kCombineSlices; ++k) M = fmaxf(M, red[k][32]);
  __syncthreads();
  float l = 0.0f;
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
    e[c] = expf(__fsub_rn(ml[(size_t(c) * H + h) * 2], M));
    l = __fmaf_rn(e[c], ml[(size_t(c) * H + h) * 2 + 1], l);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(kFull, l, off);
  if (lane == 0) red[slice][32] = l;
  __syncthreads();
  float L = 0.0f;
#pragma unroll
  for (int k = 0; k < kCombineSlices; ++k) L += red[k][32];
  float O0 = 0.0f, O1 = 0.0f;  // two chains, so that the loads of the unrolled loop overlap
  if (d < D) {
#pragma unroll 8
    for (int c = slice; c < chunks; c += 2 * kCombineSlices) {
      O0 = __fmaf_rn(e[c], __ldg(o_part + (size_t(c) * H + h) * D + d), O0);
      if (c + kCombineSlices < chunks)
        O1 = __fmaf_rn(e[c + kCombineSlices], __ldg(o_part + (size_t(c + kCombineSlices) * H + h) * D + d), O1);
    }
  }
  red[slice][lane] = O0 + O1;
  __syncthreads();
  if (slice == 0 && d < D) {
    float sum = red[0][lane];
#pragma unroll
    for (int k = 1; k < kCombineSlices; ++k) sum += red[k][lane];
    o[size_t(h) * D + d] = __fdiv_rn(sum, L);
  }
}

}  // namespace

namespace {

constexpr int kAttnTargetChunks = 304;  // two per SM of a 152-SM GPU
constexpr int kAttnMaxChunkTokens = 512;
constexpr int kAttnRingBudget = 72 * 1024;  // two CTAs per SM

struct AttnPlan {
  int sub, chunk_tokens, chunks, stage_bytes, ring_bytes, stages, k_tok, v_tok;
  size_t smem;
};

AttnPlan attn_plan(int kt, int vt, int64_t T, int64_t H, int64_t n_kv, int64_t D) {
  AttnPlan p{};
  const int nb = int(D / kQK);
  p.k_tok = int(n_kv) * nb * (kt == kTypeQ4_0 ? Fmt<kTypeQ4_0>::kBytes : Fmt<kTypeQ8_0>::kBytes);
  p.v_tok = int(n_kv) * nb * (vt == kTypeQ4_0 ? Fmt<kTypeQ4_0>::kBytes : Fmt<kTypeQ8_0>::kBytes);
  const int tok = std::max(p.k_tok, p.v_tok);
  // four stages of 16 tokens where they fit (the copies' latency is covered
  // by three stages of compute), else two stages of at least 8 tokens
  p.sub = 16;
  p.stages = 4;
  while (p.sub > 8 && p.stages * p.sub * tok > kAttnRingBudget) p.sub /= 2;
  if (p.stages * p.sub * tok > kAttnRingBudget) p.stages = 2;
  const int64_t per = (T + kAttnTargetChunks - 1) / kAttnTargetChunks;
  const int64_t ct = std::min<int64_t>(kAttnMaxChunkTokens, (per + p.sub - 1) / p.sub * p.sub);
  p.chunk_tokens = int(ct);
  p.chunks = int((T + ct - 1) / ct);
  p.stage_bytes = p.sub * tok;  // a multiple of 16: sub is a multiple of 8, a block 18 or 34 bytes
  const int units = int(H * D / 16);
  const int splits = kAttnThreads / units;
  p.ring_bytes = std::max(p.stages * p.stage_bytes, (splits - 1) * units * 16 * 4);
  p.ring_bytes = (p.ring_bytes + 15) / 16 * 16;
  p.smem = size_t(p.ring_bytes) + 32 + size_t(H) * nb * kQRecWords * 4 + size_t(H) * (p.chunk_tokens + 1) * 4 +
           size_t(H) * 8 + 16 + 8 * kMaxStages;
  return p;
}

template <int KT, int VT>
cudaError_t launch_attn_kv(int G, const AttnArgs &a, int chunks, size_t smem, cudaStream_t stream) {
  const void *fn = nullptr;
  switch (G) {
    case 1: fn = reinterpret_cast<const void *>(k_attn_chunk<KT, VT, 1>); break;
    case 2: fn = reinterpret_cast<const void *>(k_attn_chunk<KT, VT, 2>); break;
    case 4: fn = reinterpret_cast<const void *>(k_attn_chunk<KT, VT, 4>); break;
    case 8: fn = reinterpret_cast<const void *>(k_attn_chunk<KT, VT, 8>); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_smem(fn, int(smem));
  if (e != cudaSuccess) return e;
  switch (G) {
    case 1: k_attn_chunk<KT, VT, 1><<<chunks, kAttnThreads, smem, stream>>>(a); break;
    case 2: k_attn_chunk<KT, VT, 2><<<chunks, kAttnThreads, smem, stream>>>(a); break;
    case 4: k_attn_chunk<KT, VT, 4><<<chunks, kAttnThreads, smem, stream>>>(a); break;
    default: k_attn_chunk<KT, VT, 8><<<chunks, kAttnThreads, smem, stream>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

size_t attn_workspace_bytes(int kt, int vt, int64_t T, int64_t H, int64_t n_kv, int64_t D) {
  const AttnPlan p = attn_plan(kt, vt, T, H, n_kv, D);
  return (size_t(p.chunks) * size_t(H) * size_t(D + 2) * 4 + 255) / 256 * 256;
}

size_t attn_smem_bytes(int kt, int vt, int64_t T, int64_t H, int64_t n_kv, int64_t D) {
  return attn_plan(kt, vt, T, H, n_kv, D).smem;
}

cudaError_t launch_attn_decode(int kt, int vt, const float *q, const uint8_t *K, const uint8_t *V, float *o,
                               int64_t T, int64_t H, int64_t n_kv, int64_t D, float scale, void *ws,
                               cudaStream_t stream) {
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  const AttnPlan p = attn_plan(kt, vt, T, H, n_kv, D);
  AttnArgs a{};
  a.q = q;
  a.K = K;
  a.V = V;
  a.o_part = static_cast<float *>(ws);
  a.ml = a.o_part + size_t(p.chunks) * H * D;
  a.scale = scale;
  a.n_tokens = int(T);
  a.n_heads = int(H);
  a.n_kv = int(n_kv);
  a.D = int(D);
  a.nb = int(D / kQK);
  a.k_tok = p.k_tok;
  a.v_tok = p.v_tok;
  a.chunk_tokens = p.chunk_tokens;
  a.sub = p.sub;
  a.stage_bytes = p.stage_bytes;
  a.ring_bytes = p.ring_bytes;
  a.stages = p.stages;
  a.err = di->err_word;
  a.spin_limit = spin_limit();
  const int G = int(H / n_kv);
  cudaError_t e;
  if (kt == kTypeQ4_0)
    e = vt == kTypeQ4_0 ? launch_attn_kv<kTypeQ4_0, kTypeQ4_0>(G, a, p.chunks, p.smem, stream)
                        : launch_attn_kv<kTypeQ4_0, kTypeQ8_0>(G, a, p.chunks, p.smem, stream);
  else
    e = vt == kTypeQ4_0 ? launch_attn_kv<kTypeQ8_0, kTypeQ4_0>(G, a, p.chunks, p.smem, stream)
                        : launch_attn_kv<kTypeQ8_0, kTypeQ8_0>(G, a, p.chunks, p.smem, stream);
  if (e != cudaSuccess) return e;
  const size_t csmem = size_t(p.chunks) * sizeof(float);
  if ((e = ensure_smem(reinterpret_cast<const void *>(k_attn_combine), int(csmem))) != cudaSuccess) return e;
  k_attn_combine<<<dim3(unsigned(H), unsigned((D + 31) / 32)), 256, csmem, stream>>>(a.o_part, a.ml, o, p.chunks,
                                                                                  int(H), int(D));
  return cudaGetLastError();
}

}  // namespace bq
