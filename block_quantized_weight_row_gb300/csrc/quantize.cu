// quantize.cu — row quantization (Q4_0 / Q8_0), the KV-cache write with an
// optional mean-centering bias, and dequantization.
//
// Row quantize: every 32 consecutive values of a row form one block with one
// binary16 scale ("llama.cpp 原理：如何在普通硬件跑本地大模型", §量化：内存真正去哪了;
// "05. llama.cpp：从 GGUF 文件到本地推理服务", §量化类型). KV write: K is written
// to the cache quantized, optionally after subtracting a calibrated
// per-(kv-head, channel) bias (lpnh.cn KV-cache article, §解法).
//
// Design (HBM-bound: 128 B of fp32 read per 18 or 34 B written; the
// quantization arithmetic must stay well under the SMs' issue rate at that
// byte rate, so one lane owns one whole block: no shuffles, one division per
// block, full-rate rounding, one tie test per block):
//   - warp tile = 32 consecutive blocks (4 KB), copied with fully coalesced
//     16-byte asynchronous copies (cp.async; 512 contiguous bytes per
//     instruction) into one of two warp-private shared-memory tiles while the
//     warp quantizes the other, so every warp keeps 4 KB of reads in flight
//     without holding them in registers (80 registers: a persistent grid of
//     three CTAs per SM); lane i then reads block i. The tiles are
//     XOR-swizzled (16-byte chunk c of block b sits at chunk c ^ (b & 7)),
//     which keeps both the coalesced writes and the per-block reads free of
//     bank conflicts;
//   - the per-value rounding runs on fp32 pairs, and the code words are
//     built as the values are rounded;
//   - a mean-centering bias (one block per (kv-head, 32 channels), a few KB)
//     is staged once per CTA in the same swizzled layout;
//   - the tile's output (576 B Q4_0 / 1088 B Q8_0) is written back into the
//     consumed input tile with word stores and leaves as 16-byte stores.
// Hadamard-rotated K (lpnh.cn KV-cache article, §三步上手, third step: a
// quantized K cache with head_dim a multiple of 64 is rotated, and the bias
// must be measured in the same basis): every 64 channels of a head become
// H64 x / 8 before the bias is subtracted. Blocks 2m and 2m+1 of a tile are
// one group of 64, held by lanes 2m and 2m+1: the butterflies of span 1-16
// run inside a lane, span 32 across the lane pair, then the exact 1/8.
// The bias calibration (k_kv_bias) sums each channel over the tokens in fp64
// in token order, in either basis.
#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kQuantWarps = kQuantThreads / 32;
constexpr int kMaxSmemBiasBlocks = 128;  // 16 KB of bias staged per CTA

// byte offset of 16-byte chunk c of block b in a swizzled tile
__device__ __forceinline__ int swz(int b, int c) { return b * 128 + ((c ^ (b & 7)) << 4); }

// 32 values of one block (elements 32 * (lane & 1) + i of a 64-group) ->
// H64 x / 8: butterflies (a, b) -> (a + b, a - b) of span 1, 2, 4, 8, 16 in
// the lane, span 32 with lane ^ 1, then * 0.125. Every lane of the warp takes
// part. Spans 2-32 run on fp32 pairs (v[2k], v[2k+1]); a - b is the fused
// -1 * b + a, which rounds once like the subtraction, and the cross-lane
// step is s * v + p with s = +1 or -1.
__device__ __forceinline__ void hadamard64_lane_pair(float (&v)[32], int lane) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float a = v[i], b = v[i + 1];
    v[i] = __fadd_rn(a, b);
    v[i + 1] = __fsub_rn(a, b);
  }
  uint64_t P[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) P[k] = pack2(__float_as_uint(v[2 * k]), __float_as_uint(v[2 * k + 1]));
  const uint64_t m1 = pack2(__float_as_uint(-1.0f), __float_as_uint(-1.0f));
#pragma unroll
  for (int hp = 1; hp < 16; hp <<= 1)  // span 2 * hp, in pairs
#pragma unroll
    for (int k = 0; k < 16; ++k)
      if ((k & hp) == 0) {
        const uint64_t t = P[k];
        P[k] = fadd2(t, P[k + hp]);
        P[k + hp] = ffma2(m1, P[k + hp], t);
      }
  const float sg = (lane & 1) ? -1.0f : 1.0f;
  const uint64_t s2 = pack2(__float_as_uint(sg), __float_as_uint(sg));
  const uint64_t e2 = pack2(__float_as_uint(0.125f), __float_as_uint(0.125f));
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t plo = __shfl_xor_sync(kFull, uint32_t(P[k]), 1), phi = __shfl_xor_sync(kFull, uint32_t(P[k] >> 32), 1);
    P[k] = fmul2(ffma2(s2, P[k], pack2(plo, phi)), e2);
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    v[2 * k] = __uint_as_float(uint32_t(P[k]));
    v[2 * k + 1] = __uint_as_float(uint32_t(P[k] >> 32));
  }
}

// 16-byte asynchronous copy global -> shared, zero-filled when !valid (src
// must then still be a mapped address).
__device__ __forceinline__ void cp_async16_zf(void *dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}

// The fast path of quantize_block_lane on fp32 pairs, the code words built
// as the values are rounded (no per-value staging): per value the same IEEE
// operations (product by the reciprocal, rounding add of the magic number,
// subtraction back, and the distance r - (t - M) as the fused -1 * d + r,
// which rounds once like the subtraction). False when the block needs the
// exact path; the words and scale are then not final.
template <int TYPE>
__device__ __forceinline__ bool quantize_block_words_fast(const float (&v)[32], uint16_t &scale,
                                                          uint32_t (&w)[TYPE == kTypeQ4_0 ? 4 : 8]) {
  float ds;
  block_scale<TYPE>(block_amax<TYPE>(v), scale, ds);
  const float inv = ds > 0.0f ? rcp_approx(ds) : 0.0f;
  constexpr float kMagic = 12582912.0f + float(TYPE == kTypeQ4_0 ? 8 : 0);
  const uint64_t inv2 = pack2(__float_as_uint(inv), __float_as_uint(inv));
  const uint64_t mg2 = pack2(__float_as_uint(kMagic), __float_as_uint(kMagic));
  const uint64_t nmg2 = pack2(__float_as_uint(-kMagic), __float_as_uint(-kMagic));
  const uint64_t m1 = pack2(__float_as_uint(-1.0f), __float_as_uint(-1.0f));
  float dmax = 0.0f;
  // the code bytes of values j0 .. j0+3 (low byte of each t) as one word
  auto word4 = [&](int j0) {
    uint32_t t[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint64_t r = fmul2(pack2(__float_as_uint(v[j0 + 2 * h]), __float_as_uint(v[j0 + 2 * h + 1])), inv2);
      const uint64_t tt = fadd2(r, mg2);
      const uint64_t e = ffma2(m1, fadd2(tt, nmg2), r);
      t[2 * h] = uint32_t(tt);
      t[2 * h + 1] = uint32_t(tt >> 32);
      dmax = fmaxf(dmax, fmaxf(fabsf(__uint_as_float(uint32_t(e))), fabsf(__uint_as_float(uint32_t(e >> 32)))));
    }
    return pack_bytes(t[0], t[1], t[2], t[3]);
  };
  if constexpr (TYPE == kTypeQ4_0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = word4(4 * i), hi = word4(16 + 4 * i);
      w[i] = lo + (hi << 4);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = word4(4 * i);
  }
  return !(dmax > 0.4999f || (ds > 0.0f && ds < 6.103515625e-05f));
}

// Shared memory of k_quantize_rows: per warp two 4 KB input tiles (the next
// tile's asynchronous copies land in one while the other is quantized; the
// output blocks are written back into the consumed tile), the legacy types'
// output tiles, then the bias blocks when they fit.
template <int TYPE>
constexpr int quant_out_bytes() {
  return Legacy<TYPE>::kIs ? kQuantWarps * 32 * Fmt<TYPE>::kBytes : 0;
}
template <int TYPE>
size_t quant_smem_bytes(int64_t bias_smem_blocks) {
  return size_t(kQuantWarps) * 2 * 32 * 128 + size_t(quant_out_bytes<TYPE>()) + size_t(bias_smem_blocks) * 128;
}

// BMODE: where the bias lives. 0: decided at run time (staged in shared
// memory when it fits, else read from global memory); 1: staged negated in
// shared memory and added as fp32 pairs (x - b and x + (-b) are the same IEEE
// sum), with a branch-free block store; 2: global memory. The rotated writes
// with a bias take 1 or 2 (fewer instructions where the rotation already
// makes the kernel issue-bound); the others 0 (the specialised forms cost the
// plain kernel registers: at 80 registers a stack frame).
template <int TYPE, bool BIAS, bool ROT, int BMODE = 0>
__global__ void __launch_bounds__(kQuantThreads, 3)
    k_quantize_rows(const float *__restrict__ src, uint8_t *__restrict__ dst, int64_t n_blocks,
                    const float *__restrict__ bias, int64_t bias_period, int bias_smem_blocks, int pair) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  constexpr int NW = TYPE == kTypeQ4_0 ? 4 : 8;  // code words per block (Q4_0 / Q8_0)
  constexpr int kTile = 32 * 128;
  extern __shared__ __align__(128) uint8_t qsm[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t *tiles = qsm + warp * 2 * kTile;
  uint8_t *ot = qsm + kQuantWarps * 2 * kTile + warp * 32 * BB;  // legacy types only
  uint8_t *bias_tile = qsm + kQuantWarps * 2 * kTile + quant_out_bytes<TYPE>();
  const bool bias_in_smem = BMODE == 1 || (BMODE == 0 && BIAS && bias_smem_blocks > 0);
  if (bias_in_smem) {
    for (int i = threadIdx.x; i < bias_smem_blocks * 8; i += kQuantThreads) {
      float4 f = __ldg(reinterpret_cast<const float4 *>(bias) + i);
      if (BMODE == 1) f = make_float4(-f.x, -f.y, -f.z, -f.w);  // x - b is the identical sum x + (-b)
      *reinterpret_cast<float4 *>(bias_tile + swz(i >> 3, i & 7)) = f;
    }
    __syncthreads();
  }
  const bool bias_pow2 = (bias_period & (bias_period - 1)) == 0;
  // the first launch of a one-layer KV write lets the second (the other
  // tensor) be scheduled at once: it touches none of this launch's memory,
  // and its CTAs take the SMs this grid's CTAs leave. No other launch does:
  // a dependent GEMV streams its weights before its dependency wait, and
  // these may be the rows this launch writes.
  if (pair == 1) pdl_launch_dependents();
  const int64_t total_warps = int64_t(gridDim.x) * kQuantWarps;
  // coalesced: vector i = lane + 32c of a tile is chunk (i & 7) of block (i >> 3)
  auto issue_tile = [&](int64_t t, uint8_t *buf) {
    const int64_t nb = t * 32 < n_blocks ? min(int64_t(32), n_blocks - t * 32) : 0;
    const float *g = src + t * 32 * kQK;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int i = lane + 32 * c;
      const bool in = (i >> 3) < nb;
      cp_async16_zf(buf + swz(i >> 3, i & 7), in ? static_cast<const void *>(g + 4 * i) : src, in);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  int64_t tile = int64_t(blockIdx.x) * kQuantWarps + warp;
  issue_tile(tile, tiles);
  for (int k = 0; tile * 32 < n_blocks; tile += total_warps, k ^= 1) {
    uint8_t *it = tiles + k * kTile;
    issue_tile(tile + total_warps, tiles + (k ^ 1) * kTile);  // in flight while this tile is quantized
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncwarp();
    const int nblk = int(min(int64_t(32), n_blocks - tile * 32));
    float v[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 f = *reinterpret_cast<const float4 *>(it + swz(lane, c));
      v[4 * c] = f.x;
      v[4 * c + 1] = f.y;
      v[4 * c + 2] = f.z;
      v[4 * c + 3] = f.w;
    }
    if (ROT) hadamard64_lane_pair(v, lane);
    const int64_t b = tile * 32 + lane;
    // block b of row (token, head) uses bias block b mod (heads * blocks per row)
    const int64_t bb = BIAS ? (bias_pow2 ? (b & (bias_period - 1)) : b % bias_period) : 0;
    auto sub_bias = [&](float (&x)[32]) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        if constexpr (BMODE == 1) {
          const float4 f = *reinterpret_cast<const float4 *>(bias_tile + swz(int(bb), c));  // -bias
          const uint64_t a = fadd2(pack2(__float_as_uint(x[4 * c]), __float_as_uint(x[4 * c + 1])),
                                   pack2(__float_as_uint(f.x), __float_as_uint(f.y)));
          const uint64_t d = fadd2(pack2(__float_as_uint(x[4 * c + 2]), __float_as_uint(x[4 * c + 3])),
                                   pack2(__float_as_uint(f.z), __float_as_uint(f.w)));
          x[4 * c] = __uint_as_float(uint32_t(a));
          x[4 * c + 1] = __uint_as_float(uint32_t(a >> 32));
          x[4 * c + 2] = __uint_as_float(uint32_t(d));
          x[4 * c + 3] = __uint_as_float(uint32_t(d >> 32));
        } else {
          const float4 f = (BMODE == 0 && bias_in_smem) ? *reinterpret_cast<const float4 *>(bias_tile + swz(int(bb), c))
                                                        : __ldg(reinterpret_cast<const float4 *>(bias + bb * kQK) + c);
          x[4 * c] = __fsub_rn(x[4 * c], f.x);
          x[4 * c + 1] = __fsub_rn(x[4 * c + 1], f.y);
          x[4 * c + 2] = __fsub_rn(x[4 * c + 2], f.z);
          x[4 * c + 3] = __fsub_rn(x[4 * c + 3], f.w);
        }
      }
    };
    if (BIAS && b < n_blocks) sub_bias(v);
    const uint8_t *out_src;
    if constexpr (Legacy<TYPE>::kIs) {
      // legacy types: the exact rule for every block
      legacy_quantize_block<TYPE>(v, reinterpret_cast<uint16_t *>(ot + lane * BB));
      out_src = ot;
    } else {
      uint16_t scale;
      uint32_t w[NW];
      if (!quantize_block_words_fast<TYPE>(v, scale, w)) {
        // rare (a value near a tie, or a subnormal scale): the block again
        // through the exact path (rotated: from the registers, which still
        // hold the rotated, centred values)
        if constexpr (ROT) {
          quantize_block_lane_exact<TYPE>(v, scale, w);
        } else {
          float e[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 f = *reinterpret_cast<const float4 *>(it + swz(lane, c));
            e[4 * c] = f.x;
            e[4 * c + 1] = f.y;
            e[4 * c + 2] = f.z;
            e[4 * c + 3] = f.w;
          }
          if (BIAS && b < n_blocks) sub_bias(e);
          quantize_block_lane_exact<TYPE>(e, scale, w);
        }
      }
      __syncwarp();  // every lane has read its block before outputs land in the tile
      // block `lane` at byte lane*BB of the consumed tile (BB = 2 mod 4: even
      // lanes start on a word, odd lanes half a word later)
      uint8_t *ob = it + lane * BB;
      if constexpr (BMODE != 0) {
        // branch-free: odd lanes start half a word later
        const bool odd = lane & 1;
        uint32_t *o32 = reinterpret_cast<uint32_t *>(ob + (odd ? 2 : 0));
        const uint32_t sh = odd ? 32u : 16u;
        uint32_t prev = uint32_t(scale) << 16;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
          o32[i] = __funnelshift_rc(prev, w[i], sh);
          prev = w[i];
        }
        *reinterpret_cast<uint16_t *>(ob + (odd ? 0 : 4 * NW)) = odd ? scale : uint16_t(w[NW - 1] >> 16);
      } else if (lane & 1) {
        *reinterpret_cast<uint16_t *>(ob) = scale;
#pragma unroll
        for (int i = 0; i < NW; ++i) reinterpret_cast<uint32_t *>(ob + 2)[i] = w[i];
      } else {
        uint32_t *o32 = reinterpret_cast<uint32_t *>(ob);
        o32[0] = uint32_t(scale) | (w[0] << 16);
#pragma unroll
        for (int i = 1; i < NW; ++i) o32[i] = __funnelshift_r(w[i - 1], w[i], 16);
        *reinterpret_cast<uint16_t *>(ob + 4 * NW) = uint16_t(w[NW - 1] >> 16);
      }
      out_src = it;
    }
    __syncwarp();
    const int nbytes = nblk * BB;
    uint8_t *out = dst + tile * 32 * BB;  // 16-byte aligned: 32 * BB is a multiple of 16
    const int n16 = nbytes / 16;
    for (int i = lane; i < n16; i += 32)
      reinterpret_cast<uint4 *>(out)[i] = reinterpret_cast<const uint4 *>(out_src)[i];
    for (int i = n16 * 8 + lane; i < nbytes / 2; i += 32)
      reinterpret_cast<uint16_t *>(out)[i] = reinterpret_cast<const uint16_t *>(out_src)[i];
    __syncwarp();  // the next iteration refills this buffer
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy in flight at exit
  // the second launch of the pair ends only after the first has completed,
  // so that whatever follows on the stream is ordered after both
  if (pair == 2) pdl_wait();
}

// x_hat = scale * q, exact in fp32. One thread per 4 outputs.
template <int TYPE>
__global__ void __launch_bounds__(256)
    k_dequantize_rows(const uint8_t *__restrict__ blocks, float *__restrict__ dst, int64_t n_blocks) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  const int64_t n_quads = n_blocks * 8;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_quads;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t g = i >> 3;
    const int j = int(i & 7);  // elements 4j..4j+3
    const uint8_t *blk = blocks + g * BB;
    const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
    if constexpr (Legacy<TYPE>::kIs) {
      using L = Legacy<TYPE>;
      const uint16_t *h = reinterpret_cast<const uint16_t *>(blk);  // 2-byte aligned
      const float mn = L::kAffine ? half_bits_to_float(h[1]) : 0.0f;
      const uint32_t qh = L::kQh >= 0 ? (uint32_t(h[L::kQh / 2]) | (uint32_t(h[L::kQh / 2 + 1]) << 16)) : 0u;
      float r[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int el = 4 * j + e;
        const uint8_t b = blk[L::kQs + (el & 15)];
        const int uu = int((el < 16 ? (b & 0x0f) : (b >> 4)) | (((qh >> el) & 1u) << 4));
        // value d * u + m (two fp32 operations) or d * (u - 16)
        r[e] = L::kAffine ? __fadd_rn(__fmul_rn(d, float(uu)), mn) : __fmul_rn(d, float(uu - 16));
      }
      reinterpret_cast<float4 *>(dst)[i] = make_float4(r[0], r[1], r[2], r[3]);
    } else {
      int q[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (TYPE == kTypeQ4_0) {
          const int el = 4 * j + e;
          const uint8_t b = blk[2 + (el & 15)];
          q[e] = int(el < 16 ? (b & 0x0f) : (b >> 4)) - 8;
        } else {
          q[e] = int(static_cast<int8_t>(blk[2 + 4 * j + e]));
        }
      }
      float4 o;
      o.x = __fmul_rn(d, float(q[0]));
      o.y = __fmul_rn(d, float(q[1]));
      o.z = __fmul_rn(d, float(q[2]));
      o.w = __fmul_rn(d, float(q[3]));
      reinterpret_cast<float4 *>(dst)[i] = o;
    }
  }
}

// k-quants: one warp per super-block of 256 values, lane l holding values
// 8l..8l+7; the sub-block extremes and the super-block maxima are reductions
// (order-free), every other step the exact rule of the block format.
template <int TYPE>
__global__ void __launch_bounds__(256) k_quantize_kq(const float *__restrict__ src, uint8_t *__restrict__ dst,
                                                     int64_t n_sb) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  const int lane = threadIdx.x & 31;
  for (int64_t sb = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; sb < n_sb;
       sb += (int64_t(gridDim.x) * blockDim.x) >> 5) {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(src + sb * kQK_K) + 2 * lane);
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(src + sb * kQK_K) + 2 * lane + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint8_t *out = dst + sb * BB;
    if constexpr (TYPE == kTypeQ4_K) {
      float lo = v[0], hi = v[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) {
        lo = fminf(lo, v[i]);
        hi = fmaxf(hi, v[i]);
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {  // the 4 lanes of a sub-block of 32
        lo = fminf(lo, __shfl_xor_sync(kFull, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(kFull, hi, o));
      }
      const float m = lo < 0.0f ? -lo : 0.0f;
      const float sj = __fdiv_rn(__fadd_rn(hi, m), 15.0f);
      float smax = sj, mmax = m;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, o));
        mmax = fmaxf(mmax, __shfl_xor_sync(kFull, mmax, o));
      }
      const __half hd = __float2half_rn(__fdiv_rn(smax, 63.0f)), hm = __float2half_rn(__fdiv_rn(mmax, 63.0f));
      const float d = __half2float(hd), dm = __half2float(hm);
      const int sc = d == 0.0f ? 0 : min(max(int(rintf(__fdiv_rn(sj, d))), 0), 63);
      const int mn = dm == 0.0f ? 0 : min(max(int(rintf(__fdiv_rn(m, dm))), 0), 63);
      const float S = __fmul_rn(d, float(sc)), M = __fmul_rn(dm, float(mn));
      uint32_t packed = 0;  // the lane's 8 codes, 4 bits each
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int u = S == 0.0f ? 0 : min(max(int(rintf(__fdiv_rn(__fadd_rn(v[i], M), S))), 0), 15);
        packed |= uint32_t(u) << (4 * i);
      }
      // header: d, dmin and the 96-bit stream of sc[0..7], mn[0..7] (lane 4j has sub-block j's)
      uint64_t lo64 = 0;
      uint32_t hi32 = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint64_t sv = uint64_t(__shfl_sync(kFull, sc, 4 * j)), mv = uint64_t(__shfl_sync(kFull, mn, 4 * j));
        lo64 |= sv << (6 * j);  // bits 0..47
        const int bm = 48 + 6 * j;
        if (bm + 6 <= 64) lo64 |= mv << bm;
        else if (bm >= 64) hi32 |= uint32_t(mv << (bm - 64));
        else { lo64 |= mv << bm; hi32 |= uint32_t(mv >> (64 - bm)); }
      }
      const uint32_t partner = __shfl_down_sync(kFull, packed, 2);  // codes i + 16 of this lane's i
      if (lane == 0)
        *reinterpret_cast<uint4 *>(out) = make_uint4(uint32_t(__half_as_ushort(hd)) | (uint32_t(__half_as_ushort(hm)) << 16),
                                                     uint32_t(lo64), uint32_t(lo64 >> 32), hi32);
      if ((lane & 3) < 2) {
        uint32_t w0 = 0, w1 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          w0 |= (((packed >> (4 * i)) & 15u) | (((partner >> (4 * i)) & 15u) << 4)) << (8 * i);
          w1 |= (((packed >> (4 * i + 16)) & 15u) | (((partner >> (4 * i + 16)) & 15u) << 4)) << (8 * i);
        }
        *reinterpret_cast<uint2 *>(out + 16 + 16 * (lane >> 2) + 8 * (lane & 3)) = make_uint2(w0, w1);
      }
    } else {  // Q6_K
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));  // the 2 lanes of a sub-block of 16
      const float sk = __fdiv_rn(amax, 31.0f);
      float smax = sk;
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, o));
      const __half hd = __float2half_rn(__fdiv_rn(smax, 127.0f));
      const float d = __half2float(hd);
      const int sc = d == 0.0f ? 0 : min(max(int(rintf(__fdiv_rn(sk, d))), -128), 127);
      const float S = __fmul_rn(d, float(sc));
      uint32_t lo4 = 0, hi2 = 0;  // the lane's 8 codes: low 4 bits, top 2 bits
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int u = (S == 0.0f ? 0 : min(max(int(rintf(__fdiv_rn(v[i], S))), -32), 31)) + 32;
        lo4 |= uint32_t(u & 15) << (4 * i);
        hi2 |= uint32_t(u >> 4) << (2 * i);
      }
      uint16_t *o16 = reinterpret_cast<uint16_t *>(out);  // 2-byte aligned
      const uint32_t lo_up = __shfl_down_sync(kFull, lo4, 16);  // codes i + 128
      if (lane < 16) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t b0 = ((lo4 >> (8 * k)) & 15u) | (((lo_up >> (8 * k)) & 15u) << 4);
          const uint32_t b1 = ((lo4 >> (8 * k + 4)) & 15u) | (((lo_up >> (8 * k + 4)) & 15u) << 4);
          o16[4 * lane + k] = uint16_t(b0 | (b1 << 8));
        }
      }
      const uint32_t h1 = __shfl_down_sync(kFull, hi2, 8), h2 = __shfl_down_sync(kFull, hi2, 16),
                     h3 = __shfl_down_sync(kFull, hi2, 24);  // codes i + 64, i + 128, i + 192
      if (lane < 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t bb[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = 2 * k + e;
            bb[e] = ((hi2 >> (2 * i)) & 3u) | (((h1 >> (2 * i)) & 3u) << 2) | (((h2 >> (2 * i)) & 3u) << 4) |
                    (((h3 >> (2 * i)) & 3u) << 6);
          }
          o16[64 + 4 * lane + k] = uint16_t(bb[0] | (bb[1] << 8));
        }
      }
      if ((lane & 1) == 0) out[192 + (lane >> 1)] = uint8_t(int8_t(sc));
      if (lane == 0) o16[104] = __half_as_ushort(hd);
    }
  }
}

template <int TYPE>
__global__ void __launch_bounds__(256) k_dequantize_kq(const uint8_t *__restrict__ blocks, float *__restrict__ dst,
                                                       int64_t n_sb) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  const int lane = threadIdx.x & 31;
  for (int64_t sb = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; sb < n_sb;
       sb += (int64_t(gridDim.x) * blockDim.x) >> 5) {
    const uint8_t *blk = blocks + sb * BB;
    float r[8];
    if constexpr (TYPE == kTypeQ4_K) {
      const uint4 h = *reinterpret_cast<const uint4 *>(blk);
      const int j = lane >> 2;
      const float d = half_bits_to_float(h.x & 0xffffu), dm = half_bits_to_float(h.x >> 16);
      const float S = __fmul_rn(d, float(q4k_stream(h.y, h.z, h.w, j)));
      const float M = __fmul_rn(dm, float(q4k_stream(h.y, h.z, h.w, 8 + j)));
      const uint2 c = *reinterpret_cast<const uint2 *>(blk + 16 + 16 * j + 8 * (lane & 1));
      const uint32_t sh = (lane & 2) ? 4u : 0u;  // lanes 4j+2, 4j+3: the high nibbles
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t u = (((i < 4 ? c.x : c.y) >> (8 * (i & 3))) >> sh) & 15u;
        r[i] = __fsub_rn(__fmul_rn(S, float(u)), M);
      }
    } else {
      const uint16_t *b16 = reinterpret_cast<const uint16_t *>(blk);
      const float d = half_bits_to_float(b16[104]);
      const float S = __fmul_rn(d, float(int8_t(blk[192 + (lane >> 1)])));
      const int lo_off = (8 * lane) & 127, hi_off = (8 * lane) & 63;
      const uint32_t lsh = lane < 16 ? 0u : 4u, hsh = 2u * uint32_t(lane >> 3);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t ql = blk[lo_off + i], qh = blk[128 + hi_off + i];
        const int u = int(((ql >> lsh) & 15u) | (((qh >> hsh) & 3u) << 4));
        r[i] = __fmul_rn(S, float(u - 32));
      }
    }
    float4 *o = reinterpret_cast<float4 *>(dst + sb * kQK_K) + 2 * lane;
    o[0] = make_float4(r[0], r[1], r[2], r[3]);
    o[1] = make_float4(r[4], r[5], r[6], r[7]);
  }
}

// pair: 0 a launch of its own; 1 the first launch of a one-layer KV write
// (lets the second start at once); 2 the second: launched as a programmatic
// dependent of the first without waiting for it to start work (their memory
// is disjoint, and the first waited for all earlier work), and waiting for
// it to complete before ending.
template <int TYPE, bool BIAS, bool ROT, int BMODE = 0>
cudaError_t launch_q_mode(const float *src, uint8_t *dst, int64_t n_blocks, const float *bias, int64_t bias_period,
                          cudaStream_t stream, int pair) {
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  const int64_t tiles = (n_blocks + 31) / 32;
  const int64_t ctas = (tiles + kQuantWarps - 1) / kQuantWarps;
  const int64_t grid = min(ctas, int64_t(di->sm_count) * 3);  // persistent: 3 resident CTAs per SM
  const int bias_smem_blocks = (BIAS && BMODE != 2 && bias_period <= kMaxSmemBiasBlocks) ? int(bias_period) : 0;
  const size_t smem = quant_smem_bytes<TYPE>(bias_smem_blocks);
  err = ensure_smem(reinterpret_cast<const void *>(k_quantize_rows<TYPE, BIAS, ROT, BMODE>), int(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kQuantThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pair == 2 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_quantize_rows<TYPE, BIAS, ROT, BMODE>, src, dst, n_blocks, bias, bias_period,
                            bias_smem_blocks, pair);
}

// The rotated writes with a bias take instantiations specialised on where
// the bias lives (staged negated in shared memory, added as fp32 pairs; or
// read from global memory), the plain writes one that decides at run time.
template <int TYPE, bool BIAS, bool ROT>
cudaError_t launch_q(const float *src, uint8_t *dst, int64_t n_blocks, const float *bias, int64_t bias_period,
                     cudaStream_t stream, int pair = 0) {
  if constexpr (ROT && BIAS) {
    if (bias_period <= kMaxSmemBiasBlocks)
      return launch_q_mode<TYPE, true, true, 1>(src, dst, n_blocks, bias, bias_period, stream, pair);
    return launch_q_mode<TYPE, true, true, 2>(src, dst, n_blocks, bias, bias_period, stream, pair);
  } else {
    return launch_q_mode<TYPE, BIAS, ROT, 0>(src, dst, n_blocks, bias, bias_period, stream, pair);
  }
}

template <bool ROT>
cudaError_t launch_q_typed(int type, const float *src, uint8_t *dst, int64_t n_blocks, const float *bias,
                           int64_t bias_period, cudaStream_t stream) {
  // legacy types: no bias and no rotation (rejected by the ABI layer)
  if (type == kTypeQ4_1) return launch_q<kTypeQ4_1, false, false>(src, dst, n_blocks, nullptr, 1, stream);
  if (type == kTypeQ5_0) return launch_q<kTypeQ5_0, false, false>(src, dst, n_blocks, nullptr, 1, stream);
  if (type == kTypeQ5_1) return launch_q<kTypeQ5_1, false, false>(src, dst, n_blocks, nullptr, 1, stream);
  if (type == kTypeQ4_0)
    return bias ? launch_q<kTypeQ4_0, true, ROT>(src, dst, n_blocks, bias, bias_period, stream)
                : launch_q<kTypeQ4_0, false, ROT>(src, dst, n_blocks, nullptr, 1, stream);
  // a bias with Q8_0 is rejected by the ABI layer
  return launch_q<kTypeQ8_0, false, ROT>(src, dst, n_blocks, nullptr, 1, stream);
}

// One layer's KV write (lpnh.cn KV-cache article, §解法 and §三步上手): the two
// tensors' row-quantize launches, the second a programmatic dependent of the
// first that does not wait for it. K and V share no memory, so the second
// launch's CTAs may fill the SMs that the first launch's persistent CTAs
// leave as they finish; the second cannot start before the first has, and
// the first starts after every earlier launch. Order (measured): K first for
// a plain K (V's memory-bound start then overlaps K's arithmetic-heavy
// tail), V first for a rotated K (the longer K half then fills V's tail).
cudaError_t launch_kv_write_pair(int k_type, int v_type, bool k_rot, const float *k_src, uint8_t *k_dst,
                                 const float *v_src, uint8_t *v_dst, int64_t n_blocks, const float *bias,
                                 int64_t bias_period, cudaStream_t stream) {
  auto launch_k = [&](int pair) {
    if (k_type == kTypeQ4_0) {
      if (bias)
        return k_rot ? launch_q<kTypeQ4_0, true, true>(k_src, k_dst, n_blocks, bias, bias_period, stream, pair)
                     : launch_q<kTypeQ4_0, true, false>(k_src, k_dst, n_blocks, bias, bias_period, stream, pair);
      return k_rot ? launch_q<kTypeQ4_0, false, true>(k_src, k_dst, n_blocks, nullptr, 1, stream, pair)
                   : launch_q<kTypeQ4_0, false, false>(k_src, k_dst, n_blocks, nullptr, 1, stream, pair);
    }
    return k_rot ? launch_q<kTypeQ8_0, false, true>(k_src, k_dst, n_blocks, nullptr, 1, stream, pair)
                 : launch_q<kTypeQ8_0, false, false>(k_src, k_dst, n_blocks, nullptr, 1, stream, pair);
  };
  auto launch_v = [&](int pair) {
    return v_type == kTypeQ4_0 ? launch_q<kTypeQ4_0, false, false>(v_src, v_dst, n_blocks, nullptr, 1, stream, pair)
                               : launch_q<kTypeQ8_0, false, false>(v_src, v_dst, n_blocks, nullptr, 1, stream, pair);
  };
  cudaError_t e = k_rot ? launch_v(1) : launch_k(1);
  if (e != cudaSuccess) return e;
  return k_rot ? launch_k(2) : launch_v(2);
}

// bias[h][c] = fp32(sum_t r_t[h][c] / n_tokens), the sum in fp64 in token
// order; r_t the token's row, rotated per 64 channels when ROT. One warp per
// group of 64 channels (lane: channels lane and lane + 32) when ROT, else one
// thread per channel. The loads of the next tokens are issued ahead.
template <bool ROT>
__global__ void __launch_bounds__(128) k_kv_bias(const float *__restrict__ rows, float *__restrict__ bias,
                                                 int64_t n_tokens, int64_t row_len) {
  constexpr int kAhead = 8;
  if (ROT) {
    const int64_t g = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // group of 64
    const int lane = threadIdx.x & 31;
    if (g * 64 >= row_len) return;  // uniform per warp
    const float *p = rows + g * 64 + lane;
    double s0 = 0.0, s1 = 0.0;
    for (int64_t t0 = 0; t0 < n_tokens; t0 += kAhead) {
      float x0[kAhead], x1[kAhead];
#pragma unroll
      for (int k = 0; k < kAhead; ++k) {
        const bool in = t0 + k < n_tokens;
        x0[k] = in ? __ldg(p + (t0 + k) * row_len) : 0.0f;
        x1[k] = in ? __ldg(p + (t0 + k) * row_len + 32) : 0.0f;
      }
#pragma unroll
      for (int k = 0; k < kAhead; ++k) {
        float a0 = x0[k], a1 = x1[k];
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
          const float p0 = __shfl_xor_sync(kFull, a0, h), p1 = __shfl_xor_sync(kFull, a1, h);
          const bool up = (lane & h) != 0;
          a0 = up ? __fsub_rn(p0, a0) : __fadd_rn(a0, p0);
          a1 = up ? __fsub_rn(p1, a1) : __fadd_rn(a1, p1);
        }
        const float b0 = __fmul_rn(__fadd_rn(a0, a1), 0.125f), b1 = __fmul_rn(__fsub_rn(a0, a1), 0.125f);
        if (t0 + k < n_tokens) {
          s0 = __dadd_rn(s0, double(b0));
          s1 = __dadd_rn(s1, double(b1));
        }
      }
    }
    bias[g * 64 + lane] = float(__ddiv_rn(s0, double(n_tokens)));
    bias[g * 64 + lane + 32] = float(__ddiv_rn(s1, double(n_tokens)));
  } else {
    const int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= row_len) return;
    double s = 0.0;
    for (int64_t t0 = 0; t0 < n_tokens; t0 += kAhead) {
      float x[kAhead];
#pragma unroll
      for (int k = 0; k < kAhead; ++k) x[k] = t0 + k < n_tokens ? __ldg(rows + (t0 + k) * row_len + c) : 0.0f;
#pragma unroll
      for (int k = 0; k < kAhead; ++k)
        if (t0 + k < n_tokens) s = __dadd_rn(s, double(x[k]));
    }
    bias[c] = float(__ddiv_rn(s, double(n_tokens)));
  }
}

}  // namespace

cudaError_t launch_quantize_rows(int type, const float *src, uint8_t *dst, int64_t n_blocks,
                                 int64_t /*blocks_per_row*/, const float *bias, int64_t bias_period,
                                 cudaStream_t stream, bool rotate) {
  if (n_blocks == 0) return cudaSuccess;
  if (type == kTypeQ4_K || type == kTypeQ6_K) {  // n_blocks counts super-blocks here
    cudaError_t err;
    const DeviceInfo *di = device_info(&err);
    if (!di) return err;
    const unsigned grid = unsigned(min((n_blocks + 7) / 8, int64_t(di->sm_count) * 8));
    if (type == kTypeQ4_K)
      k_quantize_kq<kTypeQ4_K><<<grid, 256, 0, stream>>>(src, dst, n_blocks);
    else
      k_quantize_kq<kTypeQ6_K><<<grid, 256, 0, stream>>>(src, dst, n_blocks);
    return cudaGetLastError();
  }
  return rotate ? launch_q_typed<true>(type, src, dst, n_blocks, bias, bias_period, stream)
                : launch_q_typed<false>(type, src, dst, n_blocks, bias, bias_period, stream);
}

cudaError_t launch_kv_write(int k_type, int v_type, bool k_rot, const float *k_src, uint8_t *k_dst,
                            const float *v_src, uint8_t *v_dst, int64_t n_blocks, const float *bias,
                            int64_t bias_period, cudaStream_t stream) {
  if (n_blocks == 0) return cudaSuccess;
  return launch_kv_write_pair(k_type, v_type, k_rot, k_src, k_dst, v_src, v_dst, n_blocks, bias, bias_period, stream);
}

cudaError_t launch_kv_bias(const float *rows, float *bias, int64_t n_tokens, int64_t row_len, bool rotate,
                           cudaStream_t stream) {
  if (row_len == 0) return cudaSuccess;
  const int64_t threads = rotate ? row_len / 64 * 32 : row_len;
  const unsigned grid = unsigned((threads + 127) / 128);
  if (rotate)
    k_kv_bias<true><<<grid, 128, 0, stream>>>(rows, bias, n_tokens, row_len);
  else
    k_kv_bias<false><<<grid, 128, 0, stream>>>(rows, bias, n_tokens, row_len);
  return cudaGetLastError();
}

cudaError_t launch_dequantize_rows(int type, const uint8_t *blocks, float *dst, int64_t n_blocks,
                                   cudaStream_t stream) {
  if (n_blocks == 0) return cudaSuccess;
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  if (type == kTypeQ4_K || type == kTypeQ6_K) {  // n_blocks counts super-blocks here
    const unsigned grid = unsigned(min((n_blocks + 7) / 8, int64_t(di->sm_count) * 8));
    if (type == kTypeQ4_K)
      k_dequantize_kq<kTypeQ4_K><<<grid, 256, 0, stream>>>(blocks, dst, n_blocks);
    else
      k_dequantize_kq<kTypeQ6_K><<<grid, 256, 0, stream>>>(blocks, dst, n_blocks);
    return cudaGetLastError();
  }
  const int64_t grid = min((n_blocks * 8 + 255) / 256, int64_t(di->sm_count) * 8);
  switch (type) {
    case kTypeQ4_0: k_dequantize_rows<kTypeQ4_0><<<unsigned(grid), 256, 0, stream>>>(blocks, dst, n_blocks); break;
    case kTypeQ4_1: k_dequantize_rows<kTypeQ4_1><<<unsigned(grid), 256, 0, stream>>>(blocks, dst, n_blocks); break;
    case kTypeQ5_0: k_dequantize_rows<kTypeQ5_0><<<unsigned(grid), 256, 0, stream>>>(blocks, dst, n_blocks); break;
    case kTypeQ5_1: k_dequantize_rows<kTypeQ5_1><<<unsigned(grid), 256, 0, stream>>>(blocks, dst, n_blocks); break;
    default: k_dequantize_rows<kTypeQ8_0><<<unsigned(grid), 256, 0, stream>>>(blocks, dst, n_blocks); break;
  }
  return cudaGetLastError();
}

}  // namespace bq
