// gemv.cu — decode GEMV over block-quantized weights: y = W . x for one token.
//
// Decode reads every weight once per token, so its speed is bounded by
// memory bandwidth divided by the weight bytes ("05. llama.cpp：从 GGUF 文件到
// 本地推理服务", §性能直觉：带宽决定 Decode，算力决定 Prefill). The kernel is
// therefore built to stream W from HBM at full rate:
//
//   - x (fp32) is quantized to Q8_0 (same block rule as the row quantizer, so
//     the codes are bit-identical) either once per launch by a small prep
//     kernel into the caller's workspace, whose records every GEMV CTA copies
//     (with programmatic dependent launch the prep kernel also asks L2 for
//     the launch's weights while the previous kernel runs), or, without a
//     workspace, by every CTA itself (two lanes per block) while its weight
//     stream is already in flight. The two paths give bit-identical records.
//   - One producer warp streams the CTA's rows with 1-D bulk async copies
//     (cp.async.bulk) into a ring of shared-memory stages, completing on
//     mbarriers; 8 consumer warps wait on those barriers and release stages
//     through a second set of mbarriers.
//   - Consumer lane <-> a group of 8 consecutive blocks (144 B Q4_0 / 272 B
//     Q8_0, i.e. 9 / 17 aligned 16-byte words): the group is read with
//     conflict-free 128-bit shared loads, blocks are cut out in registers with
//     funnel shifts, and the integer dot of each block runs on dp4a against the
//     quantized x. x's codes, scales and code sums are stored per group with
//     a 16-byte pad so the 128-bit reads of 8 neighbouring lanes hit distinct
//     banks.
//   - Per block: term = (scale_w * scale_x) * sumi, one fma into a per-lane
//     fp32 partial (the scale product of two binary16 values is exact in
//     fp32, sumi is exact in int32); lanes of a row then reduce by a shuffle
//     tree. At most 16 sequential terms per lane plus 5 tree levels.
//   - Rows with K % 256 != 0 (row bytes not a multiple of 16) take a plain
//     warp-per-row kernel with 2-byte loads.
#include <algorithm>
#include <numeric>

#include "bq_device.cuh"
#include "bq_internal.h"
#include "gemv_common.cuh"

namespace bq {
namespace {

using gemv::kXRecBytes;
using gemv::kXRecWords;
using gemv::group_terms;
using gemv::quantize_x_records;
using gemv::quantize_x_records_2lane;
using gemv::GroupWords;
using gemv::q6k_group_terms;

constexpr int kConsumerWarps = 8;
constexpr int kMaxMats = BQ_GEMV_MAX_MATS;

constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kDrainLimit = 1u << 26;
constexpr int kMaxStageBytes = 64 * 1024;

struct GemvArgs {
  const uint8_t *W[kMaxMats];  // matrix i: rows [row_start[i], row_start[i+1]) of the batch
  float *y[kMaxMats];
  int row_start[kMaxMats + 1];
  int n_mats;
  const float *x;
  int M;               // total rows of the batch
  int K;
  int groups;          // K / 256
  int lanes_per_row;   // power of two <= 32
  int rows_per_warp;   // 32 / lanes_per_row: rows one warp covers per pass
  int row_bytes;
  int stage_rows;      // at most this many rows per stage (one bulk copy)
  int stages;
  int stage_bytes;     // stage_rows * row_bytes
  int row_quantum;     // rows whose bytes are a multiple of 16: CTA ranges and stages are multiples of it
  int xrec_bytes;      // groups * kXRecBytes rounded up to 128
  const uint32_t *rec;  // x's records written by k_gemv_prep, or null: quantize x here
  unsigned *err;
  uint32_t spin_limit;
};

// The CTA's rows are cut into stages of at most stage_rows rows that never
// straddle two matrices; producer and consumers walk the same sequence.
struct StageCursor {
  int row;  // global row of the batch where the next stage starts
  __device__ __forceinline__ void next(const GemvArgs &a, int r1, int &mat, int &nrows) const {
    mat = 0;
    while (row >= a.row_start[mat + 1]) ++mat;
    nrows = min(min(a.stage_rows, r1 - row), a.row_start[mat + 1] - row);
  }
};

template <int TYPE>
__global__ void __launch_bounds__(kGemvThreads, 2) k_gemv_tma(const GemvArgs a) {
  constexpr int GW = GroupWords<TYPE>::kWords;
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t *xrec = reinterpret_cast<uint32_t *>(smem);
  uint8_t *stage_base = smem + a.xrec_bytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(stage_base + size_t(a.stages) * a.stage_bytes);
  uint64_t *empty = full + a.stages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // contiguous, balanced row range of this CTA (in whole row quanta, so that
  // every bulk copy starts on a 16-byte boundary), streamed in stages
  const int nq = a.M / a.row_quantum;
  const int r0 = int(int64_t(nq) * blockIdx.x / gridDim.x) * a.row_quantum;
  const int r1 = int(int64_t(nq) * (blockIdx.x + 1) / gridDim.x) * a.row_quantum;
  const int S = a.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);  // every consumer warp releases every stage
    }
    fence_mbar_init();
  }
  __syncthreads();
  // The next kernel on the stream may start as soon as every CTA got here
  // (only when it was launched with programmatic dependent launch).
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      // without records, every CTA loads x after the wait: ask L2 for it now
      // (no data comes to the SM; the previous kernel's stores to x land in
      // L2, so the later loads cannot see stale values)
      if (!a.rec) prefetch_l2(a.x, uint32_t(a.K) * 4u);
      int issued = 0;
      const uint64_t stream_policy = l2_evict_first_policy();  // W is read once
      StageCursor cur{r0};
      for (int j = 0; cur.row < r1; ++j) {
        const int s = j % S;
        if (j >= S && !mbar_wait_bounded(&empty[s], uint32_t((j / S - 1) & 1), a.spin_limit)) {
          atomicOr(a.err, kErrTimeout);
          break;
        }
        int mat, nrows;
        cur.next(a, r1, mat, nrows);
        const uint32_t bytes = uint32_t(nrows) * uint32_t(a.row_bytes);
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s_hint(stage_base + size_t(s) * a.stage_bytes,
                      a.W[mat] + int64_t(cur.row - a.row_start[mat]) * a.row_bytes, bytes, &full[s],
                      stream_policy);
        cur.row += nrows;
        issued = j + 1;
      }
      // Never leave with a copy in flight: wait for the last use of each slot.
      for (int s = 0; s < min(S, issued); ++s) {
        const int last = s + S * ((issued - 1 - s) / S);
        if (!mbar_wait_bounded(&full[s], uint32_t((last / S) & 1), kDrainLimit))
          atomicOr(a.err, kErrTimeout);
      }
    }
  } else {
    // --------------------------------------------------------- consumers --
    // W is already streaming; x and y may belong to the previous kernel on
    // the stream, so wait for it to complete before touching them.
    pdl_wait();
    if (a.rec) {
      // x's records, ready in L2 (read past L1: written after this CTA
      // started); every CTA starts at a different offset to spread the
      // requests over L2
      const int n16 = a.groups * (kXRecBytes / 16);
      const int rot = int((blockIdx.x * 97u) % unsigned(n16));
      for (int i = threadIdx.x; i < n16; i += kConsumerWarps * 32) {
        const int k = i + rot < n16 ? i + rot : i + rot - n16;
        reinterpret_cast<uint4 *>(xrec)[k] = __ldcg(reinterpret_cast<const uint4 *>(a.rec) + k);
      }
    } else {
      quantize_x_records_2lane(a.x, a.K / kQK, xrec, threadIdx.x, kConsumerWarps * 32);
    }
    named_bar_sync(1, kConsumerWarps * 32);

    const int L = a.lanes_per_row;
    const int rr = lane / L;  // row (within the warp's pass) handled by this lane
    const int gl = lane % L;  // first group of that row handled by this lane
    StageCursor cur{r0};
    for (int j = 0; cur.row < r1; ++j) {
      const int s = j % S;
      // every warp consumes every stage in order, so a parity wait is never
      // more than one phase ahead of the barrier
      if (!mbar_wait_bounded(&full[s], uint32_t((j / S) & 1), a.spin_limit)) {
        atomicOr(a.err, kErrTimeout);
        break;
      }
      int mat, nrows;
      cur.next(a, r1, mat, nrows);
      float *yp = a.y[mat] + (cur.row - a.row_start[mat]);
      const uint8_t *stage = stage_base + size_t(s) * a.stage_bytes;
      for (int pr = warp * a.rows_per_warp; pr < nrows; pr += kConsumerWarps * a.rows_per_warp) {
        const int row = pr + rr;
        float acc = 0.0f;
        if (row < nrows) {
          const uint8_t *rowp = stage + size_t(row) * a.row_bytes;
          for (int g = gl; g < a.groups; g += L) {
            if constexpr (TYPE == kTypeQ6_K) {
              // 210-byte super-blocks: 2-byte aligned in the stage
              acc = q6k_group_terms(rowp + size_t(g) * Fmt<kTypeQ6_K>::kBytes, xrec + g * kXRecWords, acc);
            } else {
            uint32_t w[GW];
            const uint4 *src = reinterpret_cast<const uint4 *>(rowp + size_t(g) * GW * 4);
#pragma unroll
            for (int k = 0; k < GW / 4; ++k) {
              const uint4 u = src[k];
              w[4 * k] = u.x;
              w[4 * k + 1] = u.y;
              w[4 * k + 2] = u.z;
              w[4 * k + 3] = u.w;
            }
            acc = group_terms<TYPE>(w, xrec + g * kXRecWords, acc);
            }
          }
        }
        for (int off = L >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
        if (gl == 0 && row < nrows) yp[row] = acc;
      }
      cur.row += nrows;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------ prep kernel --

// Runs before k_gemv_tma in the same stream when a workspace is available:
//   1. with programmatic dependent launch, and weights of at most 64 MB,
//      asks L2 to fetch every weight byte of the launch (no dependency on
//      earlier kernels, so this overlaps the previous kernel and keeps HBM
//      busy through the launch boundary);
//   2. after the previous kernel completed, quantizes x once into records in
//      global memory (16 blocks per CTA, 8 lanes per block), which every GEMV
//      CTA then copies instead of quantizing x itself.
constexpr int kPrepThreads = 128;
constexpr int kPrepBlocksPerCta = kPrepThreads / 8;
constexpr uint32_t kPrepChunk = 64 * 1024;
constexpr int64_t kPrefetchMaxBytes = int64_t(64) << 20;  // about half of L2

struct PrepArgs {
  const uint8_t *W[kMaxMats];
  int64_t bytes[kMaxMats];            // weight bytes of matrix i
  int64_t chunk_start[kMaxMats + 1];  // first L2-prefetch chunk of matrix i
  int n_mats;
  const float *x;
  int nb;         // K / 32
  uint32_t *rec;  // groups * kXRecWords words
  int quant_ctas;
};

__global__ void __launch_bounds__(kPrepThreads) k_gemv_prep(const PrepArgs p) {
  if (threadIdx.x == 0) {
    // this CTA's part of x into L2 first: its load after the wait below is
    // then an L2 hit. A prefetch reads nothing into the SM, and L2 is where
    // the previous kernel's stores to x land, so it cannot expose stale data.
    if (int(blockIdx.x) < p.quant_ctas) {
      const int b0 = int(blockIdx.x) * kPrepBlocksPerCta;
      prefetch_l2(p.x + int64_t(b0) * kQK, uint32_t(min(kPrepBlocksPerCta, p.nb - b0)) * kQK * 4u);
    }
    for (int64_t c = blockIdx.x; c < p.chunk_start[p.n_mats]; c += gridDim.x) {
      int m = 0;
      while (c >= p.chunk_start[m + 1]) ++m;
      const int64_t off = (c - p.chunk_start[m]) * int64_t(kPrepChunk);
      prefetch_l2(p.W[m] + off, uint32_t(min(int64_t(kPrepChunk), p.bytes[m] - off)));
    }
  }
  pdl_launch_dependents();
  // x may be written by the previous kernel, which may also still read the
  // records of its own x: touch neither before it has completed
  pdl_wait();
  if (int(blockIdx.x) >= p.quant_ctas) return;  // whole CTA: the shuffles below stay converged
  quantize_x_records(p.x + int64_t(blockIdx.x) * kPrepBlocksPerCta * kQK,
                     min(kPrepBlocksPerCta, p.nb - int(blockIdx.x) * kPrepBlocksPerCta),
                     p.rec + blockIdx.x * (kPrepBlocksPerCta / 8) * kXRecWords, threadIdx.x, kPrepThreads, 0);
}

// ------------------------------------------------------ generic fallback --

// x quantized to Q8_0 once, for the generic kernel: words [8b + i], the
// scale (fp32) at [8nb + b], the code sum at [9nb + b]. One lane per block.
__device__ __forceinline__ void quantize_x_generic(const float *__restrict__ x, uint32_t *xs, int nb, int b) {
  float v[32];
  load_block<false>(x + b * kQK, v);
  uint16_t scale;
  uint32_t w[8];
  int sum;
  quantize_block_lane<kTypeQ8_0, true>(v, scale, w, sum);
#pragma unroll
  for (int i = 0; i < 8; ++i) xs[8 * b + i] = w[i];
  xs[8 * nb + b] = __float_as_uint(half_bits_to_float(scale));
  xs[9 * nb + b] = uint32_t(sum);
}

// x's records for k_gemv_generic / k_gemv_staged, 8 lanes per block (the
// same codes, scales and sums as quantize_x_generic: one block rule), 32
// blocks per CTA.
__global__ void __launch_bounds__(256) k_gemv_generic_prep(const float *__restrict__ x, uint32_t *__restrict__ xg,
                                                           int nb) {
  // k_gemv_staged, launched as a programmatic dependent, may start streaming
  // its rows now (it reads the records only after this launch completed)
  pdl_launch_dependents();
  const int b = int(blockIdx.x) * 32 + int(threadIdx.x >> 3), j = int(threadIdx.x & 7);
  if (int(blockIdx.x) * 32 >= nb) return;  // whole CTA: the shuffles below stay converged
  const float4 v = b < nb ? __ldg(reinterpret_cast<const float4 *>(x + int64_t(b) * kQK) + j)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
  uint16_t sc;
  uint32_t word;
  int sum;
  quantize_block_8lanes(v, sc, word, sum);
  if (b < nb) {
    xg[8 * b + j] = word;
    if (j == 0) {
      xg[8 * nb + b] = __float_as_uint(half_bits_to_float(sc));
      xg[9 * nb + b] = uint32_t(sum);
    }
  }
}

// Any K % 32 == 0: warp per row, lane per block (Q4_0 / Q8_0: aligned 32-bit
// loads, four blocks per lane in flight; the other types 2-byte loads). x's codes are
// stored unpadded (as quantize_x_generic writes them), in shared memory:
// quantized by the CTA itself, or copied from xg where a prep launch wrote
// them once for the whole grid.
template <int TYPE>
__global__ void __launch_bounds__(256)
    k_gemv_generic(const uint8_t *__restrict__ W, const float *__restrict__ x, const uint32_t *__restrict__ xg,
                   float *__restrict__ y, int M, int K) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  extern __shared__ __align__(16) uint32_t xs[];
  const int nb = K / kQK;
  if (xg) {
    for (int i = threadIdx.x; i < 10 * nb; i += blockDim.x) xs[i] = __ldg(xg + i);
  } else {
    for (int b = threadIdx.x; b < nb; b += blockDim.x) quantize_x_generic(x, xs, nb, b);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // k-quants: BB bytes per super-block of 8 x blocks
  const int64_t row_bytes = IsKQuant<TYPE>::kV ? int64_t(nb / 8) * BB : int64_t(nb) * BB;
  for (int64_t m = int64_t(blockIdx.x) * 8 + warp; m < M; m += int64_t(gridDim.x) * 8) {
    float acc = 0.0f;
    if constexpr (TYPE != kTypeQ4_0 && TYPE != kTypeQ8_0)
    for (int b = lane; b < nb; b += 32) {
      if constexpr (IsKQuant<TYPE>::kV) {
        // x block b meets sub-block(s) of super-block b / 8
        const uint8_t *sbp = W + m * row_bytes + int64_t(b >> 3) * BB;
        const int j = b & 7;
        const uint32_t *xw = xs + 8 * b;
        const float dx = __uint_as_float(xs[8 * nb + b]);
        const int xsum = int(xs[9 * nb + b]);
        if constexpr (TYPE == kTypeQ4_K) {
          const uint4 h = *reinterpret_cast<const uint4 *>(sbp);
          const float S = __fmul_rn(half_bits_to_float(h.x & 0xffffu), float(q4k_stream(h.y, h.z, h.w, j)));
          const float Mn = __fmul_rn(half_bits_to_float(h.x >> 16), float(q4k_stream(h.y, h.z, h.w, 8 + j)));
          const uint4 c = *reinterpret_cast<const uint4 *>(sbp + 16 + 16 * j);
          const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
          int su = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            su = dp4a_us(cw[i] & 0x0f0f0f0fu, xw[i], su);
            su = dp4a_us((cw[i] >> 4) & 0x0f0f0f0fu, xw[4 + i], su);
          }
          acc = __fmaf_rn(__fmul_rn(S, dx), float(su), acc);
          acc = __fmaf_rn(__fmul_rn(Mn, dx), float(-xsum), acc);
        } else {
          const uint16_t *b16 = reinterpret_cast<const uint16_t *>(sbp);  // 2-byte aligned
          const float d = half_bits_to_float(b16[104]);
          const int lo_off = (32 * j) & 127, hi_off = 128 + ((32 * j) & 63);
          const uint32_t lsh = j < 4 ? 0u : 4u, hsh = 2u * uint32_t(j >> 1);
          int su[2] = {0, 0}, sx[2] = {0, 0};
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            const uint32_t ql = uint32_t(b16[lo_off / 2 + 2 * w]) | (uint32_t(b16[lo_off / 2 + 2 * w + 1]) << 16);
            const uint32_t qh = uint32_t(b16[hi_off / 2 + 2 * w]) | (uint32_t(b16[hi_off / 2 + 2 * w + 1]) << 16);
            const uint32_t u = ((ql >> lsh) & 0x0f0f0f0fu) | (((qh >> hsh) & 0x03030303u) << 4);
            su[w >> 2] = dp4a_us(u, xw[w], su[w >> 2]);
            sx[w >> 2] = dp4a_ss(0x01010101u, xw[w], sx[w >> 2]);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float S = __fmul_rn(d, float(int8_t(sbp[192 + 2 * j + h])));
            acc = __fmaf_rn(__fmul_rn(S, dx), float(su[h] - 32 * sx[h]), acc);
          }
        }
        continue;
      }
      const uint16_t *blk = reinterpret_cast<const uint16_t *>(W + m * row_bytes + int64_t(b) * BB);
      if constexpr (Legacy<TYPE>::kIs) {
        // d_w d_x sum_j u_j qx_j (- 16 d_w d_x sum qx for Q5_0) + m_w d_x sum qx
        using L = Legacy<TYPE>;
        uint32_t qs[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qs[i] = uint32_t(blk[L::kQs / 2 + 2 * i]) | (uint32_t(blk[L::kQs / 2 + 2 * i + 1]) << 16);
        const uint32_t qh = L::kQh >= 0 ? (uint32_t(blk[L::kQh / 2]) | (uint32_t(blk[L::kQh / 2 + 1]) << 16)) : 0u;
        const int xsum = int(xs[9 * nb + b]);
        int sumi = legacy_sumu<TYPE>(qs, qh, xs + 8 * b);
        if (!L::kAffine) sumi -= 16 * xsum;
        const float dx = __uint_as_float(xs[8 * nb + b]);
        acc = __fmaf_rn(__fmul_rn(half_bits_to_float(blk[0]), dx), float(sumi), acc);
        if (L::kAffine) acc = __fmaf_rn(__fmul_rn(half_bits_to_float(blk[1]), dx), float(xsum), acc);
      }
    }
    if constexpr (TYPE == kTypeQ4_0 || TYPE == kTypeQ8_0) {
      // A block starts 2-byte aligned (BB = 2 mod 4): it is read as the
      // aligned 32-bit words that cover it, kQW + 1 of them, and realigned
      // with one clamped funnel shift per word. A block that starts on a
      // word ends half a word into its last one, which is then read with a
      // 16-bit load (nothing past the block is read). The lane's blocks are
      // taken kU at a time, all their loads issued before any is used.
      constexpr int kQW = (TYPE == kTypeQ4_0) ? 4 : 8;
      constexpr int kU = 4;
      const uint8_t *row = W + m * row_bytes;
      for (int b0 = lane; b0 < nb; b0 += 32 * kU) {
        uint32_t raw[kU][kQW + 1];
        uint32_t half[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int b = b0 + 32 * u;
          const uintptr_t a = reinterpret_cast<uintptr_t>(row + int64_t(b < nb ? b : 0) * BB);
          const uint32_t *wp = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
          half[u] = uint32_t(a & 2);
#pragma unroll
          for (int i = 0; i < kQW; ++i) raw[u][i] = b < nb ? __ldg(wp + i) : 0u;
          raw[u][kQW] = b >= nb ? 0u
                        : half[u] ? __ldg(wp + kQW)
                                  : uint32_t(__ldg(reinterpret_cast<const uint16_t *>(wp + kQW)));
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int b = b0 + 32 * u;
          if (b >= nb) break;
          // scale: bytes 0-1 of the block; codes: from byte 2
          const uint32_t sh = half[u] ? 32u : 16u;
          uint32_t q[kQW];
#pragma unroll
          for (int i = 0; i < kQW; ++i) q[i] = __funnelshift_rc(raw[u][i], raw[u][i + 1], sh);
          const uint32_t sbits = (half[u] ? (raw[u][0] >> 16) : raw[u][0]) & 0xffffu;
          const uint32_t *xw = xs + 8 * b;
          int sumi;
          if (TYPE == kTypeQ4_0)
            sumi = sumi_q4_q8(q, xw, int(xs[9 * nb + b]));
          else
            sumi = sumi_q8_q8(q, xw);
          const float s = __fmul_rn(half_bits_to_float(uint16_t(sbits)), __uint_as_float(xs[8 * nb + b]));
          acc = __fmaf_rn(s, float(sumi), acc);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
    if (lane == 0) y[m] = acc;
  }
}

// Rows that are not multiples of 16 bytes (K % 256 != 0) of Q4_0, Q8_0 and
// the legacy types: warp per row, the row staged in shared memory by 16-byte
// asynchronous copies of the aligned chunks that cover it (the matrix's last
// chunk copies only the matrix's bytes), two row buffers per warp: the next
// row's copies are in flight, holding no registers, while the current row's
// dot products run, lane per block (a Q4_0 / Q8_0 block read as the aligned
// 32-bit words that cover it and realigned with one clamped funnel shift per
// word, a legacy block by 16-bit shared loads). x's records (as
// quantize_x_generic writes them) come from the workspace, where a prep
// launch wrote them once: quantizing x in every CTA measured slower, and the
// one-lane-per-block quantizer would cost the row loop registers (at most 64
// here, for four or more CTAs per SM).
__device__ __forceinline__ void cp_async16_n(void *dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

// shared-memory bytes of one row buffer: the covering chunks and one word of
// slack (a lane's last word may reach 2 bytes past its block)
__host__ __device__ constexpr int staged_row_buf(int64_t row_bytes) { return int((row_bytes + 15 + 15) / 16 * 16 + 16); }
__host__ __device__ constexpr int staged_xs_bytes(int nb) { return (40 * nb + 15) / 16 * 16; }

template <int TYPE>
__global__ void __launch_bounds__(256, 4)
    k_gemv_staged(const uint8_t *__restrict__ W, const uint32_t *__restrict__ xg, float *__restrict__ y, int M,
                  int K) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  constexpr int kQW = (TYPE == kTypeQ4_0) ? 4 : 8;  // Q4_0 / Q8_0 code words (the legacy types: below)
  extern __shared__ __align__(16) uint32_t xs[];
  const int nb = K / kQK;
  const int64_t row_bytes = int64_t(nb) * BB;
  const int row_buf = staged_row_buf(row_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *buf0 = reinterpret_cast<uint8_t *>(xs) + staged_xs_bytes(nb) + size_t(warp) * 2 * row_buf;
  uint8_t *buf1 = buf0 + row_buf;
  const uint8_t *end = W + int64_t(M) * row_bytes;
  const int64_t stride = int64_t(gridDim.x) * 8;
  // row m's covering chunks into buf (one commit group, empty past the last row)
  auto issue = [&](int64_t m, uint8_t *buf) {
    if (m < M) {
      const uint8_t *a = W + m * row_bytes;
      const uint8_t *a16 = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(15));
      const int n16 = int((a + row_bytes - a16 + 15) / 16);
      for (int i = lane; i < n16; i += 32) {
        const uint8_t *src = a16 + 16 * i;
        const int64_t left = end - src;
        cp_async16_n(buf + 16 * i, src, left >= 16 ? 16 : int(left));
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  int64_t m = int64_t(blockIdx.x) * 8 + warp;
  // the first row's copies go out while the prep launch (a normal launch,
  // after all earlier work; it writes only the records) may still run
  issue(m, buf0);
  pdl_wait();
  // x's records, the code words transposed to [word][block] so that the
  // lanes' loads of consecutive blocks hit consecutive banks
  for (int i = threadIdx.x; i < 8 * nb; i += blockDim.x) xs[(i & 7) * nb + (i >> 3)] = __ldcg(xg + i);
  for (int i = 8 * nb + threadIdx.x; i < 10 * nb; i += blockDim.x) xs[i] = __ldcg(xg + i);
  __syncthreads();
  for (int k = 0; m < M; m += stride, k ^= 1) {
    const uint8_t *cur = k ? buf1 : buf0;
    issue(m + stride, k ? buf0 : buf1);
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncwarp();
    const int s16 = int(reinterpret_cast<uintptr_t>(W + m * row_bytes) & 15);
    float acc = 0.0f;
#pragma unroll 1
    for (int b = lane; b < nb; b += 32) {
      const int o = s16 + b * BB;  // 2-byte aligned
      if constexpr (Legacy<TYPE>::kIs) {
        // the legacy types' blocks by 16-bit shared loads (the same terms as
        // k_gemv_generic)
        using L = Legacy<TYPE>;
        const uint16_t *blk = reinterpret_cast<const uint16_t *>(cur + o);
        uint32_t qs[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qs[i] = uint32_t(blk[L::kQs / 2 + 2 * i]) | (uint32_t(blk[L::kQs / 2 + 2 * i + 1]) << 16);
        const uint32_t qh = L::kQh >= 0 ? (uint32_t(blk[L::kQh / 2]) | (uint32_t(blk[L::kQh / 2 + 1]) << 16)) : 0u;
        uint32_t xv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) xv[i] = xs[i * nb + b];
        const int xsum = int(xs[9 * nb + b]);
        int sumi = legacy_sumu<TYPE>(qs, qh, xv);
        if (!L::kAffine) sumi -= 16 * xsum;
        const float dx = __uint_as_float(xs[8 * nb + b]);
        acc = __fmaf_rn(__fmul_rn(half_bits_to_float(blk[0]), dx), float(sumi), acc);
        if (L::kAffine) acc = __fmaf_rn(__fmul_rn(half_bits_to_float(blk[1]), dx), float(xsum), acc);
        continue;
      }
      const uint32_t *wp = reinterpret_cast<const uint32_t *>(cur + (o & ~3));
      const uint32_t sh = (o & 2) ? 32u : 16u;
      uint32_t raw[kQW + 1];
#pragma unroll
      for (int i = 0; i <= kQW; ++i) raw[i] = wp[i];
      uint32_t q[kQW];
#pragma unroll
      for (int i = 0; i < kQW; ++i) q[i] = __funnelshift_rc(raw[i], raw[i + 1], sh);
      const uint32_t sbits = ((o & 2) ? (raw[0] >> 16) : raw[0]) & 0xffffu;
      uint32_t xw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) xw[i] = xs[i * nb + b];
      int sumi;
      if (TYPE == kTypeQ4_0)
        sumi = sumi_q4_q8(q, xw, int(xs[9 * nb + b]));
      else
        sumi = sumi_q8_q8(q, xw);
      const float sc = __fmul_rn(half_bits_to_float(uint16_t(sbits)), __uint_as_float(xs[8 * nb + b]));
      acc = __fmaf_rn(sc, float(sumi), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
    if (lane == 0) y[m] = acc;
    __syncwarp();  // every lane has read the buffer before the copies after next refill it
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy in flight at exit
}

int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

template <int TYPE>
cudaError_t launch_typed(int n, const uint8_t *const *W, float *const *y, const int64_t *M, const float *x,
                         int64_t K, uint32_t *rec_ws, cudaStream_t stream) {
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  constexpr int BB = Fmt<TYPE>::kBytes;
  const int nb = int(K / kQK);
  const int row_bytes = IsKQuant<TYPE>::kV ? (nb / 8) * BB : nb * BB;  // k-quants: BB per 8 x blocks
  int64_t M_total = 0;
  for (int i = 0; i < n; ++i) M_total += M[i];
  if (M_total == 0) return cudaSuccess;

  // Bulk copies need 16-byte aligned offsets and sizes: rows of every type are
  // whole multiples of 16 bytes for K % 256 == 0 except Q6_K's (210-byte
  // super-blocks, read 2-byte aligned by the consumers), whose stages then
  // hold whole quanta of rows (16 / gcd(row bytes, 16) rows), which every
  // matrix of the call must divide into.
  const int quantum = 16 / std::gcd(row_bytes, 16);
  bool quanta_ok = true;
  for (int i = 0; i < n; ++i) quanta_ok = quanta_ok && M[i] % quantum == 0;
  if (K % 256 == 0 && (quantum == 1 || (TYPE == kTypeQ6_K && quanta_ok))) {
    GemvArgs a{};
    int acc_rows = 0;
    a.n_mats = 0;
    for (int i = 0; i < n; ++i) {  // empty matrices are dropped from the batch
      if (M[i] == 0) continue;
      a.W[a.n_mats] = W[i];
      a.y[a.n_mats] = y[i];
      a.row_start[a.n_mats++] = acc_rows;
      acc_rows += int(M[i]);
    }
    for (int i = a.n_mats; i <= kMaxMats; ++i) a.row_start[i] = acc_rows;
    a.x = x;
    a.M = acc_rows;
    a.K = int(K);
    a.groups = nb / 8;
    a.lanes_per_row = min(32, next_pow2(a.groups));
    a.rows_per_warp = 32 / a.lanes_per_row;
    a.row_bytes = row_bytes;
    a.row_quantum = quantum;
    a.xrec_bytes = (a.groups * kXRecBytes + 127) / 128 * 128;
    a.err = di->err_word;
    a.spin_limit = spin_limit();
    a.rec = rec_ws;
    // Stages are large (one bulk copy of tens of KB): the copy engine's cost
    // is per copy, and small copies cap the stream far below HBM bandwidth.
    // A stage holds one pass of all consumer warps (8 x rows_per_warp rows),
    // cut to kMaxStageBytes for long rows.
    const int reserve = 1024;  // per-CTA system reservation
    const int half_sm = min(di->smem_per_sm / 2 - reserve, di->max_smem_optin);
    const int whole_sm = min(di->smem_per_sm - reserve, di->max_smem_optin);
    // tuning overrides, read from the environment once per process (a
    // lookup per call costs host time that a decode step of direct calls
    // cannot spare)
    static const int forced_rows = tuning_value("BQ_GEMV_STAGE_ROWS");
    static const int forced_stages = tuning_value("BQ_GEMV_STAGES");
    static const int forced_ctas = tuning_value("BQ_GEMV_CTAS_PER_SM");
    int stage_rows = forced_rows > 0 ? forced_rows : kConsumerWarps * a.rows_per_warp;
    stage_rows = min(stage_rows, max(1, kMaxStageBytes / row_bytes));
    stage_rows = int(std::min<int64_t>(stage_rows, a.M));
    stage_rows = std::max(quantum, stage_rows / quantum * quantum);
    a.stage_rows = stage_rows;
    a.stage_bytes = stage_rows * row_bytes;
    const int max_stages = forced_stages > 0 ? forced_stages : 4;
    auto ring = [&](int budget) {
      return min(max_stages, (budget - a.xrec_bytes - 16 * max_stages) / a.stage_bytes);
    };
    // Two CTAs per SM (16 consumer warps) when each fits in half an SM: the
    // consumers' shared-memory reads and dp4a work need that many warps to
    // keep up with the stream; rows too long for that take one CTA per SM.
    int ctas_per_sm = 2;
    int stages = ring(half_sm);
    if (stages < 2) {
      ctas_per_sm = 1;
      stages = ring(whole_sm);
    }
    // Launches beyond kPrefetchMaxBytes (no L2 prefetch; the ring alone keeps
    // HBM busy) stream faster with a third, slightly smaller stage where two
    // full ones leave the room (4-5% on a 203 MB launch at K = 4096; launches
    // of a decode chain, which wait on their predecessor, measured slower).
    if (forced_rows <= 0 && forced_stages <= 0 && ctas_per_sm == 2 && stages == 2 &&
        int64_t(a.M) * row_bytes > kPrefetchMaxBytes) {
      const int r3 = (half_sm - a.xrec_bytes - 16 * max_stages) / (3 * row_bytes) / quantum * quantum;
      if (r3 >= quantum && r3 >= stage_rows - 2 * quantum) {
        stage_rows = min(stage_rows - quantum, r3);
        a.stage_rows = stage_rows;
        a.stage_bytes = stage_rows * row_bytes;
        stages = 3;
      }
    }
    if (forced_ctas) ctas_per_sm = forced_ctas;
    if (stages >= 2) {
      a.stages = stages;
      const size_t smem = size_t(a.xrec_bytes) + size_t(stages) * a.stage_bytes + 2 * 8 * size_t(stages);
      cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_gemv_tma<TYPE>), int(smem));
      if (e != cudaSuccess) return e;
      // at least half a stage of rows per CTA, at most ctas_per_sm CTAs per SM
      const int64_t half_stage = std::max(1, stage_rows / 2);
      const int64_t grid = std::min((int64_t(a.M) + half_stage - 1) / half_stage,
                                    int64_t(di->sm_count) * ctas_per_sm);
      const bool pdl = weight_prefetch();
      a.rec = rec_ws;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      if (rec_ws) {
        PrepArgs p{};
        p.n_mats = a.n_mats;
        p.chunk_start[0] = 0;
        // The L2 prefetch pays only when it overlaps the previous kernel
        // (programmatic dependent launch) and the weights fit L2 beside the
        // stream of that kernel; otherwise it only competes with this
        // launch's own weight stream (measured: 14% slower decode steps
        // without dependent launch, 30% slower 200 MB launches).
        const bool l2_prefetch = pdl && int64_t(a.M) * row_bytes <= kPrefetchMaxBytes;
        for (int i = 0; i < a.n_mats; ++i) {
          p.W[i] = a.W[i];
          p.bytes[i] = int64_t(a.row_start[i + 1] - a.row_start[i]) * row_bytes;
          p.chunk_start[i + 1] = p.chunk_start[i] + (l2_prefetch ? (p.bytes[i] + kPrepChunk - 1) / kPrepChunk : 0);
        }
        for (int i = a.n_mats; i < kMaxMats; ++i) p.chunk_start[i + 1] = p.chunk_start[i];
        p.x = x;
        p.nb = nb;
        p.rec = rec_ws;
        p.quant_ctas = (nb + kPrepBlocksPerCta - 1) / kPrepBlocksPerCta;
        const int64_t pgrid =
            std::max<int64_t>(p.quant_ctas, std::min<int64_t>(di->sm_count, p.chunk_start[a.n_mats]));
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3(unsigned(pgrid));
        pc.blockDim = dim3(kPrepThreads);
        pc.stream = stream;
        pc.attrs = attr;
        pc.numAttrs = pdl ? 1 : 0;
        e = cudaLaunchKernelEx(&pc, k_gemv_prep, p);
        if (e != cudaSuccess) return e;
      }
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(unsigned(grid));
      cfg.blockDim = dim3(kGemvThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cfg.attrs = attr;
      cfg.numAttrs = pdl ? 1 : 0;
      return cudaLaunchKernelEx(&cfg, k_gemv_tma<TYPE>, a);
    }
  }
  // any K % 32 == 0 (or rows too long for two stages): one plain launch per
  // matrix; with a workspace, x is quantized once by a prep launch
  const size_t smem = size_t(nb) * 40;  // 32 code bytes + scale + sum per block
  cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_gemv_generic<TYPE>), int(smem));
  if (e != cudaSuccess) return e;
  const uint32_t *xg = nullptr;
  if (rec_ws) {
    k_gemv_generic_prep<<<unsigned((nb + 31) / 32), 256, 0, stream>>>(x, rec_ws, nb);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    xg = rec_ws;
  }
  // Q4_0, Q8_0 and the legacy types with x's records in the workspace: rows
  // staged in shared memory when two row buffers per warp fit
  const size_t staged_smem = size_t(staged_xs_bytes(int(nb))) + size_t(16) * staged_row_buf(nb * BB);
  constexpr bool kStagedType = !IsKQuant<TYPE>::kV;
  const bool staged = kStagedType && xg && staged_smem <= size_t(di->max_smem_optin);
  const void *fn = reinterpret_cast<const void *>(k_gemv_generic<TYPE>);
  if constexpr (kStagedType)
    if (staged) fn = reinterpret_cast<const void *>(k_gemv_staged<TYPE>);
  const size_t fsmem = staged ? staged_smem : smem;
  if (staged && (e = ensure_smem(fn, int(fsmem))) != cudaSuccess) return e;
  // one wave of CTAs (8 rows each in flight), as many per SM as are resident
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 256, fsmem)) != cudaSuccess) return e;
  per_sm = std::max(per_sm, 1);
  for (int i = 0; i < n; ++i) {
    if (M[i] == 0) continue;
    const int64_t grid = std::min((M[i] + 7) / 8, int64_t(di->sm_count) * per_sm);
    if constexpr (kStagedType)
      if (staged) {
        // a programmatic dependent of the prep launch (for i > 0, of the
        // previous matrix's launch, whose completion implies the prep's)
        cudaLaunchAttribute sattr[1];
        sattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        sattr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t sc = {};
        sc.gridDim = dim3(unsigned(grid));
        sc.blockDim = dim3(256);
        sc.dynamicSmemBytes = fsmem;
        sc.stream = stream;
        sc.attrs = sattr;
        sc.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&sc, k_gemv_staged<TYPE>, static_cast<const uint8_t *>(W[i]),
                                    static_cast<const uint32_t *>(xg), y[i], int(M[i]), int(K))) != cudaSuccess)
          return e;
        continue;
      }
    k_gemv_generic<TYPE><<<unsigned(grid), 256, smem, stream>>>(W[i], x, xg, y[i], int(M[i]), int(K));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}


}  // namespace

cudaError_t launch_gemv(int type, int n, const uint8_t *const *W, float *const *y, const int64_t *M,
                        const float *x, int64_t K, uint32_t *rec_ws, cudaStream_t stream) {
  if (type == kTypeQ4_K) return launch_typed<kTypeQ4_K>(n, W, y, M, x, K, rec_ws, stream);
  if (type == kTypeQ6_K) return launch_typed<kTypeQ6_K>(n, W, y, M, x, K, rec_ws, stream);
  if (type == kTypeQ4_1) return launch_typed<kTypeQ4_1>(n, W, y, M, x, K, rec_ws, stream);
  if (type == kTypeQ5_0) return launch_typed<kTypeQ5_0>(n, W, y, M, x, K, rec_ws, stream);
  if (type == kTypeQ5_1) return launch_typed<kTypeQ5_1>(n, W, y, M, x, K, rec_ws, stream);
  if (type == kTypeQ4_0) return launch_typed<kTypeQ4_0>(n, W, y, M, x, K, rec_ws, stream);
  return launch_typed<kTypeQ8_0>(n, W, y, M, x, K, rec_ws, stream);
}

size_t gemv_workspace_bytes(int64_t K) {
  if (K <= 0 || K % kQK) return 0;
  // the records of the bulk-copy kernel (K % 256 == 0), which also hold the
  // generic kernel's 40 bytes per block; else the generic layout alone
  const size_t bytes = K % 256 == 0 ? size_t(K / 256) * kXRecBytes : size_t(K / kQK) * 40;
  return (bytes + 255) / 256 * 256;
}

// ------------------------------------------------------------ block dots --

namespace {
template <int TYPE>
__global__ void __launch_bounds__(256)
    k_block_dots(const uint8_t *__restrict__ W, const uint8_t *__restrict__ xq,
                 int32_t *__restrict__ out, int64_t M, int nb) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  constexpr int kQW = (TYPE == kTypeQ4_0) ? 4 : 8;
  const int64_t total = M * nb;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int b = int(i % nb);
    const uint16_t *wb = reinterpret_cast<const uint16_t *>(W + i * BB);
    const uint16_t *xb = reinterpret_cast<const uint16_t *>(xq + int64_t(b) * Fmt<kTypeQ8_0>::kBytes);
    uint32_t q[kQW], xw[8];
#pragma unroll
    for (int k = 0; k < kQW; ++k) q[k] = uint32_t(wb[1 + 2 * k]) | (uint32_t(wb[2 + 2 * k]) << 16);
    int xsum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      xw[k] = uint32_t(xb[1 + 2 * k]) | (uint32_t(xb[2 + 2 * k]) << 16);
      xsum = dp4a_ss(xw[k], 0x01010101u, xsum);
    }
    out[i] = (TYPE == kTypeQ4_0) ? sumi_q4_q8(q, xw, xsum) : sumi_q8_q8(q, xw);
  }
}
}  // namespace

cudaError_t launch_block_dots(int type, const uint8_t *W, const uint8_t *xq, int32_t *out, int64_t M,
                              int64_t K, cudaStream_t stream) {
  if (M == 0 || K == 0) return cudaSuccess;
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  const int nb = int(K / kQK);
  const int64_t grid = min((M * nb + 255) / 256, int64_t(di->sm_count) * 8);
  if (type == kTypeQ4_0)
    k_block_dots<kTypeQ4_0><<<unsigned(grid), 256, 0, stream>>>(W, xq, out, M, nb);
  else
    k_block_dots<kTypeQ8_0><<<unsigned(grid), 256, 0, stream>>>(W, xq, out, M, nb);
  return cudaGetLastError();
}

}  // namespace bq
