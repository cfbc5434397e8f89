// gemv.cu — decode GEMV over block-quantized weights: y = W . x for one token.
//
// Decode reads every weight once per token, so its speed is bounded by
// memory bandwidth divided by the weight bytes ("05. llama.cpp：从 GGUF 文件到
// 本地推理服务", §性能直觉：带宽决定 Decode，算力决定 Prefill). The kernel is
// therefore built to stream W from HBM at full rate:
//
//   - x (fp32) is quantized to Q8_0 by each CTA into shared memory (same block
//     rule as the row quantizer, so the codes are bit-identical), while the
//     weight stream is already in flight. No workspace, no extra launch.
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
#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kXRecWords = 84;          // per group of 8 blocks: 64 code words, 8 scales, 8 sums, 4 pad
constexpr int kXRecBytes = kXRecWords * 4;
constexpr uint32_t kDrainLimit = 1u << 26;

struct GemvArgs {
  const uint8_t *W;
  const float *x;
  float *y;
  int M;
  int K;
  int groups;          // K / 256
  int lanes_per_row;   // power of two <= 32
  int rows_per_task;   // 32 / lanes_per_row
  int row_bytes;
  int n_tasks;         // ceil(M / rows_per_task)
  int stages;
  int stage_bytes;     // rows_per_task * row_bytes
  int xrec_bytes;      // groups * kXRecBytes rounded up to 128
  unsigned *err;
  uint32_t spin_limit;
};

// Quantize x (K fp32, 16-byte aligned) into the per-group records:
// word [g*84 + 8*jb + i] = codes 4i..4i+3 of block 8g+jb, [g*84 + 64 + jb] =
// fp32 scale, [g*84 + 72 + jb] = code sum. Called by `nthreads` threads.
__device__ __forceinline__ void quantize_x_records(const float *__restrict__ x, int nb,
                                                   uint32_t *rec, int tid, int nthreads) {
  const int j = tid & 7;
  for (int b0 = tid >> 3; b0 - (tid >> 3) < nb; b0 += nthreads >> 3) {
    const int b = b0;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (b < nb) v = __ldg(reinterpret_cast<const float4 *>(x + b * kQK + j * 4));
    const BlockCodes<kTypeQ8_0> c = quantize_block8<kTypeQ8_0>(v);
    if (b < nb) {
      uint32_t *r = rec + (b >> 3) * kXRecWords;
      const int jb = b & 7;
      r[8 * jb + j] = c.bytes4;
      if (j == 0) {
        r[64 + jb] = __float_as_uint(half_bits_to_float(c.scale));
        r[72 + jb] = uint32_t(c.sum);
      }
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

// Sum of the 8 block terms of one group. w: the group's bytes as words (the
// group starts 16-byte aligned, block jb starts at byte BB*jb).
template <int TYPE>
__device__ __forceinline__ float group_terms(const uint32_t *w, const uint32_t *xr, float acc) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  const uint4 dx0 = *reinterpret_cast<const uint4 *>(xr + 64);
  const uint4 dx1 = *reinterpret_cast<const uint4 *>(xr + 68);
  const uint32_t dxs[8] = {dx0.x, dx0.y, dx0.z, dx0.w, dx1.x, dx1.y, dx1.z, dx1.w};
  uint32_t sxs[8];
  if (TYPE == kTypeQ4_0) {
    const uint4 s0 = *reinterpret_cast<const uint4 *>(xr + 72);
    const uint4 s1 = *reinterpret_cast<const uint4 *>(xr + 76);
    sxs[0] = s0.x; sxs[1] = s0.y; sxs[2] = s0.z; sxs[3] = s0.w;
    sxs[4] = s1.x; sxs[5] = s1.y; sxs[6] = s1.z; sxs[7] = s1.w;
  }
#pragma unroll
  for (int jb = 0; jb < 8; ++jb) {
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
  return acc;
}

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
  const int t0 = int(int64_t(a.n_tasks) * blockIdx.x / gridDim.x);
  const int t1 = int(int64_t(a.n_tasks) * (blockIdx.x + 1) / gridDim.x);
  const int ntask = t1 - t0;
  const int S = a.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < ntask; ++i) {
        const int s = i % S;
        if (i >= S && !mbar_wait_bounded(&empty[s], uint32_t((i / S - 1) & 1), a.spin_limit)) {
          atomicOr(a.err, kErrTimeout);
          break;
        }
        const int row0 = (t0 + i) * a.rows_per_task;
        const int nrows = min(a.rows_per_task, a.M - row0);
        const uint32_t bytes = uint32_t(nrows) * uint32_t(a.row_bytes);
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(stage_base + size_t(s) * a.stage_bytes, a.W + int64_t(row0) * a.row_bytes, bytes,
                 &full[s]);
        issued = i + 1;
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
    quantize_x_records(a.x, a.K / kQK, xrec, threadIdx.x, kConsumerWarps * 32);
    named_bar_sync(1, kConsumerWarps * 32);

    const int L = a.lanes_per_row;
    const int rr = lane / L;  // row of the task handled by this lane
    const int gl = lane % L;  // first group of that row handled by this lane
    for (int i = warp; i < ntask; i += kConsumerWarps) {
      const int s = i % S;
      if (!mbar_wait_bounded(&full[s], uint32_t((i / S) & 1), a.spin_limit)) {
        atomicOr(a.err, kErrTimeout);
        break;
      }
      const int row0 = (t0 + i) * a.rows_per_task;
      const int nrows = min(a.rows_per_task, a.M - row0);
      float acc = 0.0f;
      if (rr < nrows) {
        const uint8_t *row = stage_base + size_t(s) * a.stage_bytes + size_t(rr) * a.row_bytes;
        for (int g = gl; g < a.groups; g += L) {
          uint32_t w[GW];
          const uint4 *src = reinterpret_cast<const uint4 *>(row + size_t(g) * GW * 4);
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
      for (int off = L >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
      if (gl == 0 && rr < nrows) a.y[row0 + rr] = acc;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();
}

// ------------------------------------------------------ generic fallback --

// Any K % 32 == 0: warp per row, lane per block, 2-byte loads. x's codes are
// stored unpadded: word [8b + i], scales at [8nb + b], sums at [9nb + b].
template <int TYPE>
__global__ void __launch_bounds__(256)
    k_gemv_generic(const uint8_t *__restrict__ W, const float *__restrict__ x,
                   float *__restrict__ y, int M, int K) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  extern __shared__ __align__(16) uint32_t xs[];
  const int nb = K / kQK;
  {
    const int j = threadIdx.x & 7;
    for (int b0 = threadIdx.x >> 3; b0 - int(threadIdx.x >> 3) < nb; b0 += 32) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (b0 < nb) v = __ldg(reinterpret_cast<const float4 *>(x + b0 * kQK + j * 4));
      const BlockCodes<kTypeQ8_0> c = quantize_block8<kTypeQ8_0>(v);
      if (b0 < nb) {
        xs[8 * b0 + j] = c.bytes4;
        if (j == 0) {
          xs[8 * nb + b0] = __float_as_uint(half_bits_to_float(c.scale));
          xs[9 * nb + b0] = uint32_t(c.sum);
        }
      }
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row_bytes = int64_t(nb) * BB;
  for (int64_t m = int64_t(blockIdx.x) * 8 + warp; m < M; m += int64_t(gridDim.x) * 8) {
    float acc = 0.0f;
    for (int b = lane; b < nb; b += 32) {
      const uint16_t *blk = reinterpret_cast<const uint16_t *>(W + m * row_bytes + int64_t(b) * BB);
      constexpr int kQW = (TYPE == kTypeQ4_0) ? 4 : 8;
      uint32_t q[kQW];
#pragma unroll
      for (int i = 0; i < kQW; ++i) q[i] = uint32_t(blk[1 + 2 * i]) | (uint32_t(blk[2 + 2 * i]) << 16);
      const uint32_t *xw = xs + 8 * b;
      int sumi;
      if (TYPE == kTypeQ4_0)
        sumi = sumi_q4_q8(q, xw, int(xs[9 * nb + b]));
      else
        sumi = sumi_q8_q8(q, xw);
      const float s = __fmul_rn(half_bits_to_float(blk[0]), __uint_as_float(xs[8 * nb + b]));
      acc = __fmaf_rn(s, float(sumi), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
    if (lane == 0) y[m] = acc;
  }
}

int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

template <int TYPE>
cudaError_t launch_typed(const uint8_t *W, const float *x, float *y, int64_t M, int64_t K,
                         cudaStream_t stream) {
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  constexpr int BB = Fmt<TYPE>::kBytes;
  const int nb = int(K / kQK);
  const int row_bytes = nb * BB;

  if (K % 256 == 0) {
    GemvArgs a{};
    a.W = W;
    a.x = x;
    a.y = y;
    a.M = int(M);
    a.K = int(K);
    a.groups = nb / 8;
    a.lanes_per_row = min(32, next_pow2(a.groups));
    a.rows_per_task = 32 / a.lanes_per_row;
    a.row_bytes = row_bytes;
    a.n_tasks = int((M + a.rows_per_task - 1) / a.rows_per_task);
    a.stage_bytes = a.rows_per_task * row_bytes;
    a.xrec_bytes = (a.groups * kXRecBytes + 127) / 128 * 128;
    a.err = di->err_word;
    a.spin_limit = spin_limit();
    // The ring holds a multiple of kConsumerWarps stages: consumer warp w
    // takes tasks w, w+8, ..., so the previous user of its slot is itself and
    // a parity wait can never be two phases ahead of the barrier.
    // Two CTAs per SM when the ring gets >= 16 stages, else one CTA.
    const int reserve = 1024;  // per-CTA system reservation
    const int per_cta2 = min(di->smem_per_sm / 2 - reserve, di->max_smem_optin);
    const int per_cta1 = min(di->smem_per_sm - reserve, di->max_smem_optin);
    auto ring = [&](int budget) {
      const int s = (budget - a.xrec_bytes - 16 * 32) / a.stage_bytes;
      return min(s, 32) / kConsumerWarps * kConsumerWarps;
    };
    int ctas_per_sm = 2;
    int stages = ring(per_cta2);
    if (stages < 2 * kConsumerWarps) {
      ctas_per_sm = 1;
      stages = ring(per_cta1);
    }
    if (stages >= kConsumerWarps) {
      a.stages = stages;
      const size_t smem = size_t(a.xrec_bytes) + size_t(stages) * a.stage_bytes + 2 * 8 * size_t(stages);
      cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_gemv_tma<TYPE>), int(smem));
      if (e != cudaSuccess) return e;
      const int64_t grid = min(int64_t(a.n_tasks), int64_t(di->sm_count) * ctas_per_sm);
      k_gemv_tma<TYPE><<<unsigned(grid), kGemvThreads, smem, stream>>>(a);
      return cudaGetLastError();
    }
  }
  const size_t smem = size_t(nb) * 40;  // 32 code bytes + scale + sum per block
  cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_gemv_generic<TYPE>), int(smem));
  if (e != cudaSuccess) return e;
  const int64_t grid = min((M + 7) / 8, int64_t(di->sm_count) * 4);
  k_gemv_generic<TYPE><<<unsigned(grid), 256, smem, stream>>>(W, x, y, int(M), int(K));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(int type, const uint8_t *W, const float *x, float *y, int64_t M, int64_t K,
                        cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  if (type == kTypeQ4_0) return launch_typed<kTypeQ4_0>(W, x, y, M, K, stream);
  return launch_typed<kTypeQ8_0>(W, x, y, M, K, stream);
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
