// quantize.cu — row quantization (Q4_0 / Q8_0), the KV-cache write with an
// optional mean-centering bias, and dequantization.
//
// Row quantize: every 32 consecutive values of a row form one block with one
// binary16 scale ("llama.cpp 原理：如何在普通硬件跑本地大模型", §量化：内存真正去哪了;
// "05. llama.cpp：从 GGUF 文件到本地推理服务", §量化类型). KV write: K is written
// to the cache quantized, optionally after subtracting a calibrated
// per-(kv-head, channel) bias (lpnh.cn KV-cache article, §解法).
//
// Design (HBM-bound: 128 B of fp32 read per 18 or 34 B written):
//   - a CTA owns tiles of 256 consecutive blocks (32 KB of fp32 input);
//   - 8 lanes per block, one float4 each, so every warp load instruction
//     reads 512 contiguous bytes; each thread keeps 8 loads in flight;
//   - the block's amax is a 3-step shuffle max inside the 8-lane group;
//   - codes are packed to the block layout in shared memory, and the tile's
//     4.5 KB (Q4_0) / 8.5 KB (Q8_0) of output leaves as 16-byte stores.
#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kTileBlocks = 256;  // blocks per CTA tile; 8 warps x 8 rounds x 4 blocks

template <int TYPE, bool BIAS>
__global__ void __launch_bounds__(kQuantThreads)
    k_quantize_rows(const float *__restrict__ src, uint8_t *__restrict__ dst, int64_t n_blocks,
                    const float *__restrict__ bias, int64_t bias_period) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  __shared__ __align__(16) uint8_t tile_out[kTileBlocks * BB];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int sub = lane >> 3;  // block of the 4-block round handled by this 8-lane group
  const int j = lane & 7;     // float4 of the block held by this lane

  for (int64_t tile0 = int64_t(blockIdx.x) * kTileBlocks; tile0 < n_blocks;
       tile0 += int64_t(gridDim.x) * kTileBlocks) {
    const int tile_n = int(min(int64_t(kTileBlocks), n_blocks - tile0));

    float4 v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int tb = warp * 32 + r * 4 + sub;
      v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tb < tile_n) v[r] = ld_stream_f4(src + (tile0 + tb) * kQK + j * 4);
    }
    if (BIAS) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int tb = warp * 32 + r * 4 + sub;
        if (tb < tile_n) {
          // block g of row (token, head) uses bias block g mod (heads * blocks per row)
          const int64_t bblk = (tile0 + tb) % bias_period;
          const float4 b = __ldg(reinterpret_cast<const float4 *>(bias + bblk * kQK + j * 4));
          v[r].x = __fsub_rn(v[r].x, b.x);
          v[r].y = __fsub_rn(v[r].y, b.y);
          v[r].z = __fsub_rn(v[r].z, b.z);
          v[r].w = __fsub_rn(v[r].w, b.w);
        }
      }
    }

#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int tb = warp * 32 + r * 4 + sub;
      const BlockCodes<TYPE> c = quantize_block8<TYPE>(v[r]);
      uint8_t *blk = tile_out + tb * BB;
      uint32_t word = c.bytes4;
      if (TYPE == kTypeQ4_0) word = pack_q4_nibbles(c.bytes4);
      if (tb < tile_n) {
        if (j == 0) *reinterpret_cast<uint16_t *>(blk) = c.scale;
        if (TYPE == kTypeQ8_0 || j < 4) {
          // qs bytes 4j..4j+3 live at block offset 2 + 4j: 2-byte aligned
          uint16_t *q = reinterpret_cast<uint16_t *>(blk + 2 + 4 * j);
          q[0] = uint16_t(word & 0xffffu);
          q[1] = uint16_t(word >> 16);
        }
      }
    }
    __syncthreads();

    uint8_t *out = dst + tile0 * BB;  // 16-byte aligned: tile0 is a multiple of 256
    const int nbytes = tile_n * BB;
    const int n16 = nbytes / 16;
    for (int i = threadIdx.x; i < n16; i += kQuantThreads)
      reinterpret_cast<uint4 *>(out)[i] = reinterpret_cast<const uint4 *>(tile_out)[i];
    for (int i = n16 * 8 + threadIdx.x; i < nbytes / 2; i += kQuantThreads)
      reinterpret_cast<uint16_t *>(out)[i] = reinterpret_cast<const uint16_t *>(tile_out)[i];
    __syncthreads();
  }
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

template <int TYPE, bool BIAS>
cudaError_t launch_q(const float *src, uint8_t *dst, int64_t n_blocks, const float *bias,
                     int64_t bias_period, cudaStream_t stream) {
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  const int64_t tiles = (n_blocks + kTileBlocks - 1) / kTileBlocks;
  const int64_t grid = min(tiles, int64_t(di->sm_count) * 8);
  k_quantize_rows<TYPE, BIAS><<<unsigned(grid), kQuantThreads, 0, stream>>>(src, dst, n_blocks, bias,
                                                                           bias_period);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_rows(int type, const float *src, uint8_t *dst, int64_t n_blocks,
                                 int64_t /*blocks_per_row*/, const float *bias, int64_t bias_period,
                                 cudaStream_t stream) {
  if (n_blocks == 0) return cudaSuccess;
  if (type == kTypeQ4_0)
    return bias ? launch_q<kTypeQ4_0, true>(src, dst, n_blocks, bias, bias_period, stream)
                : launch_q<kTypeQ4_0, false>(src, dst, n_blocks, nullptr, 1, stream);
  // a bias with Q8_0 is rejected by the ABI layer
  return launch_q<kTypeQ8_0, false>(src, dst, n_blocks, nullptr, 1, stream);
}

cudaError_t launch_dequantize_rows(int type, const uint8_t *blocks, float *dst, int64_t n_blocks,
                                   cudaStream_t stream) {
  if (n_blocks == 0) return cudaSuccess;
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  const int64_t grid = min((n_blocks * 8 + 255) / 256, int64_t(di->sm_count) * 8);
  if (type == kTypeQ4_0)
    k_dequantize_rows<kTypeQ4_0><<<unsigned(grid), 256, 0, stream>>>(blocks, dst, n_blocks);
  else
    k_dequantize_rows<kTypeQ8_0><<<unsigned(grid), 256, 0, stream>>>(blocks, dst, n_blocks);
  return cudaGetLastError();
}

}  // namespace bq
