// gemm.cu — prefill GEMM over Q8_0 weights: Y = X . W^T for N tokens.
//
// Prefill processes many tokens per weight read, so it is compute-bound
// ("05. llama.cpp：从 GGUF 文件到本地推理服务", §性能直觉：带宽决定 Decode，
// 算力决定 Prefill). X is first quantized to Q8_0 (into the workspace) by the
// row quantizer; the contraction then runs per 32-deep block on integer
// tensor-core MMAs.
//
// This translation unit holds the mma.sync (m16n8k32 s8) kernel: one MMA k-step
// is exactly one block, so each MMA yields one block's exact int32 dot, which
// is scaled by scale_w * scale_x (exact in fp32) and accumulated in fp32
// (partials over 16 blocks, then a running sum). Tiles: 128 weight rows x 64
// tokens per CTA, 8 blocks per stage, double-buffered cp.async copies of the
// raw 34-byte blocks; fragments are cut from the raw block bytes in shared
// memory (row pitch 272 B keeps the 32 lanes on 32 distinct banks).
#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {
namespace {

constexpr int kBM = 128;  // weight rows per CTA
constexpr int kBN = 64;   // tokens per CTA
constexpr int kKB = 8;    // blocks per stage
constexpr int kPitch = kKB * Fmt<kTypeQ8_0>::kBytes;  // 272 bytes per row per stage
constexpr int kStageA = kBM * kPitch;
constexpr int kStageB = kBN * kPitch;
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kGemmThreads = 256;

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 4 code bytes at byte offset `off` of shared memory, off % 2 == 0
template <bool ALIGNED4>
__device__ __forceinline__ uint32_t lds_codes(const uint8_t *base, int off) {
  if (ALIGNED4) return *reinterpret_cast<const uint32_t *>(base + off);
  const uint32_t *w = reinterpret_cast<const uint32_t *>(base + off - 2);
  return __funnelshift_r(w[0], w[1], 16);
}

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(0), "r"(0), "r"(0),
        "r"(0));
}

template <int JB>
__device__ __forceinline__ void block_step(const uint8_t *sA, const uint8_t *sB, int wm, int wn, int g,
                                           int t, float (&part)[2][4][4]) {
  constexpr int kOff = JB * Fmt<kTypeQ8_0>::kBytes;  // block start within the row slice
  constexpr bool kAl = ((kOff + 2) & 3) == 0;          // are its codes word aligned?
  uint32_t a[2][4], b[4][2];
  float dw[2][2], dx[4][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = (wm * 32 + mt * 16 + g) * kPitch + kOff;
    const int r1 = r0 + 8 * kPitch;
    a[mt][0] = lds_codes<kAl>(sA, r0 + 2 + 4 * t);
    a[mt][1] = lds_codes<kAl>(sA, r1 + 2 + 4 * t);
    a[mt][2] = lds_codes<kAl>(sA, r0 + 18 + 4 * t);
    a[mt][3] = lds_codes<kAl>(sA, r1 + 18 + 4 * t);
    dw[mt][0] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sA + r0));
    dw[mt][1] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sA + r1));
  }
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int c0 = (wn * 32 + nt * 8 + g) * kPitch + kOff;
    b[nt][0] = lds_codes<kAl>(sB, c0 + 2 + 4 * t);
    b[nt][1] = lds_codes<kAl>(sB, c0 + 18 + 4 * t);
    const int s0 = (wn * 32 + nt * 8 + 2 * t) * kPitch + kOff;
    dx[nt][0] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sB + s0));
    dx[nt][1] = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sB + s0 + kPitch));
  }
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      int c[4];
      mma_s8(c, a[mt], b[nt]);
      part[mt][nt][0] = __fmaf_rn(float(c[0]), __fmul_rn(dw[mt][0], dx[nt][0]), part[mt][nt][0]);
      part[mt][nt][1] = __fmaf_rn(float(c[1]), __fmul_rn(dw[mt][0], dx[nt][1]), part[mt][nt][1]);
      part[mt][nt][2] = __fmaf_rn(float(c[2]), __fmul_rn(dw[mt][1], dx[nt][0]), part[mt][nt][2]);
      part[mt][nt][3] = __fmaf_rn(float(c[3]), __fmul_rn(dw[mt][1], dx[nt][1]), part[mt][nt][3]);
    }
}

__global__ void __launch_bounds__(kGemmThreads, 2)
    k_gemm_q8_mma(const uint8_t *__restrict__ W, const uint8_t *__restrict__ Xq, float *__restrict__ Y,
                  int M, int N, int nb) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp & 3, wn = warp >> 2;
  const int g = lane >> 2, t = lane & 3;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
  const int64_t row_bytes = int64_t(nb) * Fmt<kTypeQ8_0>::kBytes;
  const int nchunks = nb / kKB;

  auto load_chunk = [&](int kc, int stage) {
    uint8_t *sA = smem + stage * kStageBytes;
    uint8_t *sB = sA + kStageA;
    constexpr int kPieces = kPitch / 16;  // 17
    for (int p = threadIdx.x; p < (kBM + kBN) * kPieces; p += kGemmThreads) {
      const int r = p / kPieces, piece = p % kPieces;
      if (r < kBM) {
        const int m = m0 + r;
        const bool ok = m < M;
        const uint8_t *src = W + (ok ? int64_t(m) * row_bytes + int64_t(kc) * kPitch + piece * 16 : 0);
        cp_async16(sA + r * kPitch + piece * 16, src, ok);
      } else {
        const int n = n0 + (r - kBM);
        const bool ok = n < N;
        const uint8_t *src = Xq + (ok ? int64_t(n) * row_bytes + int64_t(kc) * kPitch + piece * 16 : 0);
        cp_async16(sB + (r - kBM) * kPitch + piece * 16, src, ok);
      }
    }
    cp_async_commit();
  };

  float acc[2][4][4], part[2][4][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][nt][i] = part[mt][nt][i] = 0.0f;

  load_chunk(0, 0);
  for (int kc = 0; kc < nchunks; ++kc) {
    if (kc + 1 < nchunks) {
      load_chunk(kc + 1, (kc + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint8_t *sA = smem + (kc & 1) * kStageBytes;
    const uint8_t *sB = sA + kStageA;
    block_step<0>(sA, sB, wm, wn, g, t, part);
    block_step<1>(sA, sB, wm, wn, g, t, part);
    block_step<2>(sA, sB, wm, wn, g, t, part);
    block_step<3>(sA, sB, wm, wn, g, t, part);
    block_step<4>(sA, sB, wm, wn, g, t, part);
    block_step<5>(sA, sB, wm, wn, g, t, part);
    block_step<6>(sA, sB, wm, wn, g, t, part);
    block_step<7>(sA, sB, wm, wn, g, t, part);
    if ((kc & 1) || kc + 1 == nchunks) {  // fold every 16 blocks
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[mt][nt][i] += part[mt][nt][i];
            part[mt][nt][i] = 0.0f;
          }
    }
    __syncthreads();
  }

#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = m0 + wm * 32 + mt * 16 + g + ((i & 2) ? 8 : 0);
        const int n = n0 + wn * 32 + nt * 8 + 2 * t + (i & 1);
        if (m < M && n < N) Y[int64_t(n) * M + m] = acc[mt][nt][i];
      }
}

// Any K % 32 == 0: one thread per output, 2-byte loads (small or ragged shapes).
__global__ void __launch_bounds__(256)
    k_gemm_q8_generic(const uint8_t *__restrict__ W, const uint8_t *__restrict__ Xq,
                      float *__restrict__ Y, int64_t M, int64_t N, int nb) {
  constexpr int BB = Fmt<kTypeQ8_0>::kBytes;
  const int64_t total = M * N;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = idx / M, m = idx % M;
    const uint16_t *wr = reinterpret_cast<const uint16_t *>(W + m * nb * BB);
    const uint16_t *xr = reinterpret_cast<const uint16_t *>(Xq + n * nb * BB);
    float acc = 0.0f, part = 0.0f;
    for (int b = 0; b < nb; ++b) {
      const uint16_t *wb = wr + b * (BB / 2), *xb = xr + b * (BB / 2);
      uint32_t q[8], x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        q[i] = uint32_t(wb[1 + 2 * i]) | (uint32_t(wb[2 + 2 * i]) << 16);
        x[i] = uint32_t(xb[1 + 2 * i]) | (uint32_t(xb[2 + 2 * i]) << 16);
      }
      const float s = __fmul_rn(half_bits_to_float(wb[0]), half_bits_to_float(xb[0]));
      part = __fmaf_rn(s, float(sumi_q8_q8(q, x)), part);
      if ((b & 15) == 15) {
        acc += part;
        part = 0.0f;
      }
    }
    Y[idx] = acc + part;
  }
}

}  // namespace

cudaError_t launch_gemm(int type, const uint8_t *W, const uint8_t *Xq, float *Y, int64_t M, int64_t N,
                        int64_t K, cudaStream_t stream) {
  (void)type;  // Q8_0 only (checked by the ABI layer)
  if (M == 0 || N == 0) return cudaSuccess;
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  const int nb = int(K / kQK);
  if (K % 256 == 0 && M <= (int64_t(1) << 30) && N <= 65535 * int64_t(kBN)) {
    const size_t smem = 2 * size_t(kStageBytes);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_gemm_q8_mma), int(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(unsigned((M + kBM - 1) / kBM), unsigned((N + kBN - 1) / kBN));
    k_gemm_q8_mma<<<grid, kGemmThreads, smem, stream>>>(W, Xq, Y, int(M), int(N), nb);
    return cudaGetLastError();
  }
  const int64_t grid = min((M * N + 255) / 256, int64_t(di->sm_count) * 8);
  k_gemm_q8_generic<<<unsigned(grid), 256, 0, stream>>>(W, Xq, Y, M, N, nb);
  return cudaGetLastError();
}

}  // namespace bq

namespace bq {

PrefillPath prefill_path(int64_t M, int64_t N, int64_t K, size_t ws_limit, size_t *ws_bytes) {
  if (gemm_tc_supported(M, N, K)) {
    const size_t tc = (gemm_tc_workspace_bytes(N, K) + 255) / 256 * 256;
    if (tc <= ws_limit) {
      *ws_bytes = tc;
      return PrefillPath::kTc;
    }
  }
  *ws_bytes = (size_t(N) * size_t(K / kQK) * Fmt<kTypeQ8_0>::kBytes + 255) / 256 * 256;
  return PrefillPath::kMmaSync;
}

cudaError_t launch_prefill(PrefillPath path, const uint8_t *W, const float *X, float *Y, int64_t M, int64_t N,
                           int64_t K, void *ws, cudaStream_t stream) {
  if (path == PrefillPath::kTc) return launch_gemm_tc(W, X, Y, M, N, K, ws, stream);
  uint8_t *xq = static_cast<uint8_t *>(ws);
  cudaError_t e = launch_quantize_rows(BQ_TYPE_Q8_0, X, xq, N * (K / kQK), K / kQK, nullptr, 1, stream);
  if (e != cudaSuccess) return e;
  return launch_gemm(BQ_TYPE_Q8_0, W, xq, Y, M, N, K, stream);
}

}  // namespace bq
