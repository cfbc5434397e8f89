// gemm_tc.cu — prefill GEMM over Q8_0 weights on the fifth-generation tensor
// cores (tcgen05 MMA with the accumulators in tensor memory).
//
// Y[n][m] = sum over blocks b of scale_w[m][b] * scale_x[n][b] * sumi(m, n, b),
// sumi being the integer dot of the two blocks' 32 codes; the activations are
// quantized to Q8_0 first. Prefill is compute-bound ("05. llama.cpp：从 GGUF
// 文件到本地推理服务", §性能直觉：带宽决定 Decode，算力决定 Prefill), the weight
// blocks are those of §量化类型 (Q8_0: one fp16 scale per 32 weights).
//
// Exactness. Every int8 code is an exact binary16 number, each product of two
// codes has at most 15 bits and the sum of a block's 32 products stays below
// 2^24, so one kind::f16 MMA pair over a 32-deep block leaves the block's
// exact integer dot in its fp32 tensor-memory accumulator. The scales are
// then applied in fp32 (scale_w * scale_x is exact in fp32, one rounding per
// fused multiply-add), and partial sums over 16 blocks are folded into a
// running sum so that the rounding error stays below (16 + blocks/16) units
// of fp32 roundoff of the sum of the terms' magnitudes.
//
// CTA tile: 128 weight rows (the MMA's M, tensor-memory lanes) x 128 tokens
// (the MMA's N, tensor-memory columns); K in stages. 20 warps, so that every
// SM sub-partition runs one helper warp next to four epilogue warps:
//   - warp 0, lane 0: 2-D TMA copies of the raw 34-byte weight blocks, 8
//     blocks (272 bytes) of each of the 128 rows per stage, and 1-D bulk
//     copies of the tile's activation scales; lane 1: 1-D bulk copies of the
//     activation operand, which the activation quantizer already wrote as
//     binary16 codes in the MMA's 128-byte-swizzled K-major layout (16 KB per
//     2 blocks x 128 tokens);
//   - warp 1: allocates the 512 tensor-memory columns and, from one lane,
//     issues two MMAs (K = 16 each) per block into one of three 128-column
//     accumulators;
//   - warps 2, 3: each thread turns two weight rows of raw blocks into
//     binary16 codes in the same swizzled layout, and their scales into fp32;
//   - warps 4..19: the epilogue; warp w reads lanes 32 (w mod 4) .. + 31 and
//     32 of the 128 columns with one tensor-memory load, releases the
//     accumulator, multiplies by the scale products with packed fp32x2 FMAs,
//     and every 16 blocks folds its partial sums into a running sum held in
//     the last 128 tensor-memory columns. (Four warps per sub-partition
//     measured 3-4% faster than two with 64 columns each; the kernel is bound
//     by shared-memory traffic per block, not by the epilogue's warps.)
// Every wait is bounded; a wait that runs out sets the device error word and
// a CTA-wide abort flag, after which every role leaves its loop, copies and
// MMAs in flight are waited for, and the tensor memory is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {
namespace {

constexpr int kTM = 128;                        // weight rows per CTA
constexpr int kTN = 128;                        // tokens per CTA
constexpr int kChunkBlocks = 8;                 // blocks per raw weight stage
constexpr int kRawPitch = kChunkBlocks * 34;    // 272 bytes per row per stage
constexpr int kRawBytes = kTM * kRawPitch;      // 34816
constexpr int kRawStages = 2;
constexpr int kOpBytes = 128 * 128;             // one operand stage: 128 rows x 2 blocks of fp16
constexpr int kSubStages = 4;                   // operand stages (2 blocks each)
constexpr int kScaleSlots = 3;                  // scale stages (8 blocks each)
constexpr int kScaleSlotBytes = 2 * kChunkBlocks * 128 * 4;  // dx then dw, fp32
constexpr int kSBufs = 3;                       // per-block accumulators (128 columns each)
constexpr int kAccCol = kSBufs * kTN;           // running sums: columns 384..511
constexpr int kTmemCols = 512;
constexpr int kFold = 16;                       // blocks per partial sum
#ifndef BQ_GEMM_EPI_WARPS
#define BQ_GEMM_EPI_WARPS 16
#endif
constexpr int kEpiWarps = BQ_GEMM_EPI_WARPS;    // 4 per SM sub-partition
constexpr int kEpiCols = kTN / (kEpiWarps / 4); // 32 columns per epilogue warp
constexpr int kEpiChunks = kEpiCols / 32;       // 32-column tensor-memory loads per block
constexpr int kConvWarps = 2;                   // 2 weight rows per thread
constexpr int kTcThreads = (4 + kEpiWarps) * 32;
constexpr uint32_t kDrainPolls = 1u << 22;

constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kSubStages * kOpBytes;
constexpr int kOffRaw = kOffB + kSubStages * kOpBytes;
constexpr int kOffScale = kOffRaw + kRawStages * kRawBytes;
constexpr int kOffBar = kOffScale + kScaleSlots * kScaleSlotBytes;
constexpr int kNumBars = 32;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024

// barrier indices
constexpr int kRawFull = 0, kRawEmpty = 2, kBFull = 4, kAReady = 8, kSubEmpty = 12, kDxFull = 16,
              kScaleFull = 19, kScaleEmpty = 22, kTFull = 25, kTEmpty = 28, kDone = 31;

static_assert(kOffRaw % 1024 == 0 && kOffScale % 128 == 0 && kOffBar % 8 == 0, "layout");
static_assert(kDone < kNumBars, "barriers");
static_assert(kSmemBytes <= 232448, "shared memory");

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B binary16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at
// bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(kTN >> 3) << 17) | (uint32_t(kTM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: rows of 128 bytes, 8-row groups 1024 bytes apart (stride
// byte offset), start address >> 4 in bits 0-13, descriptor version 1 at bit
// 46, swizzle mode 2 (128 B) in bits 61-63. The leading byte offset is unused
// by this layout and set to 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled operand tile
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive columns of this warp's 32 lanes: thread i gets lane
// (lane base + i), columns taddr.col .. + 31. The wait is in the same asm
// statement so that no use of the registers can be scheduled before it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Shared-memory vector load kept in program order with the tensor-memory
// loads around it (volatile), so that the compiler does not hoist a whole
// block's worth of them and run out of registers.
__device__ __forceinline__ float4 lds_f4_ordered(const float4 *p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// 2-D TMA load of a box of the raw weight map into shared memory
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Bounded wait that also gives up once another thread of the CTA has given
// up. Polls do not suspend in the barrier unit (whose wake-up came hundreds
// of cycles after the phase completed); between polls the thread sleeps
// briefly, so that waiting warps leave the issue slots to working ones. The
// abort flag is read every 64 polls.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, uint32_t limit, volatile int *abort_flag,
                                        unsigned *err) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    __nanosleep(i < 64 ? 20 : 200);
    if ((i & 63) == 63 && *abort_flag) return false;
  }
  *abort_flag = 1;
  atomicOr(err, kErrTimeout);
  return false;
}
// The same for a whole warp: lane 0 polls, the result is broadcast, and the
// warp synchronizes (which orders the other lanes' later accesses after lane
// 0's observation of the phase).
__device__ __forceinline__ bool tc_wait_warp(uint64_t *bar, uint32_t parity, uint32_t limit, volatile int *abort_flag,
                                             unsigned *err) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = tc_wait(bar, parity, limit, abort_flag, err);
  ok = __shfl_sync(kFull, ok, 0);
  __syncwarp();
  return ok != 0;
}
// Wait for copies or MMAs already issued (they complete on their own).
__device__ __forceinline__ void drain(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kDrainPolls; ++i)
    if (mbar_try_wait(bar, parity)) return;
}

// One converter thread: rows r and r + 64 of operand stage k (0..3) of the
// raw chunk in `raw`, written as binary16 codes into the swizzled tile `a`.
__device__ __forceinline__ void convert_stage(const uint8_t *raw, uint8_t *a, int r, int k) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int rr = r + 64 * h;
    const uint8_t *row = raw + rr * kRawPitch;
    // bytes 68k .. 68k+67 of the row: 16-byte vectors 4k .. 4k+4, words k .. k+16 of them
    uint32_t w[20];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * (4 * k + i));
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
    uint32_t code[16];  // first block: bytes 2..33 (shifted by 2 bytes); second: words 9..16
#pragma unroll
    for (int i = 0; i < 8; ++i) code[i] = __funnelshift_r(w[k + i], w[k + i + 1], 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) code[8 + i] = w[k + 9 + i];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const uint2 lo = codes_to_f16x2(code[2 * cc]), hi = codes_to_f16x2(code[2 * cc + 1]);
      *reinterpret_cast<uint4 *>(a + sw128_off(rr, cc)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
  }
}

// Issue a 32-column tensor-memory load without waiting for it.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Wait for this thread's tensor-memory loads; the registers of the last one
// are operands so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// part[2i], part[2i+1] += S[c] * (dw * dx[c]) for the 32 columns of one chunk
__device__ __forceinline__ void scale_accumulate(uint64_t *part, const uint32_t (&s)[32], uint64_t dw2,
                                                 const float4 *dx4) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 d = lds_f4_ordered(dx4 + q);
    const uint64_t p01 = fmul2(dw2, pack2(__float_as_uint(d.x), __float_as_uint(d.y)));
    const uint64_t p23 = fmul2(dw2, pack2(__float_as_uint(d.z), __float_as_uint(d.w)));
    part[2 * q] = ffma2(pack2(s[4 * q], s[4 * q + 1]), p01, part[2 * q]);
    part[2 * q + 1] = ffma2(pack2(s[4 * q + 2], s[4 * q + 3]), p23, part[2 * q + 1]);
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    k_gemm_q8_tc(const __grid_constant__ CUtensorMap wmap, const uint8_t *__restrict__ xp,
                 const float *__restrict__ dxs, float *__restrict__ Y, int M, int N, int nb, uint32_t spin,
                 unsigned *err) {
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t base = smem_u32(smem_dyn);
  uint8_t *sm = smem_dyn + (((base + 1023u) & ~1023u) - base);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x, m0 = blockIdx.y * kTM;
  const int nchunks = nb / kChunkBlocks, nsub = nb / 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(&bar[kRawFull + i], 1);
      mbar_init(&bar[kRawEmpty + i], kConvWarps);
    }
    for (int i = 0; i < kSubStages; ++i) {
      mbar_init(&bar[kBFull + i], 1);
      mbar_init(&bar[kAReady + i], kConvWarps);
      mbar_init(&bar[kSubEmpty + i], 1);
    }
    for (int i = 0; i < kScaleSlots; ++i) {
      mbar_init(&bar[kDxFull + i], 1);
      mbar_init(&bar[kScaleFull + i], kConvWarps);
      mbar_init(&bar[kScaleEmpty + i], kEpiWarps);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&bar[kTFull + i], 1);
      mbar_init(&bar[kTEmpty + i], kEpiWarps);
    }
    mbar_init(&bar[kDone], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- producer: raw weight blocks (2-D TMA) and activation scales ----
    int raw_armed = 0, dx_armed = 0;  // chunks whose copies were issued
    for (int c = 0; c < nchunks; ++c) {
      const int rs = c % kRawStages, ss = c % kScaleSlots;
      if (!tc_wait(&bar[kRawEmpty + rs], ((c / kRawStages) & 1) ^ 1, spin, abort_flag, err)) break;
      mbar_arrive_expect_tx(&bar[kRawFull + rs], kRawBytes);
      tma_load_2d(sm + kOffRaw + rs * kRawBytes, &wmap, c * (kRawPitch / 2), m0, &bar[kRawFull + rs]);
      raw_armed = c + 1;
      if (!tc_wait(&bar[kScaleEmpty + ss], ((c / kScaleSlots) & 1) ^ 1, spin, abort_flag, err)) break;
      mbar_arrive_expect_tx(&bar[kDxFull + ss], kChunkBlocks * 128 * 4);
      bulk_g2s(sm + kOffScale + ss * kScaleSlotBytes, dxs + (int64_t(n_tile) * nb + c * kChunkBlocks) * 128,
               kChunkBlocks * 128 * 4, &bar[kDxFull + ss]);
      dx_armed = c + 1;
    }
    // wait until every issued copy has landed: the last phase armed on each
    // slot (chunk last = the largest chunk < armed that used the slot)
    for (int i = 0; i < kRawStages && i < raw_armed; ++i) {
      const int last = raw_armed - 1 - ((raw_armed - 1 - i) % kRawStages);
      drain(&bar[kRawFull + i], (last / kRawStages) & 1);
    }
    for (int i = 0; i < kScaleSlots && i < dx_armed; ++i) {
      const int last = dx_armed - 1 - ((dx_armed - 1 - i) % kScaleSlots);
      drain(&bar[kDxFull + i], (last / kScaleSlots) & 1);
    }
  } else if (warp == 0 && lane == 1) {
    // ---- producer: activation operand tiles (1-D bulk, pre-swizzled) ----
    const uint8_t *src = xp + int64_t(n_tile) * nsub * kOpBytes;
    int g = 0;
    for (; g < nsub; ++g) {
      const int as = g % kSubStages;
      if (!tc_wait(&bar[kSubEmpty + as], ((g / kSubStages) & 1) ^ 1, spin, abort_flag, err)) break;
      mbar_arrive_expect_tx(&bar[kBFull + as], kOpBytes);
      bulk_g2s(sm + kOffB + as * kOpBytes, src + int64_t(g) * kOpBytes, kOpBytes, &bar[kBFull + as]);
    }
    for (int i = 0; i < kSubStages && i < g; ++i) {
      const int last = g - 1 - ((g - 1 - i) % kSubStages);
      drain(&bar[kBFull + i], (last / kSubStages) & 1);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issue (one lane) ----
    const uint32_t a0 = smem_u32(sm + kOffA), b0 = smem_u32(sm + kOffB);
    for (int gb = 0; gb < nb; ++gb) {
      const int g = gb >> 1, j = gb & 1, as = g % kSubStages, sb = gb % kSBufs;
      if (j == 0) {
        if (!tc_wait(&bar[kAReady + as], (g / kSubStages) & 1, spin, abort_flag, err)) break;
        if (!tc_wait(&bar[kBFull + as], (g / kSubStages) & 1, spin, abort_flag, err)) break;
      }
      if (!tc_wait(&bar[kTEmpty + sb], ((gb / kSBufs) & 1) ^ 1, spin, abort_flag, err)) break;
      tc_fence_after();
      const uint64_t ad = sw128_desc(a0 + as * kOpBytes) + uint64_t(j * 4);
      const uint64_t bd = sw128_desc(b0 + as * kOpBytes) + uint64_t(j * 4);
      const uint32_t d = tmem + uint32_t(sb * kTN);
      tc_mma(d, ad, bd, 0);          // k 0..15 of the block
      tc_mma(d, ad + 2, bd + 2, 1);  // k 16..31 (32 bytes further)
      tc_commit(&bar[kTFull + sb]);
      if (j == 1) tc_commit(&bar[kSubEmpty + as]);
    }
    tc_commit(&bar[kDone]);
    drain(&bar[kDone], 0);
  } else if (warp == 2 || warp == 3) {
    // ---- converters: raw Q8_0 blocks -> binary16 codes (swizzled) + fp32 scales ----
    const int r = (warp - 2) * 32 + lane;  // rows r and r + 64
    for (int c = 0; c < nchunks; ++c) {
      const int rs = c % kRawStages, ss = c % kScaleSlots;
      if (!tc_wait_warp(&bar[kRawFull + rs], (c / kRawStages) & 1, spin, abort_flag, err)) break;
      if (!tc_wait_warp(&bar[kScaleEmpty + ss], ((c / kScaleSlots) & 1) ^ 1, spin, abort_flag, err)) break;
      const uint8_t *raw = sm + kOffRaw + rs * kRawBytes;
      float *dw = reinterpret_cast<float *>(sm + kOffScale + ss * kScaleSlotBytes) + kChunkBlocks * 128;
#pragma unroll
      for (int j = 0; j < kChunkBlocks; ++j) {
        dw[j * 128 + r] = half_bits_to_float(reinterpret_cast<const uint16_t *>(raw + r * kRawPitch)[17 * j]);
        dw[j * 128 + r + 64] = half_bits_to_float(reinterpret_cast<const uint16_t *>(raw + (r + 64) * kRawPitch)[17 * j]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kScaleFull + ss]);
      bool ok = true;
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // operand stages of this chunk (2 blocks = 68 raw bytes each)
        const int g = c * 4 + k, as = g % kSubStages;
        if (!tc_wait_warp(&bar[kSubEmpty + as], ((g / kSubStages) & 1) ^ 1, spin, abort_flag, err)) {
          ok = false;
          break;
        }
        convert_stage(raw, sm + kOffA + as * kOpBytes, r, k);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kAReady + as]);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kRawEmpty + rs]);
    }
  } else if (warp >= 4 && warp < 4 + kEpiWarps) {
    // ---- epilogue: lanes 32 (warp mod 4) .., kEpiCols columns in 32-column chunks ----
    const int lg = warp & 3, ch = (warp - 4) >> 2;
    const int row = lg * 32 + lane, col0 = ch * kEpiCols;
    const uint32_t lane_addr = tmem + (uint32_t(lg * 32) << 16);
    uint64_t part[kEpiCols / 2];  // columns col0 + 2i, 2i + 1
#pragma unroll
    for (int i = 0; i < kEpiCols / 2; ++i) part[i] = 0;
    bool first_fold = true, ok = true;
    for (int gb = 0; gb < nb && ok; ++gb) {
      const int c = gb / kChunkBlocks, jj = gb % kChunkBlocks, ss = c % kScaleSlots, sb = gb % kSBufs;
      if (jj == 0) {
        ok = tc_wait_warp(&bar[kDxFull + ss], (c / kScaleSlots) & 1, spin, abort_flag, err) &&
             tc_wait_warp(&bar[kScaleFull + ss], (c / kScaleSlots) & 1, spin, abort_flag, err);
        if (!ok) break;
      }
      if (!tc_wait_warp(&bar[kTFull + sb], (gb / kSBufs) & 1, spin, abort_flag, err)) break;
      tc_fence_after();
      const float *slot = reinterpret_cast<const float *>(sm + kOffScale + ss * kScaleSlotBytes);
      const float dwv = slot[kChunkBlocks * 128 + jj * 128 + row];
      const uint64_t dw2 = pack2(__float_as_uint(dwv), __float_as_uint(dwv));
      const float4 *dx4 = reinterpret_cast<const float4 *>(slot + jj * 128 + col0);
      if constexpr (kEpiChunks == 1) {
        // one 32-column load: the accumulator is released as soon as it is read
        uint32_t s0[32];
        tmem_ld32_issue(lane_addr + uint32_t(sb * kTN + col0), s0);
        tmem_ld_wait(s0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kTEmpty + sb]);
        scale_accumulate(part, s0, dw2, dx4);
      } else {
        uint32_t s0[32], s1[32];
        tmem_ld32_issue(lane_addr + uint32_t(sb * kTN + col0), s0);
        tmem_ld_wait(s0);
        tmem_ld32_issue(lane_addr + uint32_t(sb * kTN + col0 + 32), s1);  // lands while chunk 0 is scaled
        scale_accumulate(part, s0, dw2, dx4);
        tmem_ld_wait(s1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kTEmpty + sb]);
        scale_accumulate(part + 16, s1, dw2, dx4 + 8);
      }
      if (jj == kChunkBlocks - 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kScaleEmpty + ss]);
      }
      if ((gb % kFold) == kFold - 1 || gb == nb - 1) {
        // fold the partial sums into the running sum (tensor-memory columns 384 + col0 ..)
#pragma unroll
        for (int h = 0; h < kEpiChunks; ++h) {
          const uint32_t acc_addr = lane_addr + uint32_t(kAccCol + col0 + 32 * h);
          uint32_t v[32];
          if (first_fold) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              v[2 * i] = uint32_t(part[16 * h + i]);
              v[2 * i + 1] = uint32_t(part[16 * h + i] >> 32);
            }
          } else {
            tmem_ld32(acc_addr, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint64_t sum = fadd2(pack2(v[2 * i], v[2 * i + 1]), part[16 * h + i]);
              v[2 * i] = uint32_t(sum);
              v[2 * i + 1] = uint32_t(sum >> 32);
            }
          }
          tmem_st32(acc_addr, v);
        }
#pragma unroll
        for (int i = 0; i < kEpiCols / 2; ++i) part[i] = 0;
        first_fold = false;
      }
    }
    if (ok && !*abort_flag) {
      const int m = m0 + row;
#pragma unroll 1
      for (int h = 0; h < kEpiChunks; ++h) {
        const int nbase = n_tile * kTN + col0 + 32 * h;
        uint32_t v[32];
        tmem_ld32(lane_addr + uint32_t(kAccCol + col0 + 32 * h), v);
        if (m < M) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (nbase + i < N) Y[int64_t(nbase + i) * M + m] = __uint_as_float(v[i]);
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Activations for the kernel above: X (N x K fp32) quantized to Q8_0 codes
// (the same rule as the row quantizer), written as binary16 codes in the
// operand layout — per 128-token tile t and 2-block group a, one 16 KB
// 128-byte-swizzled tile at (t * K/64 + a) * 16 KB — and the scales as fp32 at
// dxs[(t * nb + b) * 128 + token % 128]. Tokens N .. (tiles*128 - 1) get zero
// codes and zero scales. 8 lanes per block.
__global__ void __launch_bounds__(256)
    k_quantize_x_tc(const float *__restrict__ X, int N, int nb, int n_pad, uint8_t *__restrict__ xp,
                    float *__restrict__ dxs) {
  const int j = threadIdx.x & 7;
  const int64_t total = int64_t(n_pad) * nb;  // a multiple of 128
  const int64_t step = int64_t(gridDim.x) * (blockDim.x >> 3);
  // the 4 items of a warp are consecutive and total is a multiple of 4, so
  // every lane of a warp takes the same number of trips (the quantizer shuffles)
  for (int64_t item = int64_t(blockIdx.x) * (blockDim.x >> 3) + (threadIdx.x >> 3); item < total; item += step) {
    const int64_t n = item / nb;
    const int b = int(item % nb);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (n < N) v = __ldcs(reinterpret_cast<const float4 *>(X + n * int64_t(nb) * kQK + b * kQK) + j);
    uint16_t scale;
    uint32_t word;
    int sum;
    quantize_block_8lanes(v, scale, word, sum);
    const int64_t t = n >> 7;
    const int r = int(n & 127);
    uint8_t *tile = xp + (t * (nb / 2) + (b >> 1)) * int64_t(kOpBytes);
    const int chunk = (b & 1) * 4 + (j >> 1);
    *reinterpret_cast<uint2 *>(tile + sw128_off(r, chunk) + (j & 1) * 8) = codes_to_f16x2(word);
    if (j == 0) dxs[(t * nb + b) * 128 + r] = half_bits_to_float(scale);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

bool gemm_tc_supported(int64_t M, int64_t N, int64_t K) {
  return K > 0 && K % 256 == 0 && K / kQK <= (int64_t(1) << 24) && (M + kTM - 1) / kTM <= 65535 &&
         N <= 0x7fffffffll - kTN && M <= 0x7fffffffll;
}

size_t gemm_tc_workspace_bytes(int64_t N, int64_t K) {
  const size_t tiles = size_t((N + kTN - 1) / kTN);
  return tiles * kTN * size_t(K) * 2 + tiles * size_t(K / kQK) * kTN * 4;
}

cudaError_t launch_gemm_tc(const uint8_t *W, const float *X, float *Y, int64_t M, int64_t N, int64_t K, void *ws,
                           cudaStream_t stream) {
  if (M == 0 || N == 0) return cudaSuccess;
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  const int nb = int(K / kQK);
  const int64_t n_tiles = (N + kTN - 1) / kTN;
  uint8_t *xp = static_cast<uint8_t *>(ws);
  float *dxs = reinterpret_cast<float *>(xp + n_tiles * kTN * K * 2);
  {
    const int64_t items = n_tiles * kTN * nb;
    const int64_t grid = std::min<int64_t>((items + 31) / 32, int64_t(di->sm_count) * 16);
    k_quantize_x_tc<<<unsigned(grid), 256, 0, stream>>>(X, int(N), nb, int(n_tiles * kTN), xp, dxs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {cuuint64_t(nb) * 17, cuuint64_t(M)};  // 16-bit units per row, rows
  const cuuint64_t strides[1] = {cuuint64_t(nb) * 34};
  const cuuint32_t box[2] = {kRawPitch / 2, kTM};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t *>(W), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k_gemm_q8_tc), kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(unsigned(n_tiles), unsigned((M + kTM - 1) / kTM));
  k_gemm_q8_tc<<<grid, kTcThreads, kSmemBytes, stream>>>(map, xp, dxs, Y, int(M), int(N), nb, spin_limit(),
                                                         di->err_word);
  return cudaGetLastError();
}

}  // namespace bq
