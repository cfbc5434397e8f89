// gemv_seq.cu — a decode step's GEMV batches in one persistent launch.
//
// A decode step is a run of weight-matrix products, each bounded by the
// weight bytes it reads ("05. llama.cpp：从 GGUF 文件到本地推理服务",
// §性能直觉：带宽决定 Decode，算力决定 Prefill: decode reads every weight once per
// token, so tokens/s is about bandwidth / weight bytes). Launched one batch at
// a time, the weight stream stops at every launch boundary (the next kernel
// starts, waits for the previous one, quantizes its input, refills its
// pipeline). Here one launch covers the whole run and the stream never stops.
//
// One CTA per SM:
//   producer warp    streams this CTA's rows of every batch, in batch order,
//                    with 1-D bulk copies into a ring of shared-memory stages
//                    (mbarrier-completed). It depends on nothing but free
//                    stages: the run never writes a weight.
//   consumer warps   two groups of 8 take the stages in turn; a stage is one
//                    pass of a group (each warp 32 / lanes rows, as in the
//                    per-launch kernel), so a stage is consumed by its whole
//                    group at once and released once. Every row is dotted
//                    with x's Q8_0 records, its lanes reduced, y written.
//   x warps          at the start, with the consumers, quantize x of every
//                    batch that waits for nothing (see below) into records in
//                    the workspace, each CTA a slice, and count the CTA done;
//                    then one lane copies each batch's records into a ring of
//                    record buffers (bulk copies), batches ahead of the
//                    consumers.
// Batch g has the result of one bq_gemv_multi call issued after the calls of
// batches 0..g-1. Only memory orders them: when x[g] overlaps an output of an
// earlier batch, or an output of batch g overlaps the input of an earlier
// batch, batch g waits until every CTA has finished the latest such batch (a
// per-batch counter in global memory, incremented once per CTA after a fence,
// polled with acquire loads), and then the consumers quantize x[g]
// themselves. The host derives these waits from the pointers; batches that
// share no memory never wait. All waits are bounded.
// Every CTA takes a contiguous, balanced range of each batch's rows, the
// ranges rotating over the CTAs from batch to batch so that the CTAs' total
// bytes stay level. Per row the arithmetic (records, group order, lanes per
// row, shuffle tree) is that of the per-launch kernel, so the outputs are
// bit-identical to bq_gemv_multi. The launch is cooperative (every CTA
// resident), so a wait on other CTAs cannot wait for a CTA that has not
// started.
#include <algorithm>
#include <memory>
#include <vector>

#include "bq_device.cuh"
#include "bq_internal.h"
#include "gemv_common.cuh"

namespace bq {
namespace {

using gemv::GroupWords;
using gemv::group_terms;
using gemv::kXRecBytes;
using gemv::kXRecWords;
using gemv::quantize_x_records_2lane;

constexpr int kSqConsumers = 16;  // consumer warps per CTA
constexpr int kSqXWarps = 3;      // quantize x at the start; then one lane copies records (20 warps: 96 registers)
constexpr int kSqProducer = kSqConsumers + kSqXWarps;  // warp index of the producer
constexpr int kSqWarps = kSqConsumers + kSqXWarps + 1;
constexpr int kSqThreads = kSqWarps * 32;
constexpr int kSeqMaxGroups = 256;  // per launch; longer runs take several launches
constexpr int kSeqMaxMats = 512;
constexpr uint32_t kSeqDrainLimit = 1u << 26;
constexpr int kRowRotation = 37;  // CTA range rotation per batch
constexpr int kBarConsumers = 1;  // named barrier of the consumer warps
constexpr int kBarPre = 2;        // named barrier of the warps that quantize x at the start
constexpr int kPreThreads = (kSqConsumers + kSqXWarps) * 32;
constexpr int kMaxRecBufs = 8;    // record buffers in shared memory
constexpr int kCopyWarps = 2;     // x warps that copy records (nrec is a multiple of it)
constexpr int kSyncWords = 2 + kSeqMaxGroups;  // abort flag, CTAs done quantizing, CTAs done per batch
constexpr size_t kSyncBytes = (kSyncWords * 4 + 255) / 256 * 256;
constexpr size_t kRecBytesMax = size_t(kSeqMaxGroups) * (BQ_GEMV_SEQ_MAX_K / 256) * kXRecBytes;

// One batch, as every CTA keeps it in shared memory during the launch (32
// bytes; read there, not from the kernel parameters, whose dynamically
// indexed reads miss the constant cache).
struct BatchDesc {
  const float *x;
  int rows;            // rows of all the batch's matrices
  int rec_off;         // words: x's records in SeqArgs::rec, or -1: quantized in every CTA
  int blk0;            // first block of x in the start-of-launch quantization (rec_off >= 0)
  uint16_t K;          // a multiple of 256, at most BQ_GEMV_SEQ_MAX_K
  uint16_t first_mat;  // matrices first_mat .. first_mat + n_mats - 1
  uint16_t stage_rows; // rows per stage: one pass of a consumer group, as the ring slot allows
  int16_t wait_on;     // batch (of this launch) every CTA must have finished first, or -1
  uint8_t n_mats;
  uint8_t lanes;       // lanes per row: the power of two <= 32 the per-launch kernel takes
  uint8_t signal;      // nonzero: a later batch waits for this one
  uint8_t lanes_log2;
};
static_assert(sizeof(BatchDesc) == 32, "batch descriptor");

struct MatDesc {
  const uint8_t *W;
  float *y;
  int row_start;  // first row of this matrix within its batch
  int pad;
};
static_assert(sizeof(MatDesc) == 24, "matrix descriptor");

struct SeqArgs {
  BatchDesc g[kSeqMaxGroups];
  MatDesc m[kSeqMaxMats];
  int n_groups;
  int n_mats;
  int stages;
  int slot_bytes;  // bytes of one ring stage
  int xrec_bytes;  // bytes of one record buffer (the largest K of the launch)
  int nrec;        // record buffers in shared memory: a power of two, 2..kMaxRecBufs
  int nrec_log2;
  int ngroups;     // consumer groups: 2 or 4 (kSqConsumers / ngroups warps each)
  int pre_blocks;  // blocks of x quantized at the start (every batch with rec_off >= 0)
  int n_local;     // the first n_local batches are quantized by every CTA itself
  int desc_bytes;  // shared-memory bytes of the descriptor tables (16-byte multiple)
  uint32_t *rec;   // x's records of those batches (global memory)
  unsigned *sync;  // [0]: abort flag, [1]: CTAs done quantizing, [2 + g]: CTAs done with batch g; zeroed
  unsigned *err;
  uint32_t spin_limit;
  uint32_t poll_ns;  // sleep between polls of a mbarrier
};

// A batch's fields in registers.
template <int TYPE>
struct Batch {
  const float *x;
  int rows, rec_off, blk0, K, first_mat, n_mats, stage_rows, wait_on, lanes, lanes_log2, signal, groups8, row_bytes;
  __device__ __forceinline__ explicit Batch(const BatchDesc &d)
      : x(d.x), rows(d.rows), rec_off(d.rec_off), blk0(d.blk0), K(d.K), first_mat(d.first_mat), n_mats(d.n_mats),
        stage_rows(d.stage_rows), wait_on(d.wait_on), lanes(d.lanes), lanes_log2(d.lanes_log2), signal(d.signal),
        groups8(d.K >> 8), row_bytes((d.K >> 5) * Fmt<TYPE>::kBytes) {}
};

// Rows [r0, r1) of a batch of `rows` rows taken by this CTA (the batch's
// part p, the parts rotating over the CTAs from batch to batch). Computed
// once per batch at the start of the launch into a shared-memory table: the
// 64-bit divisions cost hundreds of cycles.
__device__ __forceinline__ int2 cta_rows(int rows, int g) {
  const int G = int(gridDim.x);
  const int p = int((blockIdx.x + unsigned(g) * kRowRotation) % unsigned(G));
  return make_int2(int(int64_t(rows) * p / G), int(int64_t(rows) * (p + 1) / G));
}

// Stages of one batch's row range in order: each at most stage_rows rows,
// never past the range or a matrix's end. Producer and consumers walk the
// same sequence (incrementally: no division per stage).
struct StageWalk {
  int row, r1, mat, mat_end, last, rows, stage_rows;
  template <int TYPE>
  __device__ __forceinline__ void begin(const MatDesc *md, const Batch<TYPE> &B, int r0, int r1_) {
    row = r0;
    r1 = r1_;
    rows = B.rows;
    stage_rows = B.stage_rows;
    mat = B.first_mat;
    last = B.first_mat + B.n_mats - 1;
    while (mat < last && row >= md[mat + 1].row_start) ++mat;
    mat_end = mat < last ? md[mat + 1].row_start : rows;
  }
  // rows of the stage that starts at `row` (row < r1)
  __device__ __forceinline__ int next(const MatDesc *md) {
    if (row >= mat_end) {
      ++mat;
      mat_end = mat < last ? md[mat + 1].row_start : rows;
    }
    return min(min(stage_rows, r1 - row), mat_end - row);
  }
};

__device__ __forceinline__ bool grid_aborted(const SeqArgs &a) {
  return *reinterpret_cast<volatile unsigned *>(a.sync) != 0u;
}

__device__ __forceinline__ void seq_abort(const SeqArgs &a, volatile int *cta_abort) {
  *cta_abort = 1;
  atomicExch(a.sync, 1u);
  atomicOr(a.err, kErrTimeout);
}

// Bounded wait on one of this CTA's mbarriers that also gives up once
// another role of the CTA gave up. By default each poll may suspend the
// thread in the barrier unit until the phase completes (a waiting warp then
// issues almost nothing); with poll_ns set, polls never suspend and the warp
// sleeps poll_ns between them.
// Only the CTA's own flag (shared memory) is read here: these barriers depend
// on this CTA's roles alone, which all end; the grid-wide flag is read where a
// CTA waits for other CTAs.
__device__ __forceinline__ bool seq_wait(const SeqArgs &a, uint64_t *bar, uint32_t parity, volatile int *cta_abort) {
  // a phase that has already completed: the non-blocking test answers at
  // once (a suspending wait takes a few hundred cycles even then); a limit
  // of 0 polls gives up without looking
  if (a.spin_limit > 0 && mbar_test_wait(bar, parity)) return true;
  if (a.poll_ns == 0) {  // suspend in the barrier unit between polls
    for (uint32_t i = 0; i < a.spin_limit; ++i) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((i & 15) == 15 && *cta_abort) return false;
    }
  } else {
    for (uint32_t i = 0; i < a.spin_limit; ++i) {
      if (mbar_test_wait(bar, parity)) return true;
      __nanosleep(a.poll_ns);
      if ((i & 63) == 63 && *cta_abort) return false;
    }
  }
  seq_abort(a, cta_abort);
  return false;
}

// Until the counter `cnt` (global memory, counts CTAs) reaches every CTA of
// the grid (acquire), bounded; also gives up once the grid aborted.
__device__ __forceinline__ bool seq_count_wait(const SeqArgs &a, const unsigned *cnt, volatile int *cta_abort) {
  const unsigned target = gridDim.x;
  for (uint32_t i = 0; i < a.spin_limit; ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= target) return true;
    if (*cta_abort || grid_aborted(a)) return false;
    __nanosleep(20);
  }
  seq_abort(a, cta_abort);
  return false;
}

// Until every CTA has counted itself done with batch `g`.
__device__ __forceinline__ bool seq_batch_wait(const SeqArgs &a, int g, volatile int *cta_abort) {
  return seq_count_wait(a, a.sync + 2 + g, cta_abort);
}

// Blocks [lo, hi) of the start-of-launch quantization taken by this CTA.
__device__ __forceinline__ void pre_range(const SeqArgs &a, int &lo, int &hi) {
  const int G = int(gridDim.x);
  lo = int(int64_t(a.pre_blocks) * blockIdx.x / G);
  hi = int(int64_t(a.pre_blocks) * (blockIdx.x + 1) / G);
}

// Quantize this CTA's share of x's blocks of every batch whose records come
// from the workspace (the launch's blocks in batch order, cut evenly over the
// CTAs) into those records: two threads per block (quantize_block_pair), so
// the records are those of the per-launch kernels. tid < kPreThreads.
__device__ __forceinline__ void seq_prequantize(const SeqArgs &a, const BatchDesc *bd, int tid) {
  int lo, hi;
  pre_range(a, lo, hi);
  const int h = tid & 1;
  int g = 0;  // batch of block i (i only grows)
  for (int base = lo; base < hi; base += kPreThreads / 2) {  // uniform: every lane runs every round
    const int i = base + (tid >> 1);
    const bool valid = i < hi;
    float f[16];
    uint32_t *rg = a.rec;
    int jb = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] = 0.0f;
    if (valid) {
      while (bd[g].rec_off < 0 || i >= bd[g].blk0 + bd[g].K / kQK) ++g;
      const int bl = i - bd[g].blk0;
      const float4 *src = reinterpret_cast<const float4 *>(bd[g].x + int64_t(bl) * kQK + 16 * h);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 v = __ldcg(src + c);
        f[4 * c] = v.x;
        f[4 * c + 1] = v.y;
        f[4 * c + 2] = v.z;
        f[4 * c + 3] = v.w;
      }
      rg = a.rec + bd[g].rec_off + (bl >> 3) * kXRecWords;
      jb = bl & 7;
    }
    gemv::quantize_block_pair(f, h, rg, jb, valid);
  }
}

// L2 prefetch of this CTA's slice of the start-of-launch quantization (the
// x ranges seq_prequantize reads here) and of x of the first batches, which
// every CTA quantizes itself.
__device__ __forceinline__ void seq_prefetch_x(const SeqArgs &a, const BatchDesc *bd) {
  int lo, hi;
  pre_range(a, lo, hi);
  for (int g = 0; g < a.n_groups; ++g) {
    const BatchDesc &d = bd[g];
    if (d.rec_off < 0) {
      if (d.wait_on < 0 && g < a.n_local) prefetch_l2(d.x, uint32_t(d.K) * 4u);
      continue;
    }
    if (d.blk0 >= hi) break;
    const int b0 = max(lo, d.blk0), b1 = min(hi, d.blk0 + d.K / kQK);
    if (b0 < b1) prefetch_l2(d.x + int64_t(b0 - d.blk0) * kQK, uint32_t(b1 - b0) * kQK * 4u);
  }
}

// Consumer group cg takes stages j with j mod ngroups == cg: does it take
// one of the batch's stages here (first stage js.x, js.y stages)?
__device__ __forceinline__ bool seq_group_owns(const SeqArgs &a, int2 js, int cg) {
  return js.y >= a.ngroups || ((cg - js.x) & (a.ngroups - 1)) < js.y;
}
// Can the consumer groups with no stage of this batch here step over it? Only
// where its records come from the workspace and no other batch waits for it
// (else every group takes part: the consumers' own quantization of x and the
// signal to the grid need them all), and where some group has no stage.
__device__ __forceinline__ bool seq_batch_skippable(const SeqArgs &a, const BatchDesc &d, int2 js) {
  return d.rec_off >= 0 && !d.signal && js.y < a.ngroups;
}

// SKIP: the consumer groups step over the batches in which they own no
// stage (instantiated for launches of four groups, where a CTA's share of a
// batch is often a stage or two; with two groups the stage table and the
// extra branch cost more than they save).
template <int TYPE, bool SKIP>
__global__ void __launch_bounds__(kSqThreads, 1) k_gemv_seq(const __grid_constant__ SeqArgs a) {
  constexpr int GW = GroupWords<TYPE>::kWords;
  extern __shared__ __align__(128) uint8_t smem[];
  // record buffer b at smem + b * xrec_bytes, b < nrec; then the ring, the
  // descriptor tables, the barriers
  uint8_t *ring = smem + size_t(a.nrec) * a.xrec_bytes;
  BatchDesc *bd = reinterpret_cast<BatchDesc *>(ring + size_t(a.stages) * a.slot_bytes);
  MatDesc *md = reinterpret_cast<MatDesc *>(bd + a.n_groups);
  int2 *rr = reinterpret_cast<int2 *>(md + a.n_mats);  // this CTA's rows of batch g
  int2 *js = rr + a.n_groups;  // this CTA's first stage of batch g and its number of stages
  uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(bd) + a.desc_bytes);
  uint64_t *empty = full + a.stages;
  uint64_t *rfull = empty + a.stages;  // [nrec]: records of buffer b in place
  uint64_t *rempty = rfull + a.nrec;   // [nrec]: records of buffer b no longer read
  volatile int *cta_abort = reinterpret_cast<volatile int *>(rempty + a.nrec);
  __shared__ int s_go;  // dependency wait result, broadcast to the consumer warps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;
  const uint32_t rmask = uint32_t(a.nrec - 1);

  {
    // descriptor tables into shared memory (the words of g[] and m[] in use)
    const uint32_t *pg = reinterpret_cast<const uint32_t *>(a.g);
    const uint32_t *pm = reinterpret_cast<const uint32_t *>(a.m);
    uint32_t *sg = reinterpret_cast<uint32_t *>(bd), *sm_ = reinterpret_cast<uint32_t *>(md);
    const int ng = a.n_groups * int(sizeof(BatchDesc) / 4), nm = a.n_mats * int(sizeof(MatDesc) / 4);
    for (int i = threadIdx.x; i < ng; i += kSqThreads) sg[i] = pg[i];
    for (int i = threadIdx.x; i < nm; i += kSqThreads) sm_[i] = pm[i];
    for (int g = threadIdx.x; g < a.n_groups; g += kSqThreads) rr[g] = cta_rows(a.g[g].rows, g);
  }
  if constexpr (SKIP) {
    __syncthreads();
    // stages of every batch in this CTA (the walk the producer and the
    // consumers make), then their first stage indices by a prefix sum over the
    // batches (warp 0, 32 batches per step)
    for (int g = threadIdx.x; g < a.n_groups; g += kSqThreads) {
      const Batch<TYPE> B(bd[g]);
      int n = 0;
      if (rr[g].x < rr[g].y) {
        StageWalk wk{};
        wk.begin(md, B, rr[g].x, rr[g].y);
        while (wk.row < wk.r1) {
          wk.row += wk.next(md);
          ++n;
        }
      }
      js[g].y = n;
    }
    __syncthreads();
    if (warp == 0) {
      int base = 0;
      for (int g0 = 0; g0 < a.n_groups; g0 += 32) {
        const int g = g0 + lane;
        const int v = g < a.n_groups ? js[g].y : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int t = __shfl_up_sync(kFull, incl, off);
          if (lane >= off) incl += t;
        }
        if (g < a.n_groups) js[g].x = base + incl - v;
        base += __shfl_sync(kFull, incl, 31);
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSqConsumers / a.ngroups);  // every warp of the stage's consumer group releases it
    }
    for (int b = 0; b < a.nrec; ++b) {
      mbar_init(&rfull[b], 32);  // every lane of the copying x warp, after its record stores
      mbar_init(&rempty[b], kSqConsumers);
    }
    *cta_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp != kSqProducer && a.pre_blocks > 0) {
    // x of the batches whose records come from the workspace, quantized once
    // for the whole grid (this CTA's slice); then this CTA counts itself done
    // (release: the records are visible to the whole GPU)
    seq_prequantize(a, bd, threadIdx.x);
    named_bar_sync(kBarPre, kPreThreads);
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(a.sync + 1, 1u);
    }
  }

  if (warp == kSqProducer) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      // Before the weight stream, ask L2 for the x this CTA reads first (its
      // slice of the start-of-launch quantization, and x of the first batch,
      // which every CTA quantizes itself): these loads then do not queue
      // behind the whole GPU's weight stream.
      seq_prefetch_x(a, bd);
      int issued = 0;
      const uint64_t policy = l2_evict_first_policy();  // every weight is read once
      bool stop = false;
      int j = 0, s = 0;  // stage index, its ring slot
      uint32_t ph = 0;   // (j / S) & 1
      for (int g = 0; g < a.n_groups && !stop; ++g) {
        const Batch<TYPE> B(bd[g]);
        const int r0 = rr[g].x, r1 = rr[g].y;
        if (r0 >= r1) continue;
        StageWalk wk{};
        wk.begin(md, B, r0, r1);
        while (wk.row < r1) {
          // the slot's previous use (stage j - S) must have been released
          if (j >= S && !seq_wait(a, &empty[s], ph ^ 1u, cta_abort)) {
            stop = true;
            break;
          }
          const int nrows = wk.next(md);
          const uint32_t bytes = uint32_t(nrows) * uint32_t(B.row_bytes);
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_g2s_hint(ring + size_t(s) * a.slot_bytes,
                        md[wk.mat].W + int64_t(wk.row - md[wk.mat].row_start) * B.row_bytes, bytes, &full[s],
                        policy);
          wk.row += nrows;
          issued = ++j;
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // never leave with a copy in flight: wait for the last use of each slot
      for (int s = 0; s < min(S, issued); ++s) {
        const int last = s + S * ((issued - 1 - s) / S);
        if (!mbar_wait_bounded(&full[s], uint32_t((last / S) & 1), kSeqDrainLimit)) atomicOr(a.err, kErrTimeout);
      }
    }
  } else if (warp >= kSqConsumers) {
    // ------------------------------------------------------- record copier --
    // The x warps copy the records of every batch whose records come from
    // the workspace into the record buffers, up to nrec - 1 batches ahead of
    // the consumers, with 16-byte loads through L2 (not bulk copies: the
    // SM's bulk-copy unit, which streams the weights, takes a fixed time per
    // copy, and short batches would double its copies). Copier warp w
    // copies the CTA's batches k with k mod kCopyWarps == w, so that the
    // copies of several batches are in flight at once; as nrec is a multiple
    // of kCopyWarps, every record buffer is filled by one warp only, in the
    // order of its uses, so that a parity wait on its release is never more
    // than one phase ahead. The other batches are quantized by the consumers
    // themselves.
    const int xw = warp - kSqConsumers;
    bool ok = a.pre_blocks == 0;
    if (!ok) {
      int w = 1;
      if (lane == 0) w = seq_count_wait(a, a.sync + 1, cta_abort);
      ok = __shfl_sync(kFull, w, 0) != 0;
      __syncwarp();  // the other lanes' loads follow lane 0's acquire
    }
    for (int g = 0, k = 0; g < a.n_groups && ok && xw < kCopyWarps; ++g) {
      const BatchDesc &d = bd[g];
      const int r0 = rr[g].x, r1 = rr[g].y;
      if (r0 >= r1) continue;  // no rows here: nothing read, nothing written
      const int b = int(uint32_t(k) & rmask);
      const int use = k >> a.nrec_log2;
      const bool mine = k % kCopyWarps == xw;
      ++k;
      if (!mine) continue;
      // the buffer's previous batch is done once its consumers released it;
      // waited for also before a batch the consumers fill themselves, so that
      // this warp is never two phases ahead of the buffer's release barrier
      if (use > 0 && !seq_wait(a, &rempty[b], uint32_t((use - 1) & 1), cta_abort)) break;
      if (d.rec_off < 0) continue;
      const int n16 = (d.K / 256) * (kXRecBytes / 16);
      const uint4 *src = reinterpret_cast<const uint4 *>(a.rec + d.rec_off);
      uint4 *dst = reinterpret_cast<uint4 *>(smem + size_t(b) * a.xrec_bytes);
      int i = lane;
      for (; i + 3 * 32 < n16; i += 4 * 32) {  // four loads in flight per lane
        const uint4 v0 = __ldcg(src + i), v1 = __ldcg(src + i + 32), v2 = __ldcg(src + i + 64),
                    v3 = __ldcg(src + i + 96);
        dst[i] = v0;
        dst[i + 32] = v1;
        dst[i + 64] = v2;
        dst[i + 96] = v3;
      }
      for (; i < n16; i += 32) dst[i] = __ldcg(src + i);
      mbar_arrive(&rfull[b]);  // release: this lane's stores before the consumers' wait
    }
  } else {
    // --------------------------------------------------------- consumers --
    // ngroups groups of gw warps take the stages in turn (stage j: group
    // j mod ngroups); within a stage every warp of the group takes its rows,
    // as in the per-launch kernel, so that a stage is consumed by its whole
    // group at once and released once.
    const int gw = kSqConsumers / a.ngroups;
    const int cg = warp / gw;  // consumer group
    const int cw = warp % gw;  // warp within the group
    const int gmask = a.ngroups - 1;
    bool skip = false;  // a wait ran out: walk on without waiting or computing
    int j = 0, s = 0;   // stage index (the producer's numbering), its ring slot
    uint32_t ph = 0;    // (j / S) & 1
    uint32_t nq = 0;    // bit b: parity of the copies into buffer b so far (phases of rfull)
    for (int g = 0, k = 0; g < a.n_groups; ++g) {
      const Batch<TYPE> B(bd[g]);
      const int r0 = rr[g].x, r1 = rr[g].y;
      if (r0 < r1) {
        const int b = int(uint32_t(k) & rmask);
        if (SKIP && seq_batch_skippable(a, bd[g], js[g]) && !seq_group_owns(a, js[g], cg)) {
          // no stage of this batch for this group: step over its stages. The
          // group still waits for the batch's records and releases the buffer
          // like every other batch, so that the record copies never run more
          // than one use of a buffer ahead of any group (a later parity wait
          // on the buffer then cannot alias).
          if (!skip) skip = !seq_wait(a, &rfull[b], (nq >> b) & 1u, cta_abort);
          nq ^= 1u << b;
          j += js[g].y;
          for (s += js[g].y; s >= S; s -= S) ph ^= 1u;
          __syncwarp();
          if (!skip && lane == 0) mbar_arrive(&rempty[b]);
          ++k;
          continue;
        }
        if (B.rec_off < 0) {
          // x quantized here by all consumer threads: a batch that waits for
          // an earlier one (batch wait_on's outputs are, or overlap, its x, or
          // its outputs overwrite wait_on's x), once every CTA has finished
          // that batch; or one of the launch's first batches, whose records
          // the start-of-launch quantization has not produced yet. The
          // buffer's last batch (k - nrec) is done: the consumers run the
          // batches in order.
          if (threadIdx.x == 0)
            s_go = (!skip && (B.wait_on < 0 || seq_batch_wait(a, B.wait_on, cta_abort))) ? 1 : 0;
          named_bar_sync(kBarConsumers, kSqConsumers * 32);
          if (!s_go) skip = true;
          if (!skip)  // read past L1: x may have been written by other CTAs during this launch
            quantize_x_records_2lane(B.x, B.K / kQK, reinterpret_cast<uint32_t *>(smem + b * a.xrec_bytes),
                                     threadIdx.x, kSqConsumers * 32);
          // the records are written, and s_go is read before it is rewritten
          named_bar_sync(kBarConsumers, kSqConsumers * 32);
        } else {
          if (!skip) skip = !seq_wait(a, &rfull[b], (nq >> b) & 1u, cta_abort);
          nq ^= 1u << b;
        }
        const uint32_t *xr = reinterpret_cast<const uint32_t *>(smem + b * a.xrec_bytes);
        const int L = B.lanes, rpw = 32 >> B.lanes_log2;
        const int lr = lane >> B.lanes_log2;  // row (within the warp's pass) handled by this lane
        const int gl = lane & (L - 1);        // first group of that row handled by this lane
        StageWalk wk{};
        wk.begin(md, B, r0, r1);
        while (wk.row < r1) {
          const int nrows = wk.next(md);
          if ((j & gmask) == cg) {
            // every warp of the group consumes every stage of the group in
            // order, so a parity wait is never more than one phase ahead
            if (!skip) skip = !seq_wait(a, &full[s], ph, cta_abort);
            if (!skip) {
              float *yp = md[wk.mat].y + (wk.row - md[wk.mat].row_start);
              const uint8_t *stage = ring + size_t(s) * a.slot_bytes;
              for (int pr = cw * rpw; pr < nrows; pr += gw * rpw) {
                const int r = pr + lr;
                float acc = 0.0f;
                if (r < nrows) {
                  const uint8_t *rowp = stage + size_t(r) * B.row_bytes;
                  for (int q = gl; q < B.groups8; q += L) {
                    uint32_t w[GW];
                    const uint4 *src = reinterpret_cast<const uint4 *>(rowp + size_t(q) * GW * 4);
#pragma unroll
                    for (int c = 0; c < GW / 4; ++c) {
                      const uint4 u = src[c];
                      w[4 * c] = u.x;
                      w[4 * c + 1] = u.y;
                      w[4 * c + 2] = u.z;
                      w[4 * c + 3] = u.w;
                    }
                    acc = group_terms<TYPE>(w, xr + q * kXRecWords, acc);
                  }
                }
                for (int off = L >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
                if (gl == 0 && r < nrows) yp[r] = acc;
              }
            }
            __syncwarp();
            if (!skip && lane == 0) mbar_arrive(&empty[s]);
          }
          wk.row += nrows;
          ++j;
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        __syncwarp();
        if (!skip && lane == 0) mbar_arrive(&rempty[b]);
        ++k;
      }
      if (B.signal) {
        // every row of batch g (and of every earlier batch) this CTA owns is
        // written: count the CTA done with batch g, after a fence that makes
        // the consumers' stores visible to the whole GPU
        named_bar_sync(kBarConsumers, kSqConsumers * 32);
        if (threadIdx.x == 0 && !skip) {
          __threadfence();
          atomicAdd(a.sync + 2 + g, 1u);
        }
      }
    }
  }
  __syncthreads();
}

}  // namespace

namespace {

bool spans_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

template <int TYPE>
cudaError_t launch_seq_chunk(const std::vector<int> &groups, const std::vector<int> &mat0, const int *n_mats,
                             const uint8_t *const *W, float *const *y, const int64_t *M, const float *const *x,
                             const int64_t *K, unsigned *sync, const DeviceInfo *di, cudaStream_t stream) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  std::unique_ptr<SeqArgs> a(new SeqArgs{});
  const int n = int(groups.size());
  // Consumer groups: two of 8 warps, or four of 4 where the CTAs' share of a
  // batch is short (a stage then holds a few rows, and four stages in
  // progress instead of two hide their latency).
  int64_t wbytes = 0;
  for (int i = 0; i < n; ++i)
    for (int k = 0; k < n_mats[groups[i]]; ++k) wbytes += M[mat0[groups[i]] + k] * (K[groups[i]] / kQK) * BB;
  static const int forced_groups = tuning_value("BQ_GEMV_SEQ_GROUPS");  // read once per process
  int ngroups = wbytes < int64_t(n) * di->sm_count * (64 << 10) ? 4 : 2;
  if (forced_groups == 2 || forced_groups == 4) ngroups = forced_groups;
  const int gw = kSqConsumers / ngroups;
  const bool skip_idle = ngroups == 4;  // the kernel with the per-batch stage table
  // Per batch: the per-launch kernel's lanes per row (so that every row's
  // arithmetic is the same), and the bytes of one pass of a consumer group
  // (gw warps, 32 / lanes rows each).
  std::vector<int> lanes(n), row_bytes(n), pass_rows(n);
  int xrec_bytes = 0, max_row = 0, max_pass = 0;
  for (int i = 0; i < n; ++i) {
    const int gi = groups[i];
    const int groups8 = int(K[gi] / 256);
    int L = 1;
    while (L < groups8 && L < 32) L <<= 1;
    lanes[i] = L;
    row_bytes[i] = int(K[gi] / kQK) * BB;
    pass_rows[i] = gw * (32 / L);
    xrec_bytes = std::max(xrec_bytes, groups8 * kXRecBytes);
    max_row = std::max(max_row, row_bytes[i]);
    max_pass = std::max(max_pass, pass_rows[i] * row_bytes[i]);
  }
  xrec_bytes = (xrec_bytes + 127) / 128 * 128;
  // Record buffers: as many (2 .. kMaxRecBufs, a power of two) as fit in
  // 32 KB, so that short batches' records arrive several batches ahead.
  int nrec = 2;
  while (nrec < kMaxRecBufs && 2 * nrec * xrec_bytes <= (32 << 10)) nrec *= 2;
  // Shared memory: the record buffers, the ring, 2 (S + nrec) barriers and
  // the abort flag. A ring slot holds one pass of a consumer group (a single
  // large copy: the copy cost is per copy), capped so that the ring keeps at
  // least four stages; a batch whose pass does not fit takes the rows that do.
  const int reserve = 1024;  // per-CTA system reservation
  // descriptor tables of this launch (nm: matrices with rows)
  int nm_total = 0;
  for (int i = 0; i < n; ++i)
    for (int k = 0; k < n_mats[groups[i]]; ++k) nm_total += M[mat0[groups[i]] + k] > 0 ? 1 : 0;
  const int desc_bytes =
      (n * int(sizeof(BatchDesc)) + nm_total * int(sizeof(MatDesc)) + (skip_idle ? 2 : 1) * n * int(sizeof(int2)) +
       15) / 16 * 16;
  const int budget =
      std::min(di->smem_per_sm - reserve, di->max_smem_optin) - nrec * xrec_bytes - desc_bytes - 1024;
  static const int forced_slot = tuning_value("BQ_GEMV_SEQ_SLOT_BYTES");  // read once per process
  int slot = std::min(max_pass, budget / 4) / 16 * 16;
  if (forced_slot > 0) slot = (forced_slot + 15) / 16 * 16;
  if (slot < max_row) slot = (max_row + 15) / 16 * 16;
  // A multiple of ngroups: a ring slot then always serves the same consumer
  // group, which waits on it only for stages after the slot's previous one
  // (of the same group, so already consumed): parity waits stay one phase
  // ahead at most.
  const int stages = std::min(32, budget / slot) / ngroups * ngroups;
  if (stages < ngroups) return cudaErrorInvalidValue;  // slot <= budget / 4: does not happen
  a->n_groups = n;
  a->stages = stages;
  a->slot_bytes = slot;
  a->xrec_bytes = xrec_bytes;
  a->desc_bytes = desc_bytes;
  a->nrec = nrec;
  a->nrec_log2 = nrec == 2 ? 1 : nrec == 4 ? 2 : 3;
  a->ngroups = ngroups;
  a->sync = sync;
  a->rec = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(sync) + kSyncBytes);
  a->err = di->err_word;
  a->spin_limit = spin_limit();
  static const int forced_poll = tuning_value("BQ_GEMV_SEQ_POLL_NS");  // read once per process
  a->poll_ns = forced_poll > 0 ? uint32_t(forced_poll) : 0u;  // 0: suspend in the barrier unit
  int nm = 0;
  for (int i = 0; i < n; ++i) {
    const int gi = groups[i];
    BatchDesc &G = a->g[i];
    G.x = x[gi];
    G.K = uint16_t(K[gi]);
    G.first_mat = uint16_t(nm);
    G.wait_on = -1;
    G.lanes = uint8_t(lanes[i]);
    G.lanes_log2 = uint8_t(__builtin_ctz(unsigned(lanes[i])));
    const int pass_bytes = pass_rows[i] * row_bytes[i];
    G.stage_rows = uint16_t(pass_bytes <= slot ? pass_rows[i] * (slot / pass_bytes) : slot / row_bytes[i]);
    int rows = 0;
    for (int k = 0; k < n_mats[gi]; ++k) {
      const int mi = mat0[gi] + k;
      if (M[mi] == 0) continue;
      a->m[nm].W = W[mi];
      a->m[nm].y = y[mi];
      a->m[nm].row_start = rows;
      rows += int(M[mi]);
      ++nm;
    }
    G.n_mats = uint8_t(nm - G.first_mat);
    G.rows = rows;
  }
  a->n_mats = nm;
  // Orders that memory imposes: batch i waits for the latest earlier batch
  // whose outputs its x reads, or whose x its outputs overwrite. (Outputs
  // never overlap outputs; the ABI layer rejects that.)
  auto mat_rows = [&](const BatchDesc &B, int mi) {
    return (mi + 1 < B.first_mat + B.n_mats ? a->m[mi + 1].row_start : B.rows) - a->m[mi].row_start;
  };
  for (int i = 1; i < n; ++i) {
    const BatchDesc &G = a->g[i];
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(G.x), x1 = x0 + uintptr_t(G.K) * 4;
    for (int p = i - 1; p >= 0 && a->g[i].wait_on < 0; --p) {
      const BatchDesc &P = a->g[p];
      const uintptr_t px0 = reinterpret_cast<uintptr_t>(P.x), px1 = px0 + uintptr_t(P.K) * 4;
      bool dep = false;
      for (int mp = P.first_mat; mp < P.first_mat + P.n_mats && !dep; ++mp) {
        const uintptr_t y0 = reinterpret_cast<uintptr_t>(a->m[mp].y);
        dep = spans_overlap(x0, x1, y0, y0 + uintptr_t(mat_rows(P, mp)) * 4);
      }
      for (int mi = G.first_mat; mi < G.first_mat + G.n_mats && !dep; ++mi) {
        const uintptr_t y0 = reinterpret_cast<uintptr_t>(a->m[mi].y);
        dep = spans_overlap(px0, px1, y0, y0 + uintptr_t(mat_rows(G, mi)) * 4);
      }
      if (dep) {
        a->g[i].wait_on = int16_t(p);
        a->g[p].signal = 1;
      }
    }
  }
  // x of every batch that waits for nothing is quantized once at the start
  // of the launch, in batch order, into the records area of the workspace
  // (but the first batch, which every CTA quantizes itself while the grid
  // quantizes the rest)
  const int n_local = std::min(n, 1);
  int rec_words = 0, blocks = 0;
  for (int i = 0; i < n; ++i) {
    BatchDesc &G = a->g[i];
    G.rec_off = -1;
    G.blk0 = blocks;
    if (G.wait_on >= 0 || i < n_local) continue;
    G.rec_off = rec_words;
    rec_words += (G.K / 256) * kXRecWords;
    blocks += G.K / kQK;
  }
  a->pre_blocks = blocks;
  a->n_local = n_local;
  const size_t smem = size_t(nrec) * xrec_bytes + size_t(stages) * slot + size_t(desc_bytes) +
                     8 * (2 * size_t(stages) + 2 * size_t(nrec)) + 16;
  const void *fn = skip_idle ? reinterpret_cast<const void *>(k_gemv_seq<TYPE, true>)
                             : reinterpret_cast<const void *>(k_gemv_seq<TYPE, false>);
  cudaError_t e = ensure_smem(fn, int(smem));
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(sync, 0, sizeof(unsigned) * size_t(2 + n), stream)) != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(di->sm_count));
  cfg.blockDim = dim3(kSqThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return skip_idle ? cudaLaunchKernelEx(&cfg, k_gemv_seq<TYPE, true>, *a)
                   : cudaLaunchKernelEx(&cfg, k_gemv_seq<TYPE, false>, *a);
}

template <int TYPE>
cudaError_t launch_seq_typed(int n_groups, const int *n_mats, const uint8_t *const *W, float *const *y,
                             const int64_t *M, const float *const *x, const int64_t *K, unsigned *sync,
                             cudaStream_t stream) {
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  std::vector<int> mat0(size_t(n_groups) + 1, 0);
  for (int gi = 0; gi < n_groups; ++gi) mat0[gi + 1] = mat0[gi] + n_mats[gi];
  // batches in order, cut into launches of at most kSeqMaxGroups batches and
  // kSeqMaxMats matrices (the stream orders the launches); batches without
  // rows are left out
  std::vector<int> chunk;
  int chunk_mats = 0;
  for (int gi = 0; gi <= n_groups; ++gi) {
    int mats = 0;
    if (gi < n_groups)
      for (int k = 0; k < n_mats[gi]; ++k) mats += M[mat0[gi] + k] > 0 ? 1 : 0;
    const bool flush = gi == n_groups || int(chunk.size()) == kSeqMaxGroups || chunk_mats + mats > kSeqMaxMats;
    if (flush && !chunk.empty()) {
      cudaError_t e = launch_seq_chunk<TYPE>(chunk, mat0, n_mats, W, y, M, x, K, sync, di, stream);
      if (e != cudaSuccess) return e;
      chunk.clear();
      chunk_mats = 0;
    }
    if (gi < n_groups && mats > 0) {
      chunk.push_back(gi);
      chunk_mats += mats;
    }
  }
  return cudaSuccess;
}

}  // namespace

size_t gemv_seq_workspace_bytes() { return kSyncBytes + kRecBytesMax; }

cudaError_t launch_gemv_seq(int type, int n_groups, const int *n_mats, const uint8_t *const *W, float *const *y,
                            const int64_t *M, const float *const *x, const int64_t *K, unsigned *sync,
                            cudaStream_t stream) {
  if (type == kTypeQ4_0) return launch_seq_typed<kTypeQ4_0>(n_groups, n_mats, W, y, M, x, K, sync, stream);
  return launch_seq_typed<kTypeQ8_0>(n_groups, n_mats, W, y, M, x, K, sync, stream);
}

}  // namespace bq
