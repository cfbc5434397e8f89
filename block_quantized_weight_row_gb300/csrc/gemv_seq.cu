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
constexpr int kSqGroupWarps = 8;  // consumer warps per group (two groups take the stages in turn)
constexpr int kSqXWarps = 3;      // quantize x at the start; then one lane copies records (20 warps: 96 registers)
constexpr int kSqProducer = kSqConsumers + kSqXWarps;  // warp index of the producer
constexpr int kSqThreads = (kSqConsumers + kSqXWarps + 1) * 32;
constexpr int kSeqMaxGroups = 256;  // per launch; longer runs take several launches
constexpr int kSeqMaxMats = 512;
constexpr uint32_t kSeqDrainLimit = 1u << 26;
constexpr int kRowRotation = 37;  // CTA range rotation per batch
constexpr int kBarConsumers = 1;  // named barrier of the consumer warps
constexpr int kBarPre = 2;        // named barrier of the warps that quantize x before the stream
constexpr int kPreThreads = (kSqConsumers + kSqXWarps) * 32;
constexpr int kMaxRecBufs = 8;    // record buffers in shared memory
constexpr int kSyncWords = 2 + kSeqMaxGroups;  // abort flag, CTAs done quantizing, CTAs done per batch
constexpr size_t kSyncBytes = (kSyncWords * 4 + 255) / 256 * 256;
constexpr size_t kRecBytesMax = size_t(kSeqMaxGroups) * (BQ_GEMV_SEQ_MAX_K / 256) * kXRecBytes;
#ifndef SEQ_POLL_NS
#define SEQ_POLL_NS 32  // sleep between polls of a mbarrier
#endif

struct SeqGroup {
  const float *x;
  int K;           // a multiple of 256
  int first_mat;   // matrices first_mat .. first_mat + n_mats - 1 of SeqArgs::m
  int n_mats;
  int rows;        // rows of all the batch's matrices
  int wait_on;     // batch (of this launch) every CTA must have finished first, or -1
  int signal;      // nonzero: a later batch waits for this one
  int groups8;     // K / 256 groups of 8 blocks per row
  int lanes;       // lanes per row: the power of two <= 32 the per-launch kernel takes
  int row_bytes;
  int stage_rows;  // rows per stage: one pass of a consumer group's warps, as the ring slot allows
  int rec_off;     // words: x's records in SeqArgs::rec (batches that wait for nothing), else -1
  int blk0;        // first block of x in the launch's quantization order (rec_off >= 0)
};

struct SeqMat {
  const uint8_t *W;
  float *y;
  int row_start;  // first row of this matrix within its batch
  int pad;
};

struct SeqArgs {
  SeqGroup g[kSeqMaxGroups];
  SeqMat m[kSeqMaxMats];
  int n_groups;
  int stages;
  int slot_bytes;  // bytes of one ring stage
  int xrec_bytes;  // bytes of one record buffer (the largest K of the launch)
  int nrec;        // record buffers in shared memory: a power of two, 2..kMaxRecBufs
  int pre_blocks;  // blocks of x quantized at the start (every batch with rec_off >= 0)
  uint32_t *rec;   // x's records of those batches (global memory)
  unsigned *sync;  // [0]: abort flag, [1]: CTAs done quantizing, [2 + g]: CTAs done with batch g; zeroed
  unsigned *err;
  uint32_t spin_limit;
};

// Rows [r0, r1) of batch g taken by this CTA.
__device__ __forceinline__ void cta_rows(int rows, int g, int &r0, int &r1) {
  const int G = int(gridDim.x);
  const int p = int((blockIdx.x + unsigned(g) * kRowRotation) % unsigned(G));
  r0 = int(int64_t(rows) * p / G);
  r1 = int(int64_t(rows) * (p + 1) / G);
}

// Stages of one batch's row range in order: each at most stage_rows rows,
// never past the range or a matrix's end. Producer and consumers walk the
// same sequence (incrementally: no division per stage).
struct StageWalk {
  int row, r1, mat, mat_end, last;
  __device__ __forceinline__ void begin(const SeqArgs &a, const SeqGroup &G, int r0, int r1_) {
    row = r0;
    r1 = r1_;
    mat = G.first_mat;
    last = G.first_mat + G.n_mats - 1;
    while (mat < last && row >= a.m[mat + 1].row_start) ++mat;
    mat_end = mat < last ? a.m[mat + 1].row_start : G.rows;
  }
  // rows of the stage that starts at `row` (row < r1)
  __device__ __forceinline__ int next(const SeqArgs &a, const SeqGroup &G) {
    if (row >= mat_end) {
      ++mat;
      mat_end = mat < last ? a.m[mat + 1].row_start : G.rows;
    }
    return min(min(G.stage_rows, r1 - row), mat_end - row);
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
// another role of the CTA gave up. Polls never suspend in the barrier unit
// (whose wake-up comes long after the phase completes: with a handoff per
// stage that latency, not the work, set the pace); between polls the warp
// sleeps briefly so that waiting warps leave the issue slots to working ones.
// Only the CTA's own flag (shared memory) is read here: these barriers depend
// on this CTA's roles alone, which all end; the grid-wide flag is read where a
// CTA waits for other CTAs.
__device__ __forceinline__ bool seq_wait(const SeqArgs &a, uint64_t *bar, uint32_t parity, volatile int *cta_abort) {
  for (uint32_t i = 0; i < a.spin_limit; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if (SEQ_POLL_NS > 0) __nanosleep(SEQ_POLL_NS);
    if ((i & 63) == 63 && *cta_abort) return false;
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

// Quantize this CTA's share of x's blocks of every batch that waits for
// nothing (the launch's blocks in batch order, cut evenly over the CTAs) into
// the global records: two threads per block (quantize_block_pair), so the
// records are those of the per-launch kernels. tid < kPreThreads.
__device__ __forceinline__ void seq_prequantize(const SeqArgs &a, int tid) {
  const int G = int(gridDim.x);
  const int lo = int(int64_t(a.pre_blocks) * blockIdx.x / G);
  const int hi = int(int64_t(a.pre_blocks) * (blockIdx.x + 1) / G);
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
      while (a.g[g].rec_off < 0 || i >= a.g[g].blk0 + a.g[g].K / kQK) ++g;
      const int bl = i - a.g[g].blk0;
      const float4 *src = reinterpret_cast<const float4 *>(a.g[g].x + int64_t(bl) * kQK + 16 * h);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 v = __ldcg(src + c);
        f[4 * c] = v.x;
        f[4 * c + 1] = v.y;
        f[4 * c + 2] = v.z;
        f[4 * c + 3] = v.w;
      }
      rg = a.rec + a.g[g].rec_off + (bl >> 3) * kXRecWords;
      jb = bl & 7;
    }
    gemv::quantize_block_pair(f, h, rg, jb, valid);
  }
}

template <int TYPE>
__global__ void __launch_bounds__(kSqThreads, 1) k_gemv_seq(const __grid_constant__ SeqArgs a) {
  constexpr int GW = GroupWords<TYPE>::kWords;
  extern __shared__ __align__(128) uint8_t smem[];
  // record buffer b at smem + b * xrec_bytes, b < nrec
  uint8_t *ring = smem + size_t(a.nrec) * a.xrec_bytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(ring + size_t(a.stages) * a.slot_bytes);
  uint64_t *empty = full + a.stages;
  uint64_t *rfull = empty + a.stages;  // [nrec]: records of buffer b in place
  uint64_t *rempty = rfull + a.nrec;   // [nrec]: records of buffer b no longer read
  volatile int *cta_abort = reinterpret_cast<volatile int *>(rempty + a.nrec);
  const uint32_t rmask = uint32_t(a.nrec - 1);
  __shared__ int s_go;  // dependency wait result, broadcast to the consumer warps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSqGroupWarps);  // every warp of the stage's consumer group releases it
    }
    for (int b = 0; b < a.nrec; ++b) {
      mbar_init(&rfull[b], 1);  // the record copier (bytes on the transaction count)
      mbar_init(&rempty[b], kSqConsumers);
    }
    *cta_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp != kSqProducer && a.pre_blocks > 0) {
    // x of every batch that waits for nothing, quantized once for the whole
    // grid while the producer already streams weights; then this CTA counts
    // itself done (release: the records are visible to the whole GPU)
    seq_prequantize(a, threadIdx.x);
    named_bar_sync(kBarPre, kPreThreads);
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(a.sync + 1, 1u);
    }
  }

  if (warp == kSqProducer) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      int issued = 0;
      const uint64_t policy = l2_evict_first_policy();  // every weight is read once
      bool stop = false;
      int j = 0, s = 0;  // stage index, its ring slot
      uint32_t ph = 0;   // (j / S) & 1
      for (int g = 0; g < a.n_groups && !stop; ++g) {
        const SeqGroup &G = a.g[g];
        int r0, r1;
        cta_rows(G.rows, g, r0, r1);
        if (r0 >= r1) continue;
        StageWalk wk;
        wk.begin(a, G, r0, r1);
        while (wk.row < r1) {
          // the slot's previous use (stage j - S) must have been released
          if (j >= S && !seq_wait(a, &empty[s], ph ^ 1u, cta_abort)) {
            stop = true;
            break;
          }
          const int nrows = wk.next(a, G);
          const uint32_t bytes = uint32_t(nrows) * uint32_t(G.row_bytes);
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_g2s_hint(ring + size_t(s) * a.slot_bytes,
                        a.m[wk.mat].W + int64_t(wk.row - a.m[wk.mat].row_start) * G.row_bytes, bytes, &full[s],
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
    // One lane copies the records of every batch that waits for nothing from
    // global memory into the record buffers, up to nrec - 1 batches ahead of
    // the consumers (1-D bulk copies completing on rfull). A batch that waits
    // for an earlier one is quantized by the consumers themselves once the
    // wait is over (they are idle then).
    if (warp == kSqConsumers && lane == 0) {
      bool ok = a.pre_blocks == 0 || seq_count_wait(a, a.sync + 1, cta_abort);
      // the records were written by other threads' ordinary stores; the
      // copies read them through the asynchronous proxy
      asm volatile("fence.proxy.async.global;" ::: "memory");
      uint32_t used = 0, par = 0;  // buffers copied into; parity of each one's last copy
      for (int g = 0, k = 0; g < a.n_groups && ok; ++g) {
        const SeqGroup &G = a.g[g];
        int r0, r1;
        cta_rows(G.rows, g, r0, r1);
        if (r0 >= r1) continue;  // no rows here: nothing read, nothing written
        const int b = int(uint32_t(k) & rmask);
        const int use = k / a.nrec;
        ++k;
        if (G.rec_off < 0) continue;
        // the buffer's previous batch is done once its consumers released it
        if (use > 0 && !seq_wait(a, &rempty[b], uint32_t((use - 1) & 1), cta_abort)) break;
        const uint32_t bytes = uint32_t(G.K / 256) * kXRecBytes;
        mbar_arrive_expect_tx(&rfull[b], bytes);
        bulk_g2s(smem + size_t(b) * a.xrec_bytes, a.rec + G.rec_off, bytes, &rfull[b]);
        used |= 1u << b;
        par = (par & ~(1u << b)) | (uint32_t(use & 1) << b);
      }
      // never leave with a copy in flight
      for (int b = 0; b < a.nrec; ++b)
        if (((used >> b) & 1u) && !mbar_wait_bounded(&rfull[b], (par >> b) & 1u, kSeqDrainLimit))
          atomicOr(a.err, kErrTimeout);
    }
  } else {
    // --------------------------------------------------------- consumers --
    // Two groups of kSqGroupWarps warps take the stages in turn (stage j:
    // group j & 1); within a stage every warp of the group takes its rows,
    // as in the per-launch kernel, so that a stage is consumed by its whole
    // group at once and released once.
    const int cg = warp / kSqGroupWarps;  // consumer group
    const int cw = warp % kSqGroupWarps;  // warp within the group
    bool skip = false;  // a wait ran out: walk on without waiting or computing
    int j = 0, s = 0;   // stage index (the producer's numbering), its ring slot
    uint32_t ph = 0;    // (j / S) & 1
    uint32_t nq = 0;    // bit b: parity of the copies into buffer b so far (phases of rfull)
    for (int g = 0, k = 0; g < a.n_groups; ++g) {
      const SeqGroup &G = a.g[g];
      int r0, r1;
      cta_rows(G.rows, g, r0, r1);
      if (r0 < r1) {
        const int b = int(uint32_t(k) & rmask);
        if (G.wait_on >= 0) {
          // batch wait_on's outputs are (or overlap) this batch's x, or this
          // batch's outputs overwrite its x: once every CTA has finished it,
          // all consumer threads quantize x into the buffer (its last batch,
          // k - 2, is done: the consumers run the batches in order)
          if (threadIdx.x == 0) s_go = (!skip && seq_batch_wait(a, G.wait_on, cta_abort)) ? 1 : 0;
          named_bar_sync(kBarConsumers, kSqConsumers * 32);
          if (!s_go) skip = true;
          if (!skip)  // read past L1: x was written by other CTAs during this launch
            quantize_x_records_2lane(G.x, G.K / kQK, reinterpret_cast<uint32_t *>(smem + b * a.xrec_bytes),
                                     threadIdx.x, kSqConsumers * 32);
          // the records are written, and s_go is read before it is rewritten
          named_bar_sync(kBarConsumers, kSqConsumers * 32);
        } else {
          if (!skip) skip = !seq_wait(a, &rfull[b], (nq >> b) & 1u, cta_abort);
          nq ^= 1u << b;
        }
        const uint32_t *xr = reinterpret_cast<const uint32_t *>(smem + b * a.xrec_bytes);
        const int L = G.lanes, rpw = 32 / L;
        const int rr = lane / L;  // row (within the warp's pass) handled by this lane
        const int gl = lane % L;  // first group of that row handled by this lane
        StageWalk wk;
        wk.begin(a, G, r0, r1);
        while (wk.row < r1) {
          const int nrows = wk.next(a, G);
          if ((j & 1) == cg) {
            // every warp of the group consumes every stage of the group in
            // order, so a parity wait is never more than one phase ahead
            if (!skip) skip = !seq_wait(a, &full[s], ph, cta_abort);
            if (!skip) {
              float *yp = a.m[wk.mat].y + (wk.row - a.m[wk.mat].row_start);
              const uint8_t *stage = ring + size_t(s) * a.slot_bytes;
              for (int pr = cw * rpw; pr < nrows; pr += kSqGroupWarps * rpw) {
                const int r = pr + rr;
                float acc = 0.0f;
                if (r < nrows) {
                  const uint8_t *rowp = stage + size_t(r) * G.row_bytes;
                  for (int q = gl; q < G.groups8; q += L) {
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
      if (G.signal) {
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

// One launch over the batches `groups` (each with K % 256 == 0 and rows > 0).
template <int TYPE>
cudaError_t launch_seq_chunk(const std::vector<int> &groups, const std::vector<int> &mat0, const int *n_mats,
                             const uint8_t *const *W, float *const *y, const int64_t *M, const float *const *x,
                             const int64_t *K, unsigned *sync, const DeviceInfo *di, cudaStream_t stream) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  std::unique_ptr<SeqArgs> a(new SeqArgs{});
  const int n = int(groups.size());
  // Per batch: the per-launch kernel's lanes per row (so that every row's
  // arithmetic is the same), and the bytes of one pass of a consumer group
  // (kSqGroupWarps warps, 32 / lanes rows each).
  std::vector<int> lanes(n), row_bytes(n), pass_rows(n);
  int xrec_bytes = 0, max_row = 0, max_pass = 0;
  for (int i = 0; i < n; ++i) {
    const int gi = groups[i];
    const int groups8 = int(K[gi] / 256);
    int L = 1;
    while (L < groups8 && L < 32) L <<= 1;
    lanes[i] = L;
    row_bytes[i] = int(K[gi] / kQK) * BB;
    pass_rows[i] = kSqGroupWarps * (32 / L);
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
  const int budget = std::min(di->smem_per_sm - reserve, di->max_smem_optin) - nrec * xrec_bytes - 1024;
  static const int forced_slot = tuning_value("BQ_GEMV_SEQ_SLOT_BYTES");  // read once per process
  int slot = std::min(max_pass, budget / 4) / 16 * 16;
  if (forced_slot > 0) slot = (forced_slot + 15) / 16 * 16;
  if (slot < max_row) slot = (max_row + 15) / 16 * 16;
  const int stages = std::min(32, budget / slot);
  if (stages < 2) return cudaErrorInvalidValue;  // the ABI layer bounds K, so this does not happen
  a->n_groups = n;
  a->stages = stages;
  a->slot_bytes = slot;
  a->xrec_bytes = xrec_bytes;
  a->nrec = nrec;
  a->sync = sync;
  a->rec = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(sync) + kSyncBytes);
  a->err = di->err_word;
  a->spin_limit = spin_limit();
  int nm = 0;
  for (int i = 0; i < n; ++i) {
    const int gi = groups[i];
    SeqGroup &G = a->g[i];
    G.x = x[gi];
    G.K = int(K[gi]);
    G.first_mat = nm;
    G.wait_on = -1;
    G.groups8 = G.K / 256;
    G.lanes = lanes[i];
    G.row_bytes = row_bytes[i];
    const int pass_bytes = pass_rows[i] * row_bytes[i];
    G.stage_rows = pass_bytes <= slot ? pass_rows[i] * (slot / pass_bytes) : slot / row_bytes[i];
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
    G.n_mats = nm - G.first_mat;
    G.rows = rows;
  }
  // Orders that memory imposes: batch i waits for the latest earlier batch
  // whose outputs its x reads, or whose x its outputs overwrite. (Outputs
  // never overlap outputs; the ABI layer rejects that.)
  for (int i = 1; i < n; ++i) {
    const SeqGroup &G = a->g[i];
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(G.x), x1 = x0 + uintptr_t(G.K) * 4;
    for (int p = i - 1; p >= 0 && a->g[i].wait_on < 0; --p) {
      const SeqGroup &P = a->g[p];
      const uintptr_t px0 = reinterpret_cast<uintptr_t>(P.x), px1 = px0 + uintptr_t(P.K) * 4;
      bool dep = false;
      for (int mp = P.first_mat; mp < P.first_mat + P.n_mats && !dep; ++mp) {
        const uintptr_t y0 = reinterpret_cast<uintptr_t>(a->m[mp].y);
        const int rows = (mp + 1 < P.first_mat + P.n_mats ? a->m[mp + 1].row_start : P.rows) - a->m[mp].row_start;
        dep = spans_overlap(x0, x1, y0, y0 + uintptr_t(rows) * 4);
      }
      for (int mi = G.first_mat; mi < G.first_mat + G.n_mats && !dep; ++mi) {
        const uintptr_t y0 = reinterpret_cast<uintptr_t>(a->m[mi].y);
        const int rows = (mi + 1 < G.first_mat + G.n_mats ? a->m[mi + 1].row_start : G.rows) - a->m[mi].row_start;
        dep = spans_overlap(px0, px1, y0, y0 + uintptr_t(rows) * 4);
      }
      if (dep) {
        a->g[i].wait_on = p;
        a->g[p].signal = 1;
      }
    }
  }
  // x of every batch that waits for nothing is quantized once at the start
  // of the launch, in batch order, into the records area of the workspace
  int rec_words = 0, blocks = 0;
  for (int i = 0; i < n; ++i) {
    SeqGroup &G = a->g[i];
    G.rec_off = -1;
    G.blk0 = blocks;
    if (G.wait_on >= 0) continue;
    G.rec_off = rec_words;
    rec_words += G.groups8 * kXRecWords;
    blocks += G.K / kQK;
  }
  a->pre_blocks = blocks;
  const size_t smem =
      size_t(nrec) * xrec_bytes + size_t(stages) * slot + 8 * (2 * size_t(stages) + 2 * size_t(nrec)) + 16;
  const void *fn = reinterpret_cast<const void *>(k_gemv_seq<TYPE>);
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
  return cudaLaunchKernelEx(&cfg, k_gemv_seq<TYPE>, *a);
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
