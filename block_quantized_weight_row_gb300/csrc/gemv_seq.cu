// gemv_seq.cu — a sequence of decode GEMV batches in one persistent launch.
//
// A decode step is a chain of weight-matrix products, each bounded by the
// weight bytes it reads ("05. llama.cpp：从 GGUF 文件到本地推理服务",
// §性能直觉：带宽决定 Decode，算力决定 Prefill). Launched one batch at a time, the
// weight stream stops at every launch boundary: the next kernel's copies
// begin only after the previous one has drained and the new one has started
// and quantized its input. Here one launch covers the whole sequence and the
// stream does not stop:
//
//   - batch g has the semantics of one bq_gemv_multi call issued after the
//     calls of batches 0..g-1: its x is read only once every output of the
//     earlier batches has been written (x may be such an output). A
//     grid-wide barrier (a counter in global memory, bounded waits) separates
//     the batches for the consumer warps;
//   - the producer warp of every CTA has no such dependency (weights are
//     never written by the sequence) and keeps streaming the next batches'
//     rows into its shared-memory ring while the consumers wait at a barrier
//     and quantize the new x; the ring absorbs that pause;
//   - the consumer code (x's Q8_0 records, the group dot product) is the one
//     of the per-batch kernel, so the results are those of bq_gemv_multi.
// The launch is cooperative, so that every CTA of the grid is resident and
// the barrier cannot wait for a CTA that has not started. Every CTA takes a
// contiguous, balanced range of each batch's rows.
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
using gemv::quantize_x_records;

constexpr int kSeqConsumers = 8;  // consumer warps per CTA
constexpr int kSeqThreads = (kSeqConsumers + 1) * 32;
constexpr int kSeqMaxGroups = 256;  // per launch; longer sequences take several launches
constexpr int kSeqMaxMats = 512;
constexpr uint32_t kSeqDrainLimit = 1u << 26;

struct SeqGroup {
  const float *x;
  int K;              // a multiple of 256
  int first_mat;      // matrices first_mat .. first_mat + n_mats - 1 of SeqArgs::m
  int n_mats;
  int rows;           // rows of all the batch's matrices
  int groups8;        // K / 256: groups of 8 blocks per row
  int lanes_per_row;  // power of two <= 32
  int rows_per_warp;  // 32 / lanes_per_row
  int row_bytes;
  int stage_rows;     // rows per stage (stage_rows * row_bytes <= slot_bytes)
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
  int slot_bytes;
  int xrec_bytes;       // records of the largest K of the sequence
  unsigned *sync;       // [0]: CTAs done with a batch (counts up), [1]: abort; zeroed before the launch
  unsigned *err;
  uint32_t spin_limit;
};

// Stage sequence of one CTA over every batch: rows [r0, r1) of batch g in
// stages that never straddle two matrices. Producer and consumers walk it in
// the same order.
struct SeqCursor {
  int g, row, r1;
  __device__ __forceinline__ void start(const SeqArgs &a, int gg) {
    g = gg;
    for (; g < a.n_groups; ++g) {
      const int rows = a.g[g].rows;
      row = int(int64_t(rows) * blockIdx.x / gridDim.x);
      r1 = int(int64_t(rows) * (blockIdx.x + 1) / gridDim.x);
      if (row < r1) return;
    }
  }
  // matrix and row count of the stage at the cursor
  __device__ __forceinline__ void stage(const SeqArgs &a, int &mat, int &nrows) const {
    const SeqGroup &G = a.g[g];
    mat = G.first_mat;
    while (mat + 1 < G.first_mat + G.n_mats && row >= a.m[mat + 1].row_start) ++mat;
    const int mat_end = (mat + 1 < G.first_mat + G.n_mats) ? a.m[mat + 1].row_start : G.rows;
    nrows = min(min(G.stage_rows, r1 - row), mat_end - row);
  }
  __device__ __forceinline__ void advance(const SeqArgs &a, int nrows) {
    row += nrows;
    if (row >= r1) start(a, g + 1);
  }
};

__device__ __forceinline__ bool seq_aborted(const SeqArgs &a, volatile int *cta_abort) {
  return *cta_abort || *reinterpret_cast<volatile unsigned *>(a.sync + 1);
}

__device__ __forceinline__ void seq_abort(const SeqArgs &a, volatile int *cta_abort) {
  *cta_abort = 1;
  atomicExch(a.sync + 1, 1u);
  atomicOr(a.err, kErrTimeout);
}

// Bounded mbarrier wait that gives up early once the CTA or the grid aborted.
__device__ __forceinline__ bool seq_wait(const SeqArgs &a, uint64_t *bar, uint32_t parity, volatile int *cta_abort) {
  for (uint32_t i = 0; i < a.spin_limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15) == 15 && seq_aborted(a, cta_abort)) return false;
  }
  seq_abort(a, cta_abort);
  return false;
}

// Until `target` CTAs have arrived at the grid counter (acquire), bounded.
__device__ __forceinline__ bool seq_grid_wait(const SeqArgs &a, unsigned target, volatile int *cta_abort) {
  for (uint32_t i = 0; i < a.spin_limit; ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.sync) : "memory");
    if (v >= target) return true;
    if (seq_aborted(a, cta_abort)) return false;
    __nanosleep(32);
  }
  seq_abort(a, cta_abort);
  return false;
}

template <int TYPE>
__global__ void __launch_bounds__(kSeqThreads, 2) k_gemv_seq(const __grid_constant__ SeqArgs a) {
  constexpr int GW = GroupWords<TYPE>::kWords;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_go;
  uint32_t *xrec = reinterpret_cast<uint32_t *>(smem);
  uint8_t *ring = smem + a.xrec_bytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(ring + size_t(a.stages) * a.slot_bytes);
  uint64_t *empty = full + a.stages;
  volatile int *cta_abort = reinterpret_cast<volatile int *>(empty + a.stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSeqConsumers);  // every consumer warp releases every stage
    }
    *cta_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kSeqConsumers) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      int issued = 0;
      const uint64_t policy = l2_evict_first_policy();  // every weight is read once
      SeqCursor cur;
      cur.start(a, 0);
      for (int j = 0; cur.g < a.n_groups; ++j) {
        const int s = j % S;
        if (j >= S && !seq_wait(a, &empty[s], uint32_t((j / S - 1) & 1), cta_abort)) break;
        int mat, nrows;
        cur.stage(a, mat, nrows);
        const int row_bytes = a.g[cur.g].row_bytes;
        const uint32_t bytes = uint32_t(nrows) * uint32_t(row_bytes);
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s_hint(ring + size_t(s) * a.slot_bytes,
                      a.m[mat].W + int64_t(cur.row - a.m[mat].row_start) * row_bytes, bytes, &full[s], policy);
        cur.advance(a, nrows);
        issued = j + 1;
      }
      // never leave with a copy in flight: wait for the last use of each slot
      for (int s = 0; s < min(S, issued); ++s) {
        const int last = s + S * ((issued - 1 - s) / S);
        if (!mbar_wait_bounded(&full[s], uint32_t((last / S) & 1), kSeqDrainLimit)) atomicOr(a.err, kErrTimeout);
      }
    }
  } else {
    // --------------------------------------------------------- consumers --
    const int tid = threadIdx.x;
    SeqCursor cur;
    cur.start(a, 0);
    int j = 0;  // stage index, the producer's numbering
    bool skip = false;
    for (int g = 0; g < a.n_groups; ++g) {
      if (g > 0) {
        // every CTA has finished batch g-1, so its outputs (which this
        // batch's x may be) are written and visible
        if (tid == 0) {
          const bool ok = !skip && seq_grid_wait(a, unsigned(g) * gridDim.x, cta_abort);
          if (ok) __threadfence();
          s_go = ok ? 1 : 0;
        }
        named_bar_sync(1, kSeqConsumers * 32);
        if (!s_go) break;  // uniform: written before the barrier, rewritten only after the next one
      }
      const SeqGroup &G = a.g[g];
      const bool mine = cur.g == g;  // this CTA has rows of batch g
      if (mine) {
        quantize_x_records(G.x, G.K / kQK, xrec, tid, kSeqConsumers * 32, int(blockIdx.x) * 8);
        named_bar_sync(1, kSeqConsumers * 32);
      }
      const int L = G.lanes_per_row;
      const int rr = lane / L;  // row (within the warp's pass) handled by this lane
      const int gl = lane % L;  // first group of that row handled by this lane
      while (cur.g == g) {
        const int s = j % S;
        if (!skip) {
          // every warp consumes every stage in order, so a parity wait is
          // never more than one phase ahead of the barrier; lane 0 waits
          int ok = 1;
          if (lane == 0) ok = seq_wait(a, &full[s], uint32_t((j / S) & 1), cta_abort);
          ok = __shfl_sync(kFull, ok, 0);
          __syncwarp();
          skip = !ok;
        }
        int mat, nrows;
        cur.stage(a, mat, nrows);
        if (!skip) {
          float *yp = a.m[mat].y + (cur.row - a.m[mat].row_start);
          const uint8_t *stage = ring + size_t(s) * a.slot_bytes;
          for (int pr = warp * G.rows_per_warp; pr < nrows; pr += kSeqConsumers * G.rows_per_warp) {
            const int row = pr + rr;
            float acc = 0.0f;
            if (row < nrows) {
              const uint8_t *rowp = stage + size_t(row) * G.row_bytes;
              for (int q = gl; q < G.groups8; q += L) {
                uint32_t w[GW];
                const uint4 *src = reinterpret_cast<const uint4 *>(rowp + size_t(q) * GW * 4);
#pragma unroll
                for (int k = 0; k < GW / 4; ++k) {
                  const uint4 u = src[k];
                  w[4 * k] = u.x;
                  w[4 * k + 1] = u.y;
                  w[4 * k + 2] = u.z;
                  w[4 * k + 3] = u.w;
                }
                acc = group_terms<TYPE>(w, xrec + q * kXRecWords, acc);
              }
            }
            for (int off = L >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
            if (gl == 0 && row < nrows) yp[row] = acc;
          }
        }
        cur.advance(a, nrows);
        __syncwarp();
        if (!skip && lane == 0) mbar_arrive(&empty[s]);
        ++j;
      }
      // every row of batch g this CTA owns is written, and x's records are free
      named_bar_sync(1, kSeqConsumers * 32);
      if (tid == 0 && g + 1 < a.n_groups && !skip) {
        __threadfence();
        atomicAdd(a.sync, 1u);
      }
    }
  }
  __syncthreads();
}

}  // namespace

namespace {

int pow2_at_least(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// One launch over batches [g0, g1) (all with K % 256 == 0 and rows > 0).
template <int TYPE>
cudaError_t launch_seq_chunk(const std::vector<int> &groups, const std::vector<int> &mat0, const int *n_mats,
                             const uint8_t *const *W, float *const *y, const int64_t *M, const float *const *x,
                             const int64_t *K, unsigned *sync, const DeviceInfo *di, cudaStream_t stream) {
  constexpr int BB = Fmt<TYPE>::kBytes;
  std::unique_ptr<SeqArgs> a(new SeqArgs{});
  int xrec_bytes = 0, max_row = 0, max_pass = 0;
  for (size_t i = 0; i < groups.size(); ++i) {
    const int gi = groups[i];
    const int groups8 = int(K[gi] / 256);
    const int row_bytes = int(K[gi] / kQK) * BB;
    const int L = std::min(32, pow2_at_least(groups8));
    xrec_bytes = std::max(xrec_bytes, groups8 * kXRecBytes);
    max_row = std::max(max_row, row_bytes);
    max_pass = std::max(max_pass, kSeqConsumers * (32 / L) * row_bytes);
  }
  xrec_bytes = (xrec_bytes + 127) / 128 * 128;
  // Two CTAs per SM (16 consumer warps): a ring of at least 3 stages within
  // half an SM; a stage is one pass of the consumer warps, cut to fit.
  const int reserve = 1024 + 128;  // per-CTA system reservation and static shared memory
  const int budget = std::min(di->smem_per_sm / 2 - reserve, di->max_smem_optin) - xrec_bytes - 256;
  int slot = std::min(max_pass, budget / 3) / 16 * 16;
  if (slot < max_row) return cudaErrorInvalidValue;  // the ABI layer bounds K, so this does not happen
  const int stages = std::min(8, budget / slot);
  a->n_groups = int(groups.size());
  a->stages = stages;
  a->slot_bytes = slot;
  a->xrec_bytes = xrec_bytes;
  a->sync = sync;
  a->err = di->err_word;
  a->spin_limit = spin_limit();
  int nm = 0;
  for (size_t i = 0; i < groups.size(); ++i) {
    const int gi = groups[i];
    SeqGroup &G = a->g[i];
    G.x = x[gi];
    G.K = int(K[gi]);
    G.groups8 = G.K / 256;
    G.lanes_per_row = std::min(32, pow2_at_least(G.groups8));
    G.rows_per_warp = 32 / G.lanes_per_row;
    G.row_bytes = (G.K / kQK) * BB;
    G.stage_rows = std::max(1, std::min(kSeqConsumers * G.rows_per_warp, slot / G.row_bytes));
    G.first_mat = nm;
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
  const size_t smem = size_t(xrec_bytes) + size_t(stages) * slot + 16 * size_t(stages) + 16;
  const void *fn = reinterpret_cast<const void *>(k_gemv_seq<TYPE>);
  cudaError_t e = ensure_smem(fn, int(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemv_seq<TYPE>, kSeqThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  per_sm = std::min(per_sm, 2);
  static const int forced = tuning_value("BQ_GEMV_SEQ_CTAS_PER_SM");  // read once per process
  if (forced) per_sm = std::min(per_sm, forced);
  if ((e = cudaMemsetAsync(sync, 0, 2 * sizeof(unsigned), stream)) != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(di->sm_count * per_sm));
  cfg.blockDim = dim3(kSeqThreads);
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
  // kSeqMaxMats matrices; batches without rows are left out
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

cudaError_t launch_gemv_seq(int type, int n_groups, const int *n_mats, const uint8_t *const *W, float *const *y,
                            const int64_t *M, const float *const *x, const int64_t *K, unsigned *sync,
                            cudaStream_t stream) {
  if (type == kTypeQ4_0) return launch_seq_typed<kTypeQ4_0>(n_groups, n_mats, W, y, M, x, K, sync, stream);
  return launch_seq_typed<kTypeQ8_0>(n_groups, n_mats, W, y, M, x, K, sync, stream);
}

}  // namespace bq
