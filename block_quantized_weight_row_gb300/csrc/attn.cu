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
// two per SM; one CTA takes a chunk and every head, and each token's K and V
// rows (contiguous over the kv heads in the cache layout) arrive by 1-D bulk
// copies into a shared-memory ring. Scores are kept in base-2 units
// (s * scale * log2 e) so that every exponential is one 2^x. Two chunk kernels:
//   k_attn_warp (n_kv in {1, 2, 4, 8}, head_dim * G <= 1024): one warp per kv
//     head with its own online softmax, no block-wide barrier per tile;
//   k_attn_chunk (every other shape): the block takes all heads together,
//     scores for the chunk, one softmax per head, then the values.
// Each chunk writes (m, l, o) per head, laid out per head and 32-channel slice;
// k_attn_combine merges the chunks:
// o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c (fp32).
#include "attn_kernels.cuh"

namespace bq {
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

// Plan of the warp-per-kv-head kernel; ok = false where it does not apply.
constexpr int kWarpRingBudget = 96 * 1024;  // two CTAs per SM

struct AttnWPlan {
  bool ok;
  int lb, tw, sub, chunk_tokens, chunks, stage_bytes, stages, ring_bytes, k_tok, v_tok;
  size_t smem;
};

AttnWPlan attn_wplan(int kt, int vt, int64_t T, int64_t H, int64_t n_kv, int64_t D) {
  AttnWPlan p{};
  const int64_t G = H / n_kv;
  if (!(n_kv == 1 || n_kv == 2 || n_kv == 4 || n_kv == 8) || D * G > 1024) return p;
  const int nb = int(D / kQK);
  p.lb = 1;
  while (p.lb < nb) p.lb *= 2;
  p.k_tok = int(n_kv) * nb * (kt == kTypeQ4_0 ? Fmt<kTypeQ4_0>::kBytes : Fmt<kTypeQ8_0>::kBytes);
  p.v_tok = int(n_kv) * nb * (vt == kTypeQ4_0 ? Fmt<kTypeQ4_0>::kBytes : Fmt<kTypeQ8_0>::kBytes);
  const int WS = kWarpAttnWarps / int(n_kv);
  // the largest warp tile (at most 16 tokens) with three or four stages, else two
  for (int min_stages = 3; min_stages >= 2 && !p.ok; --min_stages)
    for (int tw = 16; tw >= 1 && !p.ok; tw /= 2) {
      const int sub = tw * WS;
      if (sub % 8) break;  // tiles must start on 16-byte boundaries
      const int stage = sub * (p.k_tok + p.v_tok);
      for (int ns = 4; ns >= min_stages && !p.ok; --ns)
        if (ns * stage <= kWarpRingBudget) {
          p.ok = true;
          p.tw = tw;
          p.sub = sub;
          p.stages = ns;
          p.stage_bytes = stage;
        }
    }
  if (!p.ok) return p;
  const int64_t per = (T + kAttnTargetChunks - 1) / kAttnTargetChunks;
  const int64_t max_ct = std::max<int64_t>(p.sub, kAttnMaxChunkTokens / p.sub * p.sub);
  p.chunk_tokens = int(std::min<int64_t>(max_ct, (per + p.sub - 1) / p.sub * p.sub));
  p.chunks = int((T + p.chunk_tokens - 1) / p.chunk_tokens);
  const int merge = kWarpAttnThreads * (32 + int(G)) * 4;  // G * (32 / G + 1) floats per thread
  p.ring_bytes = (std::max(p.stages * p.stage_bytes, merge) + 15) / 16 * 16;
  p.smem = size_t(p.ring_bytes) + size_t(H) * nb * kQRecWords2 * 4 + size_t(kWarpAttnWarps) * 32 * G * 4 +
           size_t(kWarpAttnWarps) * G * 2 * 4 + (2 + kMaxStages) * 4 + 16 + kMaxStages * 8;
  return p;
}

// fixed128: head_dim 128 with full 16-token warp tiles (the common decode
// shapes), the kv-head count fixed at compile time too (attn_fixed_*.cu)
template <int KT, int VT>
const void *attn_warp_fn(int G, bool fixed128, int n_kv) {
  if (!fixed128) return attn_warp_fn_g<KT, VT, 0, 0>(G);
  return KT == kTypeQ4_0 ? attn_warp_fixed_fn_q4k(VT, G, n_kv) : attn_warp_fixed_fn_q8k(VT, G, n_kv);
}

template <int KT, int VT>
cudaError_t launch_attn_warp(int G, bool fixed128, const AttnWArgs &a, int chunks, size_t smem, cudaStream_t stream) {
  const void *fn = attn_warp_fn<KT, VT>(G, fixed128, a.n_kv);
  if (!fn) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem(fn, int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(chunks));
  cfg.blockDim = dim3(kWarpAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[] = {const_cast<AttnWArgs *>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, args);
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

int attn_chunks(int kt, int vt, int64_t T, int64_t H, int64_t n_kv, int64_t D) {
  const AttnWPlan w = attn_wplan(kt, vt, T, H, n_kv, D);
  return w.ok ? w.chunks : attn_plan(kt, vt, T, H, n_kv, D).chunks;
}

}  // namespace

size_t attn_workspace_bytes(int kt, int vt, int64_t T, int64_t H, int64_t n_kv, int64_t D) {
  return (size_t(attn_chunks(kt, vt, T, H, n_kv, D)) * size_t(H) * size_t(D + 2) * 4 + 255) / 256 * 256;
}

size_t attn_smem_bytes(int kt, int vt, int64_t T, int64_t H, int64_t n_kv, int64_t D) {
  const AttnWPlan w = attn_wplan(kt, vt, T, H, n_kv, D);
  return w.ok ? w.smem : attn_plan(kt, vt, T, H, n_kv, D).smem;
}

cudaError_t launch_attn_decode(int kt, int vt, const float *q, const uint8_t *K, const uint8_t *V, float *o,
                               int64_t T, int64_t H, int64_t n_kv, int64_t D, float scale, void *ws,
                               cudaStream_t stream, bool k_rot) {
  cudaError_t err;
  const DeviceInfo *di = device_info(&err);
  if (!di) return err;
  const int G = int(H / n_kv);
  // scores are kept in base-2 units, s * scale * log2(e), so that every
  // exponential is one exp2
  const float scale2 = float(double(scale) * 1.4426950408889634);
  const int chunks = attn_chunks(kt, vt, T, H, n_kv, D);
  float *o_part = static_cast<float *>(ws);
  float *ml = o_part + size_t(chunks) * H * D;
  cudaError_t e;
  const AttnWPlan w = attn_wplan(kt, vt, T, H, n_kv, D);
  if (w.ok) {
    AttnWArgs a{};
    a.q = q;
    a.K = K;
    a.V = V;
    a.o_part = o_part;
    a.ml = ml;
    a.scale = scale2;
    a.n_tokens = int(T);
    a.n_heads = int(H);
    a.n_kv = int(n_kv);
    a.D = int(D);
    a.nb = int(D / kQK);
    a.k_tok = w.k_tok;
    a.v_tok = w.v_tok;
    a.lb = w.lb;
    a.chunk_tokens = w.chunk_tokens;
    a.tw = w.tw;
    a.sub = w.sub;
    a.stage_bytes = w.stage_bytes;
    a.stages = w.stages;
    a.ring_bytes = w.ring_bytes;
    a.k_rot = k_rot ? 1 : 0;
    a.err = di->err_word;
    a.spin_limit = spin_limit();
    static const int forced_poll = tuning_value("BQ_ATTN_POLL_NS");  // read once per process
    a.poll_ns = forced_poll > 0 ? uint32_t(forced_poll) : 0u;
    static const int forced_prefetch = tuning_value("BQ_ATTN_PREFETCH_TOKENS");
    a.prefetch_tokens = forced_prefetch > 0 ? forced_prefetch : w.sub;  // one tile: more competes with the previous kernel
    static const int no_fixed = tuning_value("BQ_ATTN_GENERIC");
    const bool fixed128 = D == 4 * kQK && w.tw == kFixedTW && no_fixed <= 0;
    if (kt == kTypeQ4_0)
      e = vt == kTypeQ4_0 ? launch_attn_warp<kTypeQ4_0, kTypeQ4_0>(G, fixed128, a, chunks, w.smem, stream)
                          : launch_attn_warp<kTypeQ4_0, kTypeQ8_0>(G, fixed128, a, chunks, w.smem, stream);
    else
      e = vt == kTypeQ4_0 ? launch_attn_warp<kTypeQ8_0, kTypeQ4_0>(G, fixed128, a, chunks, w.smem, stream)
                          : launch_attn_warp<kTypeQ8_0, kTypeQ8_0>(G, fixed128, a, chunks, w.smem, stream);
  } else {
    const AttnPlan p = attn_plan(kt, vt, T, H, n_kv, D);
    AttnArgs a{};
    a.q = q;
    a.K = K;
    a.V = V;
    a.o_part = o_part;
    a.ml = ml;
    a.scale = scale2;
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
    a.k_rot = k_rot ? 1 : 0;
    a.err = di->err_word;
    a.spin_limit = spin_limit();
    if (kt == kTypeQ4_0)
      e = vt == kTypeQ4_0 ? launch_attn_kv<kTypeQ4_0, kTypeQ4_0>(G, a, chunks, p.smem, stream)
                          : launch_attn_kv<kTypeQ4_0, kTypeQ8_0>(G, a, chunks, p.smem, stream);
    else
      e = vt == kTypeQ4_0 ? launch_attn_kv<kTypeQ8_0, kTypeQ4_0>(G, a, chunks, p.smem, stream)
                          : launch_attn_kv<kTypeQ8_0, kTypeQ8_0>(G, a, chunks, p.smem, stream);
  }
  if (e != cudaSuccess) return e;
  // the combine starts while the chunk kernel drains (programmatic dependent launch)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  const int csmem = combine_smem_bytes(chunks);
  if ((e = ensure_smem(reinterpret_cast<const void *>(k_attn_combine), csmem)) != cudaSuccess) return e;
  cfg.gridDim = dim3(unsigned(H), unsigned(D / 32));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = size_t(csmem);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_attn_combine, static_cast<const float *>(o_part), static_cast<const float *>(ml),
                            o, chunks, int(H), int(D));
}

}  // namespace bq
