// attn_fixed_q4k.cu — the decode-attention warp kernels with a compile-time
// shape (head_dim 128, every kv-head count and query heads per kv head) for a
// Q4_0 K cache; a file per K type so that the
// instantiations compile in parallel.
#include "attn_kernels.cuh"

namespace bq {

const void *attn_warp_fixed_fn_q4k(int vt, int G, int n_kv) {
  if (vt != kTypeQ4_0 && vt != kTypeQ8_0) return nullptr;
  switch (n_kv) {
    case 1: return vt == kTypeQ4_0 ? attn_warp_fn_g<kTypeQ4_0, kTypeQ4_0, 4, 1>(G) : attn_warp_fn_g<kTypeQ4_0, kTypeQ8_0, 4, 1>(G);
    case 2: return vt == kTypeQ4_0 ? attn_warp_fn_g<kTypeQ4_0, kTypeQ4_0, 4, 2>(G) : attn_warp_fn_g<kTypeQ4_0, kTypeQ8_0, 4, 2>(G);
    case 4: return vt == kTypeQ4_0 ? attn_warp_fn_g<kTypeQ4_0, kTypeQ4_0, 4, 4>(G) : attn_warp_fn_g<kTypeQ4_0, kTypeQ8_0, 4, 4>(G);
    case 8: return vt == kTypeQ4_0 ? attn_warp_fn_g<kTypeQ4_0, kTypeQ4_0, 4, 8>(G) : attn_warp_fn_g<kTypeQ4_0, kTypeQ8_0, 4, 8>(G);
    default: return nullptr;
  }
}

}  // namespace bq
