// paged_attention_decode_append: the fused (append + decode) instantiations
// of the split-KV decode kernel in decode_split.cuh, in a translation unit of
// their own so that they compile in parallel with the plain ones.
#include "decode_split.cuh"

namespace pa {

cudaError_t launch_split_fused(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rt,
                               cudaStream_t s) {
  const int D = p.pool.head_dim;
  if (p.kv8)
    return D == 128 ? launch_split_d<128, true, true>(p, tk, tv, rt, s) : launch_split_d<64, true, true>(p, tk, tv, rt, s);
  return D == 128 ? launch_split_d<128, false, true>(p, tk, tv, rt, s) : launch_split_d<64, false, true>(p, tk, tv, rt, s);
}

}  // namespace pa
