// The WC instantiations of the split-KV decode kernel in decode_split.cuh
// (head_dim 128, boxes of 8 KV heads, 16-row groups; plain and fused, bf16 and
// e4m3 pools): the cut of the units weighs each segment change and a publisher
// warp counts cut segments, as for 32-row groups.  Chosen by the host when
// seg_penalty > 0 (decode_segment_penalty); a translation unit of their own so
// that they compile in parallel with the others and leave their code
// generation untouched.
#include "decode_split.cuh"

namespace pa {

cudaError_t launch_split_weighted(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, bool kv8,
                                  bool fused, cudaStream_t s) {
  if (kv8)
    return fused ? launch_split<128, 8, 1, true, true, true>(p, tk, tv, s)
                 : launch_split<128, 8, 1, true, false, true>(p, tk, tv, s);
  return fused ? launch_split<128, 8, 1, false, true, true>(p, tk, tv, s)
               : launch_split<128, 8, 1, false, false, true>(p, tk, tv, s);
}

}  // namespace pa
