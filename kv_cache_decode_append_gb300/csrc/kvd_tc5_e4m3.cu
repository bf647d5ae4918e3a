// Instantiates the tcgen05 decode-attention kernels over E4M3 caches (bf16 q / out,
// D = 128, contiguous caches), with the merge pass and merging split heads themselves.
#include "kvd_attention_tc5.cuh"

namespace kvd {
bool attn_variant_tc5_e4m3(int D, AttnVariant *v) { return pick_tc5_e4m3_variant<false>(D, v); }
bool attn_variant_tc5_e4m3_tk(int D, AttnVariant *v) { return pick_tc5_e4m3_variant<true>(D, v); }
}  // namespace kvd
