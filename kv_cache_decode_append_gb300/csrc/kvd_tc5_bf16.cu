// Instantiates the bf16 tcgen05 decode-attention kernels whose split heads go to the separate merge pass
// (D in {64, 128}, 128-row blocks, contiguous and paged caches).
#include "kvd_attention_tc5.cuh"

namespace kvd {
bool attn_variant_tc5_bf16(int D, bool paged, AttnVariant *v) { return pick_tc5_variant<__nv_bfloat16, false>(D, paged, v); }
}  // namespace kvd
