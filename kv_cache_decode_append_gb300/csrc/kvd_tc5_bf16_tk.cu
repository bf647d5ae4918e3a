// Instantiates the bf16 tcgen05 decode-attention kernels that merge split heads themselves
// (D in {64, 128}, 128-row blocks, contiguous and paged caches).
#include "kvd_attention_tc5.cuh"

namespace kvd {
bool attn_variant_tc5_bf16_tk(int D, bool paged, AttnVariant *v) { return pick_tc5_variant<__nv_bfloat16, true>(D, paged, v); }
}  // namespace kvd
