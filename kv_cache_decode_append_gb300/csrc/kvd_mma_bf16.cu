// Instantiates the bf16 tensor-core decode-attention kernels with the separate merge pass
// (D in {64, 128}, 16-row blocks, contiguous and paged caches).
#include "kvd_attention_mma.cuh"

namespace kvd {
bool attn_variant_mma_bf16(int D, bool paged, AttnVariant *v) { return pick_mma_variant<__nv_bfloat16, false>(D, paged, v); }
}  // namespace kvd
