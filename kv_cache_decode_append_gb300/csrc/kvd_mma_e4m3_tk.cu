// Instantiates the tensor-core decode-attention kernels with bf16 q / out over
// an E4M3 cache that merge split heads themselves (D = 128, blocks of 16 rows, or
// of 8 in the swapped form for heads of at most 8 rows; contiguous caches).
#include "kvd_attention_mma.cuh"

namespace kvd {
bool attn_variant_mma_e4m3_tk(int D, int rows, AttnVariant *v) { return pick_mma_e4m3_variant<true>(D, rows, v); }
}  // namespace kvd
