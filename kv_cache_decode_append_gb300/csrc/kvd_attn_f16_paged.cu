// Instantiates the fp16 decode-attention kernels over a paged cache with the separate merge pass
// (D in {64, 128}, RB in {1, 2, 4, 8}).
#include "kvd_attention.cuh"

namespace kvd {
bool attn_variant_f16_paged(int D, int RB, AttnVariant *v) { return pick_variant<__half, false, true>(D, RB, v); }
}  // namespace kvd
