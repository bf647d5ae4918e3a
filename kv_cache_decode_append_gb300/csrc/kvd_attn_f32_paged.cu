// Instantiates the fp32 decode-attention kernels over a paged cache, with the
// separate merge pass (D in {64, 128}, RB in {1, 2, 4, 8}).
#include "kvd_attention.cuh"

namespace kvd {
bool attn_variant_f32_paged(int D, int RB, AttnVariant *v) { return pick_variant<float, false, true>(D, RB, v); }
}  // namespace kvd
