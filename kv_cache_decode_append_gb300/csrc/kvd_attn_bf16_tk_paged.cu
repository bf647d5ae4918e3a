// Instantiates the bf16 decode-attention kernels over a paged cache that merge
// split heads themselves (D in {64, 128}, RB in {1, 2, 4, 8}).
#include "kvd_attention.cuh"

namespace kvd {
bool attn_variant_bf16_tk_paged(int D, int RB, AttnVariant *v) { return pick_variant<__nv_bfloat16, true, true>(D, RB, v); }
}  // namespace kvd
