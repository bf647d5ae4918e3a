// Instantiates the fp16 decode-attention kernels that merge split heads themselves
// (D in {64, 128}, RB in {1, 2, 4, 8}).
#include "kvd_attention.cuh"

namespace kvd {
bool attn_variant_f16_tk(int D, int RB, AttnVariant *v) { return pick_variant<__half, true, false>(D, RB, v); }
}  // namespace kvd
