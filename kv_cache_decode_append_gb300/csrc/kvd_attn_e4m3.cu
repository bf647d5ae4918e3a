// Instantiates the decode-attention kernels with bf16 q / out over an E4M3
// cache, with the separate merge pass (D in {64, 128}, RB in {1, 2, 4}).
#include "kvd_attention.cuh"

namespace kvd {
bool attn_variant_e4m3(int D, int RB, AttnVariant *v)
{
    return pick_variant<__nv_bfloat16, false, false, __nv_fp8_e4m3>(D, RB, v);
}
}  // namespace kvd
