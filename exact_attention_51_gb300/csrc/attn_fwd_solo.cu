// One query tile per CTA (small grids): bf16 and e4m3 instantiations of the
// fused attention forward for head dims 64 and 128.
#include "launch.cuh"

namespace ea51 {
FwdVariant fwd_variant_d64_solo() { return make_variant<64, false, kShapeSolo>(); }
FwdVariant fwd_variant_d128_solo() { return make_variant<128, false, kShapeSolo>(); }
FwdVariant fwd_variant_e4m3_d64_solo() { return make_variant<64, true, kShapeSolo>(); }
FwdVariant fwd_variant_e4m3_d128_solo() { return make_variant<128, true, kShapeSolo>(); }
}  // namespace ea51
