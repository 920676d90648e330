// e4m3 (8-bit) inputs, head dims 64, 128 and 256: the fused forward with
// Q K^T and P V on tcgen05.mma kind::f8f6f4 (V read MN-major as stored); d =
// 64 also in the two-CTAs-per-SM shape for short rows, as bf16.
#include "launch.cuh"

namespace ea51 {

FwdVariant fwd_variant_e4m3_d64() { return make_variant<64, true>(); }
FwdVariant fwd_variant_e4m3_d64_two() { return make_variant<64, true, kShapeTwo>(); }
FwdVariant fwd_variant_e4m3_d128() { return make_variant<128, true>(); }
FwdVariant fwd_variant_e4m3_d256() { return make_variant<256, true>(); }

}  // namespace ea51
