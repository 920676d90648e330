// Head dim 64 instantiation of the fused attention forward with two CTAs per
// SM (one query tile each).
#include "launch.cuh"

namespace ea51 {
FwdVariant fwd_variant_d64_two() { return make_variant<64, false, kShapeTwo>(); }
}  // namespace ea51
