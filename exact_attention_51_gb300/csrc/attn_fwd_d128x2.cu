// Head dim 128 instantiation of the fused attention forward with two CTAs per
// SM (one query tile each).
#include "launch.cuh"

namespace ea51 {
FwdVariant fwd_variant_d128_two() { return make_variant<128, true>(); }
}  // namespace ea51
