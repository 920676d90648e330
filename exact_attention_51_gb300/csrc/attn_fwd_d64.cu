// Head dim 64 instantiation of the fused attention forward.
#include "launch.cuh"

namespace ea51 {
FwdVariant fwd_variant_d64() { return make_variant<64>(); }
}  // namespace ea51
