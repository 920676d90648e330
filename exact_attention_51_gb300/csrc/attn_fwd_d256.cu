// Head dim 256 instantiation of the fused attention forward.
#include "launch.cuh"

namespace ea51 {
FwdVariant fwd_variant_d256() { return make_variant<256>(); }
}  // namespace ea51
