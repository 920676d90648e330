// Head dim 128 instantiation of the fused attention forward.
#include "launch.cuh"

namespace ea51 {
FwdVariant fwd_variant_d128() { return make_variant<128>(); }
}  // namespace ea51
