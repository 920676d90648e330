// e4m3 (8-bit) inputs, head dims 64, 128 and 256: the fused forward with
// Q K^T and P V on tcgen05.mma kind::f8f6f4 (V read MN-major as stored).
#include "launch.cuh"

namespace ea51 {

namespace {

template <int D>
cudaError_t launch_e4m3(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                        const CUtensorMap* to, const FwdParams& p, bool causal, cudaStream_t stream) {
  // split-KV partial outputs use their own instantiation, as for bf16
  if (p.kv_splits > 1)
    return causal ? launch_one<D, true, true, true>(tq, tk, tv, to, p, stream)
                  : launch_one<D, false, true, true>(tq, tk, tv, to, p, stream);
  return causal ? launch_one<D, true, false, true>(tq, tk, tv, to, p, stream)
                : launch_one<D, false, false, true>(tq, tk, tv, to, p, stream);
}

}  // namespace

FwdVariant fwd_variant_e4m3_d64() {
  using L = Layout<64, true>;
  return FwdVariant{L::BN, L::NQ * BM, &launch_e4m3<64>};
}

FwdVariant fwd_variant_e4m3_d128() {
  using L = Layout<128, true>;
  return FwdVariant{L::BN, L::NQ * BM, &launch_e4m3<128>};
}

FwdVariant fwd_variant_e4m3_d256() {
  using L = Layout<256, true>;
  return FwdVariant{L::BN, L::NQ * BM, &launch_e4m3<256>};
}

}  // namespace ea51
