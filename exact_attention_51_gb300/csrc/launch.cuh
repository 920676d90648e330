// Kernel launch for one head dim (both causal flags).  Included by exactly one
// translation unit per head dim and input type so the variants compile in
// parallel.
#pragma once
#include <atomic>

#include "attn_fwd_kernel.cuh"

namespace ea51 {

template <int D, bool CAUSAL, bool SPLIT, bool F8 = false, int SK = kShapeDefault>
cudaError_t launch_one(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                       const CUtensorMap* to, const FwdParams& p, cudaStream_t stream) {
  using L = Layout<D, F8, SK>;
  auto kern = attn_fwd_kernel<D, CAUSAL, SPLIT, F8, SK>;
  // The dynamic shared-memory opt-in is per device; remember which are done.
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    // all of the unified L1 / shared memory as shared memory, so that
    // MIN_BLOCKS CTAs fit on an SM
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const unsigned grid = static_cast<unsigned>(p.n_qblk) * static_cast<unsigned>(p.BH) *
                        static_cast<unsigned>(p.kv_splits);
  kern<<<grid, L::THREADS, L::SMEM_ALLOC, stream>>>(*tq, *tk, *tv, *to, p);
  return cudaGetLastError();
}

template <int D, bool F8, int SK>
cudaError_t launch_d(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                     const CUtensorMap* to, const FwdParams& p, bool causal, cudaStream_t stream) {
  // split-KV partial outputs use their own instantiation, so the single-pass
  // kernel carries none of that epilogue
  if (p.kv_splits > 1)
    return causal ? launch_one<D, true, true, F8, SK>(tq, tk, tv, to, p, stream)
                  : launch_one<D, false, true, F8, SK>(tq, tk, tv, to, p, stream);
  return causal ? launch_one<D, true, false, F8, SK>(tq, tk, tv, to, p, stream)
                : launch_one<D, false, false, F8, SK>(tq, tk, tv, to, p, stream);
}

template <int D, bool F8 = false, int SK = kShapeDefault>
FwdVariant make_variant() {
  using L = Layout<D, F8, SK>;
  return FwdVariant{L::BN, L::NQ * BM, &launch_d<D, F8, SK>};
}

}  // namespace ea51
