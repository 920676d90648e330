// Host <-> kernel interface of the attention forward: launch parameters and
// the per-head-dim launcher table.  Plain C++ (no device code).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace ea51 {

struct FwdParams {
  void* o;               // bf16 [BH, N, D]
  float* lse;            // fp32 [BH, N]
  unsigned int* status;  // device-wide wait-timeout word (0 = clean)
  int N;
  int BH;
  int n_qblk;            // CTAs per head
  float scale_log2;      // scale * log2(e)
};

struct FwdVariant {
  int kv_rows;         // keys per K/V tile (TMA box rows of K and V)
  int q_rows_per_cta;  // query rows per CTA (multiple of the 128-row Q box)
  cudaError_t (*launch)(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                        const FwdParams& p, bool causal, cudaStream_t stream);
};

FwdVariant fwd_variant_d64();
FwdVariant fwd_variant_d128();
FwdVariant fwd_variant_d256();

}  // namespace ea51
