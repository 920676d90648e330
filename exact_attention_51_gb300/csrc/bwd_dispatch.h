// Host <-> kernel interface of the attention backward pass.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ea51 {

struct BwdParams {
  __nv_bfloat16* dq;     // bf16 [BH, N, D]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* lse2;           // workspace: -LSE * log2(e), [BH, Npad]
  float* dsum;           // workspace: -D, D = rowsum(dO o O), [BH, Npad]
  unsigned int* status;  // device-wide wait-timeout word
  int N;
  int Npad;              // N rounded up to 128
  int BH;
  int heads_per_group;   // causal launch order: heads whose blocks interleave
  float scale;
  float scale_log2;      // scale * log2(e)
};

// Preprocess + dK/dV + dQ kernels on `stream` (d = 64, 128 or 256; the maps
// have 128-row boxes of 64 columns).
cudaError_t launch_bwd(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                       const CUtensorMap* tdo, const BwdParams& p, const void* o, const void* dout,
                       const float* lse, int d, bool causal, cudaStream_t stream);

// The d = 256 kernels (dV, dK, dQ) after the preprocess.
cudaError_t launch_bwd_d256(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                            const CUtensorMap* tdo, const BwdParams& p, bool causal,
                            cudaStream_t stream);

}  // namespace ea51
