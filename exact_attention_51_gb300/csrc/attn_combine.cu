// Split-KV merge: each of kv_splits partial results of one query row is a
// normalised output O_s (fp32) with its log-sum-exp L_s over the keys that
// split saw.  The full row is their log-sum-exp weighted mean:
//   L = ln sum_s exp(L_s),   O = sum_s exp(L_s - L) O_s
// (the associative merge of per-block softmax states, "algebraic aggregates"
// in HN item 40939030; the online-softmax rescaling of "Tri Dao: prediction"
// applied across CTAs instead of across tiles).  Splits with L_s = -inf saw no
// key and are skipped.  Every row the entry points accept sees at least one
// key (causal rows need Nk >= Nq), so some split of it is non-empty; a row
// whose splits were all empty would be written as O = 0, LSE = -inf (the
// empty sum) rather than as 0/0.  One warp per row; HBM-bound.
#include <cuda_bf16.h>

#include <cstdint>

#include "fwd_dispatch.h"

namespace ea51 {
namespace {

template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           __nv_bfloat16* __restrict__ o,
                                                           float* __restrict__ lse, long long rows,
                                                           int splits) {
  constexpr int PER = D / 32;  // columns per lane
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s) m = fmaxf(m, lse_part[s * rows + row]);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  // 16-byte loads where a lane's columns allow (d >= 128), two splits in
  // flight per iteration; the branch is uniform across the warp (one row)
#pragma unroll 2
  for (int s = 0; s < splits; ++s) {
    const float ls = lse_part[s * rows + row];
    if (ls == -INFINITY) continue;
    const float wgt = expf(ls - m);
    wsum += wgt;
    const float* src = o_part + (s * rows + row) * D + lane * PER;
    if constexpr (PER % 4 == 0) {
#pragma unroll
      for (int e = 0; e < PER; e += 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + e);
        acc[e] += wgt * v.x;
        acc[e + 1] += wgt * v.y;
        acc[e + 2] += wgt * v.z;
        acc[e + 3] += wgt * v.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < PER; e += 2) {
        const float2 v = *reinterpret_cast<const float2*>(src + e);
        acc[e] += wgt * v.x;
        acc[e + 1] += wgt * v.y;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = o + row * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  if (lane == 0) lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(int d, const float* o_part, const float* lse_part, void* o, float* lse,
                           long long rows, int kv_splits, cudaStream_t stream) {
  constexpr int kWarps = 8;
  const long long blocks = (rows + kWarps - 1) / kWarps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(blocks)), block(kWarps * 32);
  auto* ob = static_cast<__nv_bfloat16*>(o);
  switch (d) {
    case 64: attn_combine_kernel<64><<<grid, block, 0, stream>>>(o_part, lse_part, ob, lse, rows, kv_splits); break;
    case 128: attn_combine_kernel<128><<<grid, block, 0, stream>>>(o_part, lse_part, ob, lse, rows, kv_splits); break;
    case 256: attn_combine_kernel<256><<<grid, block, 0, stream>>>(o_part, lse_part, ob, lse, rows, kv_splits); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ea51
