// Pieces shared by the backward kernels (head dims 64 / 128 in attn_bwd.cu,
// 256 in attn_bwd_d256.cu): warp roles, the causal launch order, and the
// elementwise steps P = exp2(S * c - LSE * log2 e) and dS = P o (dP - D) on
// 32-column chunks of a tensor-memory row.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "attn_fwd_kernel.cuh"
#include "bwd_dispatch.h"

namespace ea51 {

// Warps: 0..7 elementwise (two per tensor-memory lane quadrant, each taking
// half of a tile's columns), 8 TMA, 9 MMA.
constexpr int kComputeWarps = 8;
constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr int kBwdThreads = 320;

// 128-column tiles: packed bf16 output of column half h (64 fp32 columns at
// 64h -> 32 columns of bf16 pairs at 64h): each 32-column chunk's 16 packed
// columns land on columns this half has already read, never on the other
// half's.  a_col: the tensor-memory column of K-step k (16 rows of the other
// operand) of such a packed A operand (P^T, dS^T or dS).
__host__ __device__ constexpr int packed_col(int h) { return 64 * h; }
__host__ __device__ constexpr int a_col(int k) { return k < 4 ? k * 8 : 64 + (k - 4) * 8; }

// Causal CTA order: heaviest blocks first (longest-processing-time order)
// across a group of heads_per_group heads whose streamed operands fit in a
// share of L2 (the host sizes the group); `heavy_rank` 0 is the heaviest
// block of a head.
__device__ __forceinline__ void grouped_order(int cta, int nblk, int BH, int hpg, int& bh,
                                              int& heavy_rank) {
  const int per_group = hpg * nblk;
  const int group = cta / per_group;
  const int gs = min(hpg, BH - group * hpg);
  const int within = cta - group * per_group;
  bh = group * hpg + within % gs;
  heavy_rank = within / gs;
}

// 1-D bulk copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}

// Four consecutive fp32 values from shared memory (16-byte aligned address).
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "r"(addr));
  return r;
}

// p = exp2(s * c - lse2_q) for one 32-query chunk of one key row (dK/dV
// kernel), in place over the chunk's S^T bits, with the chunk's -lse2 at
// shared-memory address `row`; also packs P^T to bf16.  MASKED keeps queries
// q with lo <= q < lo + span (block-relative) only (causal diagonal, ragged
// tail).
template <bool MASKED>
__device__ __forceinline__ void p_chunk_t(uint32_t (&sp)[32], uint32_t row, float c, int col0,
                                          int lo, int span, uint32_t (&pk)[16]) {
  const f32x2 cc = f2_pack(c, c);
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const float4 nl = lds_f4(row + 16 * g);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = 2 * g + u;
      const f32x2 x = f2_fma(f2_pack(__uint_as_float(sp[2 * e]), __uint_as_float(sp[2 * e + 1])),
                             cc, u ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y));
      float x0, x1;
      f2_unpack(x, x0, x1);
      float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      if (MASKED) {
        p0 = static_cast<unsigned>(col0 + 2 * e - lo) < static_cast<unsigned>(span) ? p0 : 0.f;
        p1 = static_cast<unsigned>(col0 + 2 * e + 1 - lo) < static_cast<unsigned>(span) ? p1 : 0.f;
      }
      sp[2 * e] = __float_as_uint(p0);
      sp[2 * e + 1] = __float_as_uint(p1);
      pk[e] = pack_bf16x2(p0, p1);
    }
  }
}

// p = exp2(s * c - lse2) for one 32-key chunk of one query row (dQ kernel),
// in place, with the row's nl2 = -lse2; MASKED keeps keys col0 + i < lim.
template <bool MASKED>
__device__ __forceinline__ void p_chunk_q(uint32_t (&sp)[32], float c, float nl2, int col0,
                                          int lim) {
  const f32x2 cc = f2_pack(c, c), nl = f2_pack(nl2, nl2);
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const f32x2 x =
        f2_fma(f2_pack(__uint_as_float(sp[2 * e]), __uint_as_float(sp[2 * e + 1])), cc, nl);
    float x0, x1;
    f2_unpack(x, x0, x1);
    float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    if (MASKED) {
      p0 = col0 + 2 * e < lim ? p0 : 0.f;
      p1 = col0 + 2 * e + 1 < lim ? p1 : 0.f;
    }
    sp[2 * e] = __float_as_uint(p0);
    sp[2 * e + 1] = __float_as_uint(p1);
  }
}

// ds = p * (dp - D) for one 32-column chunk, packed to bf16, with -D per
// column (dK/dV kernel: four at a time from shared memory at `nd_row`).
__device__ __forceinline__ void ds_chunk_t(const uint32_t (&p)[32], const uint32_t (&dp)[32],
                                           uint32_t nd_row, uint32_t (&dk)[16]) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const float4 nd = lds_f4(nd_row + 16 * g);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = 2 * g + u;
      const f32x2 dd = f2_add(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])),
                              u ? f2_pack(nd.z, nd.w) : f2_pack(nd.x, nd.y));
      const f32x2 ds = f2_mul(f2_pack(__uint_as_float(p[2 * e]), __uint_as_float(p[2 * e + 1])), dd);
      float d0, d1;
      f2_unpack(ds, d0, d1);
      dk[e] = pack_bf16x2(d0, d1);
    }
  }
}

// The same with one -D for the whole chunk (dQ kernel: one query row).
__device__ __forceinline__ void ds_chunk_q(const uint32_t (&p)[32], const uint32_t (&dp)[32],
                                           float nds, uint32_t (&dk)[16]) {
  const f32x2 nd = f2_pack(nds, nds);
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const f32x2 ds = f2_mul(
        f2_pack(__uint_as_float(p[2 * e]), __uint_as_float(p[2 * e + 1])),
        f2_add(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])), nd));
    float d0, d1;
    f2_unpack(ds, d0, d1);
    dk[e] = pack_bf16x2(d0, d1);
  }
}

}  // namespace ea51
