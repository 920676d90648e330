// Backward pass of the fused exact attention (gradients dQ, dK, dV) for
// sm_103a.  For O = softmax(scale * Q K^T [+ causal mask]) V with upstream
// gradient dO, and P recomputed from the forward's log-sum-exp:
//
//   P = exp(scale * Q K^T - LSE),  D_i = sum_c dO_ic O_ic
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q
//
// Three kernels, none of them writing an N x N matrix to HBM:
//   preprocess  -D and -LSE * log2(e) per row into a padded workspace;
//   dK/dV       one CTA per 128-key block: for every query block it
//               recomputes S^T = K Q^T and dP^T = V dO^T in tensor memory,
//               two threads per key row (one per half of the query block)
//               form P^T, then dS^T (bf16, written over the fp32 tiles; P
//               stays in fp32 registers in between), and the tensor core
//               accumulates dV += P^T dO and dK += dS^T Q in tensor memory;
//   dQ          one CTA per 128-query block: recomputes S and dP per key
//               block, forms P then dS (two threads per query row),
//               accumulates dQ += dS K.
// In both, the MMA of the next block's S runs as soon as the elementwise
// warps are done with the current one, so their exponentials overlap the
// tensor core's other products.
// S and dP are computed twice (once per kernel) so that no kernel needs a
// transposed copy of dS or atomics: every MMA uses the operand layouts of the
// forward kernel (K-major A/B from shared memory, or A from tensor memory
// with an MN-major B).  The pages name the backward pass only as the part the
// ~100-line kernel's author had not written ("Show HN: Flash Attention in
// ~100 lines of CUDA"); the formulas are the derivative of the forward
// definition.  Head dims 64 and 128 here (the tensor memory holds S, dP and
// two d-column accumulators); 256 in attn_bwd_d256.cu.
#include <cuda_bf16.h>

#include <cstdint>

#include "bwd_common.cuh"

namespace ea51 {
namespace {

// Tiles of 128 query rows by 128 key rows throughout.

template <int D>
struct BwdLayout {
  static constexpr int PANELS = D / 64;
  static constexpr int PANEL = 128 * 128;  // one 64-column panel of a 128-row tile
  static constexpr int TILE = 128 * D * 2;
  static constexpr int STAGES = D == 64 ? 3 : 2;
  // dK/dV kernel: K, V resident; ring of {Q, dO, lse', D} per query block
  static constexpr int A_OFF_K = 0, A_OFF_V = TILE, A_OFF_RING = 2 * TILE;
  static constexpr int A_STAGE = 2 * TILE + 2 * 512;
  static constexpr int A_OFF_BAR = A_OFF_RING + STAGES * A_STAGE;
  // dQ kernel: Q, dO resident; ring of {K, V} per key block
  static constexpr int B_OFF_Q = 0, B_OFF_DO = TILE, B_OFF_RING = 2 * TILE;
  static constexpr int B_STAGE = 2 * TILE;
  static constexpr int B_OFF_BAR = B_OFF_RING + STAGES * B_STAGE;
  // barriers (both kernels): 0 resident-full, [1, 1+ST) ring full,
  // [1+ST, 1+2ST) ring empty, BAR_S: S (or S^T) computed, BAR_S + 1: dP (or
  // dP^T) computed; BAR_P: P^T packed (dK/dV) or S read out (dQ), BAR_P + 1:
  // dS (or dS^T) packed, each counted once per elementwise warp; final, drain
  static constexpr int BAR_RES = 0, BAR_FULL = 1, BAR_EMPTY = 1 + STAGES, BAR_S = 1 + 2 * STAGES,
                       BAR_P = BAR_S + 2, BAR_FINAL = BAR_P + 2, BAR_DRAIN = BAR_FINAL + 1,
                       NBAR = BAR_DRAIN + 1;
  static constexpr int A_SMEM = A_OFF_BAR + NBAR * 8 + 8 + 1024;
  static constexpr int B_SMEM = B_OFF_BAR + NBAR * 8 + 8 + 1024;
  // tensor memory: T1 = S^T or S, T2 = dP^T or dP, then the accumulators
  static constexpr int T1 = 0, T2 = 128, ACC0 = 256, ACC1 = 256 + D;
  static_assert(ACC1 + D <= 512 || D == 64, "tensor memory");
  static_assert(A_SMEM <= 232448 && B_SMEM <= 232448, "shared memory");
};


// ------------------------------------------------------------ preprocess

// D / 8 lanes per row, each summing the 8 products of one 16-byte load of O
// and one of dO (then a shuffle reduction over the row's lanes); 256 / D
// rows per warp.  Padding rows (N <= i < Npad) get 0 for both.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                          const float* __restrict__ lse, float* __restrict__ lse2,
                          float* __restrict__ dsum, int N, int Npad, long long BH) {
  constexpr int LPR = D / 8, RPW = 32 / LPR;
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long prow = w * RPW + lane / LPR;  // padded row: bh * Npad + i
  const int sub = lane % LPR;
  const bool live = prow < BH * Npad;
  float acc = 0.f;
  float l2 = 0.f;
  if (live) {
    const long long bh = prow / Npad;
    const int i = static_cast<int>(prow - bh * Npad);
    if (i < N) {
      const long long row = bh * N + i;
      const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + sub * 8);
      const uint4 g = *reinterpret_cast<const uint4*>(dout + row * D + sub * 8);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 af = __bfloat1622float2(a2[e]), gf = __bfloat1622float2(g2[e]);
        acc = fmaf(af.x, gf.x, acc);
        acc = fmaf(af.y, gf.y, acc);
      }
      l2 = -lse[row] * 1.4426950408889634f;
    }
  }
#pragma unroll
  for (int s = LPR / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (live && sub == 0) {
    lse2[prow] = l2;    // -LSE * log2(e)
    dsum[prow] = -acc;  // -D
  }
}

template <int D>
cudaError_t launch_preprocess(const void* o, const void* dout, const float* lse, const BwdParams& p,
                              cudaStream_t stream) {
  constexpr int RPW = 32 / (D / 8);
  const long long rows = static_cast<long long>(p.BH) * p.Npad;
  const long long threads = (rows + RPW - 1) / RPW * 32;
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  bwd_preprocess_kernel<D><<<blocks, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, p.lse2,
      p.dsum, p.N, p.Npad, p.BH);
  return cudaGetLastError();
}

// ------------------------------------------------------------ dK / dV

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::A_OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::A_OFF_BAR + L::NBAR * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::A_OFF_BAR + L::NBAR * 8 + 4);
  const Waiter w{abort_flag, p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tile: key block kb of head bh; causal visits query blocks kb..nblk-1
  const int nblk = (p.N + 127) / 128;
  // causal: key block kb visits nblk - kb query blocks (heaviest: kb = 0)
  int bh, kb;
  if (CAUSAL) {
    grouped_order(static_cast<int>(blockIdx.x), nblk, p.BH, p.heads_per_group, bh, kb);
  } else {
    bh = static_cast<int>(blockIdx.x) / nblk;
    kb = static_cast<int>(blockIdx.x) % nblk;
  }
  const int q_first = CAUSAL ? kb : 0;
  const int nq = nblk - q_first;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::NBAR; ++i)
      mbar_init(bar(i), (i == L::BAR_P || i == L::BAR_P + 1) ? kComputeWarps : 1u);
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      const uint32_t rb = bar(L::BAR_RES);
      mbar_arrive_expect_tx(rb, 2 * L::TILE);
      for (int pn = 0; pn < L::PANELS; ++pn) {
        tma_load_3d(sbase + L::A_OFF_K + pn * L::PANEL, &tm_k, rb, pn * 64, kb * 128, bh);
        tma_load_3d(sbase + L::A_OFF_V + pn * L::PANEL, &tm_v, rb, pn * 64, kb * 128, bh);
      }
      int issued = 0;
      for (int t = 0; t < nq; ++t) {
        const int st = t % L::STAGES;
        const uint32_t ph = static_cast<uint32_t>(t / L::STAGES) & 1u;
        if (!wait_phase(bar(L::BAR_EMPTY + st), ph ^ 1u, w, kCodeProducerEmpty)) break;
        const uint32_t fb = bar(L::BAR_FULL + st);
        const uint32_t base = sbase + L::A_OFF_RING + st * L::A_STAGE;
        const int qblk = q_first + t;
        mbar_arrive_expect_tx(fb, 2 * L::TILE + 1024);
        for (int pn = 0; pn < L::PANELS; ++pn) {
          tma_load_3d(base + pn * L::PANEL, &tm_q, fb, pn * 64, qblk * 128, bh);
          tma_load_3d(base + L::TILE + pn * L::PANEL, &tm_do, fb, pn * 64, qblk * 128, bh);
        }
        const size_t rowoff = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(qblk) * 128;
        bulk_load(base + 2 * L::TILE, p.lse2 + rowoff, 512, fb);
        bulk_load(base + 2 * L::TILE + 512, p.dsum + rowoff, 512, fb);
        ++issued;
      }
      if (*w.abort_flag) {
        drain_phase(bar(L::BAR_RES), 0u, w, kCodeDrain);
        for (int t = max(0, issued - L::STAGES); t < issued; ++t)
          drain_phase(bar(L::BAR_FULL + t % L::STAGES), static_cast<uint32_t>(t / L::STAGES) & 1u,
                      w, kCodeDrain);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    const uint32_t leader = elect_one();
    // Order per query block t: dV(t), S^T(t+1), dK(t), dP^T(t+1).  The
    // exponentials of block t+1 (waiting on S^T(t+1)) run while the tensor
    // core works on dK(t) and dP^T(t+1); dS^T(t+1) is formed while it runs
    // dV(t+1) and S^T(t+2).
    constexpr uint32_t kIdescSS = idesc_bf16_f32(128, 128, false);  // S^T, dP^T: K-major
    constexpr uint32_t kIdescTS = idesc_bf16_f32(128, D, true);      // dV, dK: B MN-major
    bool ok = warp_wait_phase(bar(L::BAR_RES), 0u, w, kCodeMmaQ);
    const uint64_t dK0 = sdesc_sw128(sbase + L::A_OFF_K, 16, 1024);
    const uint64_t dV0 = sdesc_sw128(sbase + L::A_OFF_V, 16, 1024);
    auto stage_base = [&](int t) {
      return sbase + L::A_OFF_RING + static_cast<uint32_t>((t % L::STAGES) * L::A_STAGE);
    };
    auto wait_stage = [&](int t) {
      return warp_wait_phase(bar(L::BAR_FULL + t % L::STAGES),
                             static_cast<uint32_t>(t / L::STAGES) & 1u, w, kCodeMmaKV);
    };
    // S^T = K Q^T of query block t (into T1)
    auto issue_s = [&](int t) {
      const uint64_t qK = sdesc_sw128(stage_base(t), 16, 1024);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = ((k / 4) * L::PANEL + (k % 4) * 32) >> 4;
        mma_ss(tmem + L::T1, dK0 + off, qK + off, kIdescSS, k > 0 ? 1u : 0u, leader);
      }
      mma_commit(bar(L::BAR_S), leader);
    };
    // dP^T = V dO^T of query block t (into T2)
    auto issue_dp = [&](int t) {
      const uint64_t oK = sdesc_sw128(stage_base(t) + L::TILE, 16, 1024);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = ((k / 4) * L::PANEL + (k % 4) * 32) >> 4;
        mma_ss(tmem + L::T2, dV0 + off, oK + off, kIdescSS, k > 0 ? 1u : 0u, leader);
      }
      mma_commit(bar(L::BAR_S + 1), leader);
    };
    // acc += A B over the block's 128 queries: A = packed P^T or dS^T in
    // tensor memory, B = dO or Q (MN-major)
    auto issue_acc = [&](int t, uint32_t acc_col, uint32_t a_base, uint32_t b_off) {
      const uint64_t bM = sdesc_sw128(stage_base(t) + b_off, L::PANEL, 1024);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t bo = (k * 16 * 128) >> 4;
        mma_ts(tmem + acc_col, tmem + a_base + a_col(k), bM + bo, kIdescTS,
               (t > 0 || k > 0) ? 1u : 0u, leader);
      }
    };
    if (ok && nq > 0) {
      ok = wait_stage(0);
      if (ok) {
        issue_s(0);
        issue_dp(0);
      }
    }
    for (int t = 0; t < nq && ok; ++t) {
      const uint32_t ph = static_cast<uint32_t>(t) & 1u;
      ok = warp_wait_phase(bar(L::BAR_P), ph, w, kCodeMmaP);  // P^T(t) packed in T1
      if (!ok) break;
      tc_fence_after_sync();
      issue_acc(t, L::ACC0, L::T1, L::TILE);  // dV += P^T dO
      if (t + 1 < nq) {
        ok = wait_stage(t + 1);
        if (!ok) break;
        issue_s(t + 1);  // over P^T(t), read by the MMAs above
      }
      ok = warp_wait_phase(bar(L::BAR_P + 1), ph, w, kCodeMmaP);  // dS^T(t) packed in T2
      if (!ok) break;
      tc_fence_after_sync();
      issue_acc(t, L::ACC1, L::T2, 0);  // dK += dS^T Q
      mma_commit(bar(L::BAR_EMPTY + t % L::STAGES), leader);
      if (t + 1 < nq) issue_dp(t + 1);  // over dS^T(t)
    }
    if (ok) mma_commit(bar(L::BAR_FINAL), leader);
    if (!ok) {
      mma_commit(bar(L::BAR_DRAIN), leader);
      drain_phase(bar(L::BAR_DRAIN), 0u, w, kCodeDrain);
    }
    __syncwarp();
  } else if (warp < kComputeWarps) {
    // ------------- P^T, then dS^T: one key row per thread, 64 of the queries
    const int qd = warp & 3, h = warp >> 2;  // lane quadrant, column half
    const int r = qd * 32 + lane;  // key row in the block == TMEM lane
    const int key = kb * 128 + r;
    const uint32_t lb = static_cast<uint32_t>(qd * 32) << 16;
    const float c = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < nq && ok; ++t) {
      const int st = t % L::STAGES;
      const int qblk = q_first + t;
      const uint32_t ph = static_cast<uint32_t>(t) & 1u;
      // the stage's -lse2 / -D rows were written by the TMA: wait on its
      // barrier too before reading them from shared memory
      ok = warp_wait_phase(bar(L::BAR_FULL + st), static_cast<uint32_t>(t / L::STAGES) & 1u, w,
                           kCodeSoftS);
      if (ok) ok = warp_wait_phase(bar(L::BAR_S), ph, w, kCodeSoftS);
      if (!ok) break;
      tc_fence_after_sync();
      // -lse2 and -D of the block's queries (shared memory, written by the TMA)
      const uint32_t rowv = sbase + L::A_OFF_RING + st * L::A_STAGE + 2 * L::TILE;
      const bool diag = CAUSAL && qblk == kb;     // queries < key masked
      const bool tail = qblk * 128 + 128 > p.N;  // queries >= N masked
      // visible queries of this key row: [lo, lo + span) within the block
      const int lo = diag ? r : 0;
      const int span = max(0, (tail ? p.N - qblk * 128 : 128) - lo);
      // S^T of this thread's 64 queries, then P^T in fp32 (kept for dS^T)
      uint32_t pr[2][32];
      tmem_ld_32x32b_x32(tmem + lb + L::T1 + h * 64, pr[0]);
      tmem_ld_32x32b_x32(tmem + lb + L::T1 + h * 64 + 32, pr[1]);
      tmem_ld_wait(pr[0]);
      tmem_ld_wait(pr[1]);
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t pk[16];
        const int col0 = h * 64 + c2 * 32;  // first query of the chunk within the block
        if (diag || tail)
          p_chunk_t<true>(pr[c2], rowv + 4 * col0, c, col0, lo, span, pk);
        else
          p_chunk_t<false>(pr[c2], rowv + 4 * col0, c, col0, lo, span, pk);
        tmem_st_32x32b_x16(tmem + lb + L::T1 + packed_col(h) + c2 * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::BAR_P));
      // dS^T = P^T o (dP^T - D)
      ok = warp_wait_phase(bar(L::BAR_S + 1), ph, w, kCodeSoftS);
      if (!ok) break;
      tc_fence_after_sync();
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t dp[32], dk[16];
        const int col0 = h * 64 + c2 * 32;
        tmem_ld_32x32b_x32(tmem + lb + L::T2 + col0, dp);
        tmem_ld_wait(dp);
        ds_chunk_t(pr[c2], dp, rowv + 512 + 4 * col0, dk);
        tmem_st_32x32b_x16(tmem + lb + L::T2 + packed_col(h) + c2 * 16, dk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::BAR_P + 1));
    }
    if (ok && nq > 0) ok = warp_wait_phase(bar(L::BAR_FINAL), 0u, w, kCodeSoftFinal);
    if (ok) {
      tc_fence_after_sync();
      const bool valid = key < p.N;
      const size_t row = static_cast<size_t>(bh) * p.N + (valid ? key : 0);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst_row = (which == 0 ? p.dv : p.dk) + row * D;
        const float mul = which == 0 ? 1.f : p.scale;
#pragma unroll
        for (int ch = h * (D / 64); ch < (h + 1) * (D / 64); ++ch) {
          uint32_t a[32];
          tmem_ld_32x32b_x32(tmem + lb + (which == 0 ? L::ACC0 : L::ACC1) + ch * 32, a);
          tmem_ld_wait(a);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * mul, __uint_as_float(a[2 * e + 1]) * mul);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(dst_row + ch * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------ dQ

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::B_OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::B_OFF_BAR + L::NBAR * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::B_OFF_BAR + L::NBAR * 8 + 4);
  const Waiter w{abort_flag, p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tile: query block qb of head bh (heaviest first when causal); visits key
  // blocks 0..qb (causal) or all
  const int nblk = (p.N + 127) / 128;
  int bh, qb;
  if (CAUSAL) {
    int rank;
    grouped_order(static_cast<int>(blockIdx.x), nblk, p.BH, p.heads_per_group, bh, rank);
    qb = nblk - 1 - rank;
  } else {
    // a head's blocks next to each other, so its K and V stay in L2
    bh = static_cast<int>(blockIdx.x) / nblk;
    qb = static_cast<int>(blockIdx.x) % nblk;
  }
  const int nk = CAUSAL ? qb + 1 : nblk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::NBAR; ++i)
      mbar_init(bar(i), (i == L::BAR_P || i == L::BAR_P + 1) ? kComputeWarps : 1u);
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == kTmaWarp) {
    if (lane == 0) {
      const uint32_t rb = bar(L::BAR_RES);
      mbar_arrive_expect_tx(rb, 2 * L::TILE);
      for (int pn = 0; pn < L::PANELS; ++pn) {
        tma_load_3d(sbase + L::B_OFF_Q + pn * L::PANEL, &tm_q, rb, pn * 64, qb * 128, bh);
        tma_load_3d(sbase + L::B_OFF_DO + pn * L::PANEL, &tm_do, rb, pn * 64, qb * 128, bh);
      }
      int issued = 0;
      for (int t = 0; t < nk; ++t) {
        const int st = t % L::STAGES;
        const uint32_t ph = static_cast<uint32_t>(t / L::STAGES) & 1u;
        if (!wait_phase(bar(L::BAR_EMPTY + st), ph ^ 1u, w, kCodeProducerEmpty)) break;
        const uint32_t fb = bar(L::BAR_FULL + st);
        const uint32_t base = sbase + L::B_OFF_RING + st * L::B_STAGE;
        mbar_arrive_expect_tx(fb, 2 * L::TILE);
        for (int pn = 0; pn < L::PANELS; ++pn) {
          tma_load_3d(base + pn * L::PANEL, &tm_k, fb, pn * 64, t * 128, bh);
          tma_load_3d(base + L::TILE + pn * L::PANEL, &tm_v, fb, pn * 64, t * 128, bh);
        }
        ++issued;
      }
      if (*w.abort_flag) {
        drain_phase(bar(L::BAR_RES), 0u, w, kCodeDrain);
        for (int t = max(0, issued - L::STAGES); t < issued; ++t)
          drain_phase(bar(L::BAR_FULL + t % L::STAGES), static_cast<uint32_t>(t / L::STAGES) & 1u,
                      w, kCodeDrain);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    const uint32_t leader = elect_one();
    // Order per key block t: S(t+1) as soon as the elementwise warps have
    // read S(t), then dQ(t), then dP(t+1): the exponentials of block t+1 run
    // while the tensor core works on dQ(t) and dP(t+1).
    constexpr uint32_t kIdescSS = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t kIdescTS = idesc_bf16_f32(128, D, true);
    bool ok = warp_wait_phase(bar(L::BAR_RES), 0u, w, kCodeMmaQ);
    const uint64_t qA = sdesc_sw128(sbase + L::B_OFF_Q, 16, 1024);
    const uint64_t oA = sdesc_sw128(sbase + L::B_OFF_DO, 16, 1024);
    auto stage_base = [&](int t) {
      return sbase + L::B_OFF_RING + static_cast<uint32_t>((t % L::STAGES) * L::B_STAGE);
    };
    auto wait_stage = [&](int t) {
      return warp_wait_phase(bar(L::BAR_FULL + t % L::STAGES),
                             static_cast<uint32_t>(t / L::STAGES) & 1u, w, kCodeMmaKV);
    };
    // S = Q K^T of key block t (into T1)
    auto issue_s = [&](int t) {
      const uint64_t kK = sdesc_sw128(stage_base(t), 16, 1024);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = ((k / 4) * L::PANEL + (k % 4) * 32) >> 4;
        mma_ss(tmem + L::T1, qA + off, kK + off, kIdescSS, k > 0 ? 1u : 0u, leader);
      }
      mma_commit(bar(L::BAR_S), leader);
    };
    // dP = dO V^T of key block t (into T2)
    auto issue_dp = [&](int t) {
      const uint64_t vK = sdesc_sw128(stage_base(t) + L::TILE, 16, 1024);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = ((k / 4) * L::PANEL + (k % 4) * 32) >> 4;
        mma_ss(tmem + L::T2, oA + off, vK + off, kIdescSS, k > 0 ? 1u : 0u, leader);
      }
      mma_commit(bar(L::BAR_S + 1), leader);
    };
    // dQ += dS K over the block's 128 keys (dS packed in T2)
    auto issue_dq = [&](int t) {
      const uint64_t kM = sdesc_sw128(stage_base(t), L::PANEL, 1024);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t bo = (k * 16 * 128) >> 4;
        mma_ts(tmem + L::ACC0, tmem + L::T2 + a_col(k), kM + bo, kIdescTS,
               (t > 0 || k > 0) ? 1u : 0u, leader);
      }
    };
    if (ok && nk > 0) {
      ok = wait_stage(0);
      if (ok) {
        issue_s(0);
        issue_dp(0);
      }
    }
    for (int t = 0; t < nk && ok; ++t) {
      const uint32_t ph = static_cast<uint32_t>(t) & 1u;
      ok = warp_wait_phase(bar(L::BAR_P), ph, w, kCodeMmaP);  // S(t) read out of T1
      if (!ok) break;
      if (t + 1 < nk) {
        ok = wait_stage(t + 1);
        if (!ok) break;
        tc_fence_after_sync();
        issue_s(t + 1);
      }
      ok = warp_wait_phase(bar(L::BAR_P + 1), ph, w, kCodeMmaP);  // dS(t) packed in T2
      if (!ok) break;
      tc_fence_after_sync();
      issue_dq(t);
      mma_commit(bar(L::BAR_EMPTY + t % L::STAGES), leader);
      if (t + 1 < nk) issue_dp(t + 1);  // over dS(t), read by the MMAs above
    }
    if (ok) mma_commit(bar(L::BAR_FINAL), leader);
    if (!ok) {
      mma_commit(bar(L::BAR_DRAIN), leader);
      drain_phase(bar(L::BAR_DRAIN), 0u, w, kCodeDrain);
    }
    __syncwarp();
  } else if (warp < kComputeWarps) {
    const int qd = warp & 3, h = warp >> 2;  // lane quadrant, column half
    const int r = qd * 32 + lane;  // query row in the block == TMEM lane
    const int qrow = qb * 128 + r;
    const uint32_t lb = static_cast<uint32_t>(qd * 32) << 16;
    const float c = p.scale_log2;
    const size_t prow = static_cast<size_t>(bh) * p.Npad + qrow;
    const float nl2 = p.lse2[prow];   // -LSE * log2(e)
    const float nds = p.dsum[prow];   // -D
    bool ok = true;
    for (int t = 0; t < nk && ok; ++t) {
      const uint32_t ph = static_cast<uint32_t>(t) & 1u;
      ok = warp_wait_phase(bar(L::BAR_S), ph, w, kCodeSoftS);
      if (!ok) break;
      tc_fence_after_sync();
      // S of this thread's 64 keys; T1 is free for S(t+1) once they are read
      uint32_t pr[2][32];
      tmem_ld_32x32b_x32(tmem + lb + L::T1 + h * 64, pr[0]);
      tmem_ld_32x32b_x32(tmem + lb + L::T1 + h * 64 + 32, pr[1]);
      tmem_ld_wait(pr[0]);
      tmem_ld_wait(pr[1]);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::BAR_P));
      const bool diag = CAUSAL && t == qb;
      const bool tail = t * 128 + 128 > p.N;
      int lim = 128;  // keys [0, lim) of this block are visible
      if (tail) lim = p.N - t * 128;
      if (diag) lim = min(lim, qrow - t * 128 + 1);
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col0 = h * 64 + c2 * 32;  // first key of the chunk within the block
        if (diag || tail)
          p_chunk_q<true>(pr[c2], c, nl2, col0, lim);
        else
          p_chunk_q<false>(pr[c2], c, nl2, col0, lim);
      }
      // dS = P o (dP - D), packed over the dP columns already read
      ok = warp_wait_phase(bar(L::BAR_S + 1), ph, w, kCodeSoftS);
      if (!ok) break;
      tc_fence_after_sync();
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t dp[32], dk[16];
        const int col0 = h * 64 + c2 * 32;
        tmem_ld_32x32b_x32(tmem + lb + L::T2 + col0, dp);
        tmem_ld_wait(dp);
        ds_chunk_q(pr[c2], dp, nds, dk);
        tmem_st_32x32b_x16(tmem + lb + L::T2 + packed_col(h) + c2 * 16, dk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::BAR_P + 1));
    }
    if (ok && nk > 0) ok = warp_wait_phase(bar(L::BAR_FINAL), 0u, w, kCodeSoftFinal);
    if (ok) {
      tc_fence_after_sync();
      const bool valid = qrow < p.N;
      __nv_bfloat16* dst_row = p.dq + (static_cast<size_t>(bh) * p.N + (valid ? qrow : 0)) * D;
#pragma unroll
      for (int ch = h * (D / 64); ch < (h + 1) * (D / 64); ++ch) {
        uint32_t a[32];
        tmem_ld_32x32b_x32(tmem + lb + L::ACC0 + ch * 32, a);
        tmem_ld_wait(a);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(dst_row + ch * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <typename K>
cudaError_t set_smem(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_d(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                         const CUtensorMap* tdo, const BwdParams& p, cudaStream_t stream) {
  using L = BwdLayout<D>;
  cudaError_t e;
  if ((e = set_smem(bwd_dkdv_kernel<D, CAUSAL>, L::A_SMEM)) != cudaSuccess) return e;
  if ((e = set_smem(bwd_dq_kernel<D, CAUSAL>, L::B_SMEM)) != cudaSuccess) return e;
  const unsigned nblk = static_cast<unsigned>((p.N + 127) / 128);
  const unsigned grid = nblk * static_cast<unsigned>(p.BH);
  bwd_dkdv_kernel<D, CAUSAL><<<grid, kBwdThreads, L::A_SMEM, stream>>>(*tq, *tk, *tv, *tdo, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_dq_kernel<D, CAUSAL><<<grid, kBwdThreads, L::B_SMEM, stream>>>(*tq, *tk, *tv, *tdo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                       const CUtensorMap* tdo, const BwdParams& p, const void* o, const void* dout,
                       const float* lse, int d, bool causal, cudaStream_t stream) {
  cudaError_t e = d == 64    ? launch_preprocess<64>(o, dout, lse, p, stream)
                  : d == 128 ? launch_preprocess<128>(o, dout, lse, p, stream)
                             : launch_preprocess<256>(o, dout, lse, p, stream);
  if (e != cudaSuccess) return e;
  if (d == 64) return causal ? launch_bwd_d<64, true>(tq, tk, tv, tdo, p, stream)
                             : launch_bwd_d<64, false>(tq, tk, tv, tdo, p, stream);
  if (d == 128) return causal ? launch_bwd_d<128, true>(tq, tk, tv, tdo, p, stream)
                              : launch_bwd_d<128, false>(tq, tk, tv, tdo, p, stream);
  if (d == 256) return launch_bwd_d256(tq, tk, tv, tdo, p, causal, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ea51
