// Backward pass at head dim 256 for sm_103a: dQ, dK and dV of
// O = softmax(scale * Q K^T [+ causal mask]) V, with the definitions of
// attn_bwd.cu (P recomputed from the forward's log-sum-exp, D = rowsum(dO o O),
// dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO).
//
// At d = 256 a 128-row bf16 tile is 64 KiB and one d-column fp32
// accumulator is half of the tensor memory, so the two kernels used at
// d <= 128 do not fit: K and V resident plus one {Q, dO} stage is 256 KiB of
// shared memory, and dK and dV together fill all 512 columns before S and dP
// have any.  Three kernels instead, each with one 256-column accumulator and
// a resident 128-row block, over 128-row blocks of the other side:
//
//   dV  one CTA per 128-key block, K resident:  S^T = K Q^T into one of two
//       128-column buffers, P^T packed to bf16 over it, dV += P^T dO;
//   dK  one CTA per 128-key block, K and V resident:  S^T, dP^T = V dO^T,
//       dS^T packed over dP^T, dK += dS^T Q;
//   dQ  one CTA per 128-query block, Q and dO resident:  S = Q K^T,
//       dP = dO V^T, dS packed, dQ += dS K.
//
// The streamed blocks do not fit whole next to the resident ones, so they
// pass through a ring of 16 KiB slots, one 64-column panel (128 rows x 128
// bytes) each, in the order the tensor core consumes them: the four panels
// of a block feed the four K-step groups of S (or dP) one by one, each slot
// refilled as soon as its MMAs have run; the accumulation takes all four
// panels of its block at once (one N = 256 product over four adjacent
// slots), so in dK and dQ the block used twice (Q, K) is loaded twice, the
// second time from L2.  2 x 64 + 6 x 16 = 224 KiB of shared memory (dV: 64 +
// 8 x 16).  Every product has N >= 128.  The per-query -LSE log2(e) and -D
// rows of the dK / dV kernels travel in a two-slot ring that the elementwise
// warps release.  Every wait is bounded, as in the other kernels.
#include <cuda_bf16.h>

#include <cstdint>

#include "bwd_common.cuh"

namespace ea51 {
namespace {

enum Mode : int { kDV = 0, kDK = 1, kDQ = 2 };

constexpr uint32_t kCodeSmemAlign = 0x1f2;   // shared memory not 1024-byte aligned
constexpr uint32_t kCodeRingOrder = 0x1f3;   // accumulation panels not in adjacent slots

template <int MODE>
struct Bwd256 {
  static constexpr int D = 256;
  static constexpr int PANELS = D / 64;             // 128-byte column panels per row
  static constexpr int PANEL = 128 * 128;           // one panel of a 128-row block, 16 KiB
  static constexpr int TILE = 128 * D * 2;          // a whole 128-row block, 64 KiB
  static constexpr int NRES = MODE == kDV ? 1 : 2;  // resident blocks (K; K, V; Q, dO)
  static constexpr int RING = MODE == kDV ? 8 : 6;  // panel slots
  static constexpr int AUX = 2;                     // -lse2 / -D row slots
  static constexpr int AUX_BYTES = 2 * 128 * 4;     // -lse2 at +0, -D at +512
  static constexpr int OFF_RING = NRES * TILE;
  static constexpr int OFF_AUX = OFF_RING + RING * PANEL;
  static constexpr int OFF_BAR = OFF_AUX + AUX * AUX_BYTES;
  // barriers: resident blocks; ring full / empty; aux full / empty; then
  // S0, S1 (dV: S^T in buffer 0 / 1; dK, dQ: S and dP computed), P0, P1
  // (dV: P^T of buffer 0 / 1 packed; dK, dQ: S read out, dS packed; one
  // arrival per elementwise warp), final, drain
  static constexpr int BAR_RES = 0, BAR_FULL = 1, BAR_EMPTY = BAR_FULL + RING,
                       BAR_AUXF = BAR_EMPTY + RING, BAR_AUXE = BAR_AUXF + AUX,
                       BAR_S0 = BAR_AUXE + AUX, BAR_S1 = BAR_S0 + 1, BAR_P0 = BAR_S1 + 1,
                       BAR_P1 = BAR_P0 + 1, BAR_FINAL = BAR_P1 + 1, BAR_DRAIN = BAR_FINAL + 1,
                       NBAR = BAR_DRAIN + 1;
  // + abort flag and tensor-memory slot.  No alignment slack: the kernel
  // checks that its dynamic shared memory starts on a 1024-byte boundary.
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 8;
  // tensor memory: T1, T2 (128 columns each: S^T / S and dP^T / dP; in dV
  // the two S^T buffers), the 256-column accumulator at ACC
  static constexpr int T1 = 0, T2 = 128, ACC = 256;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(TILE % 1024 == 0 && PANEL % 1024 == 0 && OFF_AUX % 1024 == 0, "alignment");
};

// Kernel MODE over 128-row blocks; `tm_*` are per-head 3-D maps with
// 64-column x 128-row boxes (one panel).
template <int MODE, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  using L = Bwd256<MODE>;
  constexpr bool KEY_ROWS = MODE != kDQ;  // tensor-memory lanes are keys (dK, dV) or queries (dQ)
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment; no slack was reserved
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, kCodeSmemAlign);
    return;
  }
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_BAR + L::NBAR * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + L::NBAR * 8 + 4);
  const Waiter w{abort_flag, p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // This CTA's 128-row block `blk` of head bh, and the blocks of the other
  // side it visits: [first, first + n).  Causal: a key block sees the queries
  // at or after its first key, a query block the keys up to its last query;
  // heaviest blocks first.
  const int nblk = (p.N + 127) / 128;
  int bh, blk;
  if (CAUSAL) {
    int rank;
    grouped_order(static_cast<int>(blockIdx.x), nblk, p.BH, p.heads_per_group, bh, rank);
    blk = KEY_ROWS ? rank : nblk - 1 - rank;
  } else {
    bh = static_cast<int>(blockIdx.x) / nblk;
    blk = static_cast<int>(blockIdx.x) % nblk;
  }
  const int first = (CAUSAL && KEY_ROWS) ? blk : 0;
  const int n = CAUSAL ? (KEY_ROWS ? nblk - blk : blk + 1) : nblk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::NBAR; ++i) {
      const bool per_warp = i == L::BAR_P0 || i == L::BAR_P1 || (i >= L::BAR_AUXE && i < L::BAR_AUXE + L::AUX);
      mbar_init(bar(i), per_warp ? kComputeWarps : 1u);
    }
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

  // Operand maps: resident R0 (S side), R1 (dP side); streamed X (S side,
  // and the accumulation's B in dK / dQ), W (dP side; dV: the accumulation's
  // B, dO).
  const CUtensorMap* map_r0 = MODE == kDQ ? &tm_q : &tm_k;
  const CUtensorMap* map_r1 = MODE == kDQ ? &tm_do : &tm_v;
  const CUtensorMap* map_x = MODE == kDQ ? &tm_k : &tm_q;
  const CUtensorMap* map_w = MODE == kDQ ? &tm_v : &tm_do;
  auto slot_addr = [&](int i) {
    return sbase + L::OFF_RING + static_cast<uint32_t>((i % L::RING) * L::PANEL);
  };
  auto aux_addr = [&](int t) {
    return sbase + L::OFF_AUX + static_cast<uint32_t>((t % L::AUX) * L::AUX_BYTES);
  };

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- TMA
    // Ring order = MMA order, four panels per block.  dV: S(0), S(1), then
    // per block t: dV(t) (dO_t), S(t+2) (Q_t+2).  dK / dQ: S(0), dP(0), then
    // per block t: S(t+1) (X), acc(t) (X_t again), dP(t+1) (W).  A block
    // is 4 items, so the accumulation's four panels start at a multiple of
    // 4 (dV, 8 slots: slot 0 or 4), or at 12 + 12t, 8 + 12t for the last
    // block (dK, dQ, 6 slots: slot 0 or 2); never across the ring's end.
    if (lane == 0) {
      const uint32_t rb = bar(L::BAR_RES);
      mbar_arrive_expect_tx(rb, L::NRES * L::TILE);
      for (int r = 0; r < L::NRES; ++r)
        for (int pn = 0; pn < L::PANELS; ++pn)
          tma_load_3d(sbase + r * L::TILE + pn * L::PANEL, r ? map_r1 : map_r0, rb, pn * 64,
                      blk * 128, bh);
      int issued = 0, aux_issued = 0;
      bool ok = true;
      auto load_block = [&](const CUtensorMap* map, int t) {  // block t's four panels
        for (int pn = 0; pn < L::PANELS && ok; ++pn) {
          const int st = issued % L::RING;
          ok = wait_phase(bar(L::BAR_EMPTY + st), (static_cast<uint32_t>(issued / L::RING) & 1u) ^ 1u,
                          w, kCodeProducerEmpty);
          if (!ok) return;
          const uint32_t fb = bar(L::BAR_FULL + st);
          mbar_arrive_expect_tx(fb, L::PANEL);
          tma_load_3d(slot_addr(issued), map, fb, pn * 64, (first + t) * 128, bh);
          ++issued;
        }
      };
      auto load_aux = [&](int t) {  // -lse2 and -D of query block t (dK, dV)
        if (!KEY_ROWS || !ok) return;
        const int s = t % L::AUX;
        ok = wait_phase(bar(L::BAR_AUXE + s), (static_cast<uint32_t>(t / L::AUX) & 1u) ^ 1u, w,
                        kCodeProducerEmpty);
        if (!ok) return;
        const uint32_t fb = bar(L::BAR_AUXF + s);
        const size_t rowoff = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(first + t) * 128;
        mbar_arrive_expect_tx(fb, L::AUX_BYTES);
        bulk_load(aux_addr(t), p.lse2 + rowoff, L::AUX_BYTES / 2, fb);
        bulk_load(aux_addr(t) + L::AUX_BYTES / 2, p.dsum + rowoff, L::AUX_BYTES / 2, fb);
        ++aux_issued;
      };
      if (MODE == kDV) {
        load_aux(0);
        load_block(map_x, 0);
        if (n > 1) {
          load_aux(1);
          load_block(map_x, 1);
        }
        for (int t = 0; t < n && ok; ++t) {
          load_block(map_w, t);
          if (t + 2 < n) {
            load_aux(t + 2);
            load_block(map_x, t + 2);
          }
        }
      } else {
        load_aux(0);
        load_block(map_x, 0);
        load_block(map_w, 0);
        for (int t = 0; t < n && ok; ++t) {
          if (t + 1 < n) {
            load_aux(t + 1);
            load_block(map_x, t + 1);
          }
          load_block(map_x, t);
          if (t + 1 < n) load_block(map_w, t + 1);
        }
      }
      if (*w.abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        drain_phase(rb, 0u, w, kCodeDrain);
        for (int i = max(0, issued - L::RING); i < issued; ++i)
          drain_phase(bar(L::BAR_FULL + i % L::RING), static_cast<uint32_t>(i / L::RING) & 1u, w,
                      kCodeDrain);
        for (int t = max(0, aux_issued - L::AUX); t < aux_issued; ++t)
          drain_phase(bar(L::BAR_AUXF + t % L::AUX), static_cast<uint32_t>(t / L::AUX) & 1u, w,
                      kCodeDrain);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    const uint32_t leader = elect_one();
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);   // S, dP: both K-major
    constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, 256, true);  // acc: B MN-major
    bool ok = warp_wait_phase(bar(L::BAR_RES), 0u, w, kCodeMmaQ);
    int it = 0;  // next ring item
    auto wait_item = [&](int i) {
      return warp_wait_phase(bar(L::BAR_FULL + i % L::RING), static_cast<uint32_t>(i / L::RING) & 1u,
                             w, kCodeMmaKV);
    };
    auto release = [&]() {
      mma_commit(bar(L::BAR_EMPTY + it % L::RING), leader);
      ++it;
    };
    // tmem[d_col] = resident block x streamed block^T over d, one panel
    // (four K-steps) per ring item; arrives on `done`
    auto s_product = [&](int d_col, uint32_t res, uint32_t done) -> bool {
      for (int pn = 0; pn < L::PANELS; ++pn) {
        if (!wait_item(it)) return false;
        tc_fence_after_sync();
        const uint64_t a0 = sdesc_sw128(res + pn * L::PANEL, 16, 1024);
        const uint64_t b0 = sdesc_sw128(slot_addr(it), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem + d_col, a0 + ((kk * 32) >> 4), b0 + ((kk * 32) >> 4), kIdescS,
                 (pn > 0 || kk > 0) ? 1u : 0u, leader);
        release();
      }
      mma_commit(done, leader);
      return true;
    };
    // ACC (+)= packed A at tmem[a_base] (the block's 128 rows as K) x the
    // streamed block (128 rows x 256 columns, MN-major) in four adjacent slots
    auto acc_product = [&](int t, int a_base) -> bool {
      if ((it % L::RING) + L::PANELS > L::RING) {
        if (lane == 0) {
          atomicCAS(p.status, 0u, kCodeRingOrder);
          *w.abort_flag = 1u;
        }
        __syncwarp();
        return false;
      }
      for (int pn = 0; pn < L::PANELS; ++pn)
        if (!wait_item(it + pn)) return false;
      tc_fence_after_sync();
      const uint64_t b0 = sdesc_sw128(slot_addr(it), L::PANEL, 1024);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_ts(tmem + L::ACC, tmem + a_base + a_col(k), b0 + ((k * 16 * 128) >> 4), kIdescAcc,
               (t > 0 || k > 0) ? 1u : 0u, leader);
      for (int pn = 0; pn < L::PANELS; ++pn) release();
      return true;
    };
    const uint32_t r0 = sbase, r1 = sbase + L::TILE;
    if (MODE == kDV) {
      // two S^T buffers: S^T(t+2) is computed while P^T(t+1) is formed
      for (int b = 0; b < 2 && b < n && ok; ++b) ok = s_product(L::T1 + 128 * b, r0, bar(L::BAR_S0 + b));
      for (int t = 0; t < n && ok; ++t) {
        const int b = t & 1;
        ok = warp_wait_phase(bar(L::BAR_P0 + b), static_cast<uint32_t>(t >> 1) & 1u, w, kCodeMmaP);
        if (!ok) break;
        tc_fence_after_sync();
        ok = acc_product(t, L::T1 + 128 * b);  // dV += P^T dO
        if (ok && t + 2 < n) ok = s_product(L::T1 + 128 * b, r0, bar(L::BAR_S0 + b));  // over P^T(t)
      }
    } else {
      if (ok) ok = s_product(L::T1, r0, bar(L::BAR_S0));
      if (ok) ok = s_product(L::T2, r1, bar(L::BAR_S1));
      for (int t = 0; t < n && ok; ++t) {
        const uint32_t ph = static_cast<uint32_t>(t) & 1u;
        ok = warp_wait_phase(bar(L::BAR_P0), ph, w, kCodeMmaP);  // S(t) read out of T1
        if (!ok) break;
        if (t + 1 < n) {
          ok = s_product(L::T1, r0, bar(L::BAR_S0));
          if (!ok) break;
        }
        ok = warp_wait_phase(bar(L::BAR_P1), ph, w, kCodeMmaP);  // dS(t) packed in T2
        if (!ok) break;
        tc_fence_after_sync();
        ok = acc_product(t, L::T2);  // dK += dS^T Q or dQ += dS K
        if (ok && t + 1 < n) ok = s_product(L::T2, r1, bar(L::BAR_S1));  // over dS(t)
      }
    }
    if (ok) mma_commit(bar(L::BAR_FINAL), leader);
    if (!ok) {
      // Let every MMA this warp issued finish before tensor memory is freed.
      mma_commit(bar(L::BAR_DRAIN), leader);
      drain_phase(bar(L::BAR_DRAIN), 0u, w, kCodeDrain);
    }
    __syncwarp();
  } else if (warp < kComputeWarps) {
    // ------ P (then dS): one row per thread, 64 of the block's 128 columns
    const int qd = warp & 3, h = warp >> 2;  // lane quadrant, column half
    const int r = qd * 32 + lane;
    const int row = blk * 128 + r;  // key (dK, dV) or query (dQ) of this lane
    const uint32_t lb = static_cast<uint32_t>(qd * 32) << 16;
    const float c = p.scale_log2;
    float nl2 = 0.f, nds = 0.f;
    if (!KEY_ROWS) {
      const size_t prow = static_cast<size_t>(bh) * p.Npad + row;  // row < Npad
      nl2 = p.lse2[prow];  // -LSE * log2(e)
      nds = p.dsum[prow];  // -D
    }
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      const int s0 = (first + t) * 128;  // first row of the streamed block
      if (KEY_ROWS) {
        ok = warp_wait_phase(bar(L::BAR_AUXF + t % L::AUX), static_cast<uint32_t>(t / L::AUX) & 1u,
                             w, kCodeSoftS);
        if (!ok) break;
      }
      const int b = MODE == kDV ? (t & 1) : 0;
      const uint32_t sph = static_cast<uint32_t>(MODE == kDV ? (t >> 1) : t) & 1u;
      ok = warp_wait_phase(bar(L::BAR_S0 + b), sph, w, kCodeSoftS);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t s_t = tmem + lb + L::T1 + 128 * b;
      uint32_t pr[2][32];
      tmem_ld_32x32b_x32(s_t + h * 64, pr[0]);
      tmem_ld_32x32b_x32(s_t + h * 64 + 32, pr[1]);
      tmem_ld_wait(pr[0]);
      tmem_ld_wait(pr[1]);
      if (MODE != kDV) {  // T1 is free for S(t+1)
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::BAR_P0));
      }
      // causal diagonal block (the first one visited) and ragged tail
      const bool diag = CAUSAL && s0 == blk * 128;
      const bool tail = s0 + 128 > p.N;
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col0 = h * 64 + c2 * 32;  // first column of the chunk within the block
        uint32_t pk[16];
        if (KEY_ROWS) {
          // queries [lo, lo + span) of the block are visible to key `row`
          const int lo = diag ? r : 0;
          const int span = max(0, (tail ? p.N - s0 : 128) - lo);
          const uint32_t nl_row = aux_addr(t) + 4 * col0;
          if (diag || tail)
            p_chunk_t<true>(pr[c2], nl_row, c, col0, lo, span, pk);
          else
            p_chunk_t<false>(pr[c2], nl_row, c, col0, lo, span, pk);
        } else {
          // keys [0, lim) of the block are visible to query `row`
          int lim = tail ? p.N - s0 : 128;
          if (diag) lim = min(lim, r + 1);
          if (diag || tail)
            p_chunk_q<true>(pr[c2], c, nl2, col0, lim);
          else
            p_chunk_q<false>(pr[c2], c, nl2, col0, lim);
        }
        // dV: P^T as bf16 over the S^T columns this half has read, the A
        // operand of dV += P^T dO
        if (MODE == kDV) tmem_st_32x32b_x16(s_t + packed_col(h) + c2 * 16, pk);
      }
      if (MODE == kDV) {
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(L::BAR_P0 + b));
          mbar_arrive(bar(L::BAR_AUXE + t % L::AUX));
        }
        continue;
      }
      // dS = P o (dP - D), packed over the dP columns already read
      ok = warp_wait_phase(bar(L::BAR_S1), static_cast<uint32_t>(t) & 1u, w, kCodeSoftS);
      if (!ok) break;
      tc_fence_after_sync();
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col0 = h * 64 + c2 * 32;
        uint32_t dp[32], ds[16];
        tmem_ld_32x32b_x32(tmem + lb + L::T2 + col0, dp);
        tmem_ld_wait(dp);
        if (KEY_ROWS)
          ds_chunk_t(pr[c2], dp, aux_addr(t) + L::AUX_BYTES / 2 + 4 * col0, ds);
        else
          ds_chunk_q(pr[c2], dp, nds, ds);
        tmem_st_32x32b_x16(tmem + lb + L::T2 + packed_col(h) + c2 * 16, ds);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(L::BAR_P1));
        if (KEY_ROWS) mbar_arrive(bar(L::BAR_AUXE + t % L::AUX));
      }
    }
    if (ok && n > 0) ok = warp_wait_phase(bar(L::BAR_FINAL), 0u, w, kCodeSoftFinal);
    if (ok) {
      // this warp's 128 of the 256 accumulator columns, scaled, as bf16
      tc_fence_after_sync();
      const bool valid = row < p.N;
      __nv_bfloat16* out = MODE == kDV ? p.dv : (MODE == kDK ? p.dk : p.dq);
      const float mul = MODE == kDV ? 1.f : p.scale;
      __nv_bfloat16* dst_row = out + (static_cast<size_t>(bh) * p.N + (valid ? row : 0)) * L::D;
#pragma unroll 1
      for (int ch = h * 4; ch < h * 4 + 4; ++ch) {
        uint32_t a[32];
        tmem_ld_32x32b_x32(tmem + lb + L::ACC + ch * 32, a);
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
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int MODE, bool CAUSAL>
cudaError_t launch_mode(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                        const CUtensorMap* tdo, const BwdParams& p, cudaStream_t stream) {
  using L = Bwd256<MODE>;
  cudaError_t e = cudaFuncSetAttribute(bwd256_kernel<MODE, CAUSAL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>((p.N + 127) / 128) * static_cast<unsigned>(p.BH);
  bwd256_kernel<MODE, CAUSAL><<<grid, kBwdThreads, L::SMEM, stream>>>(*tq, *tk, *tv, *tdo, p);
  return cudaGetLastError();
}

template <bool CAUSAL>
cudaError_t launch_all(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                       const CUtensorMap* tdo, const BwdParams& p, cudaStream_t stream) {
  cudaError_t e;
  if ((e = launch_mode<kDV, CAUSAL>(tq, tk, tv, tdo, p, stream)) != cudaSuccess) return e;
  if ((e = launch_mode<kDK, CAUSAL>(tq, tk, tv, tdo, p, stream)) != cudaSuccess) return e;
  return launch_mode<kDQ, CAUSAL>(tq, tk, tv, tdo, p, stream);
}

}  // namespace

cudaError_t launch_bwd_d256(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                            const CUtensorMap* tdo, const BwdParams& p, bool causal,
                            cudaStream_t stream) {
  return causal ? launch_all<true>(tq, tk, tv, tdo, p, stream)
                : launch_all<false>(tq, tk, tv, tdo, p, stream);
}

}  // namespace ea51
