// Fused exact attention forward for sm_103a (GB300).
//
// One CTA owns NQ query tiles of 128 rows of one (batch, head) and streams
// every visible key/value tile of that head through shared memory once:
//
//   TMA warp      Q tiles once, then K_j / V_j tiles into a STAGES-deep ring
//                 (full / empty mbarriers per slot).
//   MMA warp      one thread issues tcgen05.mma: S = Q K_j^T into tensor
//                 memory (fp32), later O += P V_j with P read from tensor
//                 memory (bf16, written over the S columns it came from).
//   softmax WGs   one warpgroup per query tile, one thread per row: loads the
//                 S row from tensor memory, applies scale and mask, keeps the
//                 running row max m and row sum l, writes P = exp2(x - m) as
//                 bf16 back to tensor memory, and rescales its O row in
//                 tensor memory when the max grew by more than 2^32.
//                 The epilogue divides by l and writes O (bf16) and LSE.
//
// The N x N score matrix only ever lives in tensor memory, one 128 x BN tile
// at a time ("Tri Dao: prediction": kernel fusion + tiling into fast memory +
// the online-softmax rescaling that "still gets the right answer").  Causal
// runs visit only key tiles at or below the diagonal ("the softmax of the
// triangular matrix", HN item 40939030) and mask inside diagonal tiles.
//
// Every mbarrier wait is bounded (about two seconds); a wait that gives up
// records a code in a device status word, sets a CTA-wide abort flag, drains
// its own in-flight copies / MMAs and lets the CTA exit, so a fault in the
// pipeline cannot hang the GPU.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "fwd_dispatch.h"
#include "ptx.cuh"

namespace ea51 {

constexpr int BM = 128;                      // query rows per tile (tcgen05 M)
// log2 units: O and l are rescaled only when a row's max grows by more than
// this; otherwise P keeps the old exponent offset (bf16 values up to 2^32).
// The range is ample: O and l accumulate in fp32, so a row of N keys with
// |V| <= Vmax stays below 2^32 * N * Vmax, far inside 2^128, and bf16 keeps
// 8 significant bits at any exponent.  A stale offset leaves a dominant
// weight at 2^x with x in (0, 32] instead of exactly 1, so its rounding to
// bf16 (up to 2^-9 relative) would not cancel against the fp32 normaliser;
// the softmax therefore gives O's normaliser each tile's largest weight as
// rounded (see softmax_role).  Rescales cost a wait for the previous P.V and
// a pass over O in tensor memory; with keys whose scores jump (a few keys
// scaled by 8) a threshold of 8 rescaled some row of most warps on most
// tiles.
constexpr float kRescaleThreshold = 32.0f;
// e4m3 P is 8 bits wide: the threshold and the shift of P share its 8
// binades of headroom below 448 (see kF8Shift).
constexpr float kRescaleThresholdF8 = 4.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// Per-head-dim tiling.  BN = keys per tile, NQ = query tiles per CTA,
// NSB = S buffers per query tile in tensor memory, STAGES = K/V ring slots.
template <int D>
struct Shape;
template <>
struct Shape<64> {
  static constexpr int BN = 128, NQ = 2, NSB = 1, STAGES = 8;
};
template <>
struct Shape<128> {
  static constexpr int BN = 128, NQ = 2, NSB = 1, STAGES = 4;
};
template <>
struct Shape<256> {
  // 2 * 128 + 256 = 512 tensor-memory columns; Q + one K and one V tile =
  // 192 KiB of shared memory
  static constexpr int BN = 128, NQ = 1, NSB = 2, STAGES = 2;
};

// e4m3 at d = 256: 128-key tiles, one query tile, two S buffers: 2 * 128 +
// 256 = 512 tensor-memory columns; the 8-bit K/V tiles (32 KiB) fit a
// four-slot ring.
struct ShapeE4M3D256 {
  static constexpr int BN = 128, NQ = 1, NSB = 2, STAGES = 2;
};
// Two CTAs per SM (d = 64, short rows): one query tile and one S buffer per
// CTA, so the two query tiles that take turns on the tensor core come from
// two CTAs.  Each CTA fits half the SM: 128 + 64 <= 256 tensor-memory
// columns, Q and a four-slot K/V ring in 80 KiB of shared memory.  Short rows
// gain a little: one CTA's set-up, first loads and epilogue overlap the other
// CTA's key tiles, and a launch has twice as many, lighter CTAs to balance.
template <int D>
struct ShapeTwo {
  static_assert(D == 64, "two CTAs per SM: head dim 64");
  static constexpr int BN = 128, NQ = 1, NSB = 1, STAGES = 4;
};
// Small grids (d = 64, 128): one query tile and two S buffers per CTA, so a
// launch whose default grid (two query tiles per CTA) would not fill the
// GPU once has twice as many CTAs.  Two query tiles per CTA hide more of
// each softmax where the grid is full (the default), but on a half-empty
// grid the idle SMs cost more: B=1 H=4 N=8192 d=128 causal e4m3 743 -> 1115
// TFLOP/s.
template <int D>
struct ShapeSolo {
  static_assert(D == 64 || D == 128, "one query tile per CTA: head dim 64 or 128");
  static constexpr int BN = 128, NQ = 1, NSB = 2, STAGES = 4;
};

// Launch shapes: the head dim's default, two CTAs per SM (d = 64 short
// rows), one query tile per CTA (small grids).
enum ShapeKind : int { kShapeDefault = 0, kShapeTwo = 1, kShapeSolo = 2 };

template <int D, bool F8, int SK>
struct ShapeOf {
  using T = Shape<D>;
};
template <>
struct ShapeOf<256, true, kShapeDefault> {
  using T = ShapeE4M3D256;
};
template <int D, bool F8>
struct ShapeOf<D, F8, kShapeTwo> {
  using T = ShapeTwo<D>;
};
template <int D, bool F8>
struct ShapeOf<D, F8, kShapeSolo> {
  using T = ShapeSolo<D>;
};

// F8: Q, K, V in e4m3 (8-bit tiles, half the bytes, twice the ring slots);
// the V tile is read MN-major as stored, as in bf16.
template <int D, bool F8 = false, int SK = kShapeDefault>
struct Layout {
  using Sh = typename ShapeOf<D, F8, SK>::T;
  static constexpr bool TWO = SK == kShapeTwo;
  static constexpr int MIN_BLOCKS = TWO ? 2 : 1;  // CTAs resident per SM
  static constexpr int EB = F8 ? 1 : 2;  // bytes per Q/K/V element
  static constexpr int BN = Sh::BN, NQ = Sh::NQ, NSB = Sh::NSB,
                       STAGES = F8 ? 2 * Sh::STAGES : Sh::STAGES;
  // Rows of Q, K and V tiles are split into column panels of SWZ bytes, each
  // swizzled over that span (128 bytes; 64 for the 64-byte rows of e4m3 at
  // d = 64); 8 rows of a panel form one swizzle atom of SBO bytes.
  static constexpr int SWZ = D * EB >= 128 ? 128 : D * EB;
  static constexpr int PANELS = D * EB / SWZ;  // column panels per Q/K/V row
  static constexpr int PANEL_ELEMS = SWZ / EB;
  static constexpr int SBO = 8 * SWZ;
  static constexpr int KPP = SWZ / 32;            // 32-byte K-steps per panel
  static constexpr int KSTEPS_QK = D * EB / 32;   // 32-byte K-steps of S = Q K^T
  static constexpr int KSTEPS_PV = BN * EB / 32;  // and of O += P V
  static constexpr int KEYS_PER_KSTEP = 32 / EB;  // rows of V one P.V K-step reads
  // P is handed to the MMA warp in P_PIECES parts (32-key chunks each) so
  // that P.V starts before the whole of P is computed
  static constexpr int P_PIECES = BN >= 128 ? 2 : 1;
  // bf16 O leaves through TMA stores staged in the Q buffer (same size) in
  // the two-CTA shape; the others store rows directly.  Measured (GB300, A/B
  // of the same build): B=8 H=12 N=1024 d=64 causal 353 -> 368 TFLOP/s with
  // the TMA stores, but B=1 H=32 N=16384 d=128 causal 1401 -> 1348 and the
  // rest within 1 %.
  static constexpr bool TMA_EPILOGUE = !F8 && TWO;
  static constexpr int Q_PANEL = BM * SWZ;
  static constexpr int Q_BYTES = BM * D * EB;
  static constexpr int KV_PANEL = BN * SWZ;
  static constexpr int KV_BYTES = BN * D * EB;
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = NQ * Q_BYTES;
  static constexpr int OFF_BAR = OFF_KV + STAGES * KV_BYTES;
  // barrier indices
  static constexpr int B_QFULL = 0;
  static constexpr int B_KVFULL = B_QFULL + NQ;
  static constexpr int B_KVEMPTY = B_KVFULL + STAGES;
  static constexpr int B_SFULL = B_KVEMPTY + STAGES;  // [NQ][NSB]
  static constexpr int B_PFULL = B_SFULL + NQ * NSB;  // [NQ][NSB][P_PIECES]
  static constexpr int B_ODONE = B_PFULL + NQ * NSB * P_PIECES;  // [NQ]
  static constexpr int B_OFINAL = B_ODONE + NQ;       // [NQ]
  static constexpr int B_DRAIN = B_OFINAL + NQ;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for 1024-byte alignment
  // tensor memory columns (fp32 each): all 512, or half for two CTAs per SM
  static constexpr int TMEM_COLS = 512 / MIN_BLOCKS;
  __host__ __device__ static constexpr int s_col(int q, int b) { return (q * NSB + b) * BN; }
  __host__ __device__ static constexpr int o_col(int q) { return NQ * NSB * BN + q * D; }
  // warps: [0, 4*NQ) softmax warpgroups, then TMA, MMA, two spare warps
  static constexpr int TMA_WARP = 4 * NQ;
  static constexpr int MMA_WARP = 4 * NQ + 1;
  // bf16 d = 256: K and V tiles loaded by two producer warps (V_WARP the V
  // tiles); the e4m3 shape's four ring slots keep up with one
  static constexpr bool SPLIT_LOAD = D == 256 && !F8;
  static constexpr int V_WARP = 4 * NQ + 2;
  static constexpr int THREADS = (NQ + 1) * 128;
  // Register split (setmaxnreg) when the launch budget per thread is tight:
  // 384 threads launch with 168 registers each (65536 / 384, rounded down to
  // 8).  The control warpgroup drops to 88 and the two softmax warpgroups
  // rise to 208: 2 * 128 * (208 - 168) = 10240 <= 128 * (168 - 88) = 10240
  // (ptxas -v: the softmax spills below 208, the MMA / TMA roles below 88).
  // Two CTAs of 256 threads per SM launch with 128 each: control 48, softmax
  // 208, 128 * (208 - 128) = 10240 <= 128 * (128 - 48) = 10240 (200 / 56
  // spilled 32-44 bytes; 208 / 48 none).
  static constexpr int LAUNCH_REGS = (65536 / (THREADS * MIN_BLOCKS)) / 8 * 8 > 255
                                         ? 255
                                         : (65536 / (THREADS * MIN_BLOCKS)) / 8 * 8;
  static constexpr int REG_SOFTMAX = NQ == 2 ? 208 : TWO ? 208 : 0;
  static constexpr int REG_CONTROL = NQ == 2 ? 88 : TWO ? 48 : 0;
  static_assert(REG_SOFTMAX == 0 ||
                    NQ * 128 * (REG_SOFTMAX - LAUNCH_REGS) <= 128 * (LAUNCH_REGS - REG_CONTROL),
                "register split exceeds the launch budget");

  static_assert(D % 64 == 0 && BN % 32 == 0, "tile shape");
  static_assert(!F8 || BN == 128, "e4m3 tiles: 128 keys");
  static_assert((BN / 32) % P_PIECES == 0 && KSTEPS_PV % P_PIECES == 0, "P parts");
  static_assert(D * EB % SWZ == 0 && (SWZ == 128 || SWZ == 64), "row panels");
  static_assert(NQ * NSB * BN + NQ * D <= TMEM_COLS, "tensor memory budget");
  static_assert(SMEM_ALLOC <= 232448 / MIN_BLOCKS - 1024, "shared memory budget");
  static_assert(!TWO || (NQ == 1 && NSB == 1), "two-CTA shape");
  static_assert(Q_BYTES % 1024 == 0 && KV_BYTES % 1024 == 0, "1024-byte tile alignment");
};

// ------------------------------------------------------------ bounded waits

struct Waiter {
  volatile uint32_t* abort_flag;  // shared memory, CTA-wide
  unsigned int* status;           // global, device-wide
  unsigned long long timeout_ns = kWaitTimeoutNs;  // limit of each wait
};

// `timeout_ns` 0: the waiter's own limit.
static __device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, Waiter w, uint32_t code,
                                       bool honour_abort, unsigned long long timeout_ns = 0) {
  if (timeout_ns == 0) timeout_ns = w.timeout_ns;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort) {
      if (*w.abort_flag) return false;
      if (*reinterpret_cast<volatile unsigned int*>(w.status) != 0u) {
        *w.abort_flag = 1u;
        return false;
      }
    }
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicCAS(w.status, 0u, code);
      *w.abort_flag = 1u;
      return false;
    }
  }
}

// Wait for the phase of parity `parity`; false if the CTA is aborting.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, Waiter w, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, w, code, true);
}

// Same, for a whole warp: all lanes agree on the outcome.
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity, Waiter w,
                                                uint32_t code) {
  const bool ok = wait_phase(bar, parity, w, code);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, Waiter w, uint32_t code) {
  if (!mbar_try_wait(bar, parity)) wait_slow(bar, parity, w, code, false);
}

// Diagnostic codes: 0x100 | role << 4 | barrier kind.
enum : uint32_t {
  kCodeProducerEmpty = 0x101,
  kCodeMmaQ = 0x111,
  kCodeMmaKV = 0x112,
  kCodeMmaP = 0x113,
  kCodeSoftS = 0x121,
  kCodeSoftO = 0x122,
  kCodeSoftFinal = 0x123,
  kCodeDrain = 0x131,
  kCodeSelfTest = 0x1f1,
};

// ---------------------------------------------------------------- roles

template <int D, bool CAUSAL, bool SPLIT>
struct Tile {
  int bh;
  int row0;                   // first query row of the CTA
  int split;                  // which share of the key tiles (split-KV), 0 otherwise
  int lo;                     // first key tile of this CTA's share
  int nkv[Shape<D>::NQ];      // key tiles [lo, lo + nkv) visited by each query tile
};

template <int D, bool CAUSAL, bool SPLIT, bool F8, int SK>
__device__ __forceinline__ Tile<D, CAUSAL, SPLIT> make_tile(const FwdParams& p, int block = -1) {
  using L = Layout<D, F8, SK>;
  static_assert(L::NQ <= Shape<D>::NQ, "tile bookkeeping sized by the bf16 shape");
  Tile<D, CAUSAL, SPLIT> t;
  const int splits = SPLIT ? p.kv_splits : 1;
  const int b = block < 0 ? static_cast<int>(blockIdx.x) : block;
  const int cta = b / splits;
  t.split = b - cta * splits;
  int qblk;
  if (CAUSAL) {
    // Heaviest query blocks first (longest-processing-time order) across a
    // group of heads_per_group heads: the light blocks fill the tail of the
    // launch, and the group's K/V stays within L2 instead of every head's
    // K/V streaming from HBM at once.
    const int per_group = p.heads_per_group * p.n_qblk;
    const int group = cta / per_group;
    const int gs = min(p.heads_per_group, p.BH - group * p.heads_per_group);
    const int within = cta - group * per_group;
    t.bh = group * p.heads_per_group + within % gs;
    qblk = p.n_qblk - 1 - within / gs;
  } else {
    t.bh = cta / p.n_qblk;
    qblk = cta % p.n_qblk;
  }
  t.row0 = qblk * L::NQ * BM;
  const int nkv_all = (p.Nk + L::BN - 1) / L::BN;
  int nkv_abs[L::NQ];
  int nkv_cta = 0;
#pragma unroll
  for (int q = 0; q < L::NQ; ++q) {
    const int r0 = t.row0 + q * BM;
    if (r0 >= p.Nq) {
      nkv_abs[q] = 0;
    } else if (CAUSAL) {
      // the last key visible to the tile's last query row (bottom-right
      // aligned diagonal: query i sees keys j <= i + Nk - Nq)
      const int last_key = min(r0 + BM - 1, p.Nq - 1) + p.causal_off;
      nkv_abs[q] = last_key / L::BN + 1;
    } else {
      nkv_abs[q] = nkv_all;
    }
    nkv_cta = max(nkv_cta, nkv_abs[q]);
  }
  // split-KV: an even share of the CTA's key tiles
  const int per = (nkv_cta + splits - 1) / splits;
  t.lo = min(t.split * per, nkv_cta);
  const int hi = min(t.lo + per, nkv_cta);
#pragma unroll
  for (int q = 0; q < L::NQ; ++q) t.nkv[q] = max(0, min(hi, nkv_abs[q]) - t.lo);
  return t;
}

// One lane runs this and loads Q, then K_0, V_0, K_1, ... in ring order.
// `drop_load` (a test hook, -1 on every product path) names a ring position
// whose copy is not issued: nothing arrives on its full barrier, so the MMA
// warp's bounded wait for it runs out and the CTA takes its abort path.
// With SPLIT_LOAD, lanes of two warps run it: `par` = 0 loads Q and the K
// tiles (even ring positions), `par` = 1 the V tiles (odd positions); with an
// even number of ring slots K and V use disjoint slots, so a K tile is never
// queued behind a V tile whose slot P.V is still reading (with one K and one
// V slot, the next K loads during P.V and the next V during the next S).
template <int D, bool CAUSAL, bool SPLIT, bool F8, int SK>
__device__ void producer_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                              const CUtensorMap* tm_v, uint32_t sbase, const Tile<D, CAUSAL, SPLIT>& t,
                              Waiter w, int par, int drop_load) {
  using L = Layout<D, F8, SK>;
  static_assert(!L::SPLIT_LOAD || L::STAGES % 2 == 0, "K and V take alternate ring slots");
  constexpr int STEP = L::SPLIT_LOAD ? 2 : 1;
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  int nkv = 0;
#pragma unroll
  for (int q = 0; q < L::NQ; ++q) {
    nkv = max(nkv, t.nkv[q]);
    if (t.nkv[q] > 0 && par == 0) {
      const uint32_t fb = bar(L::B_QFULL + q);
      mbar_arrive_expect_tx(fb, L::Q_BYTES);
#pragma unroll
      for (int pn = 0; pn < L::PANELS; ++pn)
        tma_load_3d(sbase + L::OFF_Q + q * L::Q_BYTES + pn * L::Q_PANEL, tm_q, fb,
                    pn * L::PANEL_ELEMS, t.row0 + q * BM, t.bh);
    }
  }
  const int total = 2 * nkv;  // K_0, V_0, K_1, V_1, ...
  int next = par;  // next ring position of this lane
  for (int i = par; i < total; i += STEP) {
    const int st = i % L::STAGES;
    const uint32_t ph = static_cast<uint32_t>(i / L::STAGES) & 1u;
    if (!wait_phase(bar(L::B_KVEMPTY + st), ph ^ 1u, w, kCodeProducerEmpty)) break;
    next = i + STEP;
    if (i == drop_load) continue;  // test hook: this slot never fills
    const uint32_t fb = bar(L::B_KVFULL + st);
    mbar_arrive_expect_tx(fb, L::KV_BYTES);
    const CUtensorMap* map = (i & 1) ? tm_v : tm_k;
    const int key0 = (t.lo + (i >> 1)) * L::BN;
#pragma unroll
    for (int pn = 0; pn < L::PANELS; ++pn)
      tma_load_3d(sbase + L::OFF_KV + st * L::KV_BYTES + pn * L::KV_PANEL, map, fb,
                  pn * L::PANEL_ELEMS, key0, t.bh);
  }
  if (*w.abort_flag) {
    // Let every copy this thread started land before the CTA exits.
#pragma unroll
    for (int q = 0; q < L::NQ; ++q)
      if (t.nkv[q] > 0 && par == 0) drain_phase(bar(L::B_QFULL + q), 0u, w, kCodeDrain);
    for (int i = max(par, next - L::STAGES); i < next; i += STEP)
      if (i != drop_load)
        drain_phase(bar(L::B_KVFULL + i % L::STAGES), static_cast<uint32_t>(i / L::STAGES) & 1u,
                    w, kCodeDrain);
  }
}

// Runs on a whole warp with warp-uniform control flow (so the descriptors
// stay in uniform registers); one elected lane issues every tcgen05.mma and
// tcgen05.commit.
template <int D, bool CAUSAL, bool SPLIT, bool F8, int SK>
__device__ void mma_role(uint32_t tmem, uint32_t sbase, const Tile<D, CAUSAL, SPLIT>& t, Waiter w) {
  using L = Layout<D, F8, SK>;
  constexpr int NQ = L::NQ, NSB = L::NSB, BN = L::BN;
  // A=Q, B=K: both K-major.  A=P (tmem), B=V: MN-major.
  constexpr uint32_t kIdescQK = F8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, false);
  constexpr uint32_t kIdescPV = F8 ? idesc_e4m3_f32(BM, D, true) : idesc_bf16_f32(BM, D, true);
  auto mma_s = [](uint32_t d_t, uint64_t a, uint64_t b, uint32_t acc, uint32_t issue) {
    if constexpr (F8) mma_ss_f8(d_t, a, b, kIdescQK, acc, issue);
    else mma_ss(d_t, a, b, kIdescQK, acc, issue);
  };
  auto mma_pv = [](uint32_t d_t, uint32_t a_t, uint64_t b, uint32_t acc, uint32_t issue) {
    if constexpr (F8) mma_ts_f8(d_t, a_t, b, kIdescPV, acc, issue);
    else mma_ts(d_t, a_t, b, kIdescPV, acc, issue);
  };
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t leader = elect_one();

  bool ok = true;
  int nkv = 0;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    nkv = max(nkv, t.nkv[q]);
    if (t.nkv[q] > 0 && ok) ok = warp_wait_phase(bar(L::B_QFULL + q), 0u, w, kCodeMmaQ);
  }

  // ring slot i holds K_(i/2) (even i) or V_(i/2) (odd i)
  auto slot_addr = [&](int i) {
    return sbase + L::OFF_KV + static_cast<uint32_t>((i % L::STAGES) * L::KV_BYTES);
  };
  auto wait_full = [&](int i) {
    return warp_wait_phase(bar(L::B_KVFULL + i % L::STAGES),
                           static_cast<uint32_t>(i / L::STAGES) & 1u, w, kCodeMmaKV);
  };
  auto release = [&](int i) { mma_commit(bar(L::B_KVEMPTY + i % L::STAGES), leader); };

  // S(q, b) = Q_q K^T with K in ring slot `ks`
  auto issue_s = [&](int q, int b, int ks) {
    const uint64_t a0 = sdesc_swz<L::SWZ>(sbase + L::OFF_Q + q * L::Q_BYTES, 16, L::SBO);
    const uint64_t b0 = sdesc_swz<L::SWZ>(slot_addr(ks), 16, L::SBO);
    const uint32_t d_t = tmem + L::s_col(q, b);
#pragma unroll
    for (int k = 0; k < L::KSTEPS_QK; ++k) {
      const uint32_t ao = ((k / L::KPP) * L::Q_PANEL + (k % L::KPP) * 32) >> 4;
      const uint32_t bo = ((k / L::KPP) * L::KV_PANEL + (k % L::KPP) * 32) >> 4;
      mma_s(d_t, a0 + ao, b0 + bo, k > 0 ? 1u : 0u, leader);
    }
    mma_commit(bar(L::B_SFULL + q * NSB + b), leader);
  };
  // O_q (+)= P(q, b) V with V in ring slot `vs`; waits for each half of P
  // (keys [0, BN/2) then [BN/2, BN)) before issuing its K-steps.
  auto issue_pv = [&](int q, int b, int vs, bool accumulate, uint32_t pph) {
    // V as stored: MN-major, a K-step spans 16 (bf16) or 32 (e4m3) rows of
    // SWZ bytes per column panel; a K-step of P is 8 tensor-memory columns
    // (2 bf16 or 4 e4m3 each).
    const uint64_t b0 = sdesc_swz<L::SWZ>(slot_addr(vs), L::KV_PANEL, L::SBO);
    const uint32_t d_t = tmem + L::o_col(q);
    const uint32_t a_t = tmem + L::s_col(q, b);
    constexpr int NH = L::P_PIECES;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      if (!warp_wait_phase(bar(L::B_PFULL + (q * NSB + b) * NH + h), pph, w, kCodeMmaP))
        return false;
      tc_fence_after_sync();
#pragma unroll
      for (int k = h * (L::KSTEPS_PV / NH); k < (h + 1) * (L::KSTEPS_PV / NH); ++k) {
        const uint32_t bo = (k * L::KEYS_PER_KSTEP * L::SWZ) >> 4;
        mma_pv(d_t, a_t + k * 8, b0 + bo, (accumulate || k > 0) ? 1u : 0u, leader);
      }
    }
    mma_commit(bar(L::B_ODONE + q), leader);
    return true;
  };

  if (ok && nkv > 0) {  // nkv == 0: an empty split-KV share, nothing to issue
    if constexpr (NSB == 1) {
      // Per key tile j: PV_q(j) then S_q(j+1) for q = 0, 1, so the tensor
      // core works on one query tile while the other's softmax runs.
      ok = wait_full(0);
      if (ok) {
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (t.nkv[q] > 0) issue_s(q, 0, 0);
        release(0);
      }
      for (int j = 0; j < nkv && ok; ++j) {
        const int vi = 2 * j + 1, ki = 2 * j + 2;
        ok = wait_full(vi);
        bool k_ready = false;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (!ok || j >= t.nkv[q]) continue;
          ok = issue_pv(q, 0, vi, j > 0, static_cast<uint32_t>(j) & 1u);
          if (!ok) break;
          if (j + 1 == t.nkv[q]) mma_commit(bar(L::B_OFINAL + q), leader);
          if (j + 1 < t.nkv[q]) {
            if (!k_ready) {
              ok = wait_full(ki);
              if (!ok) break;
              k_ready = true;
            }
            issue_s(q, 0, ki);
          }
        }
        if (!ok) break;
        release(vi);
        if (k_ready) release(ki);
      }
    } else {
      // Two S buffers per query tile: S_q(j+2) is computed while the softmax
      // works on S_q(j+1) and the tensor core runs PV_q(j); with two query
      // tiles their PV/S pairs interleave as well.
      for (int jj = 0; jj < 2 && jj < nkv && ok; ++jj) {
        ok = wait_full(2 * jj);
        if (!ok) break;
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (jj < t.nkv[q]) issue_s(q, jj, 2 * jj);
        release(2 * jj);
      }
      for (int j = 0; j < nkv && ok; ++j) {
        const int b = j & 1;
        const int vi = 2 * j + 1, ki = 2 * (j + 2);
        ok = wait_full(vi);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (!ok || j >= t.nkv[q]) continue;
          ok = issue_pv(q, b, vi, j > 0, static_cast<uint32_t>(j >> 1) & 1u);
          if (!ok) break;
          if (j + 1 == t.nkv[q]) mma_commit(bar(L::B_OFINAL + q), leader);
        }
        if (!ok) break;
        release(vi);
        if (j + 2 < nkv) {
          // S(j+2) reuses the buffer whose P the PV above just read
          ok = wait_full(ki);
          if (!ok) break;
#pragma unroll
          for (int q = 0; q < NQ; ++q)
            if (j + 2 < t.nkv[q]) issue_s(q, b, ki);
          release(ki);
        }
      }
    }
  }
  if (!ok) {
    // Let every MMA this warp issued finish before tensor memory is freed.
    mma_commit(bar(L::B_DRAIN), leader);
    drain_phase(bar(L::B_DRAIN), 0u, w, kCodeDrain);
  }
}

// Row maximum of raw scores; MASKED keeps only columns [0, lim).
template <int NCH, bool MASKED>
__device__ __forceinline__ float row_max(const uint32_t (&s)[NCH][32], int lim) {
  float mm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float x0 = __uint_as_float(s[ch][e]), x1 = __uint_as_float(s[ch][e + 1]);
      if (MASKED) {
        x0 = (ch * 32 + e < lim) ? x0 : -INFINITY;
        x1 = (ch * 32 + e + 1 < lim) ? x1 : -INFINITY;
      }
      mm[(e >> 1) & 3] = fmax3(mm[(e >> 1) & 3], x0, x1);
    }
  return fmax3(fmaxf(mm[0], mm[1]), mm[2], mm[3]);
}

// p = exp2(s * c - m) for 32-column chunks [CH0, CH1) of one S row, stored
// as packed bf16 pairs at columns [CH0 * 16, CH1 * 16) from `s_t` (over the
// S columns already read); returns the sum of the fp32 p.  MASKED zeroes
// columns >= lim.
template <int NCH, int CH0, int CH1, bool MASKED>
__device__ __forceinline__ float exp_store(const uint32_t (&s)[NCH][32], int lim, float c, float m,
                                           uint32_t s_t) {
  const f32x2 cc = f2_pack(c, c), nm = f2_pack(-m, -m);
  f32x2 acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
  for (int ch = CH0; ch < CH1; ++ch) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const f32x2 x =
          f2_fma(f2_pack(__uint_as_float(s[ch][2 * e]), __uint_as_float(s[ch][2 * e + 1])), cc, nm);
      float t0, t1;
      f2_unpack(x, t0, t1);
      float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
      if (MASKED) {
        p0 = (ch * 32 + 2 * e < lim) ? p0 : 0.f;
        p1 = (ch * 32 + 2 * e + 1 < lim) ? p1 : 0.f;
      }
      pk[e] = pack_bf16x2(p0, p1);
      acc[e & 1] = f2_add(acc[e & 1], f2_pack(p0, p1));
    }
    tmem_st_32x32b_x16(s_t + ch * 16, pk);
  }
  return f2_sum(f2_add(acc[0], acc[1]));
}

// e4m3 form of exp_store: 2^kF8Shift * exp2(s * c - m) as e4m3, four per
// tensor-memory column at [CH0 * 8, CH1 * 8); returns the sum of the fp32
// (shifted) values.
template <int NCH, int CH0, int CH1, bool MASKED>
__device__ __forceinline__ float exp_store_f8(const uint32_t (&s)[NCH][32], int lim, float c,
                                              float m, uint32_t s_t) {
  const f32x2 cc = f2_pack(c, c), nm = f2_pack(-m, -m);
  f32x2 acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
  for (int ch = CH0; ch < CH1; ++ch) {
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float p4[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = 4 * e + 2 * h;
        const f32x2 x =
            f2_fma(f2_pack(__uint_as_float(s[ch][i]), __uint_as_float(s[ch][i + 1])), cc, nm);
        float t0, t1;
        f2_unpack(x, t0, t1);
        float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
        if (MASKED) {
          p0 = (ch * 32 + i < lim) ? p0 : 0.f;
          p1 = (ch * 32 + i + 1 < lim) ? p1 : 0.f;
        }
        p4[2 * h] = p0;
        p4[2 * h + 1] = p1;
        acc[h] = f2_add(acc[h], f2_pack(p0, p1));
      }
      pk[e] = pack_e4m3x4(p4[0], p4[1], p4[2], p4[3]);
    }
    tmem_st_32x32b_x8(s_t + ch * 8, pk);
  }
  return f2_sum(f2_add(acc[0], acc[1]));
}

// e4m3 P is stored scaled by 2^kF8Shift: with the rescale threshold of 2^4
// its values stay at or below 2^8 (e4m3 saturates at 448), and weights down
// to 2^-10 of the exponent offset (2^-14 of the row maximum at worst) stay
// normal numbers (3 mantissa bits).  Measured against a shift of 7 with a
// threshold of 1: the same whole-tensor error within 2 %, and far fewer
// rescales (4096-row causal rows 1257 -> 1411 TFLOP/s).
constexpr float kF8Shift = 4.0f;
static_assert(kF8Shift + kRescaleThresholdF8 <= 8.0f, "e4m3 P must stay below 448");

// One weight rounded as the bf16 P stores it.
__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

template <int D, bool CAUSAL, bool SPLIT, bool F8, int SK>
// Returns true when the query tile's O has been staged in shared memory for
// the TMA store (every thread of the tile gets the same answer).
__device__ bool softmax_role(int q, uint32_t tmem, uint32_t sbase, const Tile<D, CAUSAL, SPLIT>& t,
                             const FwdParams& p, Waiter w) {
  using L = Layout<D, F8, SK>;
  constexpr int BN = L::BN, NSB = L::NSB;
  constexpr int NCH = BN / 32;  // 32-column chunks of an S row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (warp & 3) * 32 + lane;  // row inside the query tile == TMEM lane
  const int r0 = t.row0 + q * BM;
  const int grow = r0 + r;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const int n = t.nkv[q];
  const float c = p.scale_log2;
  const uint32_t o_t = tmem + lane_base + L::o_col(q);

  // Running state of this row (log2 units, scale applied): m_used is the
  // exponent offset of P, O and l; l is the sum of the fp32 p.
  float m_used = 0.f;
  float l = 0.f;
  float l_fix = 0.f;  // O's normaliser is l + l_fix (see below); LSE uses l
  if (n == 0) {
    // This split saw no key of this query tile: an empty partial.
    if (SPLIT && grow < p.Nq)
      p.lse_part[static_cast<size_t>(t.split) * p.BH * p.Nq + static_cast<size_t>(t.bh) * p.Nq + grow] =
          -INFINITY;
    return false;
  }
  bool ok = true;
  for (int j = 0; j < n && ok; ++j) {
    const int b = (NSB == 1) ? 0 : (j & 1);
    const uint32_t sph = static_cast<uint32_t>(NSB == 1 ? j : (j >> 1)) & 1u;
    ok = warp_wait_phase(bar(L::B_SFULL + q * NSB + b), sph, w, kCodeSoftS);
    if (!ok) break;
    tc_fence_after_sync();
    const uint32_t s_t = tmem + lane_base + L::s_col(q, b);
    uint32_t s[NCH][32];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) tmem_ld_32x32b_x32(s_t + ch * 32, s[ch]);
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) tmem_ld_wait(s[ch]);

    const int key0 = (t.lo + j) * BN;
    const bool masked = (CAUSAL && key0 + BN - 1 > r0 + p.causal_off) || (key0 + BN > p.Nk);
    int lim = BN;  // columns [0, lim) of this tile are visible to this row
    if (masked) {
      lim = p.Nk - key0;
      if (CAUSAL) lim = min(lim, grow + p.causal_off - key0 + 1);
    }

    // P = exp2(s * c - m_used) as bf16 (e4m3), written over the first BN/2
    // (BN/4) columns of S, in P_PIECES parts: after each part's stores have
    // completed, each warp arrives on that part's barrier, and the MMA warp
    // issues the P.V K-steps of that part.  One part for 64-key tiles (a
    // second barrier round trip costs more than it overlaps).
    constexpr int CPP = NCH / L::P_PIECES;  // 32-column chunks per part
    constexpr float kThreshold = F8 ? kRescaleThresholdF8 : kRescaleThreshold;
    auto exp_part = [&](auto part) -> float {  // the part's weights; returns their sum
      constexpr int c0 = decltype(part)::value * CPP, c1 = c0 + CPP;
      if constexpr (F8) {
        const float m_f8 = m_used - kF8Shift;
        return masked ? exp_store_f8<NCH, c0, c1, true>(s, lim, c, m_f8, s_t)
                      : exp_store_f8<NCH, c0, c1, false>(s, lim, c, m_f8, s_t);
      } else {
        return masked ? exp_store<NCH, c0, c1, true>(s, lim, c, m_used, s_t)
                      : exp_store<NCH, c0, c1, false>(s, lim, c, m_used, s_t);
      }
    };
    auto hand_over = [&](int part) {
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_PFULL + (q * NSB + b) * L::P_PIECES + part));
    };
    // Moves the exponent offset to m_new where `need`: O (once P.V(j-1) has
    // landed, o_done phase j-1) and l scale by 2^(m_used - m_new).
    auto rescale = [&](float m_new, bool need) -> bool {
      if (!warp_wait_phase(bar(L::B_ODONE + q), static_cast<uint32_t>(j - 1) & 1u, w, kCodeSoftO))
        return false;
      tc_fence_after_sync();
      const float alpha = need ? ex2_approx(m_used - m_new) : 1.f;
      if (need) m_used = m_new;
      l *= alpha;
      l_fix *= alpha;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(o_t + ch * 32, ov);
        tmem_ld_wait(ov);
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
        tmem_st_32x32b_x32(o_t + ch * 32, ov);
      }
      tmem_st_wait();
      return true;
    };

    // row maximum of the raw scores (scale >= 0 keeps the arg-max)
    const float mx = masked ? row_max<NCH, true>(s, lim) : row_max<NCH, false>(s, lim);
    const float mx_c = (mx == -INFINITY) ? -INFINITY : mx * c;
    if (j == 0) {
      m_used = (mx_c == -INFINITY) ? 0.f : mx_c;
    } else {
      const float m_new = fmaxf(m_used, mx_c);
      const bool need = m_new > m_used + kThreshold;
      if (__any_sync(0xffffffffu, need)) {
        ok = rescale(m_new, need);
        if (!ok) break;
      }
    }
    l += exp_part(std::integral_constant<int, 0>{});
    hand_over(0);
    if constexpr (L::P_PIECES > 1) {
      l += exp_part(std::integral_constant<int, 1>{});
      hand_over(1);
    }
    if constexpr (L::P_PIECES > 2) {
      l += exp_part(std::integral_constant<int, 2>{});
      hand_over(2);
      l += exp_part(std::integral_constant<int, 3>{});
      hand_over(3);
    }

    // l sums the fp32 weights while P.V uses them rounded.  O's normaliser
    // takes the tile's largest weight (the one whose rounding error can be
    // large next to l) as rounded, computed as exp_store computes it, so that
    // a row dominated by one key gets that key's V back exactly; LSE keeps the
    // unrounded sum.  Done after P is handed over, off the MMA's path.
    if (mx != -INFINITY) {
      if constexpr (F8) {
        const float pm = ex2_approx(fmaf(mx, c, -(m_used - kF8Shift)));
        l_fix += round_e4m3(pm) - pm;
      } else {
        const float pm = ex2_approx(fmaf(mx, c, -m_used));
        l_fix += round_bf16(pm) - pm;
      }
    }
  }

  // epilogue: O / l -> bf16, LSE = (m + log2 l) * ln 2; with split-KV the
  // normalised fp32 partial O and the partial LSE go to the workspace.  The
  // bf16 O tile is staged in this query tile's Q buffer -- free once o_final
  // has completed, as no later MMA reads it -- in the 128B-swizzled layout
  // the TMA loaded Q in, and the kernel writes it out with TMA stores of
  // whole 128-byte row segments (coalesced; rows past Nq are not written).
  // The e4m3 Q buffer is half the size of a bf16 O tile, so e4m3 rows are
  // stored directly.  Warps that gave up still meet the others at the
  // staging barrier, so no warp waits there for one that left.
  constexpr bool split_mode = SPLIT;
  constexpr bool tma_epilogue = Layout<D, F8, SK>::TMA_EPILOGUE && !SPLIT;
  if constexpr (!tma_epilogue) {
    if (!ok) return false;
  }
  const bool valid = grow < p.Nq;
  if constexpr (tma_epilogue) {
    if (ok) ok = warp_wait_phase(bar(L::B_OFINAL + q), 0u, w, kCodeSoftFinal);
  } else {
    ok = warp_wait_phase(bar(L::B_OFINAL + q), 0u, w, kCodeSoftFinal);
    if (!ok) return false;
  }
  if (ok) {
    tc_fence_after_sync();
    // e4m3: O and l both carry the 2^kF8Shift factor; V's dequantisation
    // scale multiplies O.
    const float inv_l = F8 ? p.o_scale / (l + l_fix) : 1.f / (l + l_fix);
    const size_t row = static_cast<size_t>(t.bh) * p.Nq + (valid ? grow : 0);
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + row * D;
    float* prow = p.o_part + (static_cast<size_t>(t.split) * p.BH * p.Nq + row) * D;
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t ov[32];
      tmem_ld_32x32b_x32(o_t + ch * 32, ov);
      tmem_ld_wait(ov);
      if constexpr (split_mode) {
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(prow + ch * 32);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            dst[v4] = make_float4(__uint_as_float(ov[4 * v4]) * inv_l, __uint_as_float(ov[4 * v4 + 1]) * inv_l,
                                  __uint_as_float(ov[4 * v4 + 2]) * inv_l, __uint_as_float(ov[4 * v4 + 3]) * inv_l);
        }
      } else {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
        if constexpr (tma_epilogue) {
          // columns [32 ch, 32 ch + 32) are 16-byte chunks 4 (ch % 2) .. +3 of
          // row r in 64-column panel ch / 2; chunk c sits at c ^ (r % 8)
          const uint32_t rowb = sbase + L::OFF_Q + q * L::Q_BYTES + (ch / 2) * L::Q_PANEL + r * 128;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            st_shared_v4(rowb + ((((ch % 2) * 4 + v4) ^ (r & 7)) << 4), pk[4 * v4], pk[4 * v4 + 1],
                         pk[4 * v4 + 2], pk[4 * v4 + 3]);
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
    }
    if (valid) {
      const float lse = (m_used + __log2f(l) - (F8 ? kF8Shift : 0.f)) * kLn2;
      if constexpr (split_mode)
        p.lse_part[static_cast<size_t>(t.split) * p.BH * p.Nq + row] = lse;
      else
        p.lse[row] = lse;
    }
  }
  if constexpr (tma_epilogue) {
    // every writer orders its shared-memory writes before the TMA's reads;
    // the tile's 128 threads then meet and learn whether all of them staged
    fence_proxy_async_smem();
    return named_barrier_and(1 + q, 128, ok);
  }
  return false;
}

template <int D, bool CAUSAL, bool SPLIT, bool F8 = false, int SK = kShapeDefault>
__global__ void __launch_bounds__(Layout<D, F8, SK>::THREADS, Layout<D, F8, SK>::MIN_BLOCKS)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p) {
  using L = Layout<D, F8, SK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Tile<D, CAUSAL, SPLIT> t = make_tile<D, CAUSAL, SPLIT, F8, SK>(p);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEMSLOT);
  const Waiter w{abort_flag, p.status, p.wait_timeout_ns ? p.wait_timeout_ns : kWaitTimeoutNs};

  if (threadIdx.x == 0) {
    const uint32_t bar0 = sbase + L::OFF_BAR;
    for (int i = 0; i < L::NBAR; ++i) {
      uint32_t count = 1;
      if (i >= L::B_PFULL && i < L::B_PFULL + L::NQ * L::NSB * L::P_PIECES) count = 4;  // per softmax warp
      mbar_init(bar0 + 8u * i, count);
    }
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == L::TMA_WARP && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_o);
    if constexpr (L::TWO && !SPLIT) {
      // short rows: the CTA that will take this one's place in the next wave
      // finds its Q tile in L2
      const int next = static_cast<int>(blockIdx.x) + L::MIN_BLOCKS * p.num_sms;
      if (p.num_sms > 0 && next < static_cast<int>(gridDim.x)) {
        const Tile<D, CAUSAL, SPLIT> tn = make_tile<D, CAUSAL, SPLIT, F8, SK>(p, next);
        if (tn.nkv[0] > 0)
          for (int pn = 0; pn < L::PANELS; ++pn)
            tma_prefetch_l2_3d(&tm_q, pn * L::PANEL_ELEMS, tn.row0, tn.bh);
      }
    }
  }
  if (warp == L::MMA_WARP) {
    tmem_alloc(smem_addr(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  // Each role runs to the end of the kernel on its own path (the register
  // split differs per path), then meets the others at the teardown barrier.
  if (warp < 4 * L::NQ) {
    if constexpr (L::REG_SOFTMAX > 0) setmaxnreg_inc<L::REG_SOFTMAX>();
    const int q = warp >> 2;
    const bool staged = softmax_role<D, CAUSAL, SPLIT, F8, SK>(q, tmem, sbase, t, p, w);
    if (staged && (warp & 3) == 0 && lane == 0) {
      // one lane stores the staged O panels and waits until the TMA has read
      // them out of shared memory, before the CTA can exit (the tile's
      // coordinates are recomputed here rather than kept through the role)
      const Tile<D, CAUSAL, SPLIT> te = make_tile<D, CAUSAL, SPLIT, F8, SK>(p);
#pragma unroll
      for (int pn = 0; pn < L::PANELS; ++pn)
        tma_store_3d(&tm_o, sbase + L::OFF_Q + q * L::Q_BYTES + pn * L::Q_PANEL,
                     pn * L::PANEL_ELEMS, te.row0 + q * BM, te.bh);
      tma_store_commit();
      tma_store_wait_read();
    }
    tc_fence_before_sync();
    __syncthreads();
  } else {
    if constexpr (L::REG_CONTROL > 0) setmaxnreg_dec<L::REG_CONTROL>();
    if (warp == L::TMA_WARP || (L::SPLIT_LOAD && warp == L::V_WARP)) {
      if (lane == 0)
        producer_role<D, CAUSAL, SPLIT, F8, SK>(&tm_q, &tm_k, &tm_v, sbase, t, w,
                                            warp == L::TMA_WARP ? 0 : 1, p.drop_load);
      __syncwarp();
    } else if (warp == L::MMA_WARP) {
      mma_role<D, CAUSAL, SPLIT, F8, SK>(tmem, sbase, t, w);
      __syncwarp();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == L::MMA_WARP) {
      tc_fence_after_sync();
      tmem_dealloc(tmem, L::TMEM_COLS);
    }
  }
}

}  // namespace ea51
