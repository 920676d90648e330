// C ABI of the fused attention forward: argument checks, TMA descriptor
// encoding and dispatch to the per-head-dim kernels.  The declarations and the
// contract of every entry point are in include/attn_fwd.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <mutex>
#include <vector>

#include "attn_bwd.h"
#include "attn_fp8.h"
#include "attn_fwd.h"
#include "bwd_dispatch.h"
#include "fwd_dispatch.h"

namespace {

thread_local int t_last_cuda_error = 0;

// Device-wide word the kernels set when a bounded wait gives up.
__device__ unsigned int g_attn_status;

constexpr int kMaxDevices = 64;

// L2 bytes a causal launch order gives one group of heads' streamed operands
// (forward: K and V; backward: Q and dO, or K and V): about a quarter of L2.
constexpr double kCausalGroupBytes = 32.0 * 1024 * 1024;

struct DeviceState {
  bool checked = false;
  bool supported = false;
  unsigned int* status = nullptr;  // device address of g_attn_status
  int sms = 148;                   // streaming multiprocessors
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return ATTN_ERR_LAUNCH;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Argument checks shared by every entry point: q, o [B,H,Nq,d] bf16; k, v
// [B,H,Nk,d] bf16; lse [B,H,Nq] fp32.  Causal needs Nk >= Nq (the diagonal
// sits at the bottom-right corner, so every query row sees a key).
int check_general(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  int B, int H, int Nq, int Nk, int d, float scale, int causal) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return ATTN_ERR_INVALID_ARG;
  if (causal && Nk < Nq) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
  // Launch limits: B*H heads fit the TMA's 32-bit dimension and the grid's
  // 31-bit x extent (with at least 128 query rows per CTA).
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t ctas = BH * ((static_cast<int64_t>(Nq) + 127) / 128);
  if (BH > 0x7fffffffLL || ctas > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  const auto al = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
  if (!al(q, 16) || !al(k, 16) || !al(v, 16) || !al(o, 16) || !al(lse, 4)) return ATTN_ERR_MISALIGNED;
  const size_t q_bytes = static_cast<size_t>(BH) * static_cast<size_t>(Nq) * d * 2;
  const size_t kv_bytes = static_cast<size_t>(BH) * static_cast<size_t>(Nk) * d * 2;
  const size_t lse_bytes = static_cast<size_t>(BH) * static_cast<size_t>(Nq) * 4;
  const void* ins[3] = {q, k, v};
  const size_t in_bytes[3] = {q_bytes, kv_bytes, kv_bytes};
  for (int i = 0; i < 3; ++i) {
    if (overlaps(o, q_bytes, ins[i], in_bytes[i])) return ATTN_ERR_ALIAS;
    if (overlaps(lse, lse_bytes, ins[i], in_bytes[i])) return ATTN_ERR_ALIAS;
  }
  if (overlaps(lse, lse_bytes, o, q_bytes)) return ATTN_ERR_ALIAS;
  return ATTN_OK;
}

int check_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
               int H, int N, int d, float scale, int causal) {
  return check_general(q, k, v, o, lse, B, H, N, N, d, scale, causal);
}

// Per-device set-up: compute capability check and the status word's address.
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.checked) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return fail_cuda(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return fail_cuda(e);
    s.supported = (major == 10 && minor == 3);
    if ((e = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail_cuda(e);
    if (s.supported) {
      void* addr = nullptr;
      if ((e = cudaGetSymbolAddress(&addr, g_attn_status)) != cudaSuccess) return fail_cuda(e);
      s.status = static_cast<unsigned int*>(addr);
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult qr{};
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &qr);
      if (e != cudaSuccess) return fail_cuda(e);
      if (qr != cudaDriverEntryPointSuccess || !fn) return fail_cuda(cudaErrorNotSupported);
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    s.checked = true;
  }
  if (!s.supported) return ATTN_ERR_UNSUPPORTED_DEVICE;
  *out = &s;
  return ATTN_OK;
}

// A [BH, rows, cols] tensor (cols innermost, `pitch` elements between rows)
// with a box of one swizzle span of columns x `box_rows` rows x one head:
// `swz` = 128 bytes with 128-byte swizzle, or 64 bytes with 64-byte swizzle
// (the kernel's Layout::SWZ).  Rows and columns past the extents read as
// zeros, so a ragged last tile never touches the next head.
int encode_tiled(CUtensorMap* map, const void* base, CUtensorMapDataType type, int elem_bytes,
                 int64_t BH, int64_t rows, int64_t cols, int64_t pitch, int box_rows,
                 int swz = 128) {
  const bool narrow = swz == 64;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch * elem_bytes),
                                 static_cast<cuuint64_t>(pitch * elem_bytes * rows)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>((narrow ? 64 : 128) / elem_bytes),
                             static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = g_encode(map, type, 3, const_cast<void*>(base), dims, strides, box, estride,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = static_cast<int>(r);
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

// [BH, N, d] bf16: box = 64 columns (one 128-byte swizzle span) x `rows` rows.
int encode_map(CUtensorMap* map, const void* base, int64_t BH, int N, int d, int rows) {
  return encode_tiled(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, N, d, d, rows);
}

}  // namespace

namespace ea51 {
unsigned int* status_word() {
  DeviceState* ds = nullptr;
  return device_state(&ds) == ATTN_OK ? ds->status : nullptr;
}
int device_ready() {
  DeviceState* ds = nullptr;
  return device_state(&ds);
}
int record_cuda_error(cudaError_t e) { return fail_cuda(e); }
}  // namespace ea51

extern "C" {

int attn_fwd_check_args(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, int B, int H, int N, int d, float scale, int causal) {
  return check_args(q, k, v, o, lse, B, H, N, d, scale, causal);
}

}  // extern "C"

namespace {

// Keys per head up to which head dim 64 runs the two-CTAs-per-SM shape (one
// query tile per CTA): with at most 8 key tiles per query tile the per-CTA
// set-up and epilogue weigh more than sharing K/V between two query tiles
// saves.  Measured (GB300, both shapes on each workload): B=8 H=12 N=1024
// causal 327 -> 354 TFLOP/s (e4m3: 365 -> 403); N=8192 2-3 % slower; d = 128
// 10-15 % slower at N = 1024..16384, so it has no two-CTA shape.
constexpr int kTwoCtaMaxKeys = 1024;

// One key-tile step of a CTA with two query tiles costs about this many
// steps of a one-tile CTA (same SM, full grids: e4m3 d = 128 1546 vs 1306
// TFLOP/s, bf16 d = 64 853 vs 665, i.e. 1.69 and 1.56).
constexpr double kTwoTileStep = 1.6;

// Modelled run time of a launch, in one-tile key steps: every CTA costs its
// key tiles (split evenly over `splits` shares) times `step`, plus 2 for
// set-up and epilogue; CTAs start heaviest first on the least-loaded SM;
// a split launch pays 5 % for the merge kernel and the workspace traffic.
double launch_makespan(int64_t BH, int Nq, int Nk, bool causal, int splits, int rows, int kv_rows,
                       double step, int num_sms) {
  const int64_t nq = (static_cast<int64_t>(Nq) + rows - 1) / rows;
  std::vector<double> work;
  work.reserve(static_cast<size_t>(nq * BH * splits));
  for (int64_t qb = 0; qb < nq; ++qb) {
    const int64_t last_key = std::min<int64_t>((qb + 1) * rows, Nq) - 1 + (Nk - Nq);
    const int64_t tiles = causal ? last_key / kv_rows + 1 : (static_cast<int64_t>(Nk) + kv_rows - 1) / kv_rows;
    const int64_t share = (tiles + splits - 1) / splits;
    for (int i = 0; i < splits; ++i) {
      const int64_t t = std::max<int64_t>(std::min<int64_t>(share, tiles - i * share), 0);
      for (int64_t h = 0; h < BH; ++h) work.push_back(static_cast<double>(t) * step + 2.0);
    }
  }
  std::sort(work.begin(), work.end(), std::greater<double>());
  std::vector<double> sm(static_cast<size_t>(num_sms), 0.0);
  std::make_heap(sm.begin(), sm.end(), std::greater<double>());
  double makespan = 0;
  for (const double wk : work) {
    std::pop_heap(sm.begin(), sm.end(), std::greater<double>());
    sm.back() += wk;
    makespan = std::max(makespan, sm.back());
    std::push_heap(sm.begin(), sm.end(), std::greater<double>());
  }
  return makespan * (splits > 1 ? 1.05 : 1.0);
}

// d = 64 and 128 run one query tile per CTA (two S buffers each) when the
// default grid (two query tiles per CTA) would not fill every SM once and
// the model above gives the one-tile grid the shorter run: twice the CTAs
// on a half-empty GPU can outweigh what two query tiles per CTA hide (B=1
// H=4 N=8192 d=128 causal 658 -> 992 TFLOP/s bf16, 743 -> 1117 e4m3; the
// same shape non-causal, 128 equal CTAs, stays on the default shape).
bool solo_shape(int64_t BH, int Nq, int Nk, bool causal, int splits, int num_sms) {
  // at most one query tile (a decoding step, split-KV or not): the second
  // tile of the default shape would have nothing to do, and two S buffers
  // let the next tile's scores overlap this tile's softmax
  if (Nq <= 128) return true;
  if (splits != 1 || BH * ((static_cast<int64_t>(Nq) + 255) / 256) >= num_sms) return false;
  return launch_makespan(BH, Nq, Nk, causal, 1, 128, 128, 1.0, num_sms) <
         launch_makespan(BH, Nq, Nk, causal, 1, 256, 128, kTwoTileStep, num_sms);
}

ea51::FwdVariant variant_for(int d, int Nq, int Nk, int64_t BH, bool causal, int splits,
                             int num_sms) {
  if (d == 64 && Nk <= kTwoCtaMaxKeys) return ea51::fwd_variant_d64_two();
  if (d != 256 && solo_shape(BH, Nq, Nk, causal, splits, num_sms))
    return d == 64 ? ea51::fwd_variant_d64_solo() : ea51::fwd_variant_d128_solo();
  if (d == 64) return ea51::fwd_variant_d64();
  return d == 128 ? ea51::fwd_variant_d128() : ea51::fwd_variant_d256();
}

// Encodes the TMA maps and launches the fused kernel; with kv_splits > 1 the
// kernel writes partials to o_part / lse_part.
int launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Nq, int Nk, int d, float scale, int causal, int kv_splits, float* o_part,
               float* lse_part, DeviceState* ds, cudaStream_t stream, int drop_load = -1,
               unsigned long long wait_timeout_ns = 0) {
  const int64_t BH = static_cast<int64_t>(B) * H;
  const ea51::FwdVariant var = variant_for(d, Nq, Nk, BH, causal != 0, kv_splits, ds->sms);
  alignas(64) CUtensorMap tq, tk, tv, to;
  int rc;
  if ((rc = encode_map(&tq, q, BH, Nq, d, 128)) != ATTN_OK) return rc;
  if ((rc = encode_map(&tk, k, BH, Nk, d, var.kv_rows)) != ATTN_OK) return rc;
  if ((rc = encode_map(&tv, v, BH, Nk, d, var.kv_rows)) != ATTN_OK) return rc;
  if ((rc = encode_map(&to, o, BH, Nq, d, 128)) != ATTN_OK) return rc;
  ea51::FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.status = ds->status;
  p.Nq = Nq;
  p.Nk = Nk;
  p.causal_off = Nk - Nq;
  p.BH = static_cast<int>(BH);
  p.n_qblk = (Nq + var.q_rows_per_cta - 1) / var.q_rows_per_cta;
  // Causal launch order interleaves the heaviest blocks of as many heads as
  // keep their K and V within about a quarter of L2 (32 MiB).  Measured on
  // B=1 H=32 N=16384 d=128 causal: DRAM bytes per launch 727 MB with half of
  // L2 (8 heads at a time), 524 MB with a quarter (4 heads; 539 MB is the
  // algorithmic minimum), same run time.
  const double kv_head = 2.0 * Nk * d * 2;
  const int64_t g = static_cast<int64_t>((kCausalGroupBytes) / kv_head);
  p.heads_per_group = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.kv_splits = kv_splits;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.drop_load = drop_load;
  p.num_sms = ds->sms;
  p.wait_timeout_ns = wait_timeout_ns;
  const cudaError_t e = var.launch(&tq, &tk, &tv, &to, p, causal != 0, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return ATTN_OK;
}

constexpr int kMaxSplits = ea51::kMaxKvSplits;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Bytes of split-KV workspace: fp32 partial O, then fp32 partial LSE.
size_t splitkv_bytes(int64_t BH, int Nq, int d, int splits, size_t* lse_offset) {
  const size_t rows = static_cast<size_t>(BH) * static_cast<size_t>(Nq);
  const size_t o_bytes = align256(static_cast<size_t>(splits) * rows * d * 4);
  if (lse_offset) *lse_offset = o_bytes;
  return o_bytes + align256(static_cast<size_t>(splits) * rows * 4);
}

int check_splits(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 int B, int H, int Nq, int Nk, int d, int splits, const void* ws, size_t ws_bytes) {
  if (splits < 1 || splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH * ((static_cast<int64_t>(Nq) + 127) / 128) * splits > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  if (splits == 1) return ATTN_OK;
  const size_t need = splitkv_bytes(BH, Nq, d, splits, nullptr);
  if (!ws || ws_bytes < need) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return ATTN_ERR_MISALIGNED;
  const size_t qb = static_cast<size_t>(BH) * Nq * d * 2, kb = static_cast<size_t>(BH) * Nk * d * 2;
  const size_t lb = static_cast<size_t>(BH) * Nq * 4;
  if (overlaps(ws, need, q, qb) || overlaps(ws, need, k, kb) || overlaps(ws, need, v, kb) ||
      overlaps(ws, need, o, qb) || overlaps(ws, need, lse, lb))
    return ATTN_ERR_ALIAS;
  return ATTN_OK;
}

// Every forward entry point lands here: checks, then the fused kernel and,
// for split-KV, the merge kernel, all on `stream`.
int fwd_general(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Nq, int Nk, int d, float scale, int causal, int splits, void* ws,
                size_t ws_bytes, void* stream) {
  int rc = check_general(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal);
  if (rc != ATTN_OK) return rc;
  if ((rc = check_splits(q, k, v, o, lse, B, H, Nq, Nk, d, splits, ws, ws_bytes)) != ATTN_OK)
    return rc;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != ATTN_OK) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (splits == 1)
    return launch_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, 1, nullptr, nullptr, ds, st);
  const int64_t BH = static_cast<int64_t>(B) * H;
  size_t lse_off = 0;
  splitkv_bytes(BH, Nq, d, splits, &lse_off);
  float* o_part = static_cast<float*>(ws);
  float* lse_part = reinterpret_cast<float*>(static_cast<char*>(ws) + lse_off);
  if ((rc = launch_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, splits, o_part, lse_part,
                       ds, st)) != ATTN_OK)
    return rc;
  const cudaError_t e = ea51::launch_combine(d, o_part, lse_part, o, lse, BH * Nq, splits, st);
  if (e != cudaSuccess) return fail_cuda(e);
  return ATTN_OK;
}

// Split count with the smallest modelled makespan (see include/attn_fwd.h).
int split_model_for(bool fp8, int d, int B, int H, int Nq, int Nk, int causal, int num_sms);

int split_model(int B, int H, int Nq, int Nk, int d, int causal, int num_sms) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || (d != 64 && d != 128 && d != 256) || num_sms < 1)
    return 1;
  if (causal && Nk < Nq) return 1;
  return split_model_for(false, d, B, H, Nq, Nk, causal, num_sms);
}

ea51::FwdVariant fp8_variant(int d, int Nq, int Nk, int64_t BH, bool causal, int splits,
                             int num_sms);

// The model for the tile shape each split count launches with.
int split_model_for(bool fp8, int d, int B, int H, int Nq, int Nk, int causal, int num_sms) {
  const int64_t BH = static_cast<int64_t>(B) * H;
  auto shape = [&](int s) {
    return fp8 ? fp8_variant(d, Nq, Nk, BH, causal != 0, s, num_sms)
               : variant_for(d, Nq, Nk, BH, causal != 0, s, num_sms);
  };
  {
    const ea51::FwdVariant var = shape(1);
    const int64_t nq = (static_cast<int64_t>(Nq) + var.q_rows_per_cta - 1) / var.q_rows_per_cta;
    if (BH * nq >= num_sms) return 1;  // a full wave already: splitting only adds the merge
  }
  double best = 0;
  int best_s = 1;
  for (int s = 1; s <= 16 && s <= kMaxSplits; ++s) {
    const ea51::FwdVariant var = shape(s);
    const double step = var.q_rows_per_cta > 128 ? kTwoTileStep : 1.0;
    const double cost = launch_makespan(BH, Nq, Nk, causal != 0, s, var.q_rows_per_cta, var.kv_rows,
                                        step, num_sms);
    if (s == 1 || cost < best) {
      best = cost;
      best_s = s;
    }
  }
  return best_s;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int d, float scale, int causal, void* stream) {
  return fwd_general(q, k, v, o, lse, B, H, N, N, d, scale, causal, 1, nullptr, 0, stream);
}

size_t attn_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits) {
  if (B < 1 || H < 1 || N < 1 || num_splits < 1 || num_splits > kMaxSplits) return 0;
  if (d != 64 && d != 128 && d != 256) return 0;
  if (num_splits == 1) return 0;
  return splitkv_bytes(static_cast<int64_t>(B) * H, N, d, num_splits, nullptr);
}

int attn_fwd_splitkv_num_splits(int B, int H, int N, int d, int causal, int num_sms) {
  return split_model(B, H, N, N, d, causal, num_sms);
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int d, float scale, int causal, int num_splits, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return fwd_general(q, k, v, o, lse, B, H, N, N, d, scale, causal, num_splits, workspace,
                     workspace_bytes, stream);
}

int attn_fwd_kvcache(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int Nq, int Nk, int d, float scale, int causal, int num_splits,
                     void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_general(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits, workspace,
                     workspace_bytes, stream);
}

int attn_fwd_kvcache_num_splits(int B, int H, int Nq, int Nk, int d, int causal, int num_sms) {
  return split_model(B, H, Nq, Nk, d, causal, num_sms);
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_MISALIGNED: return "misaligned pointer (q/k/v/o need 16 bytes, lse 4)";
    case ATTN_ERR_ALIAS: return "an output buffer overlaps another buffer";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3";
    case ATTN_ERR_LAUNCH: return "CUDA call failed (see attn_last_cuda_error)";
    case ATTN_ERR_TIMEOUT: return "a device-side wait timed out; outputs are invalid";
    case ATTN_ERR_NOALLOC_TOO_LARGE:
      return "problem needs more split-KV workspace than the fixed no-allocation buffer holds";
    default: return "unknown status";
  }
}

int attn_fwd_device_status(void* stream, unsigned int* detail) {
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != ATTN_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  unsigned int word = 0, zero = 0;
  if ((e = cudaMemcpy(&word, ds->status, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail_cuda(e);
  if (word != 0 &&
      (e = cudaMemcpy(ds->status, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
    return fail_cuda(e);
  if (detail) *detail = word;
  return word == 0 ? ATTN_OK : ATTN_ERR_TIMEOUT;
}

int attn_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"

namespace {

bool fp8_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

ea51::FwdVariant fp8_variant(int d, int Nq, int Nk, int64_t BH, bool causal, int splits,
                             int num_sms) {
  if (d == 64 && Nk <= kTwoCtaMaxKeys) return ea51::fwd_variant_e4m3_d64_two();
  if (d != 256 && solo_shape(BH, Nq, Nk, causal, splits, num_sms))
    return d == 64 ? ea51::fwd_variant_e4m3_d64_solo() : ea51::fwd_variant_e4m3_d128_solo();
  return d == 64 ? ea51::fwd_variant_e4m3_d64()
                 : d == 128 ? ea51::fwd_variant_e4m3_d128() : ea51::fwd_variant_e4m3_d256();
}

// e4m3 workspace: (split-KV only) the fp32 partial O and LSE; the kernel
// reads V as stored, so nothing else is needed.
size_t fp8_ws_bytes(int64_t BH, int Nq, int /*Nk*/, int d, int splits) {
  return splits > 1 ? splitkv_bytes(BH, Nq, d, splits, nullptr) : 0;
}

int fp8_general(const void* q, const void* k, const void* v, float descale_q, float descale_k,
                float descale_v, void* o, float* lse, int B, int H, int Nq, int Nk, int d,
                float scale, int causal, int splits, void* workspace, size_t workspace_bytes,
                void* stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || !fp8_head_dim(d)) return ATTN_ERR_INVALID_ARG;
  if (causal && Nk < Nq) return ATTN_ERR_INVALID_ARG;
  if (splits < 1 || splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
  for (const float ds : {descale_q, descale_k, descale_v})
    if (!std::isfinite(ds) || ds <= 0.f) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH > 0x7fffffffLL || BH * ((static_cast<int64_t>(Nq) + 127) / 128) * splits > 0x7fffffffLL ||
      BH * ((static_cast<int64_t>(Nk) + 127) / 128) > 0x7fffffffLL || Nk > 0x7fffffff - 16)
    return ATTN_ERR_INVALID_ARG;
  const auto al = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
  const size_t need = fp8_ws_bytes(BH, Nq, Nk, d, splits);
  if (need > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_INVALID_ARG;
  if (!al(q, 16) || !al(k, 16) || !al(v, 16) || !al(o, 16) || !al(lse, 4) ||
      (need > 0 && !al(workspace, 256)))
    return ATTN_ERR_MISALIGNED;
  // one byte per e4m3 element
  const size_t q_bytes = static_cast<size_t>(BH) * Nq * d, kv_bytes = static_cast<size_t>(BH) * Nk * d;
  const void* ins[3] = {q, k, v};
  const size_t in_bytes[3] = {q_bytes, kv_bytes, kv_bytes};
  const void* outs[3] = {o, lse, workspace};
  const size_t out_bytes[3] = {q_bytes * 2, static_cast<size_t>(BH) * Nq * 4, need};
  for (int i = 0; i < 3; ++i) {
    if (out_bytes[i] == 0) continue;
    for (int j = 0; j < 3; ++j)
      if (overlaps(outs[i], out_bytes[i], ins[j], in_bytes[j])) return ATTN_ERR_ALIAS;
    for (int j = i + 1; j < 3; ++j)
      if (out_bytes[j] > 0 && overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j]))
        return ATTN_ERR_ALIAS;
  }
  DeviceState* ds = nullptr;
  int rc;
  if ((rc = device_state(&ds)) != ATTN_OK) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const ea51::FwdVariant var = fp8_variant(d, Nq, Nk, BH, causal != 0, splits, ds->sms);
  alignas(64) CUtensorMap tq, tk, tv, to;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if ((rc = encode_map(&to, o, BH, Nq, d, 128)) != ATTN_OK) return rc;  // bf16 O (unused by e4m3 tiles)
  const int swz = d >= 128 ? 128 : d;  // one byte per element
  if ((rc = encode_tiled(&tq, q, u8, 1, BH, Nq, d, d, 128, swz)) != ATTN_OK) return rc;
  if ((rc = encode_tiled(&tk, k, u8, 1, BH, Nk, d, d, var.kv_rows, swz)) != ATTN_OK) return rc;
  // V as stored, tiled like K (the P.V MMA reads it MN-major)
  if ((rc = encode_tiled(&tv, v, u8, 1, BH, Nk, d, d, var.kv_rows, swz)) != ATTN_OK) return rc;
  ea51::FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.status = ds->status;
  p.Nq = Nq;
  p.Nk = Nk;
  p.causal_off = Nk - Nq;
  p.BH = static_cast<int>(BH);
  p.n_qblk = (Nq + var.q_rows_per_cta - 1) / var.q_rows_per_cta;
  const double kv_head = 2.0 * Nk * d;
  const int64_t g = static_cast<int64_t>((kCausalGroupBytes) / kv_head);
  p.heads_per_group = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * descale_q * descale_k *
                                    1.4426950408889634);
  p.o_scale = descale_v;
  p.kv_splits = splits;
  size_t lse_off = 0;
  if (splits > 1) {
    splitkv_bytes(BH, Nq, d, splits, &lse_off);
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + lse_off);
  }
  e = var.launch(&tq, &tk, &tv, &to, p, causal != 0, st);
  if (e != cudaSuccess) return fail_cuda(e);
  if (splits > 1) {
    e = ea51::launch_combine(d, p.o_part, p.lse_part, o, lse, BH * Nq, splits, st);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return ATTN_OK;
}

}  // namespace

extern "C" {

size_t attn_fwd_fp8_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || !fp8_head_dim(d)) return 0;
  return fp8_ws_bytes(static_cast<int64_t>(B) * H, N, N, d, 1);
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, float descale_q, float descale_k,
                 float descale_v, void* o, float* lse, int B, int H, int N, int d, float scale,
                 int causal, void* workspace, size_t workspace_bytes, void* stream) {
  return fp8_general(q, k, v, descale_q, descale_k, descale_v, o, lse, B, H, N, N, d, scale,
                     causal, 1, workspace, workspace_bytes, stream);
}

size_t attn_fwd_fp8_kvcache_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || !fp8_head_dim(d)) return 0;
  if (num_splits < 1 || num_splits > kMaxSplits) return 0;
  return fp8_ws_bytes(static_cast<int64_t>(B) * H, Nq, Nk, d, num_splits);
}

int attn_fwd_fp8_kvcache_num_splits(int B, int H, int Nq, int Nk, int d, int causal, int num_sms) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || !fp8_head_dim(d) || num_sms < 1) return 1;
  if (causal && Nk < Nq) return 1;
  return split_model_for(true, d, B, H, Nq, Nk, causal, num_sms);
}

int attn_fwd_fp8_kvcache(const void* q, const void* k, const void* v, float descale_q,
                         float descale_k, float descale_v, void* o, float* lse, int B, int H,
                         int Nq, int Nk, int d, float scale, int causal, int num_splits,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return fp8_general(q, k, v, descale_q, descale_k, descale_v, o, lse, B, H, Nq, Nk, d, scale,
                     causal, num_splits, workspace, workspace_bytes, stream);
}

size_t attn_bwd_workspace_size(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  const size_t npad = (static_cast<size_t>(N) + 127) / 128 * 128;
  return 2 * align256(static_cast<size_t>(B) * H * npad * 4);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
             float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  // the forward's checks cover q, k, v, o and lse (o and lse as outputs there:
  // here they are inputs, so only their sizes / alignment matter)
  int rc = check_general(q, k, v, o, lse, B, H, N, N, d, scale, causal);
  if (rc != ATTN_OK && rc != ATTN_ERR_ALIAS) return rc;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_INVALID_ARG;
  if (!dout || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
  const auto al = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
  if (!al(dout, 16) || !al(dq, 16) || !al(dk, 16) || !al(dv, 16) || !al(workspace, 256))
    return ATTN_ERR_MISALIGNED;
  const size_t need = attn_bwd_workspace_size(B, H, N);
  if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const size_t tb = static_cast<size_t>(BH) * N * d * 2, lb = static_cast<size_t>(BH) * N * 4;
  const void* ins[6] = {q, k, v, o, dout, lse};
  const size_t in_bytes[6] = {tb, tb, tb, tb, tb, lb};
  const void* outs[4] = {dq, dk, dv, workspace};
  const size_t out_bytes[4] = {tb, tb, tb, need};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlaps(outs[i], out_bytes[i], ins[j], in_bytes[j])) return ATTN_ERR_ALIAS;
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return ATTN_ERR_ALIAS;
  }
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != ATTN_OK) return rc;
  alignas(64) CUtensorMap tq, tk, tv, tdo;
  const int box = 128;  // 128-row blocks (at d = 256 loaded one 64-column panel at a time)
  if ((rc = encode_map(&tq, q, BH, N, d, box)) != ATTN_OK) return rc;
  if ((rc = encode_map(&tk, k, BH, N, d, box)) != ATTN_OK) return rc;
  if ((rc = encode_map(&tv, v, BH, N, d, box)) != ATTN_OK) return rc;
  if ((rc = encode_map(&tdo, dout, BH, N, d, box)) != ATTN_OK) return rc;
  ea51::BwdParams p{};
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  const int npad = (N + 127) / 128 * 128;
  p.lse2 = static_cast<float*>(workspace);
  p.dsum = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                    align256(static_cast<size_t>(BH) * npad * 4));
  p.status = ds->status;
  p.N = N;
  p.Npad = npad;
  p.BH = static_cast<int>(BH);
  {
    // each CTA streams two [N, d] bf16 operands of its head (Q and dO, or K
    // and V): group as many heads as keep them within about a quarter of L2
    // (A/B against half: long causal 1051 -> 1062 TFLOP/s, mid causal 836 ->
    // 856, dsweep128 causal 976 -> 990)
    const double per_head = 2.0 * N * d * 2;
    const int64_t g = static_cast<int64_t>((kCausalGroupBytes) / per_head);
    p.heads_per_group = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  }
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  const cudaError_t e = ea51::launch_bwd(&tq, &tk, &tv, &tdo, p, o, dout, lse, d, causal != 0,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  return ATTN_OK;
}


int attn_selftest_fwd_dropped_load(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int B, int H, int N, int d, float scale, int causal,
                                   int drop_load, unsigned int timeout_ms, void* stream) {
  if (drop_load < 0 || timeout_ms < 1 || timeout_ms > 10000) return ATTN_ERR_INVALID_ARG;
  int rc = check_general(q, k, v, o, lse, B, H, N, N, d, scale, causal);
  if (rc != ATTN_OK) return rc;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != ATTN_OK) return rc;
  return launch_fwd(q, k, v, o, lse, B, H, N, N, d, scale, causal, 1, nullptr, nullptr, ds,
                    static_cast<cudaStream_t>(stream), drop_load,
                    static_cast<unsigned long long>(timeout_ms) * 1000000ull);
}

int attn_selftest_wait_timeout(unsigned int timeout_ms, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 10000) return ATTN_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != ATTN_OK) return rc;
  const cudaError_t e = ea51::launch_wait_selftest(
      ds->status, static_cast<unsigned long long>(timeout_ms) * 1000000ull,
      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  return ATTN_OK;
}

}  // extern "C"
