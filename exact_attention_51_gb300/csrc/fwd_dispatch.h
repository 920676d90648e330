// Host <-> kernel interface of the attention forward: launch parameters and
// the per-head-dim launcher table.  Plain C++ (no device code).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace ea51 {

struct FwdParams {
  void* o;               // bf16 [BH, Nq, D]
  float* lse;            // fp32 [BH, Nq]
  unsigned int* status;  // device-wide wait-timeout word (0 = clean)
  int Nq;               // query rows per head
  int Nk;               // key / value rows per head
  int causal_off;       // Nk - Nq: query i sees keys j <= i + causal_off when causal
  int BH;
  int n_qblk;            // CTAs per head
  int heads_per_group;   // causal launch order: heads whose query blocks interleave
  float scale_log2;      // scale * log2(e) (e4m3: times the Q and K dequantisation scales)
  float o_scale;         // e4m3: V's dequantisation scale (unused for bf16)
  // Split-KV: kv_splits CTAs share the key tiles of one query block; each
  // writes its normalised partial O (fp32 [kv_splits][BH][Nq][D]) and its
  // partial LSE (fp32 [kv_splits][BH][Nq], -inf when it saw no key) instead of
  // the final outputs.  kv_splits == 1 writes o / lse directly.
  int kv_splits;
  float* o_part;
  float* lse_part;
  // Test hook of attn_selftest_fwd_dropped_load, -1 on every other path: the
  // K/V ring position whose copy the producer leaves out in every CTA.
  int drop_load = -1;
  unsigned long long wait_timeout_ns = 0;  // limit of each bounded wait (0: about 2 s)
  int num_sms = 0;  // multiprocessors of the device (L2 prefetch for the next wave's CTAs)
};

struct FwdVariant {
  int kv_rows;         // keys per K/V tile (TMA box rows of K and V)
  int q_rows_per_cta;  // query rows per CTA (multiple of the 128-row Q box)
  // tq, tk, tv: Q, K, V tiles; to: the bf16 O tensor as Q's (the epilogue's
  // TMA stores).  The grid covers kv_splits.
  cudaError_t (*launch)(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                        const CUtensorMap* to, const FwdParams& p, bool causal, cudaStream_t stream);
};

// Merges kv_splits partial results per row into bf16 O and fp32 LSE.
cudaError_t launch_combine(int d, const float* o_part, const float* lse_part, void* o, float* lse,
                           long long rows, int kv_splits, cudaStream_t stream);

// Device address of the current device's wait-timeout status word (set up by
// the C ABI's per-device initialisation; nullptr if that failed).
unsigned int* status_word();

// Largest key-split count of the split-KV entry points.
constexpr int kMaxKvSplits = 64;

// The per-device set-up and check of every entry point (compute capability
// 10.3, status word, tensor-map encoder): ATTN_OK or the status the entry
// point returns.  For entry points defined outside attn_api.cu.
int device_ready();

// Records `e` as this host thread's last CUDA error (attn_last_cuda_error)
// and returns ATTN_ERR_LAUNCH.
int record_cuda_error(cudaError_t e);

// Launches a one-block kernel that waits on an mbarrier nothing arrives on,
// with the kernel's bounded wait cut to `timeout_ns`.
cudaError_t launch_wait_selftest(unsigned int* status, unsigned long long timeout_ns,
                                 cudaStream_t stream);

FwdVariant fwd_variant_d64();
FwdVariant fwd_variant_d128();
// two CTAs per SM, one 128-row query tile each (short rows)
FwdVariant fwd_variant_d64_two();
FwdVariant fwd_variant_d256();
FwdVariant fwd_variant_e4m3_d64();
FwdVariant fwd_variant_e4m3_d128();
FwdVariant fwd_variant_e4m3_d256();
FwdVariant fwd_variant_e4m3_d64_two();
// one 128-row query tile and two S buffers per CTA (grids that the default
// shape would leave short of one wave)
FwdVariant fwd_variant_d64_solo();
FwdVariant fwd_variant_d128_solo();
FwdVariant fwd_variant_e4m3_d64_solo();
FwdVariant fwd_variant_e4m3_d128_solo();

}  // namespace ea51
