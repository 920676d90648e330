// Split-KV attention forward for callers that cannot allocate device memory.
//
// attn_fwd_splitkv needs a caller-provided device workspace for its partial
// results.  Some callers have no way to provide one: a plugin whose host
// framework hands it only the input and output tensors, or a serving loop
// that must not call cudaMalloc on its hot path (cudaMalloc can synchronise
// the whole device, and on a device whose memory is carved up by a pool
// allocator it can fail or fragment it).  This entry point keeps that
// workspace in a fixed device array reserved by the library itself, so a call
// allocates nothing.
//
// The array lives for as long as the library is loaded: every device the
// library is used on holds ATTN_NOALLOC_WORKSPACE_BYTES of memory for it from
// the first use until the process exits.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "attn_fwd.h"
#include "fwd_dispatch.h"

namespace {

static_assert(ATTN_NOALLOC_WORKSPACE_BYTES % 256 == 0, "workspace size");

// The shared split-KV workspace (fp32 partial outputs and log-sum-exps).
__device__ __align__(256) unsigned char g_noalloc_workspace[ATTN_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};  // device address of the array, per device

}  // namespace

extern "C" int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                        float* lse, int B, int H, int N, int d, float scale,
                                        int causal, int num_splits, void* stream) {
  // The checks attn_fwd_splitkv makes, in its order, so that both entry
  // points answer the same arguments with the same status; the size limit of
  // the fixed array comes before anything touches the device.
  int rc = attn_fwd_check_args(q, k, v, o, lse, B, H, N, d, scale, causal);
  if (rc != ATTN_OK) return rc;
  if (num_splits < 1 || num_splits > ea51::kMaxKvSplits) return ATTN_ERR_INVALID_ARG;
  if (num_splits > 1 &&
      attn_fwd_splitkv_workspace_size(B, H, N, d, num_splits) > ATTN_NOALLOC_WORKSPACE_BYTES)
    return ATTN_ERR_NOALLOC_TOO_LARGE;
  if ((rc = ea51::device_ready()) != ATTN_OK) return rc;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return ea51::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  void* ws = nullptr;
  {
    // One-time set-up per device, with that device current: the host-side
    // name of the array is only a stand-in, its device address comes from
    // the runtime.
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
      void* addr = nullptr;
      if ((e = cudaGetSymbolAddress(&addr, g_noalloc_workspace)) != cudaSuccess)
        return ea51::record_cuda_error(e);
      if (!addr) return ea51::record_cuda_error(cudaErrorInvalidSymbol);
      g_addr[dev] = addr;
    }
    ws = g_addr[dev];
  }
  return attn_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, num_splits, ws,
                          ATTN_NOALLOC_WORKSPACE_BYTES, stream);
}
