// Self-test of the kernels' bounded waits: one block waits on an mbarrier
// that nothing ever arrives on.  The wait gives up after the requested time,
// records its code in the device status word and the block exits, so the host
// sees ATTN_ERR_TIMEOUT from attn_fwd_device_status and the context stays
// usable.  Nothing traps, faults or spins without a limit.
#include "attn_fwd_kernel.cuh"

namespace ea51 {
namespace {

__global__ void wait_selftest_kernel(unsigned int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0u;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Waiter w{&abort_flag, status};
    // phase 0 never completes: no thread arrives and no copy is pending
    if (!mbar_try_wait(b, 0u)) wait_slow(b, 0u, w, kCodeSelfTest, false, timeout_ns);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned int* status, unsigned long long timeout_ns,
                                 cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace ea51
