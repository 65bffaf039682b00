// Self-test of the bounded device-side wait used by every pipelined kernel.
// A single CTA waits on a shared-memory mbarrier that nothing arrives on; the
// wait gives up after the given time and records DFLASH_ERR_DEVICE_TIMEOUT in
// the status word, and the kernel returns normally.
#include "common.cuh"

namespace {

__global__ void selftest_timeout_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    *status = 0;
    abort_flag = 0;
    dfl::mbar_init(&bar, 1);
    dfl::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 never completes: no thread arrives on the barrier
    (void)dfl::mbar_wait_bounded(&bar, 0, &abort_flag, status, limit_ns);
  }
  __syncthreads();
}

}  // namespace

extern "C" int dflash_selftest_timeout(void* workspace, long long limit_ns, dflash_stream_t stream) {
  if (!workspace) return DFLASH_ERR_WORKSPACE;
  if (limit_ns < 0) return DFLASH_ERR_ARG;
  if (limit_ns > 1000000000ll) limit_ns = 1000000000ll;
  selftest_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<int*>(workspace), (unsigned long long)limit_ns);
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ERR_LAUNCH;
}
