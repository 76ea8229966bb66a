// Self-test of the device failure report: a wait that nothing satisfies runs
// out under the same bounded-wait scheme as the step's kernels (mbarrier
// try-wait polled against a clock64 limit) and records DSA_ERR_TIMEOUT in the
// status word, which the host then reads; the context stays usable.
#include "kernels.h"

namespace dsa {

namespace {

__global__ void timeout_selftest_kernel(DeviceStatus* st, long long limit_cycles) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none is ever made
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  const uint32_t a = smem_u32(&bar);
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(a, 0)) return;  // cannot happen: no arrival
    if ((it & 63u) == 0 && clock64() - t0 > limit_cycles) {
      record_status(st, DSA_ERR_TIMEOUT, SITE_SELFTEST, a);
      return;
    }
  }
}

}  // namespace

cudaError_t launch_timeout_selftest(DeviceStatus* st, long long limit_cycles, cudaStream_t s) {
  timeout_selftest_kernel<<<1, 32, 0, s>>>(st, limit_cycles);
  return cudaGetLastError();
}

}  // namespace dsa
