// Bounded-wait self test: the kernels' time-limited mbarrier wait, run on a
// barrier nothing arrives on, must give up, flag MTP_ERR_TIMEOUT in the
// device error word and return.
#include "common.cuh"
#include "sm100.cuh"

namespace mtp {

namespace {

__global__ void wait_selftest_kernel(uint64_t timeout_ns, unsigned* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    sm100::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !sm100::mbar_wait_timeout(&bar, 0, timeout_ns)) raise_error(err, MTP_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t timeout_ns, unsigned* err, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(timeout_ns, err);
  return cudaGetLastError();
}

}  // namespace mtp
