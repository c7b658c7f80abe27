// Self-test of the bounded waits every kernel of this library relies on: one
// warp initialises an mbarrier that nothing will ever complete and waits on it
// with the library's own bounded wait.  The wait must give up after the limit
// and record PA_ERR_TIMEOUT in the device error word; the kernel then returns
// normally, so the context stays usable.  Nothing faults, traps or hangs.
#include "pa_device.cuh"

namespace pa {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(int *err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected, none will come
    fence_mbar_init();
  }
  __syncwarp();
  const bool done = mbar_wait(&bar, 0, limit_ns);
  if (!done && threadIdx.x == 0) set_error(err, PA_ERR_TIMEOUT, -1);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int *err, uint64_t limit_ns, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace pa
