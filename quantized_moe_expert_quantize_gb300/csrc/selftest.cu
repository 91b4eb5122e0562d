// Self-test of the bounded pipeline waits: one warp waits on an mbarrier
// that nothing ever completes, through the same wait routine the product
// kernels use, and must give up by its own bound and report
// MOE_STATUS_PIPE_TIMEOUT -- the failure path of every product-kernel wait,
// exercised without a fault, a trap or an unbounded spin.
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

__global__ void __launch_bounds__(32) wait_timeout_kernel(int32_t* status, uint64_t timeout_ns,
                                                          int sleep) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival completes phase 0; none ever comes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const bool done = mbar_wait(&bar, 0, &abort_flag, timeout_ns, sleep != 0);
  __syncwarp();
  if (threadIdx.x == 0) {
    if (!done && abort_flag) atomicOr(status, MOE_STATUS_PIPE_TIMEOUT);
    // the barrier is left as it is: shared memory dies with the CTA
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_selftest_wait_timeout(int32_t* status, int sleep, moe_stream_t stream) {
  using namespace moe;
  if (!status) return MOE_ERR_NULL;
  if (((uintptr_t)status & 3) != 0) return MOE_ERR_ALIGN;
  if (sleep != 0 && sleep != 1) return MOE_ERR_SHAPE;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      major != 10 || minor != 3)
    return MOE_ERR_DEVICE;
  // the timed wait gives up after 20 ms of global time; the polling wait
  // after its fixed count of try_wait calls (about 1.4 s on a GB300)
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, 20000000ull, sleep);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}
