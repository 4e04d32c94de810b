// Self-test of the bounded-wait mechanism every kernel of the library uses:
// a one-CTA kernel whose warps wait on an mbarrier that nothing ever arrives
// on.  Warp 0 gives up after the given limit, records
// UPIPE_ERR_DEVICE_TIMEOUT in the device error word and raises the CTA's
// abort flag; warp 1, waiting on a second such barrier, sees the flag and
// leaves too.  No fault, no trap: the context stays usable.
// A second self-test exercises the debug builds' bounds checks (below).
#include "internal.h"
#include "ptx.cuh"

namespace upipe {

__global__ void selftest_wait_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* ab = &abort_flag;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    mbar_wait_for(&bars[0], 0, err, ab, limit_ns);
  } else {
    // far longer limit: returns through the abort flag raised by warp 0
    mbar_wait_for(&bars[1], 0, err, ab, 20 * limit_ns);
  }
  __syncthreads();
}

cudaError_t launch_selftest_wait(int* err, unsigned long long limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

// Self-test of the debug builds' bounds checks.  The kernel declares a view of
// kProbeView elements over an array of twice that size and asks to write
// element kProbeView, one past the view: the check must refuse it, record
// UPIPE_ERR_BOUNDS and skip the write.  The element lies inside the array, so
// the write is harmless should a check ever let it through (and a release
// build, whose checks compile to true, performs it: that build reports
// nothing, and probe_written says so).
constexpr int kProbeView = 16;
__device__ int g_bounds_probe[2 * kProbeView];

__global__ void selftest_bounds_kernel(int* err) {
  g_bounds_probe[kProbeView] = 0;
  __threadfence();
  const long long i = kProbeView + (long long)threadIdx.x;   // one thread: kProbeView
  if (dbg_in(i, i, kProbeView, err)) g_bounds_probe[i] = 1;
}

cudaError_t launch_selftest_bounds(int* err, cudaStream_t stream) {
  selftest_bounds_kernel<<<1, 1, 0, stream>>>(err);
  return cudaGetLastError();
}

cudaError_t selftest_bounds_probe_written(int* written) {
  return cudaMemcpyFromSymbol(written, g_bounds_probe, sizeof(int), kProbeView * sizeof(int));
}

}  // namespace upipe
