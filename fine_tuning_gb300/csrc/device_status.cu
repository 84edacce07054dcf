// The library's device status word: a bit set by any kernel whose bounded
// wait ran out (kStatusWaitTimeout), read and cleared by the host.  Also a
// self-test kernel that drives the bounded wait to its limit on purpose:
// it waits on an mbarrier that nothing will ever complete, so the timeout
// path (flag set, kernel returns) runs without any fault or hang.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace ftk {

namespace {

__device__ unsigned g_status_word;

std::mutex g_mutex;
unsigned *g_status_ptr[64];

__global__ void wait_timeout_selftest(unsigned *status, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, limit, status);  // nothing arrives
}

}  // namespace

cudaError_t device_status_ptr(const DeviceInfo &dev, unsigned **out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (dev.device >= 0 && dev.device < 64 && g_status_ptr[dev.device]) {
    *out = g_status_ptr[dev.device];
    return cudaSuccess;
  }
  void *p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
  if (e != cudaSuccess) return e;
  if (dev.device >= 0 && dev.device < 64) g_status_ptr[dev.device] = (unsigned *)p;
  *out = (unsigned *)p;
  return cudaSuccess;
}

cudaError_t read_device_status(unsigned *flags, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_status_word, sizeof(unsigned));
  if (e != cudaSuccess || !clear) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_status_word, &zero, sizeof(unsigned));
}

cudaError_t launch_wait_timeout_selftest(const DeviceInfo &dev, long long limit_cycles,
                                         cudaStream_t s) {
  unsigned *status = nullptr;
  cudaError_t e = device_status_ptr(dev, &status);
  if (e != cudaSuccess) return e;
  wait_timeout_selftest<<<1, 32, 0, s>>>(status, limit_cycles);
  return cudaGetLastError();
}

}  // namespace ftk
