// Per-device cache of "resident CTAs per SM" for a kernel at a launch shape,
// with the dynamic shared memory opt-in applied once per (kernel, device).
#include <mutex>
#include <vector>

#include "launch.h"

namespace ftk {

namespace {

struct OccEntry {
  const void *kernel;
  int device, threads;
  size_t smem;
  int blocks;
};
std::mutex g_occ_mutex;
std::vector<OccEntry> g_occ;

}  // namespace

int blocks_per_sm(const void *kernel, int threads, size_t smem, const DeviceInfo &dev,
                  int cap) {
  {
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    for (const OccEntry &e : g_occ)
      if (e.kernel == kernel && e.device == dev.device && e.threads == threads && e.smem == smem)
        return e.blocks < cap ? e.blocks : cap;
  }
  int n = 0;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
      n < 1) {
    cudaGetLastError();  // clear a sticky-free error from the query itself
    n = 1;
  }
  std::lock_guard<std::mutex> lock(g_occ_mutex);
  g_occ.push_back(OccEntry{kernel, dev.device, threads, smem, n});
  return n < cap ? n : cap;
}

}  // namespace ftk
