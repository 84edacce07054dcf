// Per-device cache of "resident CTAs per SM" for a kernel at a launch shape,
// and the dynamic shared memory opt-in, applied once per (kernel, device).
#include <mutex>
#include <utility>
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
std::vector<std::pair<const void *, int>> g_raised;  // (kernel, device) opted in

// Lets `kernel` use all the dynamic shared memory the device allows next to
// its static shared memory, once per (kernel, device).  Raising it to the
// maximum (never to one launch's size) keeps every later launch of the same
// kernel valid whatever its size.
void raise_smem_limit(const void *kernel, const DeviceInfo &dev) {
  for (const auto &r : g_raised)
    if (r.first == kernel && r.second == dev.device) return;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kernel) == cudaSuccess &&
      (size_t)dev.max_smem_optin > fa.sharedSizeBytes)
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)(dev.max_smem_optin - fa.sharedSizeBytes));
  cudaGetLastError();  // a refused opt-in surfaces at launch, not here
  g_raised.emplace_back(kernel, dev.device);
}

}  // namespace

int blocks_per_sm(const void *kernel, int threads, size_t smem, const DeviceInfo &dev,
                  int cap) {
  std::lock_guard<std::mutex> lock(g_occ_mutex);
  for (const OccEntry &e : g_occ)
    if (e.kernel == kernel && e.device == dev.device && e.threads == threads && e.smem == smem)
      return e.blocks < cap ? e.blocks : cap;
  raise_smem_limit(kernel, dev);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    n = 1;
  }
  g_occ.push_back(OccEntry{kernel, dev.device, threads, smem, n});
  return n < cap ? n : cap;
}

}  // namespace ftk
