// device.cu -- per-device facts the launchers need: the SM count (grid sizing) and the dynamic
// shared-memory limit of each kernel, which belongs to the device's context and so is set once per
// (device, kernel), under a lock, rather than once per process.
#include <mutex>
#include <set>
#include <utility>

#include "kernels.h"

namespace grd {

static constexpr int kMaxDevices = 64;

int device_sm_count() {
  static std::mutex mu;
  static int count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 0;
    count[dev] = n;
  }
  return count[dev];
}

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  cudaError_t r = cudaGetDevice(&dev);
  if (r != cudaSuccess) return r;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, kernel})) return cudaSuccess;
  r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (r == cudaSuccess) done.insert({dev, kernel});
  return r;
}

}  // namespace grd
