// device.cu -- per-device facts the launchers need: the SM count (grid sizing) and the dynamic
// shared-memory limit of each kernel, which belongs to the device's context and so is kept per
// (device, kernel), under a lock, rather than per process.
#include <map>
#include <mutex>
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

// The limit only ever grows: engines on one device may need different amounts for the same kernel, and a
// limit above a launch's need is harmless.
cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> limit;
  int dev = 0;
  cudaError_t r = cudaGetDevice(&dev);
  if (r != cudaSuccess) return r;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(dev, kernel);
  const auto it = limit.find(key);
  if (it != limit.end() && it->second >= bytes) return cudaSuccess;
  r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (r == cudaSuccess) limit[key] = bytes;
  return r;
}

}  // namespace grd
