// Per-device host state (see runtime.h).
#include <map>
#include <mutex>
#include <utility>

#include "runtime.h"

namespace df {
namespace {
std::mutex mu;
std::map<int, int> sm_count;                                // device -> SMs
std::map<std::pair<int, const void*>, size_t> smem_set;     // (device, kernel) -> bytes allowed

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}
}  // namespace

int num_sms() {
  const int dev = current_device();
  std::lock_guard<std::mutex> g(mu);
  auto it = sm_count.find(dev);
  if (it != sm_count.end()) return it->second;
  int n = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  sm_count[dev] = n;
  return n;
}

cudaError_t ensure_dynamic_smem(const void* func, size_t bytes) {
  // Set even for small sizes: a kernel's static shared memory counts against the default
  // 48 KB as well, so a kernel with both needs the opt-in below that size.
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(mu);
  size_t& have = smem_set[{dev, func}];
  if (have >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

}  // namespace df
