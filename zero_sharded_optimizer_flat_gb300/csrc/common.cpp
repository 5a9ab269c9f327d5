// Error reporting, version, device properties.
#include <cuda_runtime.h>

#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace zopt {

namespace {
thread_local std::string g_last_error;
}

zopt_status fail(zopt_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

zopt_status ok() {
  g_last_error.clear();
  return ZOPT_OK;
}

int sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= static_cast<int>(cache.size())) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace zopt

extern "C" const char* zopt_last_error(void) { return zopt::g_last_error.c_str(); }

extern "C" const char* zopt_version(void) { return "zopt 0.1 (sm_103a)"; }
