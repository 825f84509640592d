// Driver entry points through cudaGetDriverEntryPointByVersion (see
// driver_api.h).
#include "driver_api.h"

#include <map>
#include <mutex>
#include <string>

namespace ft {

void* driver_fn(const char* name) {
  static std::mutex mu;
  static std::map<std::string, void*> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(name);
  if (it != cache.end()) return it->second;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    fn = nullptr;
  if (fn) cache[name] = fn;
  return fn;
}

CUcontext current_context() {
  using Fn = CUresult (*)(CUcontext*);
  auto fn = reinterpret_cast<Fn>(driver_fn("cuCtxGetCurrent"));
  CUcontext ctx = nullptr;
  if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

}  // namespace ft
