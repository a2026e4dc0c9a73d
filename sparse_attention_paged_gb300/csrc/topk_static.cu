// topk_static.cu -- a fixed device array that serves as the top-k call's
// logits workspace for callers that pass none.  It sits in a translation
// unit (a module) of its own, so that with lazy module loading (the CUDA
// default) only a process that uses it has it resident.
#include <cuda_runtime.h>

#include <mutex>

#include "dsa_common.cuh"

namespace dsa {

// 24 Mi floats (96 MiB): rows x W*64 logits, e.g. 64 rows of 4,097 pages
constexpr long long kStaticScratchFloats = 24ll << 20;

__device__ __align__(256) float g_topk_scratch[kStaticScratchFloats];

long long static_scratch_floats() { return kStaticScratchFloats; }

// The array's device address on the current device, looked up once per
// device (the lookup may load this module, so a first call belongs outside
// stream capture).
cudaError_t static_scratch(float** ptr) {
  static float* addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float*>(p);
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

}  // namespace dsa
