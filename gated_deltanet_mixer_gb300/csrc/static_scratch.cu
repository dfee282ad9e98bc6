// static_scratch.cu -- device scratch owned by the library, for the
// allocation-free prefill entry point (gdn_prefill_static).  The array lives
// in a translation unit of its own, so that with lazy module loading (the
// CUDA default) a process pays its memory only once it calls that entry.
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"
#include "launch.h"

namespace gdn {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[GDN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices];  // per device, resolved once

}  // namespace

cudaError_t static_scratch(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *ptr = g_addr[dev];
  return cudaSuccess;
}

}  // namespace gdn
