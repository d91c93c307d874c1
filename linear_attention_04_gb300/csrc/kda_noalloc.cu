// kda_noalloc.cu -- scratch area of the segment-parallel forward that is part
// of the library image, for callers that cannot hand the library a workspace.
//
// The area is one static device array per device (it exists once the library
// is loaded on that device); nothing is allocated at call time.  Its address is
// looked up with cudaGetSymbolAddress per device, on the first call made with
// that device current; only a successful lookup is kept (a failed one is
// retried by the next call).  cudaDeviceReset tears the module down and with
// it the area: the kept address is then stale, so a process that resets a
// device must not call the entry point on that device again.
#include <cuda_runtime.h>

#include <atomic>

#include "kda_internal.cuh"

namespace kda {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxScratchDevices];

}  // namespace

void* noalloc_scratch() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return nullptr;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
  g_scratch_ptr[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace kda
