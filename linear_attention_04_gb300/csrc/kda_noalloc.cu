// kda_noalloc.cu -- scratch area of the segment-parallel forward that is part
// of the library image, for callers that cannot hand the library a workspace.
//
// The area is one static device array per device (it exists once the library
// is loaded on that device); nothing is allocated at call time.  Its address is
// looked up with cudaGetSymbolAddress once per device, on the first call made
// with that device current.
#include <cuda_runtime.h>

#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::once_flag g_scratch_once[kMaxScratchDevices];
void* g_scratch_ptr[kMaxScratchDevices];

}  // namespace

void* noalloc_scratch() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return nullptr;
  std::call_once(g_scratch_once[dev], [dev]() {
    void* p = nullptr;
    g_scratch_ptr[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch) == cudaSuccess ? p : nullptr;
  });
  return g_scratch_ptr[dev];
}

}  // namespace kda
