// ba_forward_noalloc: the forward pass for callers that cannot allocate device
// memory at the point where they run attention — for example a plugin invoked
// from another framework's execution loop, where a cudaMalloc would break that
// framework's memory plan or stall its stream, or a process whose device
// memory is handed to another allocator up front.  Instead of a caller-owned
// workspace it uses one file-scope device array of BA_NOALLOC_SCRATCH_BYTES.
//
// The array exists once per GPU that loads this library and stays reserved
// until the process exits.  Every call on a device shares it and it keeps the
// last call's contents; ba_forward clears what must start at zero (the status
// word) and overwrites everything else it reads.  Calls whose work overlaps on
// the GPU (two streams, or two threads) race on the array: order them.
// No cudaMalloc, cudaFree or allocating library routine is called.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "../../include/ba.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[BA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" int ba_forward_noalloc(ba_plan_t plan, const void* q_b, const void* k_m, const void* v_m, const void* k_b,
                                  const void* v_b, void* o, float* lse, void* stream) {
  if (!plan) return BA_ERR_INVALID_ARG;
  if (ba_workspace_bytes(plan) > size_t(BA_NOALLOC_SCRATCH_BYTES)) return BA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BA_ERR_CUDA;
  void* ptr = nullptr;
  {
    // set-up, once per device, with that device current: the host-side name of
    // the array is not a device address, so ask the runtime for the real one
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return BA_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    ptr = g_scratch_ptr[dev];
  }
  return ba_forward(plan, q_b, k_m, v_m, k_b, v_b, o, lse, ptr, size_t(BA_NOALLOC_SCRATCH_BYTES), stream);
}
