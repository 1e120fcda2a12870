// Fixed workspace for kda_chunk_fwd_noalloc: callers that may not allocate
// device memory (allocators that are locked or pre-sized by the host
// application, code running where cudaMalloc is not allowed) get the chunked
// prefill with its chunk records kept in this file-scope device array instead
// of memory taken from the stream-ordered pool.
//
// The array exists once on every device that loads the library and stays
// allocated until the process exits.  Its device address is looked up once per
// device (cudaGetSymbolAddress with that device current) and cached; host code
// must never hand the array's name itself to a kernel.
#include <cuda_runtime.h>

#include <mutex>

#include "kda_internal.h"

namespace kda {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_ws[kNoallocWorkspaceBytes];

constexpr int kMaxDev = 64;
void* g_ws_ptr[kMaxDev];
std::mutex g_ws_mu;

}  // namespace

cudaError_t noalloc_workspace(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (!g_ws_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (e != cudaSuccess) return e;
    g_ws_ptr[dev] = p;
  }
  *ptr = g_ws_ptr[dev];
  return cudaSuccess;
}

}  // namespace kda
