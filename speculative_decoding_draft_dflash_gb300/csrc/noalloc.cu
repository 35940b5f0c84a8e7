// Context projection that takes its scratch from a fixed array in the library.
//
// Some callers cannot hand the library a workspace: code that runs inside
// another runtime's launch path (an inference server's custom-operator
// enqueue, say) where the host runtime owns every byte of device memory and
// any cudaMalloc would both break its accounting and synchronise the whole
// device in the middle of a latency-critical loop. For them this entry point
// needs only its inputs and outputs: the scratch lives in a file-scope
// __device__ array that every GPU loading the library holds until the process
// exits.
#include <mutex>

#include "dflash_internal.cuh"

namespace dflash {
namespace {

constexpr size_t kStaticScratchBytes = DFLASH_NOALLOC_SCRATCH_BYTES;  // 16 MiB per device

// The array's name in host code is only a host-side handle for the symbol; the
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_ctx_scratch[kStaticScratchBytes];

void* static_scratch(dflash_status* st) {
  static std::mutex mu;
  static void* ptr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    *st = DFLASH_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ctx_scratch) != cudaSuccess || !p) {
      *st = DFLASH_ERR_CUDA;
      return nullptr;
    }
    ptr[dev] = p;
  }
  *st = DFLASH_OK;
  return ptr[dev];
}

}  // namespace
}  // namespace dflash

using namespace dflash;

DFLASH_API dflash_status dflash_ctx_project_noalloc(const dflash_dims* dims,
                                                    const void* const* hidden, int M,
                                                    const void* W_fc, const void* gamma_h,
                                                    void* C_out, cudaStream_t stream) {
  dflash_status st = DFLASH_OK;
  void* scratch = static_scratch(&st);
  if (!scratch) return st;
  // Same kernels as dflash_ctx_project; a call whose scratch need exceeds the
  // array is refused there with DFLASH_ERR_WORKSPACE before anything launches.
  return dflash_ctx_project(dims, hidden, M, W_fc, gamma_h, C_out, scratch, kStaticScratchBytes,
                            stream);
}
