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

constexpr size_t kStaticScratchBytes = DFLASH_NOALLOC_SCRATCH_BYTES;  // 20 MiB per device

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
  // The fc splits K over CTAs, each split with its own fp32 partial tile: when the
  // planner's split count would not fit the array, fewer splits are used (down to one),
  // so every M whose single-split scratch fits is served: M * d * 4 bytes plus a few
  // per-row and per-tile words, 1274 rows at d = 4096.
  if (!dims) return DFLASH_ERR_INVALID_ARG;
  if (M <= 0 || ctx_scratch_bytes(dims, M, 0) == 0)  // nothing to do, or refused arguments
    return ctx_project_impl(dims, hidden, M, W_fc, gamma_h, C_out, nullptr, 0, 0, stream);
  int cap = ctx_splits(dims, M);
  while (cap > 1 && ctx_scratch_bytes(dims, M, cap) > kStaticScratchBytes) --cap;
  if (ctx_scratch_bytes(dims, M, cap) > kStaticScratchBytes) return DFLASH_ERR_WORKSPACE;
  dflash_status st = DFLASH_OK;
  void* scratch = static_scratch(&st);
  if (!scratch) return st;
  // same kernels as dflash_ctx_project, on the fixed array
  return ctx_project_impl(dims, hidden, M, W_fc, gamma_h, C_out, scratch, kStaticScratchBytes, cap,
                          stream);
}
