// Kernel tracing: CUDA event pairs around selected launches, and a launch counter.
#include <atomic>
#include <mutex>
#include <vector>

#include "dflash_internal.cuh"

namespace dflash {
namespace {

struct TraceState {
  std::mutex mu;
  bool active = false;
  unsigned mask = 0;
  int max_launches = 0;
  int count = 0;
  int base = 0;                     // first event pair of the current session
  std::vector<cudaEvent_t> events;  // 2 per launch; a session never reuses an earlier
                                    // session's events (a captured graph may still hold them)
  std::vector<int> kinds;
};

TraceState& state() {
  static TraceState s;
  return s;
}

std::atomic<unsigned long long> g_launches{0};

// Inside a stream capture an event must be recorded as an external node to carry a
// timestamp; outside a capture a plain record does that.
cudaError_t record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return cudaErrorUnknown;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal)
                                             : cudaEventRecord(e, s);
}

}  // namespace

LaunchScope::LaunchScope(int kind, cudaStream_t s) : kind_(kind), stream_(s), slot_(-1) {
  TraceState& t = state();
  if (!t.active || !(t.mask & (1u << kind))) return;
  std::lock_guard<std::mutex> lock(t.mu);
  if (!t.active || t.count >= t.max_launches) return;
  if (record(t.events[2 * (t.base + t.count)], s) != cudaSuccess) {
    cudaGetLastError();  // tracing must not turn into a launch error
    return;
  }
  slot_ = t.count++;
  t.kinds[slot_] = kind;
}

LaunchScope::~LaunchScope() {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (slot_ < 0) return;
  TraceState& t = state();
  if (record(t.events[2 * (t.base + slot_) + 1], stream_) != cudaSuccess) cudaGetLastError();
}

}  // namespace dflash

using namespace dflash;

DFLASH_API dflash_status dflash_trace_start(unsigned int kernel_mask, int max_launches) {
  if (max_launches < 0) return DFLASH_ERR_INVALID_ARG;
  TraceState& t = state();
  std::lock_guard<std::mutex> lock(t.mu);
  t.base = (int)t.events.size() / 2;
  while ((int)t.events.size() < 2 * (t.base + max_launches)) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return DFLASH_ERR_CUDA;
    t.events.push_back(e);
  }
  t.kinds.assign(max_launches, 0);
  t.mask = kernel_mask;
  t.max_launches = max_launches;
  t.count = 0;
  t.active = true;
  return DFLASH_OK;
}

DFLASH_API dflash_status dflash_trace_stop(int* kinds, float* ms, int capacity, int* count) {
  TraceState& t = state();
  std::lock_guard<std::mutex> lock(t.mu);
  t.active = false;
  if (count) *count = t.count;
  for (int i = 0; i < t.count && i < capacity; ++i) {
    const int ev = 2 * (t.base + i);
    if (cudaEventSynchronize(t.events[ev + 1]) != cudaSuccess) return DFLASH_ERR_CUDA;
    float v = 0.f;
    if (cudaEventElapsedTime(&v, t.events[ev], t.events[ev + 1]) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    if (kinds) kinds[i] = t.kinds[i];
    if (ms) ms[i] = v;
  }
  return DFLASH_OK;
}

DFLASH_API unsigned long long dflash_launch_count(void) {
  return g_launches.load(std::memory_order_relaxed);
}
