// Device buffers, streams and events reused across calls of the host-driven entry points (the
// streaming driver and the quorum executor), one idle list per device. cudaMalloc / cudaFree,
// stream and event creation cost tens to hundreds of microseconds each and cudaFree synchronises
// the device, which on a ~1 ms attention call is a large share of the end-to-end time. A call takes
// what it needs here and gives it back when all of its work has completed; cqsa_release_cache()
// frees everything idle.
#include <mutex>
#include <vector>

#include "cqsa_internal.h"

namespace cqsa {
namespace {

struct Buf {
  void* p;
  size_t n;
};

struct DevicePool {
  std::vector<Buf> bufs;                // idle buffers
  std::vector<cudaEvent_t> ev_timing;   // idle events with timing
  std::vector<cudaEvent_t> ev_plain;    // idle events without timing
  std::vector<cudaStream_t> streams;    // idle non-blocking streams
  std::vector<Buf> live;                // buffers handed out (their true size)
};

std::mutex g_mu;
std::vector<DevicePool> g_pools;

DevicePool& pool_of_current(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = 0;
  }
  if (static_cast<int>(g_pools.size()) <= dev) g_pools.resize(dev + 1);
  if (dev_out) *dev_out = dev;
  return g_pools[dev];
}

}  // namespace

int pool_alloc(void** p, size_t n) {
  std::lock_guard<std::mutex> lk(g_mu);
  DevicePool& dp = pool_of_current(nullptr);
  // best fit among idle buffers no larger than twice the request
  int best = -1;
  for (int i = 0; i < static_cast<int>(dp.bufs.size()); ++i) {
    const size_t m = dp.bufs[i].n;
    if (m >= n && m <= 2 * n + (2u << 20) && (best < 0 || m < dp.bufs[best].n)) best = i;
  }
  if (best >= 0) {
    *p = dp.bufs[best].p;
    dp.live.push_back(dp.bufs[best]);
    dp.bufs.erase(dp.bufs.begin() + best);
    return CQSA_OK;
  }
  cudaError_t e = cudaMalloc(p, n);
  if (e == cudaErrorMemoryAllocation && !dp.bufs.empty()) {
    // free the idle buffers of this device and try once more
    cudaGetLastError();
    for (const Buf& b : dp.bufs) cudaFree(b.p);
    dp.bufs.clear();
    e = cudaMalloc(p, n);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("device allocation of %zu bytes failed: %s", n, cudaGetErrorString(e));
    return e == cudaErrorMemoryAllocation ? CQSA_ERR_OOM : CQSA_ERR_CUDA;
  }
  dp.live.push_back({*p, n});
  return CQSA_OK;
}

void pool_free(void* p) {
  if (!p) return;
  std::lock_guard<std::mutex> lk(g_mu);
  DevicePool& dp = pool_of_current(nullptr);
  for (size_t i = 0; i < dp.live.size(); ++i)
    if (dp.live[i].p == p) {
      dp.bufs.push_back(dp.live[i]);
      dp.live.erase(dp.live.begin() + i);
      return;
    }
  cudaFree(p);  // not from this pool (another device): release it directly
}

int pool_event(cudaEvent_t* e, bool timing) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DevicePool& dp = pool_of_current(nullptr);
    std::vector<cudaEvent_t>& v = timing ? dp.ev_timing : dp.ev_plain;
    if (!v.empty()) {
      *e = v.back();
      v.pop_back();
      return CQSA_OK;
    }
  }
  return cuda_status(cudaEventCreateWithFlags(e, timing ? cudaEventDefault : cudaEventDisableTiming),
                     "cudaEventCreate");
}

void pool_event_free(cudaEvent_t e, bool timing) {
  if (!e) return;
  std::lock_guard<std::mutex> lk(g_mu);
  DevicePool& dp = pool_of_current(nullptr);
  (timing ? dp.ev_timing : dp.ev_plain).push_back(e);
}

int pool_stream(cudaStream_t* s) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DevicePool& dp = pool_of_current(nullptr);
    if (!dp.streams.empty()) {
      *s = dp.streams.back();
      dp.streams.pop_back();
      return CQSA_OK;
    }
  }
  return cuda_status(cudaStreamCreateWithFlags(s, cudaStreamNonBlocking), "cudaStreamCreate");
}

void pool_stream_free(cudaStream_t s) {
  if (!s) return;
  std::lock_guard<std::mutex> lk(g_mu);
  pool_of_current(nullptr).streams.push_back(s);
}

}  // namespace cqsa

extern "C" int cqsa_release_cache(void) {
  using namespace cqsa;
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    return CQSA_OK;  // no device: nothing was cached
  }
  for (int dev = 0; dev < static_cast<int>(g_pools.size()); ++dev) {
    DevicePool& dp = g_pools[dev];
    if (dp.bufs.empty() && dp.ev_timing.empty() && dp.ev_plain.empty() && dp.streams.empty()) continue;
    if (cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    for (const Buf& b : dp.bufs) cudaFree(b.p);
    for (cudaEvent_t e : dp.ev_timing) cudaEventDestroy(e);
    for (cudaEvent_t e : dp.ev_plain) cudaEventDestroy(e);
    for (cudaStream_t s : dp.streams) cudaStreamDestroy(s);
    dp.bufs.clear();
    dp.ev_timing.clear();
    dp.ev_plain.clear();
    dp.streams.clear();
  }
  cudaSetDevice(cur);
  return cuda_status(cudaGetLastError(), "release cache");
}
