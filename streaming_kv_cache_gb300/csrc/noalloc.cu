// kv_stream_insert_noalloc: the frame insert for callers that cannot allocate
// device memory.  The insert's arrival counters (one int32 per cache and
// view) live in a file-scope static device array instead of caller memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "kernels.h"
#include "skv.h"

namespace {

// Counters of kv_stream_insert's last-CTA-done head advance; every device
// that loads the library holds this array until the process exits.
static __device__ __align__(256) int32_t g_insert_counters[SKV_NOALLOC_MAX_CACHE_VIEWS];

// Device address of g_insert_counters per device ordinal, looked up once per
// device with that device current (the host-side name is only a stand-in).
// Host threads that make their first call on a device together may both look
// it up; they store the same address.  A cudaDeviceReset invalidates it.
std::atomic<int32_t*> g_counters_addr[64];

}  // namespace

extern "C" int kv_stream_insert_noalloc(const skv_cache* cache, const void* k_new,
                                        const void* v_new, void* stream) {
  if (!cache) return SKV_ERR_INVALID;
  if (cache->n_cache < 0 || cache->n_view < 1) return SKV_ERR_INVALID;
  const long long n_counters = (long long)cache->n_cache * cache->n_view;
  if (n_counters > SKV_NOALLOC_MAX_CACHE_VIEWS) return SKV_ERR_TOO_LARGE;
  // every argument and the device are checked before the array is looked up
  // (cache->sync is not read: the counters below replace it)
  int rc = skv::check_insert_args(cache, k_new, v_new);
  if (rc != SKV_OK || cache->n_cache == 0) return rc;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return skv::record_cuda_error(e);
  if (dev < 0 || dev >= 64) return SKV_ERR_UNSUPPORTED;
  int32_t* counters = g_counters_addr[dev].load(std::memory_order_relaxed);
  if (!counters) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_insert_counters);
    if (e != cudaSuccess) return skv::record_cuda_error(e);
    counters = static_cast<int32_t*>(p);
    g_counters_addr[dev].store(counters, std::memory_order_relaxed);
  }

  skv_cache local = *cache;
  local.sync = counters;
  // the counters must start at zero; the array keeps whatever the last call left
  e = cudaMemsetAsync(local.sync, 0, (size_t)n_counters * sizeof(int32_t), (cudaStream_t)stream);
  if (e != cudaSuccess) return skv::record_cuda_error(e);
  return kv_stream_insert(&local, k_new, v_new, stream);
}
