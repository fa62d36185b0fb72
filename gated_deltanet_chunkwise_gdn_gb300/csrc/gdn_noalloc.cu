// gdn_noalloc.cu — gdn_extend_chunkwise_noalloc: the prefill entry point for callers that
// cannot allocate device memory, running on a fixed scratch area compiled into the library.
//
// Who needs it: code that is handed device buffers but no allocator — a plugin inside a
// host runtime that owns all device memory, or a serving loop that forbids cudaMalloc /
// cudaFree after start-up because they can synchronise the device or fail under a fixed
// memory budget. Such a caller still passes every input and output buffer; only the
// workspace comes from here.
//
// The scratch is one file-scope __device__ array. Every GPU that loads this library
// reserves it (kNoAllocScratchBytes) for the life of the process. In host code its name is
// only a host-side stand-in, so the device address is fetched with cudaGetSymbolAddress,
// once per device, the first time the entry point runs on that device (with the device
// current). Make that first call before capturing any stream. The address is kept for the
// life of the process: after cudaDeviceReset (or anything else that destroys the device's
// primary context) it is stale, so this entry point must not be used on that device again.
//
// All calls share the one array and it keeps whatever the last call left there: nothing in
// it has to start at zero (the first kernel of a call writes every field it later reads).
// Calls that overlap on the GPU (e.g. on two streams at once) race on it and must not be
// issued.
#include <mutex>

#include "gdn_common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
gdn_status noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_extend_chunkwise_noalloc(const void* q, const void* k, const void* v, gdn_dtype dtype, const float* a,
                                        const float* b, const float* A_log, const float* dt_bias, float* state_pool,
                                        int64_t pool_size, const int64_t* cache_indices, const int64_t* cu_seqlens,
                                        int32_t batch, void* out, int64_t total_tokens, int32_t H, int32_t HV,
                                        int32_t K, int32_t V, int32_t chunk_size, float scale, int32_t* device_status,
                                        void* stream) {
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u) != 0) return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_workspace_size(total_tokens, batch, H, HV, K, V, chunk_size);
  if (need > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;  // larger than the built-in scratch
  void* scratch = nullptr;
  const gdn_status st = noalloc_scratch(&scratch);
  if (st != GDN_OK) return st;
  const gdn_status r =
      gdn_extend_chunkwise(q, k, v, dtype, a, b, A_log, dt_bias, state_pool, pool_size, cache_indices, cu_seqlens,
                           batch, out, total_tokens, H, HV, K, V, chunk_size, scale, scratch, kNoAllocScratchBytes,
                           stream);
  if (r != GDN_OK || !device_status) return r;  // an error return enqueues nothing: *device_status keeps its value
  // The call's device-side status word is the first int32 of the workspace.
  if (cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

}  // extern "C"
