// Allocation-free grouping entry point.
//
// moe_permute needs scratch memory (the per-chunk expert masks), which normally
// lives in the workspace the caller allocated for a plan.  Some callers cannot allocate device
// memory at all: engines whose memory planner owns every byte of the device and forbids a
// component from allocating outside its pool, and code on a latency-critical path, where
// cudaMalloc would synchronise the device.  moe_permute_static serves them: its scratch is a
// fixed, file-scope device array that exists as soon as the library is loaded on a device.
//
// The array is kStaticWords 32-bit words for the masks (1 MiB).  Every GPU that loads the
// library holds it until the process exits.  All calls
// on a device share it: calls that can overlap on the GPU (different streams without ordering)
// race on it.  Each call rewrites every scratch word it reads, so nothing needs clearing.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr size_t kStaticWords = size_t(1) << 18;  // mask words: group_mask_stride(n_chunks) * E <= 262144

static __device__ __align__(256) uint32_t g_static_scratch[kStaticWords];

// Device address of g_static_scratch in the current CUDA context.  The module (and the array)
// is loaded per context, so the address is cached under the context's unique id: a context that
// was destroyed and re-created (cudaDeviceReset, a released and re-retained primary context)
// gets a fresh lookup instead of a stale address.
static std::mutex g_static_mu;
struct StaticAddr {
  unsigned long long ctx_id;
  void* ptr;
};
static StaticAddr g_static_cache[64] = {};  // per device ordinal: the last context seen there

static cudaError_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  unsigned long long id = 0;
  if ((e = current_context_id(&id)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticAddr& c = g_static_cache[dev];
  if (!c.ptr || c.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    c.ptr = p;
    c.ctx_id = id;
  }
  *out = c.ptr;
  return cudaSuccess;
}

}  // namespace moe

extern "C" moe_status moe_permute_static(int E, int k, const int32_t* ids, int T, int32_t* counts, int32_t* offsets,
                                         int32_t* perm, int32_t* inv_perm, moe_stream_t stream) {
  using namespace moe;
  if (E < 1 || E > 1024 || k < 1 || k > 32 || k > E || T < 0) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || (T > 0 && (!ids || !perm || !inv_perm))) return MOE_ERR_INVALID_ARG;
  const size_t n_chunks = (static_cast<size_t>(T) + kChunk - 1) / kChunk;
  if (n_chunks > (kStaticWords >> 2) ||
      static_cast<size_t>(group_mask_stride(static_cast<int>(n_chunks))) * static_cast<size_t>(E) > kStaticWords)
    return MOE_ERR_WORKSPACE;
  void* base = nullptr;
  if (static_scratch(&base) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t* masks = static_cast<uint32_t*>(base);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T > 0 && launch_masks_from_ids(ids, T, E, k, masks, nullptr, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_group(ids, masks, T, E, k, counts, offsets, perm, inv_perm, nullptr, nullptr, 0, nullptr, st) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
