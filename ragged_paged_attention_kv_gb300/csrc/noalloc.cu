// rpa_forward_noalloc: rpa_forward for callers that cannot allocate device
// memory.
//
// Some callers have no way to hand the library a workspace: code running
// inside a memory pool or allocator callback (where allocating again would
// re-enter the allocator), plugins of runtimes that own every device
// allocation and expose none to extensions, or setups that forbid any
// allocation after start-up.  For them this entry point takes its scratch
// memory (the planner's work lists, the split-KV partial results and their
// counters) from one fixed array in device global memory, reserved when the
// library is loaded and held by every GPU that loads it until the process
// exits.  It allocates nothing itself and calls no allocating routine.
#include <mutex>

#include "common.cuh"
#include "kv_write.cuh"

#include "launch.h"

namespace rpa {

// The fixed scratch array.  Host code must not pass `g_static_workspace`
// itself to a kernel: on the host that name is only a stand-in for the
// device symbol.  Its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_static_workspace[RPA_NOALLOC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {};  // device address of the array, per device

// Resolves the array's device address on the current device (once per
// device; later calls reuse it).
cudaError_t static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ws_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess) return e;
    g_ws_addr[dev] = p;
  }
  *out = g_ws_addr[dev];
  return cudaSuccess;
}
}  // namespace
}  // namespace rpa

using namespace rpa;

extern "C" int rpa_forward_noalloc(const rpa_params_t* params, const void* queries,
                                   const void* keys, const void* values, void* kv_cache,
                                   const int32_t* kv_lens, const int32_t* block_tables,
                                   const int32_t* query_start_loc, const int32_t* distribution,
                                   const float* attention_sink, void* out, void* stream) {
  size_t need = 0;
  int rc = rpa_workspace_size(params, &need);  // also validates params
  if (rc) return rc;
  if (need > (size_t)RPA_NOALLOC_WORKSPACE_BYTES) return RPA_ERR_NOALLOC_TOO_LARGE;
  if (!queries || !keys || !values || !kv_cache || !kv_lens || !block_tables ||
      !query_start_loc || !distribution || !out)
    return RPA_ERR_INVALID_ARG;
  if (!pointers_aligned(queries, keys, values, kv_cache, out, kv_lens, block_tables,
                        query_start_loc, distribution, attention_sink))
    return RPA_ERR_INVALID_ARG;
  void* ws = nullptr;
  if (static_workspace(&ws) != cudaSuccess) return RPA_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return RPA_ERR_CUDA;
  // The planner rewrites every workspace word the kernels read (header,
  // counters of the sequences it plans, work lists), so what the previous
  // call left in the array needs no clearing.
  AttnArgs a{{*params, reinterpret_cast<const __nv_bfloat16*>(keys),
              reinterpret_cast<const __nv_bfloat16*>(values),
              reinterpret_cast<uint8_t*>(kv_cache), block_tables, reinterpret_cast<int32_t*>(ws)},
             reinterpret_cast<const __nv_bfloat16*>(queries),
             kv_lens,
             query_start_loc,
             attention_sink,
             reinterpret_cast<__nv_bfloat16*>(out)};
  rc = enqueue_forward(*params, a, distribution, sms, reinterpret_cast<cudaStream_t>(stream),
                       nullptr);
  if (rc) return rc;
  return RPA_OK;
}
