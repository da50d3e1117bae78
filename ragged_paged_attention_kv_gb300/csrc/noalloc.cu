// rpa_forward_noalloc: rpa_forward for callers that cannot allocate device
// memory.
//
// Some callers have no way to hand the library a workspace: code running
// inside a memory pool or allocator callback (where allocating again would
// re-enter the allocator), plugins of runtimes that own every device
// allocation and expose none to extensions, or setups that forbid any
// allocation after start-up.  For them this entry point takes its scratch
// memory (the planner's work lists, the split-KV partial results and their
// counters) from one fixed array in device global memory.  The array is
// reserved when the library's device code is loaded into a context and held
// there until that context is destroyed (for the primary context: process
// exit or cudaDeviceReset).  The entry point allocates nothing itself and
// calls no allocating routine.
#include "common.cuh"
#include "kv_write.cuh"

#include "launch.h"

namespace rpa {

// The fixed scratch array.  Host code must not pass `g_static_workspace`
// itself to a kernel: on the host that name is only a stand-in for the
// device symbol.  Its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_static_workspace[RPA_NOALLOC_WORKSPACE_BYTES];

namespace {
// The array's device address in the current context.  It is looked up on
// every call rather than cached: each context holds its own copy of the
// array (a context made with cuCtxCreate next to the primary one, or the
// primary context rebuilt after cudaDeviceReset, puts it at another
// address).  Once the library's module is loaded in the context, the lookup
// allocates nothing.
cudaError_t static_workspace(void** out) {
  return cudaGetSymbolAddress(out, g_static_workspace);
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
