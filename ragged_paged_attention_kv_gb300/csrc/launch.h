// Host-side launchers of the library's kernels (one definition each, in the
// kernel's own translation unit).
#pragma once

#include <cuda_runtime.h>

#include "kv_write.cuh"

namespace rpa {

cudaError_t launch_plan(const rpa_params_t& p, const int32_t* kv_lens, const int32_t* qsl,
                        const int32_t* dist, int32_t* ws, int prefill_rows, cudaStream_t stream);
cudaError_t launch_cache_write(const KvArgs& a, const int32_t* kv_lens, const int32_t* qsl,
                               int prefill_rows, int num_sms, cudaStream_t stream);
cudaError_t launch_decode(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream);
// warp-level MMA prefill (64-row tiles): pages of fewer than 8 rows, and head_dim 96/192/256
cudaError_t launch_prefill(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream);
// tcgen05 prefill (two 128-row query tiles per unit): head_dim 64 and 128, pages >= 8 rows
bool prefill_uses_tc(const rpa_params_t& p);
cudaError_t launch_prefill_tc(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream);

// The alignment the kernels' bulk and tensor copies rely on: the bf16
// tensors and the cache on 16 bytes, the int32 arrays and the sink on 4.
// Null pointers pass (each entry point checks the ones it requires).
inline bool pointers_aligned(const void* queries, const void* keys, const void* values,
                             const void* kv_cache, const void* out, const void* kv_lens,
                             const void* block_tables, const void* query_start_loc,
                             const void* distribution, const void* attention_sink) {
  auto on = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
  return on(queries, 16) && on(keys, 16) && on(values, 16) && on(kv_cache, 16) && on(out, 16) &&
         on(kv_lens, 4) && on(block_tables, 4) && on(query_start_loc, 4) && on(distribution, 4) &&
         on(attention_sink, 4);
}

// Rows of a prefill tile for these params (the planner and the kernels agree on it).
inline int prefill_rows_for(const rpa_params_t& p) { return prefill_uses_tc(p) ? 256 : kPrefillRows; }

// plan -> decode -> prefill on `stream`; events (4, or null) are recorded
// before the planner and after each kernel.
int enqueue_forward(const rpa_params_t& p, const AttnArgs& a, const int32_t* distribution,
                    int num_sms, cudaStream_t stream, void* const* events);

}  // namespace rpa
