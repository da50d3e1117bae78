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
// e4m3 cache with a tcgen05 prefill (head_dim 64/128/192/256): the new
// tokens of the sequences the prefill kernel serves go into their pages
// ahead of the attention kernels (launched right behind the planner,
// overlapping it).
cudaError_t launch_prefill_pages(const KvArgs& a, const int32_t* kv_lens, const int32_t* qsl,
                                 const int32_t* dist, int num_sms, cudaStream_t stream);
cudaError_t launch_decode(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream);
// The prefill kernel for these params:
//   kPrefillTc      tcgen05, two 128-row query tiles per unit: head_dim 64 and 128
//   kPrefillTcWide  tcgen05, one 128-row query tile per unit: head_dim 192 and 256
//   kPrefillMma     warp-level MMA, 64-row tiles: head_dim 96, and pages of
//                   fewer than 8 rows (the tcgen05 kernels' TMA warp holds
//                   one page of a key tile per lane)
enum PrefillKind { kPrefillMma = 0, kPrefillTc = 1, kPrefillTcWide = 2 };
inline PrefillKind prefill_kind(const rpa_params_t& p) {
  if (p.page_size < 8) return kPrefillMma;
  if (p.head_dim == 64 || p.head_dim == 128) return kPrefillTc;
  if (p.head_dim == 192 || p.head_dim == 256) return kPrefillTcWide;
  return kPrefillMma;
}
cudaError_t launch_prefill(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream);
cudaError_t launch_prefill_tc(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream);
cudaError_t launch_prefill_tc_wide(const AttnArgs& a, int max_units, int num_sms,
                                   cudaStream_t stream);

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

// Rows of a prefill unit for these params (the planner and the kernels agree on it).
inline int prefill_rows_for(const rpa_params_t& p) {
  switch (prefill_kind(p)) {
    case kPrefillTc: return 256;
    case kPrefillTcWide: return 128;
    default: return kPrefillRows;
  }
}

// plan -> decode -> prefill on `stream`; events (4, or null) are recorded
// before the planner and after each kernel.
int enqueue_forward(const rpa_params_t& p, const AttnArgs& a, const int32_t* distribution,
                    int num_sms, cudaStream_t stream, void* const* events);

}  // namespace rpa
