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

// Rows of a prefill tile for these params (the planner and the kernels agree on it).
inline int prefill_rows_for(const rpa_params_t& p) { return prefill_uses_tc(p) ? 256 : kPrefillRows; }

// plan -> decode -> prefill on `stream`; events (4, or null) are recorded
// before the planner and after each kernel.
int enqueue_forward(const rpa_params_t& p, const AttnArgs& a, const int32_t* distribution,
                    int num_sms, cudaStream_t stream, void* const* events);

}  // namespace rpa
