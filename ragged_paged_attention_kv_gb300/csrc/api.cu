// C ABI entry points (declared in include/rpa.h): argument checks, workspace
// sizing and the launch sequence plan -> decode -> prefill on the caller's
// stream.  No entry point allocates device memory or synchronises (except
// rpa_get_status).
#include <cfloat>
#include <cstring>

#include "common.cuh"
#include "kv_write.cuh"

#include "launch.h"

namespace rpa {

static bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

static int check_params(const rpa_params_t* p) {
  if (!p) return RPA_ERR_INVALID_ARG;
  if (p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0 || p->page_size <= 0 ||
      p->num_pages <= 0 || p->pages_per_seq <= 0 || p->max_num_seqs <= 0 || p->total_tokens < 0 ||
      p->sliding_window < 0)
    return RPA_ERR_INVALID_ARG;
  if (p->num_q_heads % p->num_kv_heads != 0) return RPA_ERR_UNSUPPORTED;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (!(G == 1 || G == 2 || G == 4 || G == 8 || G == 16)) return RPA_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 96 && p->head_dim != 128 && p->head_dim != 192 &&
      p->head_dim != 256)
    return RPA_ERR_UNSUPPORTED;
  if (!is_pow2(p->page_size) || p->page_size > 1024) return RPA_ERR_UNSUPPORTED;
  if (p->kv_dtype != RPA_KV_BF16 && p->kv_dtype != RPA_KV_FP8_E4M3) return RPA_ERR_UNSUPPORTED;
  // fp8 rows of 64 or 96 bytes need at least two rows per page for 128-byte
  // aligned copies
  if (p->kv_dtype == RPA_KV_FP8_E4M3 && (p->head_dim == 64 || p->head_dim == 96) &&
      p->page_size < 2)
    return RPA_ERR_UNSUPPORTED;
  if (!(p->softmax_scale > 0.f) || !(p->logits_soft_cap >= 0.f))
    return RPA_ERR_INVALID_ARG;
  if (!(p->q_scale >= 0.f) || !(p->q_scale <= FLT_MAX) ||
      (p->q_scale > 0.f && p->kv_dtype != RPA_KV_FP8_E4M3))
    return RPA_ERR_INVALID_ARG;
  if (p->kv_dtype == RPA_KV_FP8_E4M3) {
    if (!(p->k_scale > 0.f) || !(p->v_scale > 0.f)) return RPA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p->k_scale_heads) & 3) != 0 ||
        (reinterpret_cast<uintptr_t>(p->v_scale_heads) & 3) != 0)
      return RPA_ERR_INVALID_ARG;
  } else if (p->k_scale != 1.f || p->v_scale != 1.f || p->k_scale_heads || p->v_scale_heads) {
    return RPA_ERR_INVALID_ARG;
  }
  // pool byte offsets and token rows must stay inside int64 / int32 ranges
  const int64_t pool_rows = (int64_t)p->num_pages * p->page_size;
  if (pool_rows > (int64_t)1 << 31) return RPA_ERR_UNSUPPORTED;
  if ((int64_t)p->pages_per_seq * p->page_size > (int64_t)1 << 30) return RPA_ERR_UNSUPPORTED;
  if ((int64_t)p->total_tokens * p->num_q_heads > (int64_t)1 << 31) return RPA_ERR_UNSUPPORTED;
  return RPA_OK;
}

static int check_ws(const rpa_params_t* p, const void* ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0) return RPA_ERR_WORKSPACE;
  const WorkspaceLayout L(*p);
  if (bytes < L.total) return RPA_ERR_WORKSPACE;
  return RPA_OK;
}

static int num_sms_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return n;
}

}  // namespace rpa

using namespace rpa;

namespace rpa {
int enqueue_forward(const rpa_params_t& p, const AttnArgs& a, const int32_t* distribution,
                    int num_sms, cudaStream_t s, void* const* events) {
  const WorkspaceLayout L(p);
  const PrefillKind kind = prefill_kind(p);
  auto mark = [&](int i) -> bool {
    return !events || cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
  };
  if (!mark(0)) return RPA_ERR_CUDA;
  if (launch_plan(p, a.kv_lens, a.qsl, distribution, a.kv.ws, prefill_rows_for(p), s) !=
      cudaSuccess)
    return RPA_ERR_CUDA;
  // e4m3 cache, tcgen05 prefills: they read the step's new tokens from their
  // pages, written here once (timed with the planner)
  if (kind != kPrefillMma && p.kv_dtype == RPA_KV_FP8_E4M3 &&
      launch_prefill_pages(a.kv, a.kv_lens, a.qsl, distribution, num_sms, s) != cudaSuccess)
    return RPA_ERR_CUDA;
  if (!mark(1)) return RPA_ERR_CUDA;
  if (launch_decode(a, (int)L.max_decode_units, num_sms, s) != cudaSuccess) return RPA_ERR_CUDA;
  if (!mark(2)) return RPA_ERR_CUDA;
  const int mu = (int)L.max_prefill_units;
  const cudaError_t e = kind == kPrefillTc       ? launch_prefill_tc(a, mu, num_sms, s)
                        : kind == kPrefillTcWide ? launch_prefill_tc_wide(a, mu, num_sms, s)
                                                 : launch_prefill(a, mu, num_sms, s);
  if (e != cudaSuccess) return RPA_ERR_CUDA;
  if (!mark(3)) return RPA_ERR_CUDA;
  return RPA_OK;
}
}  // namespace rpa

static int forward_impl(const rpa_params_t* params, const void* queries, const void* keys,
                        const void* values, void* kv_cache, const int32_t* kv_lens,
                        const int32_t* block_tables, const int32_t* query_start_loc,
                        const int32_t* distribution, const float* attention_sink, void* out,
                        void* workspace, size_t workspace_bytes, void* stream,
                        void* const* events) {
  int rc = check_params(params);
  if (rc) return rc;
  if (!queries || !keys || !values || !kv_cache || !kv_lens || !block_tables ||
      !query_start_loc || !distribution || !out)
    return RPA_ERR_INVALID_ARG;
  if (!pointers_aligned(queries, keys, values, kv_cache, out, kv_lens, block_tables,
                        query_start_loc, distribution, attention_sink))
    return RPA_ERR_INVALID_ARG;
  rc = check_ws(params, workspace, workspace_bytes);
  if (rc) return rc;
  const int sms = num_sms_current();
  if (sms <= 0) return RPA_ERR_CUDA;
  AttnArgs a{{*params, reinterpret_cast<const __nv_bfloat16*>(keys),
              reinterpret_cast<const __nv_bfloat16*>(values), reinterpret_cast<uint8_t*>(kv_cache),
              block_tables, reinterpret_cast<int32_t*>(workspace)},
             reinterpret_cast<const __nv_bfloat16*>(queries),
             kv_lens,
             query_start_loc,
             attention_sink,
             reinterpret_cast<__nv_bfloat16*>(out)};
  return enqueue_forward(*params, a, distribution, sms, reinterpret_cast<cudaStream_t>(stream),
                         events);
}

extern "C" {

int rpa_workspace_size(const rpa_params_t* params, size_t* bytes) {
  const int rc = check_params(params);
  if (rc) return rc;
  if (!bytes) return RPA_ERR_INVALID_ARG;
  *bytes = WorkspaceLayout(*params).total;
  return RPA_OK;
}

int rpa_update_cache(const rpa_params_t* params, const void* keys, const void* values,
                     void* kv_cache, const int32_t* kv_lens, const int32_t* block_tables,
                     const int32_t* query_start_loc, const int32_t* distribution,
                     void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_params(params);
  if (rc) return rc;
  if (!keys || !values || !kv_cache || !kv_lens || !block_tables || !query_start_loc ||
      !distribution)
    return RPA_ERR_INVALID_ARG;
  if (!pointers_aligned(nullptr, keys, values, kv_cache, nullptr, kv_lens, block_tables,
                        query_start_loc, distribution, nullptr))
    return RPA_ERR_INVALID_ARG;
  rc = check_ws(params, workspace, workspace_bytes);
  if (rc) return rc;
  const int sms = num_sms_current();
  if (sms <= 0) return RPA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* ws = reinterpret_cast<int32_t*>(workspace);
  if (launch_plan(*params, kv_lens, query_start_loc, distribution, ws, kPrefillRows, s) !=
      cudaSuccess)
    return RPA_ERR_CUDA;
  KvArgs a{*params, reinterpret_cast<const __nv_bfloat16*>(keys),
           reinterpret_cast<const __nv_bfloat16*>(values), reinterpret_cast<uint8_t*>(kv_cache),
           block_tables, ws};
  if (launch_cache_write(a, kv_lens, query_start_loc, kPrefillRows, sms, s) != cudaSuccess)
    return RPA_ERR_CUDA;
  return RPA_OK;
}

int rpa_forward(const rpa_params_t* params, const void* queries, const void* keys,
                const void* values, void* kv_cache, const int32_t* kv_lens,
                const int32_t* block_tables, const int32_t* query_start_loc,
                const int32_t* distribution, const float* attention_sink, void* out,
                void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(params, queries, keys, values, kv_cache, kv_lens, block_tables,
                      query_start_loc, distribution, attention_sink, out, workspace,
                      workspace_bytes, stream, nullptr);
}

int rpa_forward_timed(const rpa_params_t* params, const void* queries, const void* keys,
                      const void* values, void* kv_cache, const int32_t* kv_lens,
                      const int32_t* block_tables, const int32_t* query_start_loc,
                      const int32_t* distribution, const float* attention_sink, void* out,
                      void* workspace, size_t workspace_bytes, void* stream,
                      void* const* events) {
  if (!events) return RPA_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i)
    if (!events[i]) return RPA_ERR_INVALID_ARG;
  return forward_impl(params, queries, keys, values, kv_cache, kv_lens, block_tables,
                      query_start_loc, distribution, attention_sink, out, workspace,
                      workspace_bytes, stream, events);
}

int rpa_get_status(const void* workspace, void* stream, int32_t* device_status) {
  if (!workspace || !device_status) return RPA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(device_status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return RPA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RPA_ERR_CUDA;
  return RPA_OK;
}

const char* rpa_status_string(int code) {
  switch (code) {
    case RPA_OK: return "ok";
    case RPA_ERR_INVALID_ARG: return "invalid argument";
    case RPA_ERR_UNSUPPORTED: return "unsupported configuration";
    case RPA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case RPA_ERR_CUDA: return "CUDA runtime error";
    case RPA_ERR_NOALLOC_TOO_LARGE:
      return "params need more scratch than rpa_forward_noalloc's fixed device array";
    default: return "unknown code";
  }
}

}  // extern "C"
