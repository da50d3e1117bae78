/*
 * rpa.h -- C ABI of the GB300 ragged paged attention library (librpa.so).
 *
 * One call attends a batch that mixes decode steps and (chunked) prefills,
 * reading each sequence's keys/values from pages of an HBM pool and writing
 * the step's new keys/values into their pages in the same call.  The
 * arguments follow the ejkernel ragged_page_attention_v3 interface (queries /
 * keys / values concatenated over the batch, kv_cache, kv_lens,
 * block_tables, query_start_loc, a 3-entry distribution, optional
 * attention_sink, softmax_scale, sliding_window, logits_soft_cap, k_scale,
 * v_scale); the cache is updated in place instead of being returned.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers named as device arrays must be device memory of the current CUDA
 * device (or managed memory).  All computation is enqueued on `stream`
 * (a cudaStream_t passed as void*; NULL = the legacy default stream) and is
 * asynchronous: a call returns before the GPU work finishes, and no call
 * synchronises except rpa_get_status.  The caller owns every buffer; the
 * library allocates no device memory and keeps no per-call state.
 *
 * Shapes (T = params.total_tokens, Hq/Hkv = query/kv heads, D = head_dim,
 * P = page_size, all row-major, no padding):
 *   queries      [T, Hq, D]   bf16
 *   keys, values [T, Hkv, D]  bf16 (the step's new keys/values)
 *   kv_cache     [num_pages, P, 2*Hkv, D]  bf16 or fp8 e4m3 (raw bytes):
 *                channel 2h holds key head h, channel 2h+1 value head h
 *                (tpu-inference RPA v3 kernel.py: keys and values are
 *                packed together per kv head).
 *   kv_lens      [max_num_seqs] int32: tokens of each sequence INCLUDING
 *                the new ones (vLLM differential_flash_attn.py metadata:
 *                seq_len = context_len + query_len).
 *   block_tables [max_num_seqs * pages_per_seq] int32: logical page k of
 *                sequence s is physical page block_tables[s*pages_per_seq+k];
 *                entries past ceil(kv_len/P) are never read.
 *   query_start_loc [max_num_seqs + 1] int32: cumulative query lengths; the
 *                new tokens of sequence s are rows [qsl[s], qsl[s+1]).
 *   distribution [3] int32: cumulative ends (d0 <= d1 <= d2) of the
 *                decode-only, chunked-prefill and mixed classes; d2 is the
 *                number of sequences S.  It only selects tile shapes:
 *                results never depend on it.
 *   attention_sink [Hq] fp32 or NULL.
 *   out          [T, Hq, D] bf16; rows >= qsl[S] are left untouched.
 * Alignment: queries, keys, values, kv_cache and out start on 16 bytes (the
 * kernels move them with bulk and tensor copies); the int32 arrays and
 * attention_sink on 4 bytes.  A misaligned pointer is refused with
 * RPA_ERR_INVALID_ARG before anything is enqueued.
 *
 * Semantics (per sequence s, new token i, q-head hq, kv head h = hq/(Hq/Hkv);
 * k_scale and v_scale below are those of head h when per-head scales are
 * given):
 *   position p = kv_len - q_len + i; keys j with j <= p and, when
 *   sliding_window W > 0, p - j < W (vLLM's window_size = (W-1, 0));
 *   logit = softmax_scale * k_scale * (q . k_j), then cap*tanh(logit/cap) when
 *   logits_soft_cap > 0; the sink logit (if given) joins the normaliser with
 *   no value; out = sum_j softmax_j * v_scale * v_j.  fp8 caches hold
 *   e4m3 codes of x / scale (round to nearest even, saturating at +-448) and
 *   the new tokens are attended through exactly those codes (tpu-inference
 *   layers/vllm/attention.py: keys/values are quantised before the kernel).
 *   For bf16 caches k_scale and v_scale must be 1.
 *
 * Errors: a nonzero return means nothing was enqueued.  Problems that depend
 * on device data (a page id outside the pool, kv_len < q_len, a malformed
 * query_start_loc or distribution) cannot be seen on the host: the kernels
 * skip the affected sequence, leave its outputs and pages untouched, and set
 * a bit in the workspace's status word (read it with rpa_get_status).  No
 * kernel traps.
 */
#ifndef RPA_H_
#define RPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
#define RPA_OK 0
#define RPA_ERR_INVALID_ARG 1  /* null or misaligned pointer, negative size,
                                  bad scale, per-head scales or q_scale
                                  with a bf16 cache                        */
#define RPA_ERR_UNSUPPORTED 2  /* head_dim not 64/96/128/192/256, Hq/Hkv not in {1,2,4,8,16},
                                  page_size not a power of two in [1,1024],
                                  or an fp8 cache with head_dim 64/96 and
                                  page_size 1 */
#define RPA_ERR_WORKSPACE 3    /* workspace NULL, misaligned or too small   */
#define RPA_ERR_CUDA 4         /* a CUDA runtime call failed                */

/* Bits of the device status word (rpa_get_status). */
#define RPA_STATUS_BAD_PAGE 0x1          /* block_tables entry outside [0, num_pages) */
#define RPA_STATUS_BAD_KV_LEN 0x2        /* kv_len < q_len or kv_len > pages_per_seq*P */
#define RPA_STATUS_BAD_QUERY_START_LOC 0x4 /* qsl[0] != 0, decreasing, or qsl[S] > T */
#define RPA_STATUS_BAD_DISTRIBUTION 0x8  /* not 0 <= d0 <= d1 <= d2 <= max_num_seqs */
#define RPA_STATUS_DECODE_QLEN 0x10      /* a decode-class sequence with q_len != 1
                                            (informational: it is still computed) */
#define RPA_STATUS_TIMEOUT 0x20          /* a bounded device wait gave up */
#define RPA_STATUS_BAD_SCALE 0x40        /* a per-head scale not finite and > 0 */

typedef enum { RPA_KV_BF16 = 0, RPA_KV_FP8_E4M3 = 1 } rpa_kv_dtype_t;

typedef struct {
  int32_t num_q_heads;    /* Hq; Hq % Hkv == 0                              */
  int32_t num_kv_heads;   /* Hkv                                            */
  int32_t head_dim;       /* D: 64, 96, 128, 192 or 256                     */
  int32_t page_size;      /* P: power of two, 1..1024                       */
  int32_t num_pages;      /* pages in the pool                              */
  int32_t pages_per_seq;  /* row length of block_tables                     */
  int32_t max_num_seqs;   /* length of kv_lens; query_start_loc has one more */
  int32_t total_tokens;   /* T: rows of queries/keys/values/out             */
  int32_t kv_dtype;       /* rpa_kv_dtype_t                                 */
  int32_t sliding_window; /* W > 0 keeps p - j < W; 0 = no window           */
  float softmax_scale;    /* > 0; applied to q.k as given                   */
  float logits_soft_cap;  /* > 0 enables cap*tanh(x/cap); 0 = none          */
  float k_scale;          /* fp8: dequantisation scales; bf16: must be 1    */
  float v_scale;
  /* Optional per-kv-head scales (fp8 caches only), device arrays of
   * num_kv_heads fp32, 4-byte aligned, read by the kernels: when non-NULL,
   * k_scale_heads[h] (v_scale_heads[h]) replaces k_scale (v_scale) for kv
   * head h in the quantisation of the new keys (values), in the logits and
   * in the output.  Each must be finite and > 0: otherwise the call sets
   * RPA_STATUS_BAD_SCALE and that head's outputs and pages are unspecified.
   * NULL for bf16 caches.  (vLLM's fp8 caches use one scale per layer; one
   * per kv head is the finer variant.) */
  const float* k_scale_heads;
  const float* v_scale_heads;
  /* fp8 caches only, optional (w8a8 attention; the ejkernel
   * ragged_page_attention_v3 interface's q_scale): when > 0, every query
   * element is quantised exactly as the keys are -- x / q_scale in fp32,
   * e4m3 with round to nearest even, saturating at +-448 -- and the scores
   * are formed from the codes: logit = softmax_scale * q_scale * k_scale *
   * (q_codes . k_codes).  0 = the queries are used as given (bf16).  Must be
   * finite and >= 0; > 0 with a bf16 cache is refused (RPA_ERR_INVALID_ARG). */
  float q_scale;
} rpa_params_t;

/* Bytes of device workspace rpa_forward / rpa_update_cache need for these
 * params (an upper bound over all metadata the params allow).  The workspace
 * must be 256-byte aligned; its contents need no initialisation and are
 * overwritten by every call (one workspace per stream in flight). */
int rpa_workspace_size(const rpa_params_t* params, size_t* bytes);

/* The page write alone: stores keys/values of the first distribution[2]
 * sequences' new tokens into their pages (bf16 copy, or fp8 quantisation
 * x / scale).  tpu-inference RPA v3 kernel.py _update_kv_cache; vLLM's
 * reshape_and_cache_flash is the same operation.  Every other byte of
 * kv_cache is left untouched. */
int rpa_update_cache(const rpa_params_t* params, const void* keys,
                     const void* values, void* kv_cache,
                     const int32_t* kv_lens, const int32_t* block_tables,
                     const int32_t* query_start_loc,
                     const int32_t* distribution, void* workspace,
                     size_t workspace_bytes, void* stream);

/* The whole step: page write of the new keys/values fused with ragged paged
 * attention for every new token of the first distribution[2] sequences.
 * tpu-inference RPA v3 kernel.py (_ragged_paged_attention_kernel) and the
 * ejkernel ragged_page_attention_v3 interface define the operation. */
int rpa_forward(const rpa_params_t* params, const void* queries,
                const void* keys, const void* values, void* kv_cache,
                const int32_t* kv_lens, const int32_t* block_tables,
                const int32_t* query_start_loc, const int32_t* distribution,
                const float* attention_sink, void* out, void* workspace,
                size_t workspace_bytes, void* stream);

/* rpa_forward that also records four caller-created CUDA events (cudaEvent_t,
 * passed as void*) on `stream`: events[0] before the planner, [1] after the
 * planner, [2] after the decode kernel, [3] after the prefill kernel, so a
 * caller can time each kernel on the stream it runs on.  The computation is
 * exactly rpa_forward's.  No page has a counterpart: this is instrumentation. */
int rpa_forward_timed(const rpa_params_t* params, const void* queries,
                      const void* keys, const void* values, void* kv_cache,
                      const int32_t* kv_lens, const int32_t* block_tables,
                      const int32_t* query_start_loc,
                      const int32_t* distribution, const float* attention_sink,
                      void* out, void* workspace, size_t workspace_bytes,
                      void* stream, void* const* events);

/* rpa_forward for callers that cannot allocate device memory.  The pages
 * describe no such call; it exists for code that has no way to obtain a
 * workspace: a caller running inside a memory-pool or allocator callback
 * (allocating there would re-enter the allocator), a plugin of a runtime that
 * owns every device allocation, or a deployment that forbids allocation
 * after start-up.
 *
 * Instead of a caller workspace it uses one fixed array of
 * RPA_NOALLOC_WORKSPACE_BYTES in device global memory, reserved when the
 * library's device code is loaded into a context and held there until the
 * context is destroyed (for the primary context of a device: process exit
 * or cudaDeviceReset), so every GPU that uses the library holds it.  The caller still passes all inputs and outputs, exactly as for
 * rpa_forward, and gets the same results.  The call allocates nothing and
 * calls no allocating routine.
 *
 * - Params whose workspace (rpa_workspace_size) exceeds the array are
 *   refused with RPA_ERR_NOALLOC_TOO_LARGE; nothing is enqueued.
 * - Every call looks up the array's device address in the current context
 *   (cudaGetSymbolAddress; each context has its own copy of the array, so
 *   the address is never cached).  The first call in a context may load the
 *   library's device code into it; make that first call before any stream
 *   capture.  Once loaded, the lookup allocates nothing.
 * - Every call in a context shares the one array and leaves its contents
 *   behind; the planner rewrites every word the kernels read, so nothing has
 *   to be cleared between calls.  Calls whose GPU work overlaps (on
 *   different streams, or different host threads without ordering) race on
 *   the array and give undefined results: serialise them.
 * - The device status word of these calls is not readable (there is no
 *   caller workspace to pass to rpa_get_status).  The problems it reports
 *   -- page ids outside the pool, inconsistent kv_lens / query_start_loc /
 *   distribution, bad per-head scales, a bounded device wait that gave up --
 *   therefore go unreported: callers of this entry point must check their
 *   metadata themselves, and a sequence the kernels skip keeps whatever its
 *   output rows held. */
#define RPA_NOALLOC_WORKSPACE_BYTES (32u << 20)
#define RPA_ERR_NOALLOC_TOO_LARGE 5
int rpa_forward_noalloc(const rpa_params_t* params, const void* queries,
                        const void* keys, const void* values, void* kv_cache,
                        const int32_t* kv_lens, const int32_t* block_tables,
                        const int32_t* query_start_loc,
                        const int32_t* distribution,
                        const float* attention_sink, void* out, void* stream);

/* Copies the status word of the last call that used `workspace` on `stream`
 * to *device_status (a host int32) and synchronises the stream.  0 = clean. */
int rpa_get_status(const void* workspace, void* stream, int32_t* device_status);

/* Static text for a return code (RPA_OK ... RPA_ERR_NOALLOC_TOO_LARGE). */
const char* rpa_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* RPA_H_ */
