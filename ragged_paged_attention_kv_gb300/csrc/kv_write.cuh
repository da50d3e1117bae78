// New-KV page write shared by the standalone cache update and the fused
// attention kernels (tpu-inference RPA v3 kernel.py, _update_kv_cache: the
// step's keys/values land at positions ctx .. kv_len-1 of their sequence).
#pragma once

#include "common.cuh"

namespace rpa {

struct KvArgs {
  rpa_params_t p;
  const __nv_bfloat16* keys;    // [T, Hkv, D]
  const __nv_bfloat16* values;  // [T, Hkv, D]
  uint8_t* cache;               // [num_pages, P, 2*Hkv, D] (bf16 or e4m3 bytes)
  const int32_t* block_tables;  // [max_num_seqs * pages_per_seq]
  int32_t* ws;                  // workspace header
};

// Scales of kv head h: the per-head arrays when given, else the scalars.
__device__ __forceinline__ float k_scale_of(const rpa_params_t& p, int h) {
  return p.k_scale_heads ? __ldg(p.k_scale_heads + h) : p.k_scale;
}
__device__ __forceinline__ float v_scale_of(const rpa_params_t& p, int h) {
  return p.v_scale_heads ? __ldg(p.v_scale_heads + h) : p.v_scale;
}

// Physical page of logical position `pos` of sequence `seq`, or -1 (and the
// BAD_PAGE status bit) if the table entry lies outside the pool.
__device__ __forceinline__ int32_t lookup_page(const KvArgs& a, int seq, int pos) {
  const int32_t page =
      __ldg(a.block_tables + (int64_t)seq * a.p.pages_per_seq + (pos / a.p.page_size));
  if (page < 0 || page >= a.p.num_pages) {
    set_status(a.ws, RPA_STATUS_BAD_PAGE);
    return -1;
  }
  return page;
}

// Byte offset of (page, row, channel) in the pool.
__device__ __forceinline__ int64_t pool_offset(const rpa_params_t& p, int64_t page, int row,
                                               int channel, int elem_bytes) {
  return ((page * p.page_size + row) * (2 * (int64_t)p.num_kv_heads) + channel) *
         (int64_t)p.head_dim * elem_bytes;
}

// One warp writes key and value head `h` of input token `t` (sequence `seq`,
// position `pos`) into the pool: a bf16 copy or fp8 quantisation x / scale.
template <bool FP8>
__device__ __forceinline__ void write_token_kv(const KvArgs& a, int seq, int t, int pos, int h,
                                               int lane) {
  const int D = a.p.head_dim;
  const int chunks = D / 8;  // 16-byte chunks of one bf16 input row
  const int32_t page = lookup_page(a, seq, pos);
  if (page < 0) return;
  const int64_t src = ((int64_t)t * a.p.num_kv_heads + h) * D;
  const int64_t dst = pool_offset(a.p, page, pos % a.p.page_size, 2 * h, FP8 ? 1 : 2);
  for (int i = lane; i < 2 * chunks; i += 32) {
    const int kv = i / chunks, c = i % chunks;
    const __nv_bfloat16* in = (kv ? a.values : a.keys) + src + c * 8;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(in));
    if (FP8) {
      const float scale = kv ? v_scale_of(a.p, h) : k_scale_of(a.p, h);
      *reinterpret_cast<uint2*>(a.cache + dst + (int64_t)kv * D + c * 8) = quantize8(x, scale);
    } else {
      *reinterpret_cast<uint4*>(a.cache + dst + ((int64_t)kv * D + c * 8) * 2) = x;
    }
  }
}

// The same write for one token split into its two halves, so that a caller
// can issue the page-id and input loads early and store later: lane l holds
// 16-byte chunks l, l + 32, ... of the token's key row followed by its value
// row (one chunk per lane up to head_dim 128, two at 256).  Nothing reads
// the loaded values before token_kv_store, so the loads do not stall the
// caller in between.
template <int D>
struct TokenKv {
  static constexpr int kChunks = D / 8;                   // 16-byte chunks of one row
  static constexpr int kPerLane = (2 * kChunks + 31) / 32;  // chunks held by each lane
  int32_t page;        // block-table entry of the token's slot
  uint4 x[kPerLane];   // the chunks' bf16 inputs
};
template <bool FP8, int D>
__device__ __forceinline__ TokenKv<D> token_kv_load(const KvArgs& a, int seq, int t, int pos,
                                                    int h, int lane) {
  using T = TokenKv<D>;
  T r;
  r.page = __ldg(a.block_tables + (int64_t)seq * a.p.pages_per_seq + pos / a.p.page_size);
#pragma unroll
  for (int j = 0; j < T::kPerLane; ++j) {
    const int i = lane + 32 * j;
    r.x[j] = make_uint4(0, 0, 0, 0);
    if (i < 2 * T::kChunks) {
      const int kv = i / T::kChunks, c = i % T::kChunks;
      r.x[j] = __ldg(reinterpret_cast<const uint4*>(
          (kv ? a.values : a.keys) + ((int64_t)t * a.p.num_kv_heads + h) * D + c * 8));
    }
  }
  return r;
}
template <bool FP8, int D>
__device__ __forceinline__ void token_kv_store(const KvArgs& a, const TokenKv<D>& r, int pos,
                                               int h, int lane) {
  using T = TokenKv<D>;
  if (lane >= 2 * T::kChunks) return;
  if (r.page < 0 || r.page >= a.p.num_pages) {
    set_status(a.ws, RPA_STATUS_BAD_PAGE);
    return;
  }
#pragma unroll
  for (int j = 0; j < T::kPerLane; ++j) {
    const int i = lane + 32 * j;
    if (i >= 2 * T::kChunks) continue;
    const int kv = i / T::kChunks, c = i % T::kChunks;
    const int64_t dst = pool_offset(a.p, r.page, pos % a.p.page_size, 2 * h + kv, FP8 ? 1 : 2);
    if (FP8)
      *reinterpret_cast<uint2*>(a.cache + dst + c * 8) =
          quantize8(r.x[j], kv ? v_scale_of(a.p, h) : k_scale_of(a.p, h));
    else
      *reinterpret_cast<uint4*>(a.cache + dst + c * 16) = r.x[j];
  }
}

// One warp writes key and value head `h` of the n consecutive input tokens
// t0 .. t0+n-1 (positions pos0 .. pos0+n-1 of sequence `seq`) into the pool.
// Lanes take consecutive 16-byte chunks (a token's key row, then its value
// row), and each lane issues the block-table and input loads of kBatch
// chunks before any of their stores, so the loads' latencies overlap.
template <bool FP8, int D, int kBatch>
__device__ __forceinline__ void write_tokens_kv(const KvArgs& a, int seq, int t0, int pos0, int n,
                                                int h, int lane) {
  constexpr int kChunks = D / 8;       // 16-byte chunks of one bf16 row
  constexpr int kItems = 2 * kChunks;  // key and value chunks of one token
  const int total = n * kItems;
  const int32_t* bt = a.block_tables + (int64_t)seq * a.p.pages_per_seq;
  for (int base = 0; base < total; base += 32 * kBatch) {
    uint4 x[kBatch];
    int32_t page[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int idx = base + 32 * b + lane;
      if (idx < total) {
        const int i = idx / kItems, kv = (idx % kItems) / kChunks, c = idx % kChunks;
        page[b] = __ldg(bt + (pos0 + i) / a.p.page_size);
        x[b] = __ldg(reinterpret_cast<const uint4*>(
            (kv ? a.values : a.keys) + ((int64_t)(t0 + i) * a.p.num_kv_heads + h) * D + c * 8));
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int idx = base + 32 * b + lane;
      if (idx >= total) continue;
      if (page[b] < 0 || page[b] >= a.p.num_pages) {
        set_status(a.ws, RPA_STATUS_BAD_PAGE);
        continue;
      }
      const int i = idx / kItems, kv = (idx % kItems) / kChunks, c = idx % kChunks;
      const int pos = pos0 + i;
      const int64_t dst = pool_offset(a.p, page[b], pos % a.p.page_size, 2 * h + kv, FP8 ? 1 : 2);
      if (FP8) {
        *reinterpret_cast<uint2*>(a.cache + dst + c * 8) =
            quantize8(x[b], kv ? v_scale_of(a.p, h) : k_scale_of(a.p, h));
      } else {
        *reinterpret_cast<uint4*>(a.cache + dst + c * 16) = x[b];
      }
    }
  }
}

// Arguments of the attention kernels.
struct AttnArgs {
  KvArgs kv;
  const __nv_bfloat16* queries;  // [T, Hq, D]
  const int32_t* kv_lens;        // [max_num_seqs]
  const int32_t* qsl;            // [max_num_seqs + 1]
  const float* sink;             // [Hq] or null
  __nv_bfloat16* out;            // [T, Hq, D]
};

}  // namespace rpa
