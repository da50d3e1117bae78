// Planner, the page write ahead of the prefill (e4m3 caches), and the
// standalone page write.
//
// The planner reads the ragged metadata on the device (no host round trip),
// checks it, and splits the batch into work units by class: sequences of the
// decode-only class (distribution[0]) become (sequence, kv head, key split)
// units with one new token each; the chunked-prefill and mixed classes become
// (sequence, tile of new tokens, kv head) units.  The ejkernel
// ragged_page_attention_v3 interface's `distribution` argument defines the
// classes; results never depend on it (a decode-class sequence with
// q_len != 1 is flagged and planned as a prefill).  It also decides whether
// the decode kernel leaves part of the SMs to the prefill kernel.
#include <cfloat>

#include "common.cuh"
#include "kv_write.cuh"
#include "launch.h"
#include "tma_host.h"

namespace rpa {

constexpr int kSizeClasses = 16;  // decode sequences are ordered by these, longest first

// A batch with both kinds of work runs its decode units on part of the SMs
// (the decode kernel's CTAs on the other SMs leave at once) and the prefill
// kernel's CTAs, launched behind it and waiting for no part of it, on the
// rest from the start: the decode stays HBM-bound on fewer SMs (measured on
// GB300: 80 of the 152 SMs keep about 70 % of its bandwidth) while the prefill
// is bound by the tensor cores.  Only worth it when the prefill is big enough
// to keep the freed SMs busy: at least kShareFlopsPerByte prefill flops per
// byte of keys / values the decode reads (the chunked-prefill mixed batch has
// about 140, the fp8 windowed batch about 60; a small chunk beside a decode
// batch well under 1).
constexpr double kShareFlopsPerByte = 32.0;

// Block-wide exclusive scan of two ints per thread (one set of barriers for
// both); returns the prefixes and writes the block totals to *total.  All
// threads of the block must call it.
__device__ int2 block_exclusive_scan2(int2 v, int2* total, int2* smem /* 33 int2 */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int2 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yx = __shfl_up_sync(0xffffffffu, x.x, o), yy = __shfl_up_sync(0xffffffffu, x.y, o);
    if (lane >= o) {
      x.x += yx;
      x.y += yy;
    }
  }
  if (lane == 31) smem[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int2 w = lane < (int)(blockDim.x >> 5) ? smem[lane] : make_int2(0, 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yx = __shfl_up_sync(0xffffffffu, w.x, o), yy = __shfl_up_sync(0xffffffffu, w.y, o);
      if (lane >= o) {
        w.x += yx;
        w.y += yy;
      }
    }
    smem[lane] = w;  // inclusive prefix over warps
    if (lane == 31) smem[32] = w;
  }
  __syncthreads();
  const int2 before = warp > 0 ? smem[warp - 1] : make_int2(0, 0);
  const int2 excl = make_int2(x.x - v.x + before.x, x.y - v.y + before.y);
  *total = smem[32];
  __syncthreads();
  return excl;
}

// Largest i < n with off[i] <= x (off is nondecreasing, off[0] == 0 <= x).
__device__ __forceinline__ int last_at_or_below(const int* off, int n, int x) {
  int lo = 0, hi = n;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

struct SeqPlan {
  int cls;        // 0 none, 1 decode, 2 prefill
  int q0, q_len, kv_len, lo;
  int flags;      // RPA_STATUS_* bits raised by this sequence
};

// Sequence s's metadata: query_start_loc[s], [s + 1] and kv_lens[s].
struct SeqMeta {
  int a, b, kv;
};
__device__ __forceinline__ SeqMeta load_meta(int s, const int32_t* kv_lens, const int32_t* qsl) {
  return SeqMeta{__ldg(qsl + s), __ldg(qsl + s + 1), __ldg(kv_lens + s)};
}

__device__ SeqPlan classify(const rpa_params_t& p, int s, int d0, const SeqMeta& m) {
  SeqPlan sp{0, 0, 0, 0, 0, 0};
  const int a = m.a, b = m.b;
  const int kv = m.kv;
  if (a < 0 || b < a || b > p.total_tokens) {
    sp.flags = RPA_STATUS_BAD_QUERY_START_LOC;
    return sp;
  }
  const int q_len = b - a;
  if (kv < q_len || (int64_t)kv > (int64_t)p.pages_per_seq * p.page_size) {
    sp.flags = RPA_STATUS_BAD_KV_LEN;
    return sp;
  }
  sp.q0 = a;
  sp.q_len = q_len;
  sp.kv_len = kv;
  if (q_len == 0) return sp;
  bool decode = s < d0;
  if (decode && q_len != 1) {
    sp.flags = RPA_STATUS_DECODE_QLEN;
    decode = false;
  }
  sp.cls = decode ? 1 : 2;
  sp.lo = (p.sliding_window > 0 && kv - p.sliding_window > 0) ? kv - p.sliding_window : 0;
  return sp;
}

// kT threads (256 or 1024) handle the sequences in batches of kT; fewer
// threads make the block's barriers cheaper when the batch is small.
template <int kT>
__global__ void __launch_bounds__(kT) plan_kernel(rpa_params_t p, const int32_t* kv_lens,
                                                            const int32_t* qsl,
                                                            const int32_t* dist, int32_t* ws,
                                                            int prefill_rows) {
  __shared__ int s_flags;
  __shared__ int2 s_scan[33];
  __shared__ unsigned long long s_keys, s_pairs;
  constexpr int kWarps = kT / 32;
  static_assert((kSizeClasses + 1) * kWarps <= kT, "one scan covers the class counts");
  __shared__ int s_doff[kT], s_poff[kT], s_nsplit[kT], s_ntiles[kT], s_lo[kT], s_len[kT],
      s_q0[kT], s_seq[kT], s_wbase[kT];
  __shared__ int s_maxkey;
  const WorkspaceLayout L(p);
  DecodeUnit* dunits = reinterpret_cast<DecodeUnit*>(reinterpret_cast<char*>(ws) + L.decode_units_off);
  PrefillUnit* punits =
      reinterpret_cast<PrefillUnit*>(reinterpret_cast<char*>(ws) + L.prefill_units_off);
  int32_t* counters = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) + L.counters_off);
  const int tid = threadIdx.x;
  const int Hkv = p.num_kv_heads, G = p.num_q_heads / p.num_kv_heads;
  const int tile_tokens = prefill_rows / G;  // new tokens per prefill tile
  // the attention kernels launched behind this one may start their launch
  // now; they wait for this grid to complete before reading its output
  griddep_launch_dependents();

  // the first batch's metadata is loaded together with the distribution
  // (every index below max_num_seqs is inside the arrays)
  SeqMeta meta0{0, 0, 0};
  if (tid < p.max_num_seqs) meta0 = load_meta(tid, kv_lens, qsl);
  const int d0 = __ldg(dist), d1 = __ldg(dist + 1), d2 = __ldg(dist + 2);
  if (tid == 0) {
    s_flags = 0;
    s_keys = 0ull;
    s_pairs = 0ull;
    s_maxkey = 0;
  }
  __syncthreads();
  int S = d2;
  if (!(0 <= d0 && d0 <= d1 && d1 <= d2 && d2 <= p.max_num_seqs)) {
    if (tid == 0) atomicOr(&s_flags, RPA_STATUS_BAD_DISTRIBUTION);
    S = 0;
  }
  if (tid == 0 && S > 0 && meta0.a != 0) atomicOr(&s_flags, RPA_STATUS_BAD_QUERY_START_LOC);
  // per-head scales must be finite and positive
  if (p.k_scale_heads || p.v_scale_heads) {
    for (int h = tid; h < Hkv; h += kT) {
      const float ks = p.k_scale_heads ? __ldg(p.k_scale_heads + h) : 1.f;
      const float vs = p.v_scale_heads ? __ldg(p.v_scale_heads + h) : 1.f;
      if (!(ks > 0.f && ks <= FLT_MAX && vs > 0.f && vs <= FLT_MAX))
        atomicOr(&s_flags, RPA_STATUS_BAD_SCALE);
    }
  }

  // Pass 1: total decode keys (per kv head) to size the splits.
  // ... and the prefill's (query token, visible key) pairs, for the SM share
  unsigned long long my_keys = 0, my_pairs = 0;
  int my_max = 0;
  for (int s = tid; s < S; s += kT) {
    SeqPlan sp = classify(p, s, d0, s == tid ? meta0 : load_meta(s, kv_lens, qsl));
    if (sp.flags) atomicOr(&s_flags, sp.flags);
    if (sp.cls == 1) {
      my_keys += (unsigned long long)(sp.kv_len - sp.lo);
      my_max = max(my_max, sp.kv_len - sp.lo);
    }
    if (sp.cls == 2) {
      // token i sees min(ctx + i + 1, W) keys: sum over k = a .. b of min(k, W)
      const unsigned long long a = (unsigned long long)(sp.kv_len - sp.q_len) + 1, b = sp.kv_len;
      const unsigned long long w = p.sliding_window > 0 ? (unsigned long long)p.sliding_window : b;
      if (w >= b)
        my_pairs += (a + b) * (b - a + 1) / 2;
      else if (w < a)
        my_pairs += (b - a + 1) * w;
      else
        my_pairs += (a + w) * (w - a + 1) / 2 + (b - w) * w;
    }
  }
  my_max = __reduce_max_sync(0xffffffffu, my_max);
  if ((tid & 31) == 0 && my_max) atomicMax(&s_maxkey, my_max);
  // warp sums first: one shared atomic per warp, not per thread
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    my_keys += __shfl_xor_sync(0xffffffffu, my_keys, o);
    my_pairs += __shfl_xor_sync(0xffffffffu, my_pairs, o);
  }
  if ((tid & 31) == 0 && my_keys) atomicAdd(&s_keys, my_keys);
  if ((tid & 31) == 0 && my_pairs) atomicAdd(&s_pairs, my_pairs);
  __syncthreads();
  const unsigned long long want =
      (s_keys * (unsigned long long)Hkv + kDecodeUnitsTarget - 1) / kDecodeUnitsTarget;
  // splits are whole 64-key stages of the decode kernel
  int chunk = (int)((want + 63) / 64 * 64);
  if (chunk < kDecodeChunkMin) chunk = kDecodeChunkMin;

  // Pass 2, per batch of kT sequences: scan the unit counts, then
  // emit the units cooperatively (one thread per unit, coalesced stores).
  // Prefill units are ordered head-major, each head's tiles last-first, so the
  // CTAs running at the same time share one head's keys in L2 and the longest
  // causal tiles start first under the dynamic scheduler.
  int dec_base = 0, pf_base = 0;
  for (int base = 0; base < S; base += kT) {
    const int s = base + tid;
    SeqPlan sp{0, 0, 0, 0, 0, 0};
    int nsplit = 0, ntiles = 0;
    if (s < S) {
      // flags were taken in pass 1
      sp = classify(p, s, d0, s == tid ? meta0 : load_meta(s, kv_lens, qsl));
      if (sp.cls == 1) nsplit = (sp.kv_len - (sp.lo & ~63) + chunk - 1) / chunk;
      if (sp.cls == 2) ntiles = (sp.q_len + tile_tokens - 1) / tile_tokens;
    }
    s_nsplit[tid] = nsplit;
    s_ntiles[tid] = ntiles;
    s_lo[tid] = sp.lo;
    s_len[tid] = sp.cls == 1 ? sp.kv_len : sp.q_len;
    s_q0[tid] = sp.q0;
    // Decode sequences are ranked longest first (16 size classes of the
    // keys they read, the sequence index inside a class; the other
    // sequences last), so the dynamic scheduler hands out the longest decode
    // units first and the kernel's tail is made of short ones.  Counting
    // sort: rank = base of (class, warp) + rank among the warp's lanes of
    // the same class.
    {
      const int kb = sp.cls == 1 ? (int)((int64_t)(s_maxkey - (sp.kv_len - sp.lo)) * kSizeClasses /
                                         ((int64_t)s_maxkey + 1))
                                 : kSizeClasses;
      const unsigned same = __match_any_sync(0xffffffffu, kb);
      const int lane = tid & 31, warp = tid >> 5;
      s_wbase[tid] = 0;
      __syncthreads();
      if (lane == __ffs(same) - 1) s_wbase[kb * kWarps + warp] = __popc(same);
      __syncthreads();
      // (class, warp) counts in class-major order -> exclusive bases
      int2 cb_total;
      const int2 cb = block_exclusive_scan2(make_int2(s_wbase[tid], 0), &cb_total, s_scan);
      __syncthreads();
      s_wbase[tid] = cb.x;
      __syncthreads();
      s_seq[s_wbase[kb * kWarps + warp] + __popc(same & ((1u << lane) - 1u))] = tid;
    }
    __syncthreads();
    const int si = s_seq[tid];  // sequence at rank tid
    int2 totals;
    const int2 offs = block_exclusive_scan2(make_int2(s_nsplit[si] * Hkv, ntiles * Hkv), &totals, s_scan);
    const int dec_off = offs.x, pf_off = offs.y, dec_total = totals.x, pf_total = totals.y;
    s_doff[tid] = dec_off;  // by rank
    s_poff[tid] = pf_off;   // by sequence
    __syncthreads();
    for (int u = tid; u < dec_total; u += kT) {
      const int ri = last_at_or_below(s_doff, kT, u);
      const int i = s_seq[ri];
      const int ns = s_nsplit[i], r = u - s_doff[ri];
      const int h = r / ns, k = r % ns;
      const int lo = s_lo[i], kv = s_len[i];
      const int stage0 = lo & ~63;  // split boundaries on 64-key stages
      DecodeUnit du;
      du.seq = base + i;
      du.head = h;
      du.k_begin = max(lo, stage0 + k * chunk);
      du.k_end = min(kv, stage0 + (k + 1) * chunk);
      du.split = k;
      du.nsplit = ns;
      du.q0 = s_q0[i];
      du.kv_len = kv;
      dunits[dec_base + u] = du;
      if (k == 0) counters[(int64_t)(base + i) * Hkv + h] = 0;
    }
    for (int u = tid; u < pf_total; u += kT) {
      const int i = last_at_or_below(s_poff, kT, u);
      const int nt = s_ntiles[i], r = u - s_poff[i];
      const int h = r / nt, t = nt - 1 - r % nt;
      PrefillUnit pu;
      pu.seq = base + i;
      pu.t_begin = t * tile_tokens;
      pu.t_end = min(s_len[i], (t + 1) * tile_tokens);
      pu.head = h;
      punits[pf_base + u] = pu;
    }
    dec_base += dec_total;
    pf_base += pf_total;
    __syncthreads();  // the per-sequence arrays are rewritten by the next batch
  }
  __syncthreads();
  if (tid == 0) {
    ws[kHdrStatus] = s_flags;
    ws[kHdrNumDecode] = dec_base;
    ws[kHdrNumPrefill] = pf_base;
    ws[kHdrDecodeChunk] = chunk;
    ws[kHdrDecodeNext] = 0;
    ws[kHdrPrefillNext] = 0;
    const double dec_bytes = (double)s_keys * Hkv * 2.0 * p.head_dim *
                             (p.kv_dtype == RPA_KV_FP8_E4M3 ? 1.0 : 2.0);
    const double pf_flops = (double)s_pairs * 4.0 * p.head_dim * p.num_q_heads;
    ws[kHdrDecodeShare] =
        dec_base > 0 && pf_base > 0 && pf_flops >= kShareFlopsPerByte * dec_bytes ? 1 : 0;
  }
}

// Standalone page write: one warp per (token, kv head) of every planned unit.
template <bool FP8>
__global__ void __launch_bounds__(256) cache_write_kernel(KvArgs a, const int32_t* kv_lens,
                                                          const int32_t* qsl, int prefill_rows) {
  const WorkspaceLayout L(a.p);
  const DecodeUnit* dunits =
      reinterpret_cast<const DecodeUnit*>(reinterpret_cast<const char*>(a.ws) + L.decode_units_off);
  const PrefillUnit* punits =
      reinterpret_cast<const PrefillUnit*>(reinterpret_cast<const char*>(a.ws) + L.prefill_units_off);
  const int n_dec = a.ws[kHdrNumDecode], n_pf = a.ws[kHdrNumPrefill];
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  // decode units: split 0 of each (seq, head) writes the single new token
  for (int u = gw; u < n_dec; u += warps) {
    const DecodeUnit d = dunits[u];
    if (d.split != 0) continue;
    const int t = qsl[d.seq];
    write_token_kv<FP8>(a, d.seq, t, kv_lens[d.seq] - 1, d.head, lane);
  }
  // prefill units: every token of the tile for the unit's head
  const int tile_tokens = prefill_rows / (a.p.num_q_heads / a.p.num_kv_heads);
  const int64_t n_items = (int64_t)n_pf * tile_tokens;
  for (int64_t it = gw; it < n_items; it += warps) {
    const PrefillUnit pu = punits[it / tile_tokens];
    const int i = pu.t_begin + (int)(it % tile_tokens);
    if (i >= pu.t_end) continue;
    const int q0 = qsl[pu.seq];
    const int q_len = qsl[pu.seq + 1] - q0;
    const int ctx = kv_lens[pu.seq] - q_len;
    write_token_kv<FP8>(a, pu.seq, q0 + i, ctx + i, pu.head, lane);
  }
}

// ------------------------------------------------------------ host launch
cudaError_t launch_plan(const rpa_params_t& p, const int32_t* kv_lens, const int32_t* qsl,
                        const int32_t* dist, int32_t* ws, int prefill_rows, cudaStream_t stream) {
  if (p.max_num_seqs <= 256)
    plan_kernel<256><<<1, 256, 0, stream>>>(p, kv_lens, qsl, dist, ws, prefill_rows);
  else
    plan_kernel<1024><<<1, 1024, 0, stream>>>(p, kv_lens, qsl, dist, ws, prefill_rows);
  return cudaGetLastError();
}

// Page write ahead of the attention kernels (e4m3 cache, tcgen05 prefills:
// head_dim 64/128/192/256).  The new tokens of every sequence the planner gives to
// the prefill kernel -- the planner's own classification, on the same
// metadata -- are quantised into their pages once, so that kernel reads every
// key and value tile from the pool as codes and no unit quantises a tile of
// new tokens again.  It runs right behind the planner and overlaps it: it
// needs only the metadata, which it checks itself (invalid sequences and
// out-of-range page ids are skipped; the prefill kernel reads, checks and
// reports the same block-table entries when it loads those tiles).  It
// completes only after the planner, so the kernel waiting for it also finds
// the plan.  Each warp takes a contiguous run of tokens: it finds the
// sequence of its first token with a 32-way search of query_start_loc, then
// walks forward, and writes every kv head's key and value row of each token
// (one 16-byte chunk of bf16 inputs per lane and step, four steps in flight).
template <int D>
__global__ void __launch_bounds__(256) prefill_pages_kernel(KvArgs a, const int32_t* kv_lens,
                                                            const int32_t* qsl,
                                                            const int32_t* dist) {
  griddep_launch_dependents();  // the decode kernel waits for this grid itself
  const rpa_params_t& p = a.p;
  const int lane = threadIdx.x & 31;
  const int d0 = __ldg(dist), d1 = __ldg(dist + 1), d2 = __ldg(dist + 2);
  const int S = (0 <= d0 && d0 <= d1 && d1 <= d2 && d2 <= p.max_num_seqs) ? d2 : 0;
  const int T = p.total_tokens;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int per = (T + warps - 1) / warps;
  const int t0 = gw * per, t1 = min(T, t0 + per);
  if (S > 0 && t0 < t1) {
    // the last sequence s < S with query_start_loc[s] <= t0
    int lo = 0, hi = S;
    while (hi - lo > 1) {
      const int step = (hi - lo + 31) / 32;
      const int idx = lo + lane * step;
      const unsigned m = __ballot_sync(0xffffffffu, idx < hi && __ldg(qsl + idx) <= t0);
      lo += m ? (31 - __clz(m)) * step : 0;
      hi = min(hi, lo + step);
    }
    int s = lo;
    SeqPlan sp = classify(p, s, d0, load_meta(s, kv_lens, qsl));
    int a_s = __ldg(qsl + s), b_s = __ldg(qsl + s + 1);
    constexpr int kChunks = D / 8, kU = 4;
    const int Hkv = p.num_kv_heads;
    const int items = Hkv * 2 * kChunks;  // (head, key / value, chunk) of one token
    for (int t = t0; t < t1; ++t) {
      while (t >= b_s && s + 1 < S) {
        ++s;
        sp = classify(p, s, d0, load_meta(s, kv_lens, qsl));
        a_s = __ldg(qsl + s);
        b_s = __ldg(qsl + s + 1);
      }
      if (sp.cls != 2 || t < a_s || t >= b_s) continue;
      const int pos = sp.kv_len - sp.q_len + (t - sp.q0);
      const int page = __ldg(a.block_tables + (int64_t)s * p.pages_per_seq + pos / p.page_size);
      if (page < 0 || page >= p.num_pages) continue;
      const int row = pos % p.page_size;
      for (int i0 = 0; i0 < items; i0 += 32 * kU) {
        uint4 x[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int i = i0 + 32 * u + lane;
          if (i < items) {
            const int h = i / (2 * kChunks), kv = (i / kChunks) & 1, c = i % kChunks;
            x[u] = __ldg(reinterpret_cast<const uint4*>(
                (kv ? a.values : a.keys) + ((int64_t)t * Hkv + h) * D + c * 8));
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int i = i0 + 32 * u + lane;
          if (i < items) {
            const int h = i / (2 * kChunks), kv = (i / kChunks) & 1, c = i % kChunks;
            *reinterpret_cast<uint2*>(a.cache + pool_offset(p, page, row, 2 * h + kv, 1) + c * 8) =
                quantize8(x[u], kv ? v_scale_of(p, h) : k_scale_of(p, h));
          }
        }
      }
    }
  }
  griddep_wait();  // complete only after the planner
}

cudaError_t launch_prefill_pages(const KvArgs& a, const int32_t* kv_lens, const int32_t* qsl,
                                 const int32_t* dist, int num_sms, cudaStream_t stream) {
  const int T = a.p.total_tokens > 0 ? a.p.total_tokens : 1;
  int grid = (T + 7) / 8;  // at least one token per warp
  if (grid > 2 * num_sms) grid = 2 * num_sms;
  switch (a.p.head_dim) {
    case 64:
      return launch_dependent(prefill_pages_kernel<64>, grid, 256, 0, stream, a, kv_lens, qsl, dist);
    case 128:
      return launch_dependent(prefill_pages_kernel<128>, grid, 256, 0, stream, a, kv_lens, qsl,
                              dist);
    case 192:
      return launch_dependent(prefill_pages_kernel<192>, grid, 256, 0, stream, a, kv_lens, qsl,
                              dist);
    default:
      return launch_dependent(prefill_pages_kernel<256>, grid, 256, 0, stream, a, kv_lens, qsl,
                              dist);
  }
}

cudaError_t launch_cache_write(const KvArgs& a, const int32_t* kv_lens, const int32_t* qsl,
                               int prefill_rows, int num_sms, cudaStream_t stream) {
  const int grid = num_sms * 4;
  if (a.p.kv_dtype == RPA_KV_FP8_E4M3)
    cache_write_kernel<true><<<grid, 256, 0, stream>>>(a, kv_lens, qsl, prefill_rows);
  else
    cache_write_kernel<false><<<grid, 256, 0, stream>>>(a, kv_lens, qsl, prefill_rows);
  return cudaGetLastError();
}

}  // namespace rpa
