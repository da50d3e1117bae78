// Decode path: one new token per sequence, HBM-bound.
//
// Work unit = (sequence, kv head, split of the key range).  The q-heads of the
// kv head (the GQA group, tpu-inference RPA v3 kernel.py stacks them as rows
// of one q block) form a 16-row tile, so every key/value byte fetched from a
// page feeds all of them through one tensor-core MMA.  Keys/values stream
// page by page from the pool into shared memory with 16-byte cp.async
// (3-stage pipeline of 64 keys); the new token's key/value is taken from the
// step's inputs, not from the cache (RPA v3 _fetch_bkv does the same), and
// split 0 of each (sequence, kv head) writes it into its page.  Each warp
// keeps an online-softmax state over its quarter of every stage (running max
// m, sum l, accumulator O as in RPA v3 flash_attention_step1_qk_softmax /
// step2_pv); the four warps merge in shared memory, and when a sequence's
// keys are split over several units, the unit that finishes last merges the
// partial (m, l, O) of all splits with a log-sum-exp combine.
#include "common.cuh"
#include "kv_write.cuh"

namespace rpa {

namespace dec {

constexpr int kThreads = 128;
constexpr int kWarps = 4;
constexpr int kBN = 64;       // keys per stage
constexpr int kStages = 3;
constexpr int kKeysPerWarp = kBN / kWarps;  // 16

template <int D, bool FP8>
struct Smem {
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;          // one key (or value) row in the stage
  static constexpr int kStageBytes = 2 * kBN * kRowBytes;
  static constexpr int kQBytes = kDecodeRows * D * 2;
  static constexpr int kConvBytes = FP8 ? kWarps * 2 * kKeysPerWarp * D * 2 : 0;
  static constexpr int kMergeBytes = kWarps * kDecodeRows * (D + 2) * 4;
  static constexpr int kStagesBytes = kStages * kStageBytes;
  static constexpr int kLoopBytes = kStagesBytes + kConvBytes;
  static constexpr int kBytes =
      kQBytes + (kLoopBytes > kMergeBytes ? kLoopBytes : kMergeBytes);
};

// Issue the loads of one stage: keys [kb, kb + kBN) clipped to [k_begin, k_end).
// Cached keys (j < ctx) come from pages; the new key (j >= ctx) from the inputs.
template <int D, bool FP8>
__device__ __forceinline__ void load_stage(const AttnArgs& a, uint8_t* stage, int seq, int h,
                                           int kb, int k_begin, int k_end, int ctx, int q0,
                                           int tid) {
  using S = Smem<D, FP8>;
  constexpr int kChunks = S::kRowBytes / 16;  // per key row
  const int Hkv = a.kv.p.num_kv_heads;
  for (int idx = tid; idx < kBN * 2 * kChunks; idx += kThreads) {
    const int key = idx / (2 * kChunks);
    const int rem = idx % (2 * kChunks);
    const int kv = rem / kChunks, c = rem % kChunks;
    const int j = kb + key;
    uint8_t* tile = stage + kv * kBN * S::kRowBytes;
    const uint32_t dst_off = FP8 ? (uint32_t)(key * S::kRowBytes + c * 16) : swz(key, c, S::kRowBytes);
    if (j < k_begin || j >= k_end) {
      *reinterpret_cast<uint4*>(tile + dst_off) = make_uint4(0, 0, 0, 0);
      continue;
    }
    if (j < ctx) {
      const int32_t page = lookup_page(a.kv, seq, j);
      if (page < 0) {
        *reinterpret_cast<uint4*>(tile + dst_off) = make_uint4(0, 0, 0, 0);
        continue;
      }
      const uint8_t* src =
          a.kv.cache + pool_offset(a.kv.p, page, j % a.kv.p.page_size, 2 * h + kv, S::kElem) + c * 16;
      cp_async_16(smem_u32(tile + dst_off), src);
    } else {
      const __nv_bfloat16* in = (kv ? a.kv.values : a.kv.keys) +
                                ((int64_t)(q0 + (j - ctx)) * Hkv + h) * D;
      if (FP8) {
        // 16 codes = two 8-value bf16 chunks, quantised exactly as the page write does
        const float scale = kv ? a.kv.p.v_scale : a.kv.p.k_scale;
        const uint2 lo = quantize8(__ldg(reinterpret_cast<const uint4*>(in + c * 16)), scale);
        const uint2 hi = quantize8(__ldg(reinterpret_cast<const uint4*>(in + c * 16 + 8)), scale);
        *reinterpret_cast<uint4*>(tile + dst_off) = make_uint4(lo.x, lo.y, hi.x, hi.y);
      } else {
        cp_async_16(smem_u32(tile + dst_off), in + c * 8);
      }
    }
  }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads) decode_kernel(AttnArgs a) {
  using S = Smem<D, FP8>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sStages = smem + S::kQBytes;
  uint8_t* sConv = sStages + S::kStagesBytes;
  float* sMerge = reinterpret_cast<float*>(smem + S::kQBytes);  // reused after the loop
  __shared__ int s_unit, s_last;

  const rpa_params_t& p = a.kv.p;
  int32_t* hdr = a.kv.ws;
  const WorkspaceLayout L(p);
  const DecodeUnit* units =
      reinterpret_cast<const DecodeUnit*>(reinterpret_cast<const char*>(hdr) + L.decode_units_off);
  int32_t* counters = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(hdr) + L.counters_off);
  float* part_o = reinterpret_cast<float*>(reinterpret_cast<char*>(hdr) + L.partial_o_off);
  float2* part_ml = reinterpret_cast<float2*>(reinterpret_cast<char*>(hdr) + L.partial_ml_off);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int n_units = hdr[kHdrNumDecode];
  const LogitXform xf{p.softmax_scale * p.k_scale, p.logits_soft_cap,
                      p.logits_soft_cap > 0.f ? 1.f / p.logits_soft_cap : 0.f,
                      p.softmax_scale * p.k_scale * kLog2e};

  if (tid == 0) s_unit = atomicAdd(hdr + kHdrDecodeNext, 1);
  __syncthreads();
  int u = s_unit;
  while (u < n_units) {
    int next = 0;
    if (tid == 0) next = atomicAdd(hdr + kHdrDecodeNext, 1);  // prefetch the next unit
    const DecodeUnit du = units[u];
    const int seq = du.seq, h = du.head;
    const int q0 = a.qsl[seq];
    const int kv_len = a.kv_lens[seq];
    const int ctx = kv_len - 1;

    // split 0 stores the new token's key/value into its page
    if (du.split == 0 && warp == 0) write_token_kv<FP8>(a.kv, seq, q0, ctx, h, lane);

    // Q tile: rows = the G q-heads of kv head h (rows >= G are zero)
    for (int idx = tid; idx < kDecodeRows * (D / 8); idx += kThreads) {
      const int r = idx / (D / 8), c = idx % (D / 8);
      uint8_t* dst = sQ + swz(r, c, D * 2);
      if (r < G) {
        cp_async_16(smem_u32(dst), a.queries + ((int64_t)q0 * p.num_q_heads + h * G + r) * D + c * 8);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    const int kb0 = du.k_begin;
    const int n_stages = (du.k_end - du.k_begin + kBN - 1) / kBN;
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {
      if (st < n_stages)
        load_stage<D, FP8>(a, sStages + st * S::kStageBytes, seq, h, kb0 + st * kBN, du.k_begin,
                           du.k_end, ctx, q0, tid);
      cp_async_commit();
    }

    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    uint32_t qa[D / 16][4];

    for (int st = 0; st < n_stages; ++st) {
      cp_async_wait<kStages - 2>();
      __syncthreads();
      if (st == 0) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int mi = lane >> 3;
          const int row = (lane & 7) + ((mi & 1) << 3);
          const int chunk = 2 * ks + (mi >> 1);
          ldmatrix_x4(smem_u32(sQ + swz(row, chunk, D * 2)), qa[ks][0], qa[ks][1], qa[ks][2],
                      qa[ks][3]);
        }
      }
      {
        const int nst = st + kStages - 1;
        if (nst < n_stages)
          load_stage<D, FP8>(a, sStages + (nst % kStages) * S::kStageBytes, seq, h,
                             kb0 + nst * kBN, du.k_begin, du.k_end, ctx, q0, tid);
        cp_async_commit();
      }
      const uint8_t* stage = sStages + (st % kStages) * S::kStageBytes;
      const uint8_t* tK;
      const uint8_t* tV;
      int krow0;  // first row of this warp's keys in tK/tV
      if (FP8) {
        // convert this warp's 16 keys and values to bf16 (exact) in its own buffer
        uint8_t* cK = sConv + warp * 2 * kKeysPerWarp * D * 2;
        uint8_t* cV = cK + kKeysPerWarp * D * 2;
        for (int idx = lane; idx < 2 * kKeysPerWarp * (D / 8); idx += 32) {
          const int kv = idx / (kKeysPerWarp * (D / 8));
          const int rem = idx % (kKeysPerWarp * (D / 8));
          const int r = rem / (D / 8), c = rem % (D / 8);
          const uint2 codes = *reinterpret_cast<const uint2*>(
              stage + kv * kBN * S::kRowBytes + (warp * kKeysPerWarp + r) * S::kRowBytes + c * 8);
          *reinterpret_cast<uint4*>((kv ? cV : cK) + swz(r, c, D * 2)) = dequant8(codes);
        }
        __syncwarp();
        tK = cK;
        tV = cV;
        krow0 = 0;
      } else {
        tK = stage;
        tV = stage + kBN * S::kRowBytes;
        krow0 = warp * kKeysPerWarp;
      }

      // S = Q K^T for this warp's 16 keys (two n8 tiles)
      float s[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int mi = lane >> 3;
        const int key = krow0 + (lane & 7) + ((mi >> 1) << 3);
        const int chunk = 2 * ks + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(smem_u32(tK + swz(key, chunk, D * 2)), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qa[ks], b0, b1);
        mma_bf16_16816(s[1], qa[ks], b2, b3);
      }
      // logits, mask, online softmax (rows gq and gq + 8)
      const int kw = kb0 + st * kBN + warp * kKeysPerWarp;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = kw + n * 8 + 2 * tq + (e & 1);
          const float x = (j >= du.k_begin && j < du.k_end) ? xf(s[n][e]) : -INFINITY;
          s[n][e] = x;
          mx[e >> 1] = fmaxf(mx[e >> 1], x);
        }
      float alpha[2], msafe[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float mnew = fmaxf(m_run[r], quad_max(mx[r]));
        msafe[r] = mnew == -INFINITY ? 0.f : mnew;
        alpha[r] = exp2f(m_run[r] - msafe[r]);
        m_run[r] = mnew;
      }
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pe = exp2f(s[n][e] - msafe[e >> 1]);
          s[n][e] = pe;
          rs[e >> 1] += pe;
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) l_run[r] = l_run[r] * alpha[r] + rs[r];
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
      // O += P V (P as the A operand straight from the score registers)
      uint32_t pa[4];
      pa[0] = pack_bf16(s[0][0], s[0][1]);
      pa[1] = pack_bf16(s[0][2], s[0][3]);
      pa[2] = pack_bf16(s[1][0], s[1][1]);
      pa[3] = pack_bf16(s[1][2], s[1][3]);
#pragma unroll
      for (int cp = 0; cp < D / 16; ++cp) {
        const int mi = lane >> 3;
        const int key = krow0 + (lane & 7) + ((mi & 1) << 3);
        const int chunk = 2 * cp + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(smem_u32(tV + swz(key, chunk, D * 2)), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * cp], pa, b0, b1);
        mma_bf16_16816(o[2 * cp + 1], pa, b2, b3);
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // stage memory becomes the merge area

    // per-warp state -> shared memory: rows [warp][16] of (m, l, O[D])
    {
      float* mw = sMerge + warp * kDecodeRows * (D + 2);
      const float l0 = quad_sum(l_run[0]), l1 = quad_sum(l_run[1]);
      if (tq == 0) {
        mw[gq * (D + 2) + 0] = m_run[0];
        mw[gq * (D + 2) + 1] = l0;
        mw[(gq + 8) * (D + 2) + 0] = m_run[1];
        mw[(gq + 8) * (D + 2) + 1] = l1;
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const int d = n * 8 + 2 * tq;
        mw[gq * (D + 2) + 2 + d] = o[n][0];
        mw[gq * (D + 2) + 2 + d + 1] = o[n][1];
        mw[(gq + 8) * (D + 2) + 2 + d] = o[n][2];
        mw[(gq + 8) * (D + 2) + 2 + d + 1] = o[n][3];
      }
    }
    __syncthreads();

    // merge the four warps; one (row, 4 dims) per thread-iteration
    const bool single = du.nsplit == 1;
    for (int idx = tid; idx < G * (D / 4); idx += kThreads) {
      const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sMerge[(w * kDecodeRows + r) * (D + 2)]);
      float Lsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float* row = sMerge + (w * kDecodeRows + r) * (D + 2);
        const float sc = row[0] == -INFINITY ? 0.f : exp2f(row[0] - M);
        Lsum += sc * row[1];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] += sc * row[2 + d + e];
      }
      const int hq = h * G + r;
      if (single) {
        if (a.sink) {
          const float sk = a.sink[hq] * kLog2e;
          const float M2 = fmaxf(M, sk);
          const float sc = exp2f(M - M2);
          Lsum = Lsum * sc + exp2f(sk - M2);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] *= sc;
        }
        const float inv = p.v_scale / Lsum;
        __nv_bfloat16* dst = a.out + ((int64_t)q0 * p.num_q_heads + hq) * D + d;
        uint2 pk;
        pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
        pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(dst) = pk;
      } else {
        float* po = part_o + ((int64_t)u * G + r) * D + d;
        *reinterpret_cast<float4*>(po) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        if (d == 0) part_ml[(int64_t)u * G + r] = make_float2(M, Lsum);
      }
    }

    if (!single) {
      // the last split of (seq, head) to finish combines all of them
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int prev = atomicAdd(counters + (int64_t)seq * p.num_kv_heads + h, 1);
        s_last = prev == du.nsplit - 1;
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        for (int idx = tid; idx < G * (D / 4); idx += kThreads) {
          const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
          const int hq = h * G + r;
          float M = a.sink ? a.sink[hq] * kLog2e : -INFINITY;
          for (int k = 0; k < du.nsplit; ++k)
            M = fmaxf(M, __ldcg(&part_ml[(int64_t)(du.first_unit + k) * G + r].x));
          float Lsum = a.sink ? exp2f(a.sink[hq] * kLog2e - M) : 0.f;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int k = 0; k < du.nsplit; ++k) {
            const int64_t pu = (int64_t)(du.first_unit + k) * G + r;
            const float2 ml = __ldcg(&part_ml[pu]);
            const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
            Lsum += sc * ml.y;
            const float4 po = __ldcg(reinterpret_cast<const float4*>(part_o + pu * D + d));
            acc[0] += sc * po.x;
            acc[1] += sc * po.y;
            acc[2] += sc * po.z;
            acc[3] += sc * po.w;
          }
          const float inv = p.v_scale / Lsum;
          __nv_bfloat16* dst = a.out + ((int64_t)q0 * p.num_q_heads + hq) * D + d;
          uint2 pk;
          pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
          pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
          *reinterpret_cast<uint2*>(dst) = pk;
        }
      }
    }
    __syncthreads();
    if (tid == 0) s_unit = next;
    __syncthreads();
    u = s_unit;
  }
}

}  // namespace dec

template <int D, bool FP8>
static cudaError_t launch_decode_t(const AttnArgs& a, int max_units, int num_sms,
                                   cudaStream_t stream) {
  using S = dec::Smem<D, FP8>;
  auto kern = dec::decode_kernel<D, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, dec::kThreads, S::kBytes);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  int grid = num_sms * per_sm;
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;
  kern<<<grid, dec::kThreads, S::kBytes, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream) {
  const bool fp8 = a.kv.p.kv_dtype == RPA_KV_FP8_E4M3;
  if (a.kv.p.head_dim == 64)
    return fp8 ? launch_decode_t<64, true>(a, max_units, num_sms, stream)
               : launch_decode_t<64, false>(a, max_units, num_sms, stream);
  return fp8 ? launch_decode_t<128, true>(a, max_units, num_sms, stream)
             : launch_decode_t<128, false>(a, max_units, num_sms, stream);
}

}  // namespace rpa
