// Prefill / chunked-prefill path (warp-level MMA version).
//
// Work unit = (sequence, tile of new tokens, kv head).  The tile's rows are
// (token, q-head of the GQA group) pairs, token-major: row r is token
// t_begin + r / G, q-head h*G + r % G (tpu-inference RPA v3 kernel.py stacks a
// q block's heads of one kv head the same way), so each key/value tile read
// from the pages serves all G heads.  Keys stream in tiles of 64 from pages
// (cached context) or from the step's inputs (the new tokens, as RPA v3
// _fetch_bkv does); the tile's own new tokens are written into their pages by
// the same unit.  Online softmax in fp32 per row (RPA v3
// flash_attention_step1_qk_softmax / step2_pv), with the causal and sliding
// window masks applied only on tiles that cross a mask edge.
#include "common.cuh"
#include "kv_write.cuh"
#include "tma_host.h"

namespace rpa {

namespace pf {

constexpr int kThreads = 128;
constexpr int kWarps = 4;
constexpr int kBM = kPrefillRows;  // 64 rows
constexpr int kBN = 64;            // keys per tile
constexpr int kStages = 2;

template <int D>
struct Smem {
  static constexpr int kDp = (D + 63) / 64 * 64;  // head_dim 96 runs as 128 (zero columns)
  static constexpr int kRowBytes = kDp * 2;        // tiles are held as bf16
  static constexpr int kQBytes = kBM * kRowBytes;
  static constexpr int kStageBytes = 2 * kBN * kRowBytes;
  static constexpr int kBytes = kQBytes + kStages * kStageBytes;
};

// Loads keys [kb, kb + kBN) (clipped to [lo, hi]) of kv head h into a stage.
template <int D, bool FP8>
__device__ __forceinline__ void load_tile(const AttnArgs& a, uint8_t* stage, int seq, int h,
                                          int kb, int lo, int hi, int ctx, int q0, int tid) {
  constexpr int kDp = Smem<D>::kDp;
  constexpr int kChunks = kDp / 8;  // 16-byte bf16 chunks per padded row
  const int Hkv = a.kv.p.num_kv_heads;
  for (int idx = tid; idx < kBN * 2 * kChunks; idx += kThreads) {
    const int key = idx / (2 * kChunks);
    const int rem = idx % (2 * kChunks);
    const int kv = rem / kChunks, c = rem % kChunks;
    const int j = kb + key;
    uint8_t* dst = stage + kv * kBN * (kDp * 2) + swz(key, c, kDp * 2);
    if (j < lo || j > hi || c >= D / 8) {  // masked key, or a padding column
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      continue;
    }
    if (j < ctx) {
      const int32_t page = lookup_page(a.kv, seq, j);
      if (page < 0) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        continue;
      }
      const uint8_t* src =
          a.kv.cache + pool_offset(a.kv.p, page, j % a.kv.p.page_size, 2 * h + kv, FP8 ? 1 : 2);
      if (FP8) {  // keys bf16, values fp16 (exact for e4m3)
        const uint2 codes = __ldg(reinterpret_cast<const uint2*>(src + c * 8));
        *reinterpret_cast<uint4*>(dst) = kv ? dequant8_f16(codes) : dequant8(codes);
      } else {
        cp_async_16(smem_u32(dst), src + c * 16);
      }
    } else {
      const __nv_bfloat16* in =
          (kv ? a.kv.values : a.kv.keys) + ((int64_t)(q0 + (j - ctx)) * Hkv + h) * D + c * 8;
      if (FP8) {
        const float scale = kv ? v_scale_of(a.kv.p, h) : k_scale_of(a.kv.p, h);
        const uint2 codes = quantize8(__ldg(reinterpret_cast<const uint4*>(in)), scale);
        *reinterpret_cast<uint4*>(dst) = kv ? dequant8_f16(codes) : dequant8(codes);
      } else {
        cp_async_16(smem_u32(dst), in);
      }
    }
  }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads) prefill_kernel(AttnArgs a) {
  using S = Smem<D>;
  constexpr int Dp = S::kDp;  // head_dim as laid out in shared memory
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sStages = smem + S::kQBytes;
  __shared__ int s_unit;

  const rpa_params_t& p = a.kv.p;
  int32_t* hdr = a.kv.ws;
  const WorkspaceLayout L(p);
  const PrefillUnit* units =
      reinterpret_cast<const PrefillUnit*>(reinterpret_cast<const char*>(hdr) + L.prefill_units_off);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int W = p.sliding_window;
  // No wait on the kernel ahead (the decode kernel) before the work: this
  // kernel needs nothing it writes, so its CTAs may start on the SMs the
  // decode tail frees.  The planner's output is complete and visible: every
  // decode CTA lets this grid launch only after its own wait on the planner
  // (and a launch starts with a fresh L1).  Every CTA waits for the decode
  // grid before it exits, so this grid never completes before it: whatever
  // follows on the stream still finds both kernels done.
  const int n_units = __ldcg(hdr + kHdrNumPrefill);

  if (tid == 0) s_unit = atomicAdd(hdr + kHdrPrefillNext, 1);
  __syncthreads();
  int u = s_unit;
  while (u < n_units) {
    int next = 0;
    if (tid == 0) next = atomicAdd(hdr + kHdrPrefillNext, 1);
    const PrefillUnit pu = units[u];
    const int seq = pu.seq, h = pu.head;
    const float ks = k_scale_of(p, h);  // this kv head's key scale
    const LogitXform xf = make_xform(p.softmax_scale, qk_scale(p, ks), p.logits_soft_cap);
    const int q0 = a.qsl[seq];
    const int q_len = a.qsl[seq + 1] - q0;
    const int ctx = a.kv_lens[seq] - q_len;
    const int n_tok = pu.t_end - pu.t_begin;

    // this unit's new tokens -> their pages (one warp per token)
    for (int i = warp; i < n_tok; i += kWarps)
      write_token_kv<FP8>(a.kv, seq, q0 + pu.t_begin + i, ctx + pu.t_begin + i, h, lane);

    // Q tile (rows past the tile's tokens are zero)
    for (int idx = tid; idx < kBM * (Dp / 8); idx += kThreads) {
      const int r = idx / (Dp / 8), c = idx % (Dp / 8);
      const int ti = r / G;
      uint8_t* dst = sQ + swz(r, c, Dp * 2);
      if (ti < n_tok && c < D / 8) {
        const int t = q0 + pu.t_begin + ti;
        cp_async_16(smem_u32(dst), a.queries + ((int64_t)t * p.num_q_heads + h * G + r % G) * D + c * 8);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    // key range of the whole tile
    const int pos_first = ctx + pu.t_begin, pos_last = ctx + pu.t_end - 1;
    const int lo = (W > 0 && pos_first - W + 1 > 0) ? pos_first - W + 1 : 0;
    const int hi = pos_last;
    const int n_kt = (hi - lo + 1 + kBN - 1) / kBN;
    load_tile<D, FP8>(a, sStages, seq, h, lo, lo, hi, ctx, q0, tid);
    cp_async_commit();

    // the two rows this thread owns: positions (clamped for padding rows)
    int rpos[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = warp * 16 + gq + 8 * r;
      const int ti = min(row / G, n_tok - 1);
      rpos[r] = ctx + pu.t_begin + ti;
    }

    float o[Dp / 8][4];
#pragma unroll
    for (int n = 0; n < Dp / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    // query fragment ks of this warp's 16 rows; up to head_dim 128 they are
    // held in registers for the whole unit, from 192 on (48 / 64 registers)
    // they are re-read from the swizzled Q tile for every key tile
    constexpr bool kQFromSmem = Dp > 128;
    auto load_q = [&](int ks, uint32_t (&f)[4]) {
      const int mi = lane >> 3;
      const int row = warp * 16 + (lane & 7) + ((mi & 1) << 3);
      const int chunk = 2 * ks + (mi >> 1);
      ldmatrix_x4(smem_u32(sQ + swz(row, chunk, Dp * 2)), f[0], f[1], f[2], f[3]);
    };
    uint32_t qa[kQFromSmem ? 1 : Dp / 16][4];

    for (int kt = 0; kt < n_kt; ++kt) {
      if (kt + 1 < n_kt)
        load_tile<D, FP8>(a, sStages + ((kt + 1) % kStages) * S::kStageBytes, seq, h,
                          lo + (kt + 1) * kBN, lo, hi, ctx, q0, tid);
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      if (FP8 && kt == 0 && p.q_scale > 0.f) {  // q_scale needs an e4m3 cache
        // quantised queries: the tile becomes its e4m3 codes' values
        for (int i = tid; i < S::kQBytes / 16; i += kThreads)
          quantize_q8(reinterpret_cast<uint4*>(sQ) + i, p.q_scale);
        __syncthreads();
      }
      if constexpr (!kQFromSmem) {
        if (kt == 0) {
#pragma unroll
          for (int ks = 0; ks < (kQFromSmem ? 1 : Dp / 16); ++ks) load_q(ks, qa[ks]);
        }
      }
      const uint8_t* tK = sStages + (kt % kStages) * S::kStageBytes;
      const uint8_t* tV = tK + kBN * (Dp * 2);
      const int kb = lo + kt * kBN;

      float s[kBN / 8][4];
#pragma unroll
      for (int n = 0; n < kBN / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < Dp / 16; ++ks) {
        uint32_t qf[4];
        if constexpr (kQFromSmem) {
          load_q(ks, qf);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) qf[i] = qa[kQFromSmem ? 0 : ks][i];
        }
#pragma unroll
        for (int np = 0; np < kBN / 16; ++np) {
          const int mi = lane >> 3;
          const int key = np * 16 + (lane & 7) + ((mi >> 1) << 3);
          const int chunk = 2 * ks + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(smem_u32(tK + swz(key, chunk, Dp * 2)), b0, b1, b2, b3);
          mma_bf16_16816(s[2 * np], qf, b0, b1);
          mma_bf16_16816(s[2 * np + 1], qf, b2, b3);
        }
      }
      // does any key of this tile need masking for this warp's rows?
      const int wpos_lo = ctx + pu.t_begin + min((warp * 16) / G, n_tok - 1);
      const int wpos_hi = ctx + pu.t_begin + min((warp * 16 + 15) / G, n_tok - 1);
      const bool full = (kb + kBN - 1 <= wpos_lo) && (W == 0 || wpos_hi - kb < W) && (kb + kBN - 1 <= hi);
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < kBN / 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = xf(s[n][e]);
          if (!full) {
            const int j = kb + n * 8 + 2 * tq + (e & 1);
            const int pos = rpos[e >> 1];
            const bool ok = j <= pos && j >= lo && (W == 0 || pos - j < W);
            x = ok ? x : -INFINITY;
          }
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
      // P packed as the P V product takes it (fp16 with an e4m3 cache,
      // else bf16); the row sums add exactly those rounded weights
      float rs[2] = {0.f, 0.f};
      uint32_t pk[kBN / 8][2];
#pragma unroll
      for (int n = 0; n < kBN / 8; ++n)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          pk[n][r] = pack_p<FP8>(exp2f(s[n][2 * r] - msafe[r]), exp2f(s[n][2 * r + 1] - msafe[r]));
          rs[r] += pair_sum<FP8>(pk[n][r]);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) l_run[r] = l_run[r] * alpha[r] + rs[r];
#pragma unroll
      for (int n = 0; n < Dp / 8; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint32_t pa[4] = {pk[2 * kk][0], pk[2 * kk][1], pk[2 * kk + 1][0],
                                pk[2 * kk + 1][1]};
#pragma unroll
        for (int cp = 0; cp < Dp / 16; ++cp) {
          const int mi = lane >> 3;
          const int key = kk * 16 + (lane & 7) + ((mi & 1) << 3);
          const int chunk = 2 * cp + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(smem_u32(tV + swz(key, chunk, Dp * 2)), b0, b1, b2, b3);
          mma_p_16816<FP8>(o[2 * cp], pa, b0, b1);
          mma_p_16816<FP8>(o[2 * cp + 1], pa, b2, b3);
        }
      }
      __syncthreads();  // the stage is refilled next iteration
    }
    cp_async_wait<0>();

    // finalize: sink, 1/l, v_scale, bf16 store
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = warp * 16 + gq + 8 * r;
      const int ti = row / G;
      float l = quad_sum(l_run[r]);
      float m = m_run[r];
      float sc = 1.f;
      const int hq = h * G + row % G;
      if (a.sink) {
        const float sk = a.sink[hq] * kLog2e;
        const float m2 = fmaxf(m, sk);
        sc = exp2f(m - m2);
        l = l * sc + exp2f(sk - m2);
      }
      if (ti >= n_tok) continue;
      const float inv = sc * v_scale_of(p, h) / l;
      __nv_bfloat16* dst = a.out + ((int64_t)(q0 + pu.t_begin + ti) * p.num_q_heads + hq) * D;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const int d = n * 8 + 2 * tq;
        *reinterpret_cast<uint32_t*>(dst + d) = pack_bf16(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
      }
    }
    __syncthreads();
    if (tid == 0) s_unit = next;
    __syncthreads();
    u = s_unit;
  }
  griddep_wait();  // complete only after the decode kernel ahead
}

}  // namespace pf

template <int D, bool FP8>
static cudaError_t launch_prefill_t(const AttnArgs& a, int max_units, int num_sms,
                                    cudaStream_t stream) {
  using S = pf::Smem<D>;
  auto kern = pf::prefill_kernel<D, FP8>;
  static std::atomic<unsigned long long> attr_done{0};
  static std::atomic<int> per_sm_cached{0};
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), S::kBytes, &attr_done);
  if (e != cudaSuccess) return e;
  int per_sm = per_sm_cached.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, pf::kThreads, S::kBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    per_sm_cached.store(per_sm, std::memory_order_relaxed);
  }
  int grid = num_sms * per_sm;
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;
  return launch_dependent(kern, grid, pf::kThreads, S::kBytes, stream, a);
}

cudaError_t launch_prefill(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream) {
  const bool fp8 = a.kv.p.kv_dtype == RPA_KV_FP8_E4M3;
  if (a.kv.p.head_dim == 64)
    return fp8 ? launch_prefill_t<64, true>(a, max_units, num_sms, stream)
               : launch_prefill_t<64, false>(a, max_units, num_sms, stream);
  if (a.kv.p.head_dim == 96)
    return fp8 ? launch_prefill_t<96, true>(a, max_units, num_sms, stream)
               : launch_prefill_t<96, false>(a, max_units, num_sms, stream);
  if (a.kv.p.head_dim == 192)
    return fp8 ? launch_prefill_t<192, true>(a, max_units, num_sms, stream)
               : launch_prefill_t<192, false>(a, max_units, num_sms, stream);
  if (a.kv.p.head_dim == 256)
    return fp8 ? launch_prefill_t<256, true>(a, max_units, num_sms, stream)
               : launch_prefill_t<256, false>(a, max_units, num_sms, stream);
  return fp8 ? launch_prefill_t<128, true>(a, max_units, num_sms, stream)
             : launch_prefill_t<128, false>(a, max_units, num_sms, stream);
}

}  // namespace rpa
