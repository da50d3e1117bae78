// Prefill / chunked-prefill path on the 5th-generation tensor cores for
// head_dim 192 and 256.
//
// At these head sizes two 128-row query tiles would need their O
// accumulators alone to fill the 512 tensor-memory columns (2 x 256), so a
// unit here is ONE query tile of 128 (token, q-head) rows, token-major (row R
// is token t_begin + R / G, q-head h*G + R % G: tpu-inference RPA v3
// kernel.py stacks a q block's heads of one kv head the same way).  Keys come
// in tiles of 64, and S is double-buffered in tensor memory instead:
//   O    columns [0, D)      fp32 accumulator of P V
//   S_0  columns [256, 320)  scores of key tiles 0, 2, 4, ... (then P, bf16)
//   S_1  columns [320, 384)  scores of key tiles 1, 3, 5, ...
//   Q    columns [384, 384 + D/2)  the bf16 query tile, the A operand of S
//        (placed by the softmax warps at the unit's start; with quantised
//        queries S reads an e4m3 code tile from shared memory instead)
// The MMA thread issues S(0), S(1), then per key tile j: P V(j), S(j+2).  So
// the tensor core computes the scores of tile j+1 (and j+2) while the softmax
// warpgroup works on tile j -- the overlap the RPA v3 kernel gets by
// pipelining flash_attention_step1_qk_softmax of one step with
// flash_attention_step2_pv of the previous one.  S(j+2) overwrites P(j) only
// after P V(j) has read it (one thread's tcgen05 products run in order).
//
// The softmax (one thread per row) keeps the running max m and sum l in
// fp32 and moves m -- rescaling O in tensor memory -- only when a row's max
// grows by more than 2^8.  Because S(j) may complete before P V(j-1) has,
// such a rescale first waits for P V(j-1) (a barrier committed after every
// P V product); rescales are rare, so the wait almost never happens.
//
// Keys [lo, ctx) come page by page from the pool (one TMA box per page and
// 64-column block of head_dim), the step's new keys [ctx, ...) from the
// keys/values inputs (RPA v3 _fetch_bkv does the same).  Value rows no row
// of the unit may see are zeroed before the P V product.  The unit's own new
// tokens are written into their pages by two otherwise idle warps while the
// unit runs.  With an e4m3 cache the step's new tokens were written into
// their pages ahead of this kernel, every tile comes from the pool, and the
// pages' codes land in a staging buffer and are decoded into the operand
// stage: keys as bf16 (the queries' type), values as fp16 (exact for e4m3),
// with P packed as fp16 to match.  With quantised queries (q_scale) S = Q K^T
// runs on the e4m3 codes themselves (tcgen05.mma kind::f8f6f4): the query
// tile is quantised once per unit into a code tile, key pages land as codes
// in code-tile key stages, and the logit scale carries q_scale * k_scale.
#include "async.cuh"
#include "common.cuh"
#include "kv_write.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma_host.h"

namespace rpa {
namespace tcw {

// warp 0: TMA (+ fp8 decoding); warp 1: MMA (one thread) and tensor-memory
// allocation; warps 2-3: fp8 decoding, or with a bf16 cache the unit's page
// write; warps 4-7: softmax, one thread per row of the query tile
constexpr int kThreads = 256;
constexpr int kM = 128;                         // rows per unit (one query tile)
constexpr int kN = 64;                          // keys per tile
constexpr uint32_t kHalfQ = 128 * 128;          // [128 rows][64 bf16], 16 KB
constexpr uint32_t kHalfKV = 64 * 128;          // [64 rows][64 bf16], 8 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS = 256;    // S slot b at kTmemS + 64 b
constexpr uint32_t kTmemQ = 384;                // bf16 query tile (D/2 columns)
constexpr int kRescaleLog2 = 8;

// With quantised queries (Q8) the query tile and the key stages are e4m3 code
// tiles in blocks of 64 bytes (D/64 per row, 64-byte swizzle): the query
// code tile [D/64][128 rows][64 B] and key stages [D/64][64 rows][64 B]; only
// the values are staged.
template <int D, bool FP8, bool Q8 = false>
struct Cfg {
  static_assert(!Q8 || FP8, "quantised queries need an e4m3 cache");
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kQBytes = kHalves * kHalfQ;
  static constexpr uint32_t kOperand = kHalves * kHalfKV;  // one bf16 / fp16 operand stage
  static constexpr uint32_t kStaging = FP8 ? (uint32_t)kN * D : 0u;  // e4m3 codes of a tile
  static constexpr uint32_t kBlkQ = 128 * 64, kBlkK = kN * 64;  // one 64-byte block of codes
  static constexpr uint32_t kKStage = Q8 ? (uint32_t)kN * D : kOperand;  // key stage stride
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffQ8 = kQBytes;                          // Q8: query codes
  static constexpr uint32_t kOffK = kQBytes + (Q8 ? 128u * D : 0u);    // + s*kKStage
  static constexpr uint32_t kOffV = kOffK + 2 * kKStage;               // + s*kOperand
  static constexpr uint32_t kOffStg = kOffV + 2 * kOperand;  // staging kv at + kv*kStaging
  static constexpr int kStgOps = Q8 ? 1 : 2;                  // (Q8: values only, at kv 0)
  static constexpr uint32_t kOffBar = (kOffStg + kStgOps * kStaging + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = (int)kOffBar + 256 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "fits one CTA's shared memory");
};

// Byte offset of the codes of elements 8*c8 .. 8*c8+7 of row r in a 64-byte
// block of an e4m3 code tile (64-byte swizzle: 16-byte chunk XOR address
// bits 7-8).
__device__ __forceinline__ uint32_t sw64_codes(int r, int c8) {
  return (uint32_t)r * 64 + (((((uint32_t)c8 & 7u) >> 1) ^ ((uint32_t)(r >> 1) & 3u)) << 4) +
         ((uint32_t)(c8 & 1) << 3);
}

enum Bar {
  kBarQFull = 0,    // the query tile landed
  kBarKFull = 1,    // [2] key TMA landed
  kBarVFull = 3,    // [2] value TMA landed
  kBarVReady = 5,   // [2] values fixed up / decoded, MMA may read
  kBarVEmpty = 7,   // [2] value stage free: its P V product done (every P V product
                    // completes one of the two in turn, which also orders O rescales)
  kBarKReady = 9,   // [2] fp8 cache: keys decoded, MMA may read
  kBarSFull = 11,   // [2] per S slot: S computed (and its key stage free)
  kBarPReady = 13,  // [2] per S slot: P written (and O corrected)
  kBarODone = 15,   // the unit's last P V product done
  kBarDrain = 16,   // once, at exit: every tcgen05 product the MMA thread issued is done
  kBarQReady = 17,  // the softmax warps placed the query tile: in tensor memory (bf16),
                    // or as its e4m3 code tile (quantised queries, q_scale)
  kNumBars = 18,
};

struct Maps {
  CUtensorMap q;      // queries [T][Hq][D], box {64, G, 128/G}
  CUtensorMap cache;  // pool [num_pages*P][2*Hkv][D], box {64, 1, min(P,64)} (fp8: {D, 1, ..})
  CUtensorMap knew;   // keys [T][Hkv][D], box {64, 1, 64}
  CUtensorMap vnew;   // values [T][Hkv][D], box {64, 1, 64}
  CUtensorMap cache8; // Q8 only: the pool's codes, box {64, 1, min(P,64)}, 64-byte swizzle
};

// Geometry of one unit, computed identically by every role: key tiles of
// 64, from the pool from c_start = lo rounded down to 64 up to k_end (= ctx,
// or with an e4m3 cache the unit's last position + 1: the step's new tokens
// are already in their pages), then new ones from the inputs aligned to ctx.
struct Geom {
  int seq, h, q0, q_len, kv_len, ctx, t_begin, t_end;
  int lo;  // first key any row of the unit may see
  int c_start, k_end, n_cached, i0, n_tiles;
  __device__ int lead(int key0) const { return lo > key0 ? lo - key0 : 0; }
  __device__ void tile(int j, bool& is_new, int& key0, int& valid) const {
    if (j < n_cached) {
      is_new = false;
      key0 = c_start + kN * j;
      valid = min(kN, k_end - key0);
    } else {
      is_new = true;
      key0 = ctx + kN * (i0 + j - n_cached);
      valid = min(kN, kv_len - key0);
    }
  }
};

template <bool FROM_PAGES>
__device__ __forceinline__ Geom unit_geom(const AttnArgs& a, const PrefillUnit& pu) {
  Geom g;
  g.seq = pu.seq;
  g.h = pu.head;
  g.q0 = a.qsl[pu.seq];
  g.q_len = a.qsl[pu.seq + 1] - g.q0;
  g.kv_len = a.kv_lens[pu.seq];
  g.ctx = g.kv_len - g.q_len;
  g.t_begin = pu.t_begin;
  g.t_end = pu.t_end;
  const int W = a.kv.p.sliding_window;
  const int pos_first = g.ctx + g.t_begin, pos_last = g.ctx + g.t_end - 1;
  g.lo = (W > 0 && pos_first - W + 1 > 0) ? pos_first - W + 1 : 0;
  g.k_end = FROM_PAGES ? pos_last + 1 : g.ctx;
  if (g.lo < g.k_end) {
    g.c_start = g.lo & ~(kN - 1);
    g.n_cached = (g.k_end - g.c_start + kN - 1) / kN;
  } else {
    g.c_start = 0;
    g.n_cached = 0;
  }
  g.i0 = g.lo > g.ctx ? (g.lo - g.ctx) / kN : 0;
  const int i1 = (pos_last - g.ctx) / kN;
  g.n_tiles = g.n_cached + (FROM_PAGES ? 0 : i1 - g.i0 + 1);
  return g;
}

template <int D, bool FP8, bool PH, bool Q8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_wide_kernel(const __grid_constant__ Maps maps, AttnArgs a) {
  using C = Cfg<D, FP8, Q8>;
  constexpr int kDecWarps = FP8 ? 3 : 1;  // warps that decode fp8 operands
  constexpr uint32_t kOperand = C::kOperand;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + C::kOffBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  __shared__ uint32_t s_tmem;
  __shared__ int s_unit, s_abort;

  const rpa_params_t& p = a.kv.p;
  int32_t* hdr = a.kv.ws;
  const WorkspaceLayout L(p);
  const PrefillUnit* units =
      reinterpret_cast<const PrefillUnit*>(reinterpret_cast<const char*>(hdr) + L.prefill_units_off);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int P = p.page_size;
  const int W = p.sliding_window;
  // No wait on the kernel ahead (the decode kernel) before the work: this
  // kernel needs nothing it writes, so its CTAs may start on the SMs the
  // decode tail frees.  The planner's output is complete and visible: every
  // decode CTA lets this grid launch only after its own wait on the planner
  // (and a launch starts with a fresh L1).  Every CTA waits for the decode
  // grid before it exits, so this grid never completes before it: whatever
  // follows on the stream still finds both kernels done.
  const int n_units = __ldcg(hdr + kHdrNumPrefill);
  if (n_units == 0) {  // a decode-only batch: nothing to set up
    griddep_wait();     // complete only after the decode kernel ahead
    return;
  }

  if (tid == 0) {
    s_abort = 0;
    mbar_init(bar(kBarQFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVReady + s), FP8 ? kDecWarps : 1);
      mbar_init(bar(kBarVEmpty + s), 1);
      mbar_init(bar(kBarKReady + s), kDecWarps);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarPReady + s), 4);
    }
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarQReady), 4);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&maps.q);
    prefetch_tensormap(&maps.cache);
    prefetch_tensormap(&maps.knew);
    prefetch_tensormap(&maps.vnew);
    if (Q8) prefetch_tensormap(&maps.cache8);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  const uint32_t idesc_qk = Q8 ? idesc_e4m3(kM, kN) : idesc_bf16(kM, kN, false, false);
  // P and the values are fp16 with an e4m3 cache, bf16 otherwise
  const uint32_t idesc_pv = idesc_bf16(kM, D, false, true, FP8);
  const bool has_cap = p.logits_soft_cap > 0.f;
  const LogitXform xf0 = make_xform(p.softmax_scale, qk_scale(p, p.k_scale), p.logits_soft_cap);

  // fp8 cache: decoding of a landed operand of tile j (the staged codes:
  // every tile of an e4m3 unit comes from the pages, the step's new tokens
  // were written there ahead of this kernel) into its operand stage, shared
  // by kDecWarps warps.  Value rows no row of the unit may see (past the
  // valid range, or before the window) become zero; key rows there are
  // masked by the softmax.
  auto decode_fp8 = [&](const Geom& g, uint32_t tc, int j, int kv, int part) {
    if (Q8 && kv == 0) return;  // the key codes landed in their stage as they are
    bool is_new;
    int key0, valid;
    g.tile(j, is_new, key0, valid);
    uint8_t* op = smem + (kv ? C::kOffV + (tc & 1) * kOperand : C::kOffK + (tc & 1) * C::kKStage);
    const uint8_t* stg = smem + C::kOffStg + (Q8 ? 0 : kv) * C::kStaging;
    const int rows = kv ? kN : valid;
    const int lead = kv ? g.lead(key0) : 0;
    for (int idx = 32 * part + lane; idx < rows * (D / 8); idx += 32 * kDecWarps) {
      const int r = idx / (D / 8), c = idx % (D / 8);
      uint4* dst = reinterpret_cast<uint4*>(op + (c >> 3) * kHalfKV + sw128(r, c & 7));
      if (r >= valid || r < lead) {
        *dst = make_uint4(0, 0, 0, 0);
      } else {
        const uint2 codes = *reinterpret_cast<const uint2*>(stg + r * D + c * 8);
        *dst = kv ? dequant8_f16(codes) : dequant8(codes);
      }
    }
  };

  // Every role runs this loop over the CTA's units with its own body; all
  // threads meet at the same two barriers per unit.  tcount counts the key
  // tiles and ucount the units the CTA has processed so far (all roles
  // agree), and give the barriers' phases.
  auto unit_loop = [&](auto&& body) {
    uint32_t tcount = 0, ucount = 0;
    for (;;) {
      if (tid == 0) s_unit = atomicAdd(hdr + kHdrPrefillNext, 1);
      __syncthreads();
      const int u = s_unit;
      if (u >= n_units || s_abort) break;
      const Geom g = unit_geom<FP8>(a, units[u]);
      body(g, tcount, ucount);
      tcount += g.n_tiles;
      ucount += 1;
      tc_fence_before();
      __syncthreads();  // the next unit reuses Q, the stages and tensor memory
      tc_fence_after();
    }
  };

  if (warp == 0) {
    // the last query copy (unit count) and the last key / value copy (tile
    // count) per stage this warp issued, for the drain at exit
    int q_last = -1, k_last0 = -1, k_last1 = -1, v_last0 = -1, v_last1 = -1;
    unit_loop([&](const Geom& g, const uint32_t tcount, const uint32_t ucount) {
      const int nt = g.n_tiles;
      // ----------------------------------------------------- TMA producer
      if (RPA_TEST_STALL_QUERY == 0) {
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(kBarQFull), C::kQBytes);
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(sb + C::kOffQ + hf * kHalfQ, &maps.q, bar(kBarQFull), hf * 64, g.h * G,
                        g.q0 + g.t_begin);
        }
        q_last = (int)ucount;
      }
      // page ids of a cached tile: lane l holds page pg0 + l (a 64-key tile
      // spans at most 64/P <= 8 pages for P >= 8), loaded one tile ahead
      const int64_t bt_row = (int64_t)g.seq * p.pages_per_seq;
      auto load_ids = [&](int j) -> int {
        bool is_new;
        int key0, valid;
        g.tile(j, is_new, key0, valid);
        if (is_new) return 0;
        const int pg0 = key0 / P, npg = (key0 + valid - 1) / P - pg0 + 1;
        return lane < npg ? __ldg(a.kv.block_tables + bt_row + pg0 + lane) : 0;
      };
      auto issue = [&](int j, int kv, uint32_t tc, int page) {
        const uint32_t s = tc & 1;
        bool is_new;
        int key0, valid;
        g.tile(j, is_new, key0, valid);
        const uint32_t dst = sb + (kv ? C::kOffV + s * kOperand : C::kOffK + s * C::kKStage);
        const uint32_t fullbar = bar((kv ? kBarVFull : kBarKFull) + s);
        if (is_new) {
          if (lane == 0) {
            mbar_arrive_expect_tx(fullbar, kOperand);
            const int row = g.q0 + (key0 - g.ctx);
            for (int hf = 0; hf < C::kHalves; ++hf)
              tma_load_3d(dst + hf * kHalfKV, kv ? &maps.vnew : &maps.knew, fullbar, hf * 64, g.h,
                          row);
          }
        } else {
          const int rows = P < kN ? P : kN;
          const int pg0 = key0 / P, npg = (key0 + valid - 1) / P - pg0 + 1;
          if (lane == 0)
            mbar_arrive_expect_tx(fullbar, (uint32_t)(npg * rows * D * (FP8 ? 1 : 2)));
          __syncwarp();
          if (lane < npg) {
            if (page < 0 || page >= p.num_pages) {
              set_status(hdr, RPA_STATUS_BAD_PAGE);
              page = 0;
            }
            const int srow = P < kN ? (pg0 + lane) * P - key0 : 0;
            const int z = page * P + (P < kN ? 0 : key0 % P);
            if (Q8 && kv == 0) {
              for (int hf = 0; hf < C::kHalves; ++hf)
                tma_load_3d(dst + hf * C::kBlkK + srow * 64, &maps.cache8, fullbar, hf * 64, 2 * g.h,
                            z);
            } else if (FP8) {
              tma_load_3d(sb + C::kOffStg + (Q8 ? 0 : kv) * C::kStaging + srow * D, &maps.cache,
                          fullbar, 0, 2 * g.h + kv, z);
            } else {
              for (int hf = 0; hf < C::kHalves; ++hf)
                tma_load_3d(dst + hf * kHalfKV + srow * 128, &maps.cache, fullbar, hf * 64,
                            2 * g.h + kv, z);
            }
          }
        }
      };
      auto finalize_k = [&](uint32_t tc, int j) -> bool {
        const int s = tc & 1;
        if (!mbar_wait_warp(bar(kBarKFull + s), (tc >> 1) & 1, &s_abort)) return false;
        decode_fp8(g, tc, j, 0, 0);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarKReady + s));
        return true;
      };
      auto finalize_v = [&](uint32_t tc, int j) -> bool {
        const int s = tc & 1;
        if (!mbar_wait_warp(bar(kBarVFull + s), (tc >> 1) & 1, &s_abort)) return false;
        if (FP8) {
          decode_fp8(g, tc, j, 1, 0);
          fence_proxy_async();
        } else {
          bool is_new;
          int key0, valid;
          g.tile(j, is_new, key0, valid);
          const int lead = g.lead(key0);
          if (valid < kN || lead > 0) {
            // zero the value rows [0, lead) and [valid, kN): their keys are
            // masked, but their bytes may be anything (0 * NaN poisons P V)
            uint8_t* v = smem + C::kOffV + s * kOperand;
            constexpr int kRowChunks = 8 * C::kHalves;
            const int tail = kN - valid;
            for (int idx = lane; idx < (lead + tail) * kRowChunks; idx += 32) {
              const int i = idx / kRowChunks, c = idx % kRowChunks;
              const int r = i < lead ? i : valid + (i - lead);
              *reinterpret_cast<uint4*>(v + (c >> 3) * kHalfKV + r * 128 + (c & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarVReady + s));
        return true;
      };
      // bf16 cache: the keys run one tile ahead of the values.  S(j+2) is
      // issued right after P V(j), so the keys of tile j+2 are fetched as
      // soon as S(j) has freed their stage, not behind the values of tile
      // j+1 (whose stage frees only with P V(j-1)).  Per step j: keys of j+1,
      // values of j, then finalize values of j-1.
      bool ok = true;
      if constexpr (!FP8) {
        int ids_j = load_ids(0);
        int ids_j1 = nt > 1 ? load_ids(1) : 0;
        if (nt >= 1) {
          if (!mbar_wait_warp(bar(kBarSFull + (tcount & 1)), ((tcount >> 1) & 1) ^ 1, &s_abort))
            ok = false;
          else {
            issue(0, 0, tcount, ids_j);
            ((tcount & 1) ? k_last1 : k_last0) = (int)tcount;
          }
        }
        for (int j = 0; j < nt && ok; ++j) {
          const uint32_t tc = tcount + j;
          const int s = tc & 1;
          if (j + 1 < nt) {
            const uint32_t tn = tc + 1;
            if (!mbar_wait_warp(bar(kBarSFull + (tn & 1)), ((tn >> 1) & 1) ^ 1, &s_abort)) {
              ok = false;
              break;
            }
            issue(j + 1, 0, tn, ids_j1);
            ((tn & 1) ? k_last1 : k_last0) = (int)tn;
          }
          const int ids_j2 = j + 2 < nt ? load_ids(j + 2) : 0;
          if (!mbar_wait_warp(bar(kBarVEmpty + s), ((tc >> 1) & 1) ^ 1, &s_abort)) {
            ok = false;
            break;
          }
          issue(j, 1, tc, ids_j);
          (s ? v_last1 : v_last0) = (int)tc;
          __syncwarp();
          if (j >= 1) ok = finalize_v(tc - 1, j - 1);
          ids_j = ids_j1;
          ids_j1 = ids_j2;
        }
        if (ok && nt >= 1) ok = finalize_v(tcount + nt - 1, nt - 1);
        if (!ok && lane == 0) {
          set_status(hdr, RPA_STATUS_TIMEOUT);
          s_abort = 1;
        }
        return;
      }
      // e4m3 cache, per tile j: keys of j, decode keys of j-1, values of j,
      // then finalize values of j-1.  With the one staging buffer per
      // operand, the codes of tile j-1 are decoded (by every decoding warp)
      // before those of tile j are fetched.
      int ids_next = load_ids(0);
      for (int j = 0; j < nt && ok; ++j) {
        const uint32_t tc = tcount + j;
        const int s = tc & 1;
        const uint32_t par = ((tc >> 1) & 1) ^ 1;
        const int ids = ids_next;
        if (j + 1 < nt) ids_next = load_ids(j + 1);
        if (FP8 && j >= 1) {
          ok = finalize_k(tc - 1, j - 1) &&
               mbar_wait_warp(bar(kBarKReady + ((tc - 1) & 1)), ((tc - 1) >> 1) & 1, &s_abort);
          if (!ok) break;
        }
        if (!mbar_wait_warp(bar(kBarSFull + s), par, &s_abort)) {
          ok = false;
          break;
        }
        issue(j, 0, tc, ids);
        (s ? k_last1 : k_last0) = (int)tc;
        if (FP8 && j >= 1) {
          ok = finalize_v(tc - 1, j - 1) &&
               mbar_wait_warp(bar(kBarVReady + ((tc - 1) & 1)), ((tc - 1) >> 1) & 1, &s_abort);
          if (!ok) break;
        }
        if (!mbar_wait_warp(bar(kBarVEmpty + s), par, &s_abort)) {
          ok = false;
          break;
        }
        issue(j, 1, tc, ids);
        (s ? v_last1 : v_last0) = (int)tc;
        __syncwarp();
        if (!FP8 && j >= 1) ok = finalize_v(tc - 1, j - 1);
      }
      if (FP8 && ok && nt >= 1) ok = finalize_k(tcount + nt - 1, nt - 1);
      if (ok && nt >= 1) ok = finalize_v(tcount + nt - 1, nt - 1);
      if (!ok && lane == 0) {
        set_status(hdr, RPA_STATUS_TIMEOUT);
        s_abort = 1;
      }
    });
    // every copy this warp issued lands before the CTA may free its shared
    // memory: an aborted unit leaves copies nobody waits for
    if (lane == 0) {
      bool drained = q_last < 0 || mbar_drain(bar(kBarQFull), q_last & 1);
      const int kl[2] = {k_last0, k_last1}, vl[2] = {v_last0, v_last1};
      for (int s = 0; s < 2; ++s) {
        if (kl[s] >= 0) drained &= mbar_drain(bar(kBarKFull + s), (kl[s] >> 1) & 1);
        if (vl[s] >= 0) drained &= mbar_drain(bar(kBarVFull + s), (vl[s] >> 1) & 1);
      }
      if (!drained) set_status(hdr, RPA_STATUS_TIMEOUT);
    }
  } else if (warp == 1) {
    unit_loop([&](const Geom& g, const uint32_t tcount, const uint32_t ucount) {
      const int nt = g.n_tiles;
      // ------------------------------------------------------------ MMA
      // S(0), S(1), then per tile j: P V(j), S(j+2).  Key stage and S slot
      // of tile j are both (tcount + j) & 1.
      if (lane == 0) {
        bool ok = mbar_wait(bar(kBarQReady), ucount & 1, &s_abort);
        tc_fence_after();
        auto qk = [&](uint32_t tc) -> bool {
          const int s = tc & 1;
          if (!mbar_wait(bar((FP8 ? kBarKReady : kBarKFull) + s), (tc >> 1) & 1, &s_abort))
            return false;
          tc_fence_after();
          const uint32_t sK = sb + C::kOffK + s * C::kKStage, dS = tmem + kTmemS + 64 * s;
          // one thread issues every product: its descriptors are the tiles'
          // (built once here) advanced by constants, so the issue keeps pace
          // with the tensor core
          if constexpr (Q8) {
            // e4m3 codes: 32 per product, two products per 64-byte block
            const uint64_t dq = sdesc_sw64(sb + C::kOffQ8, 16, 512), dk = sdesc_sw64(sK, 16, 512);
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
              const uint32_t off = (uint32_t)(k & 1) * 32;
              umma_ss_e4m3(dS, sdesc_advance(dq, (k >> 1) * C::kBlkQ + off),
                           sdesc_advance(dk, (k >> 1) * C::kBlkK + off), idesc_qk,
                           k > 0 ? 1u : 0u);
            }
          } else {
            // bf16 queries from tensor memory (16 of D per product = 8
            // columns), keys from the stage: only the keys cross the
            // shared-memory port
            const uint64_t dk = sdesc_sw128(sK, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              umma_ts(dS, tmem + kTmemQ + 8 * k,
                      sdesc_advance(dk, (k >> 2) * kHalfKV + (k & 3) * 32), idesc_qk,
                      k > 0 ? 1u : 0u);
          }
          umma_commit(bar(kBarSFull + s));  // S ready, and the key stage free
          return true;
        };
        auto pv = [&](uint32_t tc, int j) -> bool {
          const int s = tc & 1;
          if (!mbar_wait(bar(kBarPReady + s), (tc >> 1) & 1, &s_abort)) return false;
          if (!mbar_wait(bar(kBarVReady + s), (tc >> 1) & 1, &s_abort)) return false;
          tc_fence_after();
          const uint64_t dv = sdesc_sw128(sb + C::kOffV + s * kOperand, kHalfKV, 1024);
          const uint32_t tP = tmem + kTmemS + 64 * s;
#pragma unroll
          for (int k = 0; k < kN / 16; ++k)
            umma_ts(tmem + kTmemO, tP + 8 * k, sdesc_advance(dv, k * 16 * 128), idesc_pv,
                    (j > 0 || k > 0) ? 1u : 0u);
          umma_commit(bar(kBarVEmpty + s));  // value stage free, O holds P V(j)
          return true;
        };
        if (ok && nt >= 1) ok = qk(tcount);
        if (ok && nt >= 2) ok = qk(tcount + 1);
        for (int j = 0; j < nt && ok; ++j) {
          const uint32_t tc = tcount + j;
          ok = pv(tc, j);
          if (ok && j + 1 == nt) umma_commit(bar(kBarODone));
          if (ok && j + 2 < nt) ok = qk(tc + 2);
        }
        if (!ok) {
          set_status(hdr, RPA_STATUS_TIMEOUT);
          s_abort = 1;
        }
      }
    });
    // every product this thread issued completes before tensor memory is
    // freed (an aborted unit can leave some in flight)
    if (lane == 0) {
      umma_commit(bar(kBarDrain));
      if (!mbar_drain(bar(kBarDrain), 0)) set_status(hdr, RPA_STATUS_TIMEOUT);
    }
  } else if (warp < 4) {
    if (FP8) {
      // warps 2 and 3: their shares of the fp8 decoding, tile by tile
      const int part = warp - 1;
      unit_loop([&](const Geom& g, const uint32_t tcount, const uint32_t) {
        bool ok = true;
        for (int j = 0; j < g.n_tiles && ok; ++j) {
          const uint32_t tc = tcount + j;
          const int s = tc & 1;
          for (int kv = 0; kv < 2 && ok; ++kv) {
            ok = mbar_wait_warp(bar((kv ? kBarVFull : kBarKFull) + s), (tc >> 1) & 1, &s_abort);
            if (!ok) break;
            decode_fp8(g, tc, j, kv, part);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar((kv ? kBarVReady : kBarKReady) + s));
          }
        }
        if (!ok && lane == 0) {
          set_status(hdr, RPA_STATUS_TIMEOUT);
          s_abort = 1;
        }
      });
    } else {
      // bf16 cache: warps 2 and 3 write this unit's new tokens into their
      // pages, half of them each, while the other roles run the unit (no
      // tile of this step reads those slots: the unit's new keys and values
      // come from the inputs, and the pool's tiles end at the step's
      // context).  An e4m3 cache had them written ahead of this kernel.
      unit_loop([&](const Geom& g, uint32_t, uint32_t) {
        const int n = g.t_end - g.t_begin, w = warp - 2;
        const int i0 = n * w / 2, i1 = n * (w + 1) / 2;
        write_tokens_kv<FP8, D, 4>(a.kv, g.seq, g.q0 + g.t_begin + i0, g.ctx + g.t_begin + i0,
                                   i1 - i0, g.h, lane);
      });
    }
  } else {
    unit_loop([&](const Geom& g, const uint32_t tcount, const uint32_t ucount) {
      const int nt = g.n_tiles;
      // ------------------------------------------------------- softmax
      const int q4 = warp & 3;                // tensor-memory lane quarter
      const int r = 32 * q4 + lane;           // row of the query tile
      const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
      const int ti = r / G;                   // token of the row, from t_begin
      const bool row_valid = g.t_begin + ti < g.t_end;
      const int i_tok = g.t_begin + min(ti, g.t_end - g.t_begin - 1);
      const int pos = g.ctx + i_tok;
      const int hq = g.h * G + r % G;
      const uint32_t tO = tmem + lane_off + kTmemO;
      if (!mbar_wait_warp(bar(kBarQFull), ucount & 1, &s_abort)) {
        if (lane == 0) {
          set_status(hdr, RPA_STATUS_TIMEOUT);
          s_abort = 1;
        }
        return;
      }
      if constexpr (!Q8) {
        // the query tile into tensor memory, the A operand of S: each thread
        // moves its own row (lane r of the tile), 64 elements (32 columns)
        // at a time; the previous unit's products are all done (its O was
        // read), so the columns are free
#pragma unroll 1
        for (int hf = 0; hf < C::kHalves; ++hf) {
          uint32_t qv[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v =
                *reinterpret_cast<const uint4*>(smem + C::kOffQ + hf * kHalfQ + sw128(r, c));
            qv[4 * c] = v.x;
            qv[4 * c + 1] = v.y;
            qv[4 * c + 2] = v.z;
            qv[4 * c + 3] = v.w;
          }
          tmem_st32p(tmem + lane_off + kTmemQ + 32 * hf, qv);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQReady));
      } else {
        // quantised queries: the four softmax warps turn the bf16 query tile
        // into its e4m3 code tile (q / q_scale rounded to e4m3) before the MMA
        // thread reads it
        constexpr int kChunks = D / 8;  // 8 elements per chunk
        for (int i = tid - 128; i < kM * kChunks; i += 128) {
          const int rr = i / kChunks, c = i % kChunks;
          const uint4 v = *reinterpret_cast<const uint4*>(smem + C::kOffQ + (c >> 3) * kHalfQ +
                                                          sw128(rr, c & 7));
          *reinterpret_cast<uint2*>(smem + C::kOffQ8 + (c >> 3) * C::kBlkQ + sw64_codes(rr, c)) =
              quantize8(v, p.q_scale);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQReady));
      }

      float m_run = a.sink ? a.sink[hq] * kLog2e : -INFINITY;
      float l_run = a.sink ? 1.f : 0.f;
      bool ok = true;
      for (int j = 0; j < nt; ++j) {
        const uint32_t tc = tcount + j;
        const int s = tc & 1;
        if (!mbar_wait_warp(bar(kBarSFull + s), (tc >> 1) & 1, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        bool is_new;
        int key0, valid;
        g.tile(j, is_new, key0, valid);
        const LogitXform xf =
            PH ? make_xform(p.softmax_scale,
                            qk_scale(p, p.k_scale_heads ? p.k_scale_heads[g.h] : p.k_scale),
                            p.logits_soft_cap)
               : xf0;
        const float sc = has_cap ? 1.f : xf.mul;  // raw score -> log2-domain logit
        const uint32_t tS = tmem + lane_off + kTmemS + 64 * s;
        uint32_t sr[kN];
        tmem_ld64(tS, sr);
        const bool full = valid == kN && key0 + kN - 1 <= pos && (W == 0 || pos - key0 < W);
        if (has_cap) {
#pragma unroll
          for (int c = 0; c < kN; ++c) sr[c] = __float_as_uint(xf(__uint_as_float(sr[c])));
        }
        if (!full) {
#pragma unroll
          for (int c = 0; c < kN; ++c) {
            const int jk = key0 + c;
            const bool okk = c < valid && jk <= pos && (W == 0 || pos - jk < W);
            if (!okk) sr[c] = __float_as_uint(-INFINITY);
          }
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kN; c += 2)
          mx[(c >> 1) & 3] =
              max3f(mx[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
        // lazy rescale: move the max only when it grows by more than 2^8
        const bool need = mt > m_run + (float)kRescaleLog2;
        float alpha = 1.f;
        if (need) {
          alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - mt);
          m_run = mt;
          l_run *= alpha;
        }
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // O holds P V of tiles < j once P V(j-1) is done: S(j) may have
          // completed before it, so wait for that product first
          if (!mbar_wait_warp(bar(kBarVEmpty + ((tc - 1) & 1)), ((tc - 1) >> 1) & 1, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 4
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t oc[16];
            tmem_ld16(tO + c0, oc);
#pragma unroll
            for (int c = 0; c < 16; ++c) oc[c] = __float_as_uint(__uint_as_float(oc[c]) * alpha);
            tmem_st16(tO + c0, oc);
          }
        }
        const float nm = m_run == -INFINITY ? 0.f : -m_run;
        const uint64_t sc2 = f2_pack(sc, sc), nm2 = f2_pack(nm, nm);
        // P packed as pairs into sr[0..kN/2): bf16, or fp16 with an e4m3 cache
        // (the values' type).  Scale-and-subtract uses packed f32x2
        // arithmetic, the exponentials the hardware ex2.
#pragma unroll
        for (int c = 0; c < kN; c += 2) {
          const uint64_t x2 =
              f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, nm2);
          float x0, x1;
          f2_unpack(x2, x0, x1);
          sr[c >> 1] = pack_p<FP8>(fast_exp2(x0), fast_exp2(x1));
        }
        tmem_st32p(tS, sr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPReady + s));
        // the row sum adds exactly the rounded weights just stored; it is
        // formed after P is handed over, off the tensor core's wait
        {
          float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < kN / 2; ++c)
            add_halves_f32<FP8>(rs[2 * (c & 1)], rs[2 * (c & 1) + 1], sr[c]);
          l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
        }
      }
      // epilogue: O / l -> bf16 rows
      if (ok && !mbar_wait_warp(bar(kBarODone), ucount & 1, &s_abort)) ok = false;
      if (ok) {
        tc_fence_after();
        const float inv = (PH ? v_scale_of(p, g.h) : p.v_scale) / l_run;
        __nv_bfloat16* dst = a.out + ((int64_t)(g.q0 + g.t_begin + ti) * p.num_q_heads + hq) * D;
#pragma unroll 2
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t oc[32];
          tmem_ld32(tO + c0, oc);
          if (row_valid) {
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(oc[c]) * inv, __uint_as_float(oc[c + 1]) * inv);
              v.y = pack_bf16(__uint_as_float(oc[c + 2]) * inv, __uint_as_float(oc[c + 3]) * inv);
              v.z = pack_bf16(__uint_as_float(oc[c + 4]) * inv, __uint_as_float(oc[c + 5]) * inv);
              v.w = pack_bf16(__uint_as_float(oc[c + 6]) * inv, __uint_as_float(oc[c + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + c0 + c) = v;
            }
          }
        }
      } else if (lane == 0) {
        set_status(hdr, RPA_STATUS_TIMEOUT);
        s_abort = 1;
      }
    });
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  griddep_wait();  // complete only after the decode kernel ahead
}

}  // namespace tcw

template <int D, bool FP8, bool PH, bool Q8>
static cudaError_t launch_wide_t(const AttnArgs& a, int max_units, int num_sms,
                                 cudaStream_t stream) {
  using C = tcw::Cfg<D, FP8, Q8>;
  static std::atomic<unsigned long long> attr_done{0};
  auto kern = tcw::prefill_tc_wide_kernel<D, FP8, PH, Q8>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemBytes, &attr_done);
  if (e != cudaSuccess) return e;
  const rpa_params_t& p = a.kv.p;
  const int G = p.num_q_heads / p.num_kv_heads;
  tcw::Maps maps{};
  const uint64_t T = (uint64_t)(p.total_tokens > 0 ? p.total_tokens : 1);
  const uint64_t rows = (uint64_t)p.num_pages * p.page_size;
  const uint32_t prow = p.page_size < tcw::kN ? (uint32_t)p.page_size : (uint32_t)tcw::kN;
  bool ok = encode_map_3d(&maps.q, a.queries, 2, D, (uint64_t)p.num_q_heads, T, 64u, (uint32_t)G,
                          (uint32_t)(tcw::kM / G), true) &&
            encode_map_3d(&maps.cache, a.kv.cache, FP8 ? 1 : 2, D, 2 * (uint64_t)p.num_kv_heads,
                          rows, FP8 ? (uint32_t)D : 64u, 1u, prow, !FP8) &&
            encode_map_3d(&maps.knew, a.kv.keys, 2, D, (uint64_t)p.num_kv_heads, T, 64u, 1u,
                          (uint32_t)tcw::kN, true) &&
            encode_map_3d(&maps.vnew, a.kv.values, 2, D, (uint64_t)p.num_kv_heads, T, 64u, 1u,
                          (uint32_t)tcw::kN, true) &&
            (!Q8 || encode_map_3d_swizzle(&maps.cache8, a.kv.cache, 1, D,
                                          2 * (uint64_t)p.num_kv_heads, rows, 64u, 1u, prow, 64));
  if (!ok) return cudaErrorInvalidValue;
  int grid = num_sms;
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;
  return launch_dependent(kern, grid, tcw::kThreads, C::kSmemBytes, stream, maps, a);
}

template <int D>
static cudaError_t launch_wide_d(const AttnArgs& a, int max_units, int num_sms,
                                 cudaStream_t stream) {
  const rpa_params_t& p = a.kv.p;
  if (p.kv_dtype != RPA_KV_FP8_E4M3)
    return launch_wide_t<D, false, false, false>(a, max_units, num_sms, stream);
  // quantised queries (an e4m3 cache only) run Q K^T on the codes
  const bool ph = p.k_scale_heads != nullptr || p.v_scale_heads != nullptr;
  if (p.q_scale > 0.f)
    return ph ? launch_wide_t<D, true, true, true>(a, max_units, num_sms, stream)
              : launch_wide_t<D, true, false, true>(a, max_units, num_sms, stream);
  return ph ? launch_wide_t<D, true, true, false>(a, max_units, num_sms, stream)
            : launch_wide_t<D, true, false, false>(a, max_units, num_sms, stream);
}

cudaError_t launch_prefill_tc_wide(const AttnArgs& a, int max_units, int num_sms,
                                   cudaStream_t stream) {
  return a.kv.p.head_dim == 192 ? launch_wide_d<192>(a, max_units, num_sms, stream)
                                : launch_wide_d<256>(a, max_units, num_sms, stream);
}

}  // namespace rpa
