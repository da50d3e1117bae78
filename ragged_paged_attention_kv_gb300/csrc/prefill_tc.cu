// Prefill / chunked-prefill path on the 5th-generation tensor cores.
//
// Work unit = (sequence, run of new tokens, kv head) of 256 rows: two tiles
// A and B of 128 (token, q-head of the GQA group) rows each, token-major (row
// R is token t_begin + R / G, q-head h*G + R % G), as tpu-inference RPA v3
// kernel.py stacks a q block's heads of one kv head, so every key/value tile
// serves all G heads of both tiles.  Per 128-key tile j and each of A, B:
//   S = Q K^T      tcgen05.mma, A operand = the tile's queries and B operand
//                  = the keys, from 128-byte swizzled shared memory; fp32
//                  accumulator in tensor memory;
//   P = softmax    one thread per row (a warpgroup per tile) reads S from
//                  tensor memory, applies scale / soft cap / causal + window
//                  mask, keeps the running max m and sum l in fp32 (RPA v3
//                  flash_attention_step1_qk_softmax), and writes P as bf16
//                  back over S;
//   O += P V       tcgen05.mma with A operand = P from tensor memory and B =
//                  the values (RPA v3 flash_attention_step2_pv); O stays in
//                  tensor memory and is rescaled there only when a row's max
//                  grows by more than 2^8.
// The RPA v3 kernel overlaps step2 of one kv head with step1 of the next.
// Here the two tiles play that part: the MMA thread issues PV_A(j), S_A(j+1),
// PV_B(j), S_B(j+1), so the tensor core works on one tile while the other
// tile's warpgroup computes its softmax (the ping-pong FlashAttention-4 uses
// on Blackwell).  A TMA warp feeds two-stage key and value rings; the keys
// and values of a tile are fetched once for both query tiles.
//
// Keys come in two kinds of tiles: cached keys [lo, ctx) are fetched page by
// page from the pool (one TMA box per page and 64-wide half of head_dim);
// the step's new keys [ctx, ...) are fetched from the keys/values inputs (RPA
// v3 _fetch_bkv does the same), in tiles aligned to ctx.  Value rows outside
// a tile's valid range are zeroed before the PV product.  The unit's own new
// tokens are written into their pages by the softmax warps.
//
// With an e4m3 cache the step's new tokens are quantised into their pages
// once, by a small kernel ahead of this one, and every key and value tile
// comes from the pool as codes (a tile of new tokens is read by many units:
// each would otherwise quantise it again); the codes are decoded into the
// MMA operands.  With quantised queries as well (q_scale, the w8a8 mode of
// the ragged_paged_attention_v3 signature) S = Q K^T runs on the codes
// themselves (tcgen05.mma kind::f8f6f4): the query tiles are quantised once
// per unit, cached keys go from the page straight into the key stage, and
// the logit scale carries q_scale * k_scale.
#include "async.cuh"
#include "common.cuh"
#include "kv_write.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma_host.h"

namespace rpa {
namespace tc {

// warpgroup 0: warp 0 TMA (+ fp8 decoding), warp 1 MMA, warps 2-3 fp8 decoding
// (idle for bf16 caches);
// warpgroups 1 and 2: softmax of query tiles A and B
constexpr int kThreads = 384;
constexpr int kM = 128;         // rows per query tile (two per unit)
constexpr int kN = 128;         // keys per tile
constexpr uint32_t kHalf = 128 * 128;          // [128 rows][64 bf16], 16 KB
constexpr uint32_t kTmemCols = 512;            // O_A, O_B, S_A, S_B: 128 columns each
constexpr uint32_t kTmemO = 0, kTmemS = 256;   // tile X: O at kTmemO + 128X, S at kTmemS + 128X
constexpr int kRescaleLog2 = 8;
// registers per thread after the split: the launch gives 384 x 168; the
// TMA/MMA warpgroup drops to 56 and the softmax warpgroups take 224 (no
// role spills at this split)
constexpr int kRegsControl = 56, kRegsSoftmax = 224;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= 384 * 168, "register split");

// Shared-memory layout for head_dim D (64 or 128) and cache type.  Operands
// are [128 rows][D] bf16 in 128-byte swizzled halves of 64 columns: query
// tiles A and B, then two key and two value stages.  An fp8 cache adds
// staging buffers that receive the pages' e4m3 codes ([128 rows][D] bytes)
// before they are decoded into the bf16 operands: one per stage and operand
// where they fit, else one per operand (head_dim 128).
// With quantised queries (Q8) the Q K^T product runs on the e4m3 codes
// themselves: the query tiles become code tiles [128 rows][D bytes] (rows
// swizzled over 128 bytes at head_dim 128, 64 at head_dim 64), the key stages
// are code tiles too (the pages' codes land there as they are), and only the
// values have staging buffers.
template <int D, bool FP8, bool Q8 = false>
struct TcCfg {
  static_assert(!Q8 || FP8, "quantised queries need an e4m3 cache");
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kOperand = kHalves * kHalf;
  static constexpr uint32_t kStaging = FP8 ? 128u * D : 0u;
  static constexpr uint32_t kTile8 = 128u * D;                    // one e4m3 code tile
  static constexpr uint32_t kKStage = Q8 ? kTile8 : kOperand;     // key stage stride
  static constexpr int kStgOps = Q8 ? 1 : 2;                      // operands with staging
  static constexpr uint32_t kFixed = 4 * kOperand + 2 * kKStage + (Q8 ? 2 * kTile8 : 0);
  static constexpr uint32_t bytes_for(int stg) {
    return (kFixed + kStgOps * stg * kStaging + 1023) / 1024 * 1024 + 256 + 1024;
  }
  static constexpr int kStgPerOp = !FP8 ? 0 : (bytes_for(2) <= 227 * 1024 ? 2 : 1);
  static constexpr uint32_t kOffQ = 0;                  // query tile X at kOffQ + X*kOperand
  static constexpr uint32_t kOffQ8 = 2 * kOperand;      // Q8: code tile X at kOffQ8 + X*kTile8
  static constexpr uint32_t kOffK = 2 * kOperand + (Q8 ? 2 * kTile8 : 0);  // + s*kKStage
  static constexpr uint32_t kOffV = kOffK + 2 * kKStage;                   // + s*kOperand
  static constexpr uint32_t kOffStg = kOffV + 2 * kOperand;
  static constexpr uint32_t kOffBar =
      (kOffStg + kStgOps * kStgPerOp * kStaging + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = (int)kOffBar + 256 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "fits one CTA's shared memory");
  static_assert(!Q8 || kStgPerOp == 2, "Q8: a value staging buffer per stage");
};

// Byte offset of the codes of elements 8*c8 .. 8*c8+7 of row r in an e4m3
// code tile [128 rows][D bytes], in the swizzle the tensor map writes and
// the MMA descriptor reads: 16-byte chunk (c8/2) of the row XOR-ed with
// address bits 7-9 (128-byte swizzle, head_dim 128) or 7-8 (64-byte
// swizzle, head_dim 64).
template <int D>
__device__ __forceinline__ uint32_t sw_e4m3(int r, int c8) {
  static_assert(D == 64 || D == 128, "code tiles for head_dim 64 and 128");
  const uint32_t phase = D == 128 ? (uint32_t)(r & 7) : (uint32_t)((r >> 1) & 3);
  return (uint32_t)r * D + ((((uint32_t)c8 >> 1) ^ phase) << 4) + ((uint32_t)(c8 & 1) << 3);
}

enum Bar {
  kBarQFull = 0,    // both query tiles landed
  kBarKFull = 1,    // [2] key TMA landed
  kBarKEmpty = 3,   // [2] key stage free (S products of both tiles done)
  kBarVFull = 5,    // [2] value TMA landed
  kBarVReady = 7,   // [2] values fixed up / decoded, MMA may read
  kBarVEmpty = 9,   // [2] value stage free (PV products of both tiles done)
  kBarKReady = 11,  // [2] fp8 cache: keys decoded, MMA may read
  kBarSFull = 13,   // [2] per query tile: S computed
  kBarPReady = 15,  // [2] per query tile: P written (and O corrected)
  kBarODone = 17,   // [2] per query tile: the unit's last PV product done
  kBarDrain = 19,   // once, at exit: every tcgen05 product the MMA thread issued is done
  kBarQReady = 20,  // quantised queries (q_scale): the softmax warps converted the tiles
  kNumBars = 21,
};

struct TcMaps {
  CUtensorMap q;      // queries [T][Hq][D], box {64, G, 128/G}
  CUtensorMap cache;  // pool [num_pages*P][2*Hkv][D], box {64, 1, min(P,128)} (fp8: {D, 1, ..})
  CUtensorMap knew;   // keys [T][Hkv][D], box {64, 1, 128}
  CUtensorMap vnew;   // values [T][Hkv][D], box {64, 1, 128}
  CUtensorMap cache8; // Q8 only: the pool's codes, box {D, 1, min(P,128)}, swizzled as sw_e4m3
};

// Geometry of one unit, computed identically by every role.  Keys
// [c_start, k_end) come from the pool in 128-key tiles aligned to 128 (k_end
// = ctx, or with an e4m3 cache the unit's last position + 1: the step's new
// tokens are already in their pages), the rest from the keys/values inputs in
// tiles aligned to ctx.
struct UnitGeom {
  int seq, h, q0, q_len, kv_len, ctx, t_begin, t_end;
  int lo;              // first key any row of the tile may see
  int c_start, k_end, n_cached, i0, n_tiles;
  // rows of a tile starting at key0 that lie before every row's window
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
__device__ __forceinline__ UnitGeom unit_geom(const AttnArgs& a, const PrefillUnit& pu) {
  UnitGeom g;
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
    prefill_tc_kernel(const __grid_constant__ TcMaps maps, AttnArgs a) {
  using C = TcCfg<D, FP8, Q8>;
  // warps that decode fp8 operands: the TMA warp and warps 2, 3
  constexpr int kDecWarps = FP8 ? 3 : 1;
  constexpr uint32_t kOperand = C::kOperand, kOffQ = C::kOffQ, kOffK = C::kOffK,
                     kOffV = C::kOffV, kOffBar = C::kOffBar;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + kOffBar;
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
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVReady + s), FP8 ? kDecWarps : 1);
      mbar_init(bar(kBarVEmpty + s), 1);
      mbar_init(bar(kBarKReady + s), kDecWarps);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarPReady + s), 4);
      mbar_init(bar(kBarODone + s), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarQReady), 8);
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
  // the logit transform of the scalar key scale (used unless per-head scales)
  const LogitXform xf0 = make_xform(p.softmax_scale, qk_scale(p, p.k_scale), p.logits_soft_cap);

  // Every role runs this loop over the CTA's units with its own body, so
  // the code of each role stays within its register budget; all threads meet
  // at the same two barriers per unit.  The counters (all roles agree) give
  // the mbarrier phases: tcount counts the key tiles and ucount the units
  // the CTA has processed so far, for the barriers every unit uses; tcount_b
  // and ucount_b count only the units with a query tile B, for tile B's
  // own barriers (S full, P ready, O done), which other units leave alone.
  // fp8 cache: the staging buffer of an operand of tile tc, and the decoding
  // of a landed operand of tile j into its stage, shared by kDecWarps warps
  // (part 0..kDecWarps-1).  Every tile of an e4m3 unit comes from the pages
  // (the step's new tokens were written there ahead of this kernel): keys
  // are decoded to bf16 (the queries' type), values to fp16 (exact for e4m3,
  // so that the P V product carries P in fp16).  Value rows no row of the
  // unit may see (past the valid range, or before the window) become zero;
  // key rows there are masked by the softmax.  With Q8 only the values are
  // staged and decoded; the keys land as codes in their stage.
  auto staging = [&](uint32_t tc, int kv) -> uint32_t {
    return C::kOffStg +
           (C::kStgOps * (C::kStgPerOp == 2 ? (tc & 1) : 0) + (Q8 ? 0 : kv)) * C::kStaging;
  };
  auto decode_fp8 = [&](const UnitGeom& g, uint32_t tc, int j, int kv, int part) {
    if (Q8 && kv == 0) return;
    bool is_new;
    int key0, valid;
    g.tile(j, is_new, key0, valid);
    uint8_t* op = smem + (kv ? kOffV : kOffK) + (tc & 1) * (kv ? kOperand : C::kKStage);
    const uint8_t* stg = smem + staging(tc, kv);
    const int rows = kv ? kN : valid;
    const int lead = kv ? g.lead(key0) : 0;
    for (int idx = 32 * part + lane; idx < rows * (D / 8); idx += 32 * kDecWarps) {
      const int r = idx / (D / 8), c = idx % (D / 8);
      uint4* dst = reinterpret_cast<uint4*>(op + (c >> 3) * kHalf + sw128(r, c & 7));
      if (r >= valid || r < lead) {
        *dst = make_uint4(0, 0, 0, 0);
      } else {
        const uint2 codes = *reinterpret_cast<const uint2*>(stg + r * D + c * 8);
        *dst = kv ? dequant8_f16(codes) : dequant8(codes);
      }
    }
  };

  struct Counts {
    uint32_t tcount, ucount, tcount_b, ucount_b;
    // phase counters of query tile x's own barriers
    __device__ uint32_t tiles(int x) const { return x ? tcount_b : tcount; }
    __device__ uint32_t units(int x) const { return x ? ucount_b : ucount; }
  };
  auto unit_loop = [&](auto&& body) {
    Counts n{0, 0, 0, 0};
    for (;;) {
      if (tid == 0) s_unit = atomicAdd(hdr + kHdrPrefillNext, 1);
      __syncthreads();
      const int u = s_unit;
      if (u >= n_units || s_abort) break;
      const UnitGeom g = unit_geom<FP8>(a, units[u]);
      body(g, n);
      n.tcount += g.n_tiles;
      n.ucount += 1;
      if (g.t_begin + kM / G < g.t_end) {  // the unit has a query tile B
        n.tcount_b += g.n_tiles;
        n.ucount_b += 1;
      }
      tc_fence_before();
      __syncthreads();  // the next unit reuses Q, the stages and tensor memory
      tc_fence_after();
    }
  };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0) {
      // the last query copy (unit count) and the last key / value copy (tile
      // count) per stage this warp issued, for the drain at exit
      int q_last = -1, k_last0 = -1, k_last1 = -1, v_last0 = -1, v_last1 = -1;
      unit_loop([&](const UnitGeom& g, const Counts& n) {
      const uint32_t tcount = n.tcount, ucount = n.ucount;
      const int nt = g.n_tiles;
      // ------------------------------------------------------- TMA producer
      // Keys of tile j go into key stage j%2 once both S products of tile
      // j-2 are done; values into value stage j%2 once both PV products of
      // tile j-2 are done; after the values of a tile land, rows outside its
      // valid range are zeroed.
      if (RPA_TEST_STALL_QUERY == 0) {
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(kBarQFull), 2 * kOperand);
          for (int x = 0; x < 2; ++x)
            for (int hf = 0; hf < C::kHalves; ++hf)
              tma_load_3d(sb + kOffQ + x * kOperand + hf * kHalf, &maps.q, bar(kBarQFull),
                          hf * 64, g.h * G, g.q0 + g.t_begin + x * (kM / G));
        }
        q_last = (int)ucount;
      }
      // Page ids of a cached tile: lane l holds page pg0 + l (a tile spans at
      // most 128/P + 1 <= 17 pages for P >= 8), loaded one tile ahead so the
      // block-table reads overlap the wait for a free stage.
      const int64_t bt_row = (int64_t)g.seq * p.pages_per_seq;
      auto load_ids = [&](int j) -> int {
        bool is_new;
        int key0, valid;
        g.tile(j, is_new, key0, valid);
        if (is_new) return 0;
        const int pg0 = key0 / P, npg = (key0 + valid - 1) / P - pg0 + 1;
        return lane < npg ? __ldg(a.kv.block_tables + bt_row + pg0 + lane) : 0;
      };
      // issue the boxes of one operand (kv = 0 keys, 1 values) of tile j; each
      // lane copies its own page.  New tokens come as bf16 straight into the
      // operand stage; cached pages too for a bf16 cache, or as e4m3 codes
      // into the staging buffer for an fp8 cache.
      auto issue = [&](int j, int kv, uint32_t tc, int page) {
        const uint32_t s = tc & 1;
        bool is_new;
        int key0, valid;
        g.tile(j, is_new, key0, valid);
        const uint32_t dst = sb + (kv ? kOffV + s * kOperand : kOffK + s * C::kKStage);
        const uint32_t fullbar = bar((kv ? kBarVFull : kBarKFull) + s);
        if (is_new) {
          if (lane == 0) {
            mbar_arrive_expect_tx(fullbar, kOperand);
            const int row = g.q0 + (key0 - g.ctx);
            for (int hf = 0; hf < C::kHalves; ++hf)
              tma_load_3d(dst + hf * kHalf, kv ? &maps.vnew : &maps.knew, fullbar, hf * 64, g.h,
                          row);
          }
        } else {
          const int rows = P < kN ? P : kN;
          const int pg0 = key0 / P, npg = (key0 + valid - 1) / P - pg0 + 1;
          if (lane == 0) mbar_arrive_expect_tx(fullbar, (uint32_t)(npg * rows * D * 2 / (FP8 ? 2 : 1)));
          __syncwarp();
          if (lane < npg) {
            if (page < 0 || page >= p.num_pages) {
              set_status(hdr, RPA_STATUS_BAD_PAGE);
              page = 0;
            }
            const int srow = P < kN ? (pg0 + lane) * P - key0 : 0;
            const int z = page * P + (P < kN ? 0 : key0 % P);
            if (Q8 && kv == 0) {
              tma_load_3d(dst + srow * D, &maps.cache8, fullbar, 0, 2 * g.h, z);
            } else if (FP8) {
              tma_load_3d(sb + staging(tc, kv) + srow * D, &maps.cache, fullbar, 0, 2 * g.h + kv, z);
            } else {
              for (int hf = 0; hf < C::kHalves; ++hf)
                tma_load_3d(dst + hf * kHalf + srow * 128, &maps.cache, fullbar, hf * 64,
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
            uint8_t* v = smem + kOffV + s * kOperand;
            constexpr int kRowChunks = 8 * C::kHalves;
            const int tail = kN - valid;
            for (int idx = lane; idx < (lead + tail) * kRowChunks; idx += 32) {
              const int i = idx / kRowChunks, c = idx % kRowChunks;
              const int r = i < lead ? i : valid + (i - lead);
              *reinterpret_cast<uint4*>(v + (c >> 3) * kHalf + r * 128 + (c & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarVReady + s));
        return true;
      };
      // Per tile j: keys of j, then (fp8) decode keys of j-1, values of j,
      // then values of j-1 -- in this order no role waits on another in a
      // cycle (the MMA needs keys of j+1 before the values of j are used by
      // the second query tile).  With one staging buffer per operand the
      // codes of tile j-1 are decoded before those of tile j are fetched.
      constexpr bool kStg1 = FP8 && C::kStgPerOp == 1;
      bool ok = true;
      int ids_next = load_ids(0);
      for (int j = 0; j < nt && ok; ++j) {
        const uint32_t tc = tcount + j;
        const int s = tc & 1;
        const uint32_t par = ((tc >> 1) & 1) ^ 1;
        const int ids = ids_next;
        if (j + 1 < nt) ids_next = load_ids(j + 1);
        if (kStg1 && j >= 1) {
          // the single staging buffer is refilled once every decoding warp
          // is done with tile j-1's codes
          ok = finalize_k(tc - 1, j - 1) &&
               mbar_wait_warp(bar(kBarKReady + ((tc - 1) & 1)), ((tc - 1) >> 1) & 1, &s_abort);
          if (!ok) break;
        }
        if (!mbar_wait_warp(bar(kBarKEmpty + s), par, &s_abort)) {
          ok = false;
          break;
        }
        issue(j, 0, tc, ids);
        (s ? k_last1 : k_last0) = (int)tc;
        if (FP8 && !kStg1 && j >= 1) {
          ok = finalize_k(tc - 1, j - 1);
          if (!ok) break;
        }
        if (kStg1 && j >= 1) {
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
        if (!kStg1 && j >= 1) ok = finalize_v(tc - 1, j - 1);
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
      unit_loop([&](const UnitGeom& g, const Counts& n) {
      const uint32_t tcount = n.tcount, ucount = n.ucount;
      const int nt = g.n_tiles;
      const bool has_b = g.t_begin + kM / G < g.t_end;
      // ------------------------------------------------------------ MMA
      // Order: S_A(0), S_B(0), then for each tile j: PV_A(j), S_A(j+1),
      // PV_B(j), S_B(j+1).  S_X(j+1) overwrites P_X(j) only after PV_X(j)
      // has read it (the tensor core runs one thread's products in order),
      // and its completion also tells the softmax of tile X that PV_X(j) is
      // done, so O_X may be rescaled.
      if (lane == 0) {
        bool ok = mbar_wait_poll(bar(Q8 ? kBarQReady : kBarQFull), ucount & 1, &s_abort);
        tc_fence_after();
        auto qk = [&](uint32_t tc, int x, bool last_of_stage) -> bool {
          const int s = tc & 1;
          if (x == 0) {
            if (!mbar_wait_poll(bar((FP8 ? kBarKReady : kBarKFull) + s), (tc >> 1) & 1,
                                &s_abort))
              return false;
            tc_fence_after();
          }
          const uint32_t sK = sb + kOffK + s * C::kKStage, dS = tmem + kTmemS + 128 * x;
          // one thread issues every product: its descriptors are the tiles'
          // (built once here) advanced by constants, so the issue keeps pace
          // with the tensor core
          if constexpr (Q8) {
            // e4m3 codes, 32 per product along the row (rows of D bytes)
            const uint32_t sQ = sb + C::kOffQ8 + x * C::kTile8;
            const uint64_t dq = D == 128 ? sdesc_sw128(sQ, 16, 1024) : sdesc_sw64(sQ, 16, 512);
            const uint64_t dk = D == 128 ? sdesc_sw128(sK, 16, 1024) : sdesc_sw64(sK, 16, 512);
#pragma unroll
            for (int k = 0; k < D / 32; ++k)
              umma_ss_e4m3(dS, sdesc_advance(dq, 32 * k), sdesc_advance(dk, 32 * k), idesc_qk,
                           k > 0 ? 1u : 0u);
          } else {
            const uint64_t dq = sdesc_sw128(sb + kOffQ + x * kOperand, 16, 1024),
                           dk = sdesc_sw128(sK, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
              umma_ss(dS, sdesc_advance(dq, off), sdesc_advance(dk, off), idesc_qk,
                      k > 0 ? 1u : 0u);
            }
          }
          umma_commit(bar(kBarSFull + x));
          if (last_of_stage) umma_commit(bar(kBarKEmpty + s));
          return true;
        };
        auto pv = [&](uint32_t tc, int j, int x, bool last_of_stage) -> bool {
          const int s = tc & 1;
          if (!mbar_wait_poll(bar(kBarPReady + x), (n.tiles(x) + j) & 1, &s_abort)) return false;
          if (x == 0 && !mbar_wait_poll(bar(kBarVReady + s), (tc >> 1) & 1, &s_abort))
            return false;
          tc_fence_after();
          const uint64_t dv = sdesc_sw128(sb + kOffV + s * kOperand, kHalf, 1024);
          const uint32_t tO = tmem + kTmemO + 128 * x, tP = tmem + kTmemS + 128 * x;
#pragma unroll
          for (int k = 0; k < kN / 16; ++k)
            umma_ts(tO, tP + 8 * k, sdesc_advance(dv, k * 16 * 128), idesc_pv,
                    (j > 0 || k > 0) ? 1u : 0u);
          if (last_of_stage) umma_commit(bar(kBarVEmpty + s));
          return true;
        };
        if (ok && nt >= 1) ok = qk(tcount, 0, !has_b);
        if (ok && nt >= 1 && has_b) ok = qk(tcount, 1, true);
        for (int j = 0; j < nt && ok; ++j) {
          const uint32_t tc = tcount + j;
          ok = pv(tc, j, 0, !has_b);
          if (ok && j + 1 == nt) umma_commit(bar(kBarODone + 0));
          if (ok && j + 1 < nt) ok = qk(tc + 1, 0, !has_b);
          if (ok && has_b) {
            ok = pv(tc, j, 1, true);
            if (ok && j + 1 == nt) umma_commit(bar(kBarODone + 1));
            if (ok && j + 1 < nt) ok = qk(tc + 1, 1, true);
          }
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
    } else {
      if (FP8) {
        // warps 2 and 3: their shares of the fp8 decoding, tile by tile
        const int part = warp - 1;
        unit_loop([&](const UnitGeom& g, const Counts& n) {
          const uint32_t tcount = n.tcount;
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
        unit_loop([](const UnitGeom&, const Counts&) {});
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    unit_loop([&](const UnitGeom& g, const Counts& n) {
    const uint32_t ucount = n.ucount;
    const int nt = g.n_tiles;
    // tile B holds tokens t_begin + 128/G onwards; it may be empty
    const bool has_b = g.t_begin + kM / G < g.t_end;
    bool q_ok = true;
    if constexpr (Q8) {
      // quantised queries: all eight softmax warps turn both bf16 query
      // tiles into e4m3 code tiles (q / q_scale rounded to e4m3) before the
      // MMA thread reads them
      q_ok = mbar_wait_warp(bar(kBarQFull), ucount & 1, &s_abort);
      if (q_ok) {
        constexpr int kChunks = D / 8;  // 8 elements per chunk
        for (int i = tid - 128; i < 2 * kM * kChunks; i += 256) {
          const int x = i / (kM * kChunks), r = (i / kChunks) % kM, c = i % kChunks;
          const uint4 v = *reinterpret_cast<const uint4*>(smem + kOffQ + x * kOperand +
                                                          (c >> 3) * kHalf + sw128(r, c & 7));
          *reinterpret_cast<uint2*>(smem + C::kOffQ8 + x * C::kTile8 + sw_e4m3<D>(r, c)) =
              quantize8(v, p.q_scale);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQReady));
      } else if (lane == 0) {
        set_status(hdr, RPA_STATUS_TIMEOUT);
        s_abort = 1;
      }
    }
    if (q_ok && (warp < 8 || has_b)) {
      // ---------------------------------------------- softmax of tile x
      const int x = (warp - 4) >> 2;           // query tile of this warpgroup
      const int q4 = warp & 3;                 // tensor-memory lane quarter
      const int r = 32 * q4 + lane;            // row of the tile
      const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
      const int ti = (kM * x + r) / G;         // token of the row, from t_begin
      const bool row_valid = g.t_begin + ti < g.t_end;
      const int i_tok = g.t_begin + min(ti, g.t_end - g.t_begin - 1);
      const int pos = g.ctx + i_tok;
      const int hq = g.h * G + r % G;
      const uint32_t tS = tmem + lane_off + kTmemS + 128 * x;
      const uint32_t tO = tmem + lane_off + kTmemO + 128 * x;

      // this unit's new tokens -> their pages (an eighth of them per warp, a
      // quarter when tile B is empty); the loads are batched, so the write
      // fits in the time the first S tile of the unit takes to arrive.  An
      // e4m3 cache had its new tokens written ahead of this kernel.
      if constexpr (!FP8) {
        const int n = g.t_end - g.t_begin, nw = has_b ? 8 : 4, w = warp - 4;
        const int i0 = n * w / nw, i1 = n * (w + 1) / nw;
        write_tokens_kv<FP8, D, 4>(a.kv, g.seq, g.q0 + g.t_begin + i0, g.ctx + g.t_begin + i0,
                                   i1 - i0, g.h, lane);
      }

      float m_run = a.sink ? a.sink[hq] * kLog2e : -INFINITY;
      float l_run = a.sink ? 1.f : 0.f;
      bool ok = true;
      for (int j = 0; j < nt; ++j) {
        if (!mbar_wait_warp(bar(kBarSFull + x), (n.tiles(x) + j) & 1, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        bool is_new;
        int key0, valid;
        g.tile(j, is_new, key0, valid);
        // with per-head scales the logit transform is formed per tile from a
        // plain load of this head's scale (reissued after every barrier wait)
        // rather than held in registers across the tile loop
        const LogitXform xf =
            PH ? make_xform(p.softmax_scale,
                            qk_scale(p, p.k_scale_heads ? p.k_scale_heads[g.h] : p.k_scale),
                            p.logits_soft_cap)
               : xf0;
        const float sc = has_cap ? 1.f : xf.mul;  // raw score -> log2-domain logit
        uint32_t sr[128];
        tmem_ld128(tS, sr);
        // logits in the log2 domain are fma(s, sc, -m): with a soft cap the
        // capped logit is formed first and sc is 1
        uint32_t dead = 0;  // (e4m3 caches) bit k: chunk k masked for every row of the warp
        if constexpr (!FP8) {
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
        } else {
          // e4m3 caches (compiled there only: in the bf16 kernels this path
          // cost long-prefill throughput).  A tile that crosses a mask edge is
          // taken in chunks of 16 keys: the rows of one warp are at most a few
          // tokens apart, so a chunk is usually masked (or kept) whole for all
          // of them -- a wholly masked chunk skips the cap and the mask (and,
          // below, the exponentials), a wholly kept one the mask.  Whether the
          // tile needs masking at all is decided for the whole warp (the rows'
          // positions differ), so the warp collectives run in warp-uniform
          // control flow.
          const bool full = __all_sync(0xffffffffu, valid == kN && key0 + kN - 1 <= pos &&
                                                        (W == 0 || pos - key0 < W));
          if (full) {
            if (has_cap) {
#pragma unroll
              for (int c = 0; c < kN; ++c) sr[c] = __float_as_uint(xf(__uint_as_float(sr[c])));
            }
          } else {
#pragma unroll
            for (int k = 0; k < kN / 16; ++k) {
              const int c0 = 16 * k, j0 = key0 + c0, j1 = j0 + 15;
              const bool row_dead = c0 >= valid || j0 > pos || (W > 0 && pos - j1 >= W);
              const bool row_live = c0 + 15 < valid && j1 <= pos && (W == 0 || pos - j0 < W);
              if (__all_sync(0xffffffffu, row_dead)) {
                dead |= 1u << k;
#pragma unroll
                for (int c = c0; c < c0 + 16; ++c) sr[c] = __float_as_uint(-INFINITY);
              } else {
                if (has_cap) {
#pragma unroll
                  for (int c = c0; c < c0 + 16; ++c)
                    sr[c] = __float_as_uint(xf(__uint_as_float(sr[c])));
                }
                if (!__all_sync(0xffffffffu, row_live)) {
#pragma unroll
                  for (int c = c0; c < c0 + 16; ++c) {
                    const int jk = key0 + c;
                    const bool okk = c < valid && jk <= pos && (W == 0 || pos - jk < W);
                    if (!okk) sr[c] = __float_as_uint(-INFINITY);
                  }
                }
              }
            }
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
          // O holds P V of every earlier tile: S_X(j) completed after PV_X(j-1)
          // in chunks of 16 columns: the S tile is live in registers meanwhile
#pragma unroll
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
        if (!FP8 || dead == 0) {
#pragma unroll
          for (int c = 0; c < kN; c += 2) {
            const uint64_t x2 =
                f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, nm2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            sr[c >> 1] = pack_p<FP8>(fast_exp2(x0), fast_exp2(x1));
          }
        } else {
#pragma unroll
          for (int k = 0; k < kN / 16; ++k) {
            if (dead & (1u << k)) {
#pragma unroll
              for (int c = 16 * k; c < 16 * k + 16; c += 2) sr[c >> 1] = 0u;  // P = 0
            } else {
#pragma unroll
              for (int c = 16 * k; c < 16 * k + 16; c += 2) {
                const uint64_t x2 =
                    f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, nm2);
                float x0, x1;
                f2_unpack(x2, x0, x1);
                sr[c >> 1] = pack_p<FP8>(fast_exp2(x0), fast_exp2(x1));
              }
            }
          }
        }
        tmem_st64p(tS, sr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPReady + x));
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
      if (ok && !mbar_wait_warp(bar(kBarODone + x), n.units(x) & 1, &s_abort)) ok = false;
      if (ok) {
        tc_fence_after();
        const float inv = (PH ? v_scale_of(p, g.h) : p.v_scale) / l_run;
        __nv_bfloat16* dst = a.out + ((int64_t)(g.q0 + g.t_begin + ti) * p.num_q_heads + hq) * D;
#pragma unroll
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
    }
    });
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  griddep_wait();  // complete only after the decode kernel ahead
}

}  // namespace tc

template <int D, bool FP8, bool PH, bool Q8>
static cudaError_t launch_prefill_tc_t(const AttnArgs& a, int max_units, int num_sms,
                                       cudaStream_t stream) {
  using C = tc::TcCfg<D, FP8, Q8>;
  static std::atomic<unsigned long long> attr_done{0};
  auto kern = tc::prefill_tc_kernel<D, FP8, PH, Q8>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemBytes, &attr_done);
  if (e != cudaSuccess) return e;
  const rpa_params_t& p = a.kv.p;
  const int G = p.num_q_heads / p.num_kv_heads;
  tc::TcMaps maps{};
  const uint64_t T = (uint64_t)(p.total_tokens > 0 ? p.total_tokens : 1);
  const uint64_t rows = (uint64_t)p.num_pages * p.page_size;
  const uint32_t prow = p.page_size < tc::kN ? (uint32_t)p.page_size : (uint32_t)tc::kN;
  bool ok = encode_map_3d(&maps.q, a.queries, 2, D, (uint64_t)p.num_q_heads, T, 64u, (uint32_t)G,
                          (uint32_t)(tc::kM / G), true) &&
            encode_map_3d(&maps.cache, a.kv.cache, FP8 ? 1 : 2, D, 2 * (uint64_t)p.num_kv_heads,
                          rows, FP8 ? (uint32_t)D : 64u, 1u, prow, !FP8) &&
            encode_map_3d(&maps.knew, a.kv.keys, 2, D, (uint64_t)p.num_kv_heads, T, 64u, 1u, 128u,
                          true) &&
            encode_map_3d(&maps.vnew, a.kv.values, 2, D, (uint64_t)p.num_kv_heads, T, 64u, 1u,
                          128u, true) &&
            (!Q8 || encode_map_3d_swizzle(&maps.cache8, a.kv.cache, 1, D,
                                          2 * (uint64_t)p.num_kv_heads, rows, (uint32_t)D, 1u,
                                          prow, D));
  if (!ok) return cudaErrorInvalidValue;
  int grid = num_sms;
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;
  return launch_dependent(kern, grid, tc::kThreads, C::kSmemBytes, stream, maps, a);
}

template <int D>
static cudaError_t launch_prefill_tc_d(const AttnArgs& a, int max_units, int num_sms,
                                       cudaStream_t stream) {
  const rpa_params_t& p = a.kv.p;
  if (p.kv_dtype != RPA_KV_FP8_E4M3)
    return launch_prefill_tc_t<D, false, false, false>(a, max_units, num_sms, stream);
  // per-head scales get their own instantiation, so the common cases keep
  // their logit transform loop-invariant; quantised queries (an e4m3 cache
  // only) run Q K^T on the codes
  const bool ph = p.k_scale_heads != nullptr || p.v_scale_heads != nullptr;
  if (p.q_scale > 0.f)
    return ph ? launch_prefill_tc_t<D, true, true, true>(a, max_units, num_sms, stream)
              : launch_prefill_tc_t<D, true, false, true>(a, max_units, num_sms, stream);
  return ph ? launch_prefill_tc_t<D, true, true, false>(a, max_units, num_sms, stream)
            : launch_prefill_tc_t<D, true, false, false>(a, max_units, num_sms, stream);
}

cudaError_t launch_prefill_tc(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream) {
  return a.kv.p.head_dim == 64 ? launch_prefill_tc_d<64>(a, max_units, num_sms, stream)
                               : launch_prefill_tc_d<128>(a, max_units, num_sms, stream);
}

}  // namespace rpa
