// Decode path: one new token per sequence, HBM-bound.
//
// Work unit = (sequence, kv head, split of the key range).  The q-heads of the
// kv head (the GQA group; tpu-inference RPA v3 kernel.py stacks them as rows
// of one q block) form a 16-row tile, so every key/value byte fetched from a
// page feeds all of them through one tensor-core MMA.
//
// The kernel is persistent and warp-specialised.  One producer warp walks the
// planner's unit list (dynamic atomic counter) and streams each unit's pages
// into a ring of shared-memory stages with TMA: per page, one 128-byte
// swizzled box per (key | value, 64-wide half of head_dim), so consecutive
// keys of one head land in consecutive conflict-free rows.  The query rows
// arrive with a bulk copy.  Four consumer warps each take 16 keys of every
// stage: S = Q K^T and O += P V with mma.sync, an online softmax in fp32
// (RPA v3 flash_attention_step1_qk_softmax / step2_pv) whose running max is
// only moved -- and O only rescaled -- when it grows by more than 2^8.
//
// The new token's key/value is taken from the step's inputs, not from its
// page (RPA v3 _fetch_bkv reads new keys from the inputs too), and split 0
// of each (sequence, kv head) writes it into the page.  When a sequence's
// keys are split over several units, the unit that finishes last merges the
// partial (m, l, O) of all splits with a log-sum-exp combine.
#include "async.cuh"
#include "common.cuh"
#include "kv_write.cuh"
#include "tma_host.h"

namespace rpa {
namespace dec {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kBN = 64;                       // keys per stage
constexpr int kKeysPerWarp = kBN / kConsumerWarps;  // 16
constexpr int kRescaleLog2 = 8;               // lazy-rescale threshold (log2 units)

template <int D, bool FP8>
struct Cfg {
  // Several CTAs per SM put several consumer warps on each scheduler, so one
  // warp's ldmatrix -> MMA -> softmax chain hides behind another's, and
  // multiply the units in flight when short units make the path
  // latency-bound.  head_dim 64 runs three (128 registers; the e4m3 kernel
  // spills 16 bytes; four, at 96 registers, spilled 92 bytes and ran 16 %
  // slower); bf16 head_dim 128 runs two in 168 registers (12 bytes of spills)
  // with two 32 KB stages per CTA (128 KB in flight per SM), 4 % faster than
  // one CTA with five stages.  fp8 at 128 (more conversion registers) and
  // head_dim 256 keep one CTA per SM.
  // head_dim 96 runs as 128 in shared memory (a multiple of 64 columns):
  // past the real row, bf16 stages hold TMA's zero fill and fp8 ones the
  // conversion's zeros; the query rows land at the padded stride; only the
  // real columns are read from or written to global memory
  static constexpr int kDp = (D + 63) / 64 * 64;
  static constexpr int kCtasPerSm = kDp == 64 ? 3 : ((kDp == 128 && !FP8) ? 2 : 1);
  // bytes of one box row in smem: an fp8 stage keeps the real head_dim (the
  // conversion to the padded bf16 operand zero-fills the rest)
  static constexpr int kRowBytes = FP8 ? D : 128;
  static constexpr int kHalves = FP8 ? 1 : kDp / 64;     // 64-column boxes of a stage
  // a stage holds, per 64-wide half of head_dim, 2*kBN rows: key j at row 2j,
  // value j at row 2j+1 (one TMA box brings both for a page)
  static constexpr int kHalfBytes = 2 * kBN * kRowBytes;
  static constexpr int kStageBytes = kHalves * kHalfBytes;
  // head_dim 192 and 256: the query fragments (48 / 64 registers) are
  // re-read from the slot every stage instead of being held, and each row
  // lands with its own bulk copy at a 16-byte padded stride, so those
  // ldmatrix reads are free of bank conflicts; the slot is then released at
  // the end of the unit
  static constexpr bool kQFromSmem = kDp > 128;
  static constexpr int kQRow = kQFromSmem ? kDp * 2 + 16 : kDp * 2;  // bytes per query row
  static constexpr bool kQPerRow = kQFromSmem || D != kDp;  // one bulk copy per query row
  static constexpr int kQBytes = kDecodeRows * kQRow;    // one query slot
  static constexpr int kConvBytes = FP8 ? kConsumerWarps * 2 * kKeysPerWarp * kDp * 2 : 0;
  static constexpr int kMergeBytes = kConsumerWarps * kDecodeRows * (kDp + 2) * 4;
  // as many stages as fit next to the other buffers (at most 12, 160 KB)
  static constexpr int kBudget =
      (kCtasPerSm == 3 ? 72 : kCtasPerSm == 2 ? 110 : 220) * 1024 - 2 * kQBytes - kConvBytes -
      kMergeBytes - 1024 - 256;
  static constexpr int kStages1 = (kBudget < 160 * 1024 ? kBudget : 160 * 1024) / kStageBytes;
  static constexpr int kStages = kStages1 > 12 ? 12 : (kStages1 < 2 ? 2 : kStages1);
  // layout: [stages][q slots 2][conv][merge][unit info 2][barriers]
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffConv = kOffQ + 2 * kQBytes;
  static constexpr int kOffMerge = kOffConv + kConvBytes;
  static constexpr int kOffInfo = kOffMerge + kMergeBytes;
  static constexpr int kOffBar = kOffInfo + 2 * 64;  // two UnitInfo slots
  static constexpr int kBytes = kOffBar + (2 * kStages + 4) * 8 + 1024;  // + base alignment
  static_assert(kBytes <= 227 * 1024 / kCtasPerSm, "decode shared memory over budget");
};

// What the producer tells the consumers about the unit in a query slot.
struct UnitInfo {
  DecodeUnit du;  // du.seq < 0 means "no more units"
  int q0, ctx;    // the sequence's token row and the new token's position
  int pad[6];     // pad[0]: the unit's index (its partial results live there)
};
static_assert(sizeof(UnitInfo) == 64, "two UnitInfo slots take 128 bytes");

struct DecodeMaps {
  CUtensorMap cache;  // pool [num_pages*P][2*Hkv][D]
};

// Address of 16-byte chunk `c` (of D/8) of the key (kv = 0) or value (kv = 1)
// row of key `r` in a bf16 stage written by 128-byte swizzled boxes.
__device__ __forceinline__ uint32_t kv_addr(uint32_t stage, int r, int kv, int c) {
  return stage + (uint32_t)((c >> 3) * 2 * kBN * 128) + sw128(2 * r + kv, c & 7);
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads, Cfg<D, FP8>::kCtasPerSm)
    decode_kernel(const __grid_constant__ DecodeMaps maps, AttnArgs a) {
  using C = Cfg<D, FP8>;
  constexpr int Dp = C::kDp;  // head_dim as laid out in shared memory
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  UnitInfo* info = reinterpret_cast<UnitInfo*>(smem + C::kOffInfo);
  float* sMerge = reinterpret_cast<float*>(smem + C::kOffMerge);
  const uint32_t bar_full = s_base + C::kOffBar;                 // [kStages]
  const uint32_t bar_empty = bar_full + 8 * C::kStages;          // [kStages]
  const uint32_t bar_qfull = bar_empty + 8 * C::kStages;         // [2]
  const uint32_t bar_qempty = bar_qfull + 16;                    // [2]
  __shared__ int s_abort, s_last;

  const rpa_params_t& p = a.kv.p;
  int32_t* hdr = a.kv.ws;
  const WorkspaceLayout L(p);
  const DecodeUnit* units =
      reinterpret_cast<const DecodeUnit*>(reinterpret_cast<const char*>(hdr) + L.decode_units_off);
  int32_t* counters = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(hdr) + L.counters_off);
  float* part_o = reinterpret_cast<float*>(reinterpret_cast<char*>(hdr) + L.partial_o_off);
  float2* part_ml = reinterpret_cast<float2*>(reinterpret_cast<char*>(hdr) + L.partial_ml_off);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int P = p.page_size;
  griddep_wait();  // the planner's unit list and counters are complete
  // only now may the prefill kernel behind launch: it reads the planner's
  // output without a wait of its own
  griddep_launch_dependents();
  if (hdr[kHdrNumDecode] == 0) return;  // a prefill-only batch: nothing to set up
  // A batch with enough prefill work as well (the planner's decision): the
  // CTAs on 8 of every 16 SMs (by %smid: 72 of the 152) leave at once, so
  // the prefill kernel's CTAs,
  // launched behind this grid and waiting for no part of it, run there from
  // the start while the decode stays HBM-bound on the other SMs.  Only with
  // more CTAs than the leaving SMs can hold, so that some always stay: the
  // units go to whichever CTAs run.
  if (hdr[kHdrDecodeShare] && gridDim.x > 72 * C::kCtasPerSm) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    if ((smid & 15u) >= 8u) return;
  }

  // zero both query slots (rows >= G stay zero), init barriers; the bulk
  // copies that later fill rows < G are async-proxy writes of the same bytes
  for (int i = tid; i < 2 * C::kQBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + C::kOffQ)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_qfull + 8 * s, 1);
      mbar_init(bar_qempty + 8 * s, kConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; lane l looks up and copies pages l and
    // l + 32 of each stage, with the page ids of the next stage loaded while
    // the current one waits for a free slot.
    if (lane == 0) prefetch_tensormap(&maps.cache);
    const int n_units = hdr[kHdrNumDecode];
    const int rows = P < kBN ? P : kBN;  // rows of one box
    uint32_t g = 0;                      // stages issued so far
    uint32_t nq = 0;                     // query-slot copies issued so far
    bool ended = false;                  // the "no more units" signal was posted
    bool ok = true;
    for (uint32_t uq = 0; ok; ++uq) {
      const int slot = uq & 1;
      int u = 0;
      if (lane == 0) u = atomicAdd(hdr + kHdrDecodeNext, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      DecodeUnit du{};
      int q0 = 0, kv_len = 0;
      if (u < n_units) {
        du = units[u];
        q0 = du.q0;
        kv_len = du.kv_len;
      }
      const int kb0 = du.k_begin & ~(kBN - 1);
      const int n_st = u < n_units ? (du.k_end - kb0 + kBN - 1) / kBN : 0;
      const int64_t bt_row = (int64_t)du.seq * p.pages_per_seq;
      auto stage_pages = [&](int st, int& pg0, int& npg) {
        const int kb = kb0 + st * kBN;
        const int lo = max(kb, du.k_begin), hi = min(kb + kBN, du.k_end);
        pg0 = lo / P;
        npg = (hi - 1) / P - pg0 + 1;
      };
      auto load_ids = [&](int st, int* ids) {
        int pg0, npg;
        stage_pages(st, pg0, npg);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int k = lane + 32 * i;
          ids[i] = k < npg ? __ldg(a.kv.block_tables + bt_row + pg0 + k) : 0;
        }
      };
      int ids_next[2] = {0, 0};
      if (n_st > 0) load_ids(0, ids_next);
      if (!mbar_wait_warp(bar_qempty + 8 * slot, ((uq >> 1) & 1) ^ 1, &s_abort)) {
        ok = false;
        break;
      }
      if (u >= n_units) {
        if (lane == 0) {
          info[slot].du.seq = -1;
          mbar_arrive(bar_qfull + 8 * slot);
        }
        ended = true;
        break;
      }
      constexpr bool kIssueQ = RPA_TEST_STALL_QUERY == 0;
      if (lane == 0) {
        UnitInfo ui;
        ui.du = du;
        ui.pad[0] = u;
        ui.q0 = q0;
        ui.ctx = kv_len - 1;
        info[slot] = ui;
        const uint32_t qbytes = (uint32_t)(G * D * 2);
        if (kIssueQ) mbar_arrive_expect_tx(bar_qfull + 8 * slot, qbytes);
        if (kIssueQ && !C::kQPerRow)
          bulk_load(s_base + C::kOffQ + slot * C::kQBytes,
                    a.queries + ((int64_t)q0 * p.num_q_heads + du.head * G) * D, qbytes,
                    bar_qfull + 8 * slot);
      }
      if (kIssueQ && C::kQPerRow) {  // one row per lane at the padded stride
        __syncwarp();                // the expected bytes are posted first
        if (lane < G)
          bulk_load(s_base + C::kOffQ + slot * C::kQBytes + lane * C::kQRow,
                    a.queries + ((int64_t)q0 * p.num_q_heads + du.head * G + lane) * D,
                    (uint32_t)(D * 2), bar_qfull + 8 * slot);
      }
      if (kIssueQ) ++nq;
      for (int st = 0; st < n_st; ++st, ++g) {
        int ids[2] = {ids_next[0], ids_next[1]};
        if (st + 1 < n_st) load_ids(st + 1, ids_next);
        const int s = g % C::kStages;
        if (!mbar_wait_warp(bar_empty + 8 * s, ((g / C::kStages) & 1) ^ 1, &s_abort)) {
          ok = false;
          break;
        }
        int pg0, npg;
        stage_pages(st, pg0, npg);
        const int kb = kb0 + st * kBN;
        if (lane == 0)
          mbar_arrive_expect_tx(bar_full + 8 * s,
                                (uint32_t)(npg * rows * C::kRowBytes * C::kHalves * 2));
        __syncwarp();
        const uint32_t stage = s_base + s * C::kStageBytes;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int k = lane + 32 * i;
          if (k >= npg) continue;
          int page = ids[i];
          if (page < 0 || page >= p.num_pages) {
            set_status(hdr, RPA_STATUS_BAD_PAGE);
            page = 0;  // keep the byte count; the data is never trusted
          }
          const int row_in_stage = P < kBN ? (pg0 + k) * P - kb : 0;
          const int z = page * P + (P < kBN ? 0 : kb % P);
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(stage + hf * C::kHalfBytes + 2 * row_in_stage * C::kRowBytes, &maps.cache,
                        bar_full + 8 * s, FP8 ? 0 : hf * 64, 2 * du.head, z);
        }
      }
    }
    if (!ok && lane == 0) {
      set_status(hdr, RPA_STATUS_TIMEOUT);
      s_abort = 1;
    }
    // Let every copy this warp issued land before the CTA may exit (on an
    // abort the consumers stop waiting for them): the last query copy of
    // each slot and the last stage of each ring slot.  A slot's earlier
    // copies completed before it was refilled -- by a later unit, or by the
    // "no more units" signal, which also completes a phase of the slot's
    // barrier (so the copy before it must not be waited on by parity).
    if (lane == 0) {
      bool drained = true;
      for (uint32_t i = nq > 2 ? nq - 2 : 0; i < nq; ++i)
        if (!(ended && i + 2 == nq))
          drained &= mbar_drain(bar_qfull + 8 * (i & 1), (i >> 1) & 1);
      for (uint32_t i = g > (uint32_t)C::kStages ? g - C::kStages : 0; i < g; ++i)
        drained &= mbar_drain(bar_full + 8 * (i % C::kStages), (i / C::kStages) & 1);
      if (!drained) set_status(hdr, RPA_STATUS_TIMEOUT);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t g = 0;
  for (uint32_t uq = 0;; ++uq) {
    const int slot = uq & 1;
    // the consumer warps leave together or not at all: a warp that left
    // alone would leave the others at the next named barrier
    const bool q_ok = mbar_wait(bar_qfull + 8 * slot, (uq >> 1) & 1, &s_abort);
    if (FP8 && q_ok && p.q_scale > 0.f) {  // q_scale needs an e4m3 cache
      // quantised queries: the slot's rows become their e4m3 codes' values
      // before any warp reads them (the vote below is a barrier)
      uint8_t* qslot = smem + C::kOffQ + slot * C::kQBytes;
      for (int idx = tid; idx < G * (D / 8); idx += kConsumerWarps * 32)
        quantize_q8(reinterpret_cast<uint4*>(qslot + (idx / (D / 8)) * C::kQRow +
                                             (idx % (D / 8)) * 16),
                    p.q_scale);
    }
    if (!named_bar_all(1, kConsumerWarps * 32, q_ok)) {
      if (!q_ok && lane == 0) set_status(hdr, RPA_STATUS_TIMEOUT);
      s_abort = 1;
      break;
    }
    const DecodeUnit du = info[slot].du;
    if (du.seq < 0) break;
    const int u_idx = info[slot].pad[0];  // read now: the slot is refilled once Q is taken
    const int seq = du.seq, h = du.head;
    const int q0 = info[slot].q0;
    const int ctx = info[slot].ctx;
    const float ks = k_scale_of(p, h), vs = v_scale_of(p, h);  // this kv head's scales
    const LogitXform xf = make_xform(p.softmax_scale, qk_scale(p, ks), p.logits_soft_cap);
    // split 0 stores the new token's key/value into its page after the
    // stages; the page id and the inputs are loaded now so that store does
    // not wait for them
    TokenKv<D> tkv{};
    if (du.split == 0 && warp == 0) tkv = token_kv_load<FP8, D>(a.kv, seq, q0, ctx, h, lane);

    // query fragment ks of this warp's 16-row tile
    const uint32_t sq = s_base + C::kOffQ + slot * C::kQBytes;
    auto load_q = [&](int ks, uint32_t (&f)[4]) {
      const int mi = lane >> 3;
      const int row = (lane & 7) + ((mi & 1) << 3);
      const int col = (2 * ks + (mi >> 1)) * 16;
      ldmatrix_x4(sq + row * C::kQRow + col, f[0], f[1], f[2], f[3]);
    };
    uint32_t qa[C::kQFromSmem ? 1 : Dp / 16][4];
    if constexpr (!C::kQFromSmem) {
#pragma unroll
      for (int ks = 0; ks < (C::kQFromSmem ? 1 : Dp / 16); ++ks) load_q(ks, qa[ks]);
      // The slot is refilled by a bulk copy (async proxy) once all warps
      // have arrived, and nothing reads qa before the first stage lands, so
      // the ldmatrix reads may still be in flight here: a proxy fence orders
      // them before the release (without it, a short unit's later column
      // blocks were seen to hold the next query routed to this slot).
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_qempty + 8 * slot);
    }

    float o[Dp / 8][4];
#pragma unroll
    for (int n = 0; n < Dp / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    const int kb0 = du.k_begin & ~(kBN - 1);
    const int n_st = (du.k_end - kb0 + kBN - 1) / kBN;
    bool ok = true;
    for (int st = 0; st < n_st; ++st, ++g) {
      const int s = g % C::kStages;
      if (!mbar_wait_warp(bar_full + 8 * s, (g / C::kStages) & 1, &s_abort)) {
        ok = false;
        break;
      }
      const uint32_t stage = s_base + s * C::kStageBytes;
      const int kw = kb0 + st * kBN + warp * kKeysPerWarp;  // this warp's first key
      uint32_t tK, tV;
      int krow0;
      if (FP8) {
        // convert this warp's 16 keys/values to bf16 in its own buffer; keys
        // outside the unit become zero, the new token comes from the inputs
        const uint32_t cK = s_base + C::kOffConv + warp * 2 * kKeysPerWarp * Dp * 2;
        const uint32_t cV = cK + kKeysPerWarp * Dp * 2;
        uint8_t* gK = smem + (cK - s_base);
        uint8_t* gV = smem + (cV - s_base);
        // a stage whose 16 keys of this warp are all inside the unit and are
        // not the new token (the usual case) converts in groups: the code
        // loads of a group are issued before any conversion, so their
        // latencies overlap
        // (head_dim 64 only: at larger head_dims the group's registers spill)
        const bool interior = D == 64 && kw >= du.k_begin && kw + kKeysPerWarp <= du.k_end &&
                              !(ctx >= kw && ctx < kw + kKeysPerWarp);
        if (D == 64 && interior) {
          constexpr int kItems = 2 * kKeysPerWarp * (Dp / 8) / 32;  // chunks per lane
          constexpr int kGroup = kItems < 8 ? kItems : 8;
          const uint8_t* st8 = smem + (stage - s_base);
#pragma unroll
          for (int i0 = 0; i0 < kItems; i0 += kGroup) {
            uint2 codes[kGroup];
#pragma unroll
            for (int i = 0; i < kGroup; ++i) {
              const int idx = lane + 32 * (i0 + i);
              const int kv = idx / (kKeysPerWarp * (Dp / 8));
              const int rem = idx % (kKeysPerWarp * (Dp / 8));
              const int r = rem / (Dp / 8), c = rem % (Dp / 8);
              codes[i] = *reinterpret_cast<const uint2*>(
                  st8 + (2 * (warp * kKeysPerWarp + r) + kv) * C::kRowBytes + c * 8);
            }
#pragma unroll
            for (int i = 0; i < kGroup; ++i) {
              const int idx = lane + 32 * (i0 + i);
              const int kv = idx / (kKeysPerWarp * (Dp / 8));
              const int rem = idx % (kKeysPerWarp * (Dp / 8));
              const int r = rem / (Dp / 8), c = rem % (Dp / 8);
              *reinterpret_cast<uint4*>((kv ? gV : gK) + swz(r, c, Dp * 2)) =
                  kv ? dequant8_f16(codes[i]) : dequant8(codes[i]);
            }
          }
        } else
        for (int idx = lane; idx < 2 * kKeysPerWarp * (Dp / 8); idx += 32) {
          const int kv = idx / (kKeysPerWarp * (Dp / 8));
          const int rem = idx % (kKeysPerWarp * (Dp / 8));
          const int r = rem / (Dp / 8), c = rem % (Dp / 8);
          const int j = kw + r;
          uint4 val;
          // keys become bf16 (the queries' type), values fp16 (exact for
          // e4m3, and the P V product then carries P in fp16)
          if (j < du.k_begin || j >= du.k_end || c >= D / 8) {
            val = make_uint4(0, 0, 0, 0);  // masked key, or a padding column
          } else {
            uint2 codes;
            if (j == ctx) {
              const __nv_bfloat16* in = (kv ? a.kv.values : a.kv.keys) +
                                        ((int64_t)q0 * p.num_kv_heads + h) * D + c * 8;
              codes = quantize8(__ldg(reinterpret_cast<const uint4*>(in)), kv ? vs : ks);
            } else {
              codes = *reinterpret_cast<const uint2*>(
                  smem + (stage - s_base) + (2 * (warp * kKeysPerWarp + r) + kv) * C::kRowBytes +
                  c * 8);
            }
            val = kv ? dequant8_f16(codes) : dequant8(codes);
          }
          *reinterpret_cast<uint4*>((kv ? gV : gK) + swz(r, c, Dp * 2)) = val;
        }
        __syncwarp();
        tK = cK;
        tV = cV;
        krow0 = 0;
      } else {
        tK = stage;  // keys and values interleaved: see kv_addr
        tV = stage;
        krow0 = warp * kKeysPerWarp;
        // rows outside [k_begin, k_end): zero the values (masked keys may hold
        // anything, and 0 * NaN would poison P V); the new token's row: inputs
        const bool edge = kw < du.k_begin || kw + kKeysPerWarp > du.k_end ||
                          (ctx >= kw && ctx < kw + kKeysPerWarp);
        if (edge) {
          for (int idx = lane; idx < kKeysPerWarp * (Dp / 8); idx += 32) {
            const int r = idx / (Dp / 8), c = idx % (Dp / 8);
            const int j = kw + r;
            if (j < du.k_begin || j >= du.k_end) {
              *reinterpret_cast<uint4*>(smem + (kv_addr(stage, krow0 + r, 1, c) - s_base)) =
                  make_uint4(0, 0, 0, 0);
            } else if (j == ctx && c < D / 8) {  // its padding columns hold TMA's zeros
              const int64_t off = ((int64_t)q0 * p.num_kv_heads + h) * D + c * 8;
              *reinterpret_cast<uint4*>(smem + (kv_addr(stage, krow0 + r, 0, c) - s_base)) =
                  __ldg(reinterpret_cast<const uint4*>(a.kv.keys + off));
              *reinterpret_cast<uint4*>(smem + (kv_addr(stage, krow0 + r, 1, c) - s_base)) =
                  __ldg(reinterpret_cast<const uint4*>(a.kv.values + off));
            }
          }
          __syncwarp();
        }
      }

      // S = Q K^T for this warp's 16 keys (two n8 tiles)
      float sc[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < Dp / 16; ++ks) {
        const int mi = lane >> 3;
        const int key = krow0 + (lane & 7) + ((mi >> 1) << 3);
        const int chunk = 2 * ks + (mi & 1);
        const uint32_t addr = FP8 ? tK + swz(key, chunk, Dp * 2) : kv_addr(tK, key, 0, chunk);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(addr, b0, b1, b2, b3);
        if constexpr (C::kQFromSmem) {
          uint32_t qf[4];
          load_q(ks, qf);
          mma_bf16_16816(sc[0], qf, b0, b1);
          mma_bf16_16816(sc[1], qf, b2, b3);
        } else {
          mma_bf16_16816(sc[0], qa[C::kQFromSmem ? 0 : ks], b0, b1);
          mma_bf16_16816(sc[1], qa[C::kQFromSmem ? 0 : ks], b2, b3);
        }
      }
      // logits, mask, online softmax (rows gq and gq + 8)
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = kw + n * 8 + 2 * tq + (e & 1);
          const float x = (j >= du.k_begin && j < du.k_end) ? xf(sc[n][e]) : -INFINITY;
          sc[n][e] = x;
          mx[e >> 1] = fmaxf(mx[e >> 1], x);
        }
      float alpha[2];
      bool rescale = false;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float mt = quad_max(mx[r]);
        alpha[r] = 1.f;
        if (mt > m_run[r] + (float)kRescaleLog2) {  // also true on the first finite tile
          alpha[r] = m_run[r] == -INFINITY ? 0.f : exp2f(m_run[r] - mt);
          m_run[r] = mt;
          rescale = true;
        }
      }
      const float ms0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
      const float ms1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[n][e] = exp2f(sc[n][e] - ((e >> 1) ? ms1 : ms0));
      // P as the P V product takes it (fp16 for an e4m3 cache, else bf16);
      // the row sums add exactly those rounded weights
      uint32_t pa[4];
      pa[0] = pack_p<FP8>(sc[0][0], sc[0][1]);
      pa[1] = pack_p<FP8>(sc[0][2], sc[0][3]);
      pa[2] = pack_p<FP8>(sc[1][0], sc[1][1]);
      pa[3] = pack_p<FP8>(sc[1][2], sc[1][3]);
      const float rs[2] = {pair_sum<FP8>(pa[0]) + pair_sum<FP8>(pa[2]),
                           pair_sum<FP8>(pa[1]) + pair_sum<FP8>(pa[3])};
      if (rescale) {
#pragma unroll
        for (int n = 0; n < Dp / 8; ++n) {
          o[n][0] *= alpha[0];
          o[n][1] *= alpha[0];
          o[n][2] *= alpha[1];
          o[n][3] *= alpha[1];
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) l_run[r] = l_run[r] * alpha[r] + rs[r];
#pragma unroll
      for (int cp = 0; cp < Dp / 16; ++cp) {
        const int mi = lane >> 3;
        const int key = krow0 + (lane & 7) + ((mi & 1) << 3);
        const int chunk = 2 * cp + (mi >> 1);
        const uint32_t addr = FP8 ? tV + swz(key, chunk, Dp * 2) : kv_addr(tV, key, 1, chunk);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(addr, b0, b1, b2, b3);
        mma_p_16816<FP8>(o[2 * cp], pa, b0, b1);
        mma_p_16816<FP8>(o[2 * cp + 1], pa, b2, b3);
      }
      // this warp's reads of the stage (and its edge stores) precede the
      // next TMA into it: the generic-to-async proxy fence orders them
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    if constexpr (C::kQFromSmem) {  // the query slot was read up to the last stage
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_qempty + 8 * slot);
    }
    if (du.split == 0 && warp == 0) token_kv_store<FP8, D>(a.kv, tkv, ctx, h, lane);

    // per-warp state -> shared memory rows [warp][row] of (m, l, O[D]); only
    // the G rows of the GQA group are real, the rest of the 16-row tile is
    // padding and is not stored
    {
      float* mw = sMerge + warp * kDecodeRows * (Dp + 2);
      const float l0 = quad_sum(l_run[0]), l1 = quad_sum(l_run[1]);
      if (gq < G) {
        float* row = mw + gq * (Dp + 2);
        if (tq == 0) *reinterpret_cast<float2*>(row) = make_float2(m_run[0], l0);
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
          *reinterpret_cast<float2*>(row + 2 + n * 8 + 2 * tq) = make_float2(o[n][0], o[n][1]);
      }
      if (gq + 8 < G) {
        float* row = mw + (gq + 8) * (Dp + 2);
        if (tq == 0) *reinterpret_cast<float2*>(row) = make_float2(m_run[1], l1);
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
          *reinterpret_cast<float2*>(row + 2 + n * 8 + 2 * tq) = make_float2(o[n][2], o[n][3]);
      }
    }
    // the barrier before the merge is also a vote: the consumer warps go on
    // only if every one of them saw all its stages, else all leave together
    if (!named_bar_all(1, kConsumerWarps * 32, ok)) {
      if (!ok && lane == 0) set_status(hdr, RPA_STATUS_TIMEOUT);
      s_abort = 1;
      break;
    }

    const bool single = du.nsplit == 1;
    const int ctid = tid;  // consumers are threads 0..127
    for (int idx = ctid; idx < G * (D / 4); idx += kConsumerWarps * 32) {
      const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sMerge[(w * kDecodeRows + r) * (Dp + 2)]);
      float Lsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float* row = sMerge + (w * kDecodeRows + r) * (Dp + 2);
        const float scw = row[0] == -INFINITY ? 0.f : exp2f(row[0] - M);
        Lsum += scw * row[1];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] += scw * row[2 + d + e];
      }
      const int hq = h * G + r;
      if (single) {
        if (a.sink) {
          const float sk = a.sink[hq] * kLog2e;
          const float M2 = fmaxf(M, sk);
          const float scs = exp2f(M - M2);
          Lsum = Lsum * scs + exp2f(sk - M2);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] *= scs;
        }
        const float inv = vs / Lsum;
        __nv_bfloat16* dst = a.out + ((int64_t)q0 * p.num_q_heads + hq) * D + d;
        uint2 pk;
        pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
        pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(dst) = pk;
      } else {
        float* po = part_o + ((int64_t)u_idx * G + r) * D + d;
        *reinterpret_cast<float4*>(po) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        if (d == 0) part_ml[(int64_t)u_idx * G + r] = make_float2(M, Lsum);
      }
    }

    if (!single) {
      // the last split of (seq, head) to finish combines all of them
      // publish: CTA barrier, then one thread fences and counts (the
      // fence after the barrier covers every consumer's partial stores)
      named_bar(1, kConsumerWarps * 32);
      if (ctid == 0) {
        __threadfence();
        const int prev = atomicAdd(counters + (int64_t)seq * p.num_kv_heads + h, 1);
        s_last = prev == du.nsplit - 1;
        if (s_last) __threadfence();
      }
      named_bar(1, kConsumerWarps * 32);
      if (s_last) {
        for (int idx = ctid; idx < G * (D / 4); idx += kConsumerWarps * 32) {
          const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
          const int hq = h * G + r;
          float M = a.sink ? a.sink[hq] * kLog2e : -INFINITY;
          for (int k = 0; k < du.nsplit; ++k)
            M = fmaxf(M, __ldcg(&part_ml[(int64_t)(u_idx - du.split + k) * G + r].x));
          float Lsum = a.sink ? exp2f(a.sink[hq] * kLog2e - M) : 0.f;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int k = 0; k < du.nsplit; ++k) {
            const int64_t pu = (int64_t)(u_idx - du.split + k) * G + r;
            const float2 ml = __ldcg(&part_ml[pu]);
            const float scs = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
            Lsum += scs * ml.y;
            const float4 po = __ldcg(reinterpret_cast<const float4*>(part_o + pu * D + d));
            acc[0] += scs * po.x;
            acc[1] += scs * po.y;
            acc[2] += scs * po.z;
            acc[3] += scs * po.w;
          }
          const float inv = vs / Lsum;
          __nv_bfloat16* dst = a.out + ((int64_t)q0 * p.num_q_heads + hq) * D + d;
          uint2 pk;
          pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
          pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
          *reinterpret_cast<uint2*>(dst) = pk;
        }
      }
    }
    named_bar(1, kConsumerWarps * 32);  // the merge area is rewritten by the next unit
  }
}

}  // namespace dec

template <int D, bool FP8>
static cudaError_t launch_decode_t(const AttnArgs& a, int max_units, int num_sms,
                                   cudaStream_t stream) {
  using C = dec::Cfg<D, FP8>;
  static std::atomic<unsigned long long> attr_done{0};
  auto kern = dec::decode_kernel<D, FP8>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::kBytes, &attr_done);
  if (e != cudaSuccess) return e;
  const rpa_params_t& p = a.kv.p;
  dec::DecodeMaps maps;
  const uint32_t rows = p.page_size < dec::kBN ? (uint32_t)p.page_size : (uint32_t)dec::kBN;
  // bf16 boxes are 64 columns wide (at head_dim 96 the second one reads TMA's
  // zero fill past the row); an fp8 box spans the real row
  if (!encode_map_3d(&maps.cache, a.kv.cache, FP8 ? 1 : 2, (uint64_t)D,
                     2 * (uint64_t)p.num_kv_heads, (uint64_t)p.num_pages * p.page_size,
                     FP8 ? (uint32_t)D : 64u, 2u, rows, !FP8))
    return cudaErrorInvalidValue;
  int grid = num_sms * C::kCtasPerSm;
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;
  return launch_dependent(kern, grid, dec::kThreads, C::kBytes, stream, maps, a);
}

cudaError_t launch_decode(const AttnArgs& a, int max_units, int num_sms, cudaStream_t stream) {
  const bool fp8 = a.kv.p.kv_dtype == RPA_KV_FP8_E4M3;
  if (a.kv.p.head_dim == 64)
    return fp8 ? launch_decode_t<64, true>(a, max_units, num_sms, stream)
               : launch_decode_t<64, false>(a, max_units, num_sms, stream);
  if (a.kv.p.head_dim == 96)
    return fp8 ? launch_decode_t<96, true>(a, max_units, num_sms, stream)
               : launch_decode_t<96, false>(a, max_units, num_sms, stream);
  if (a.kv.p.head_dim == 192)
    return fp8 ? launch_decode_t<192, true>(a, max_units, num_sms, stream)
               : launch_decode_t<192, false>(a, max_units, num_sms, stream);
  if (a.kv.p.head_dim == 256)
    return fp8 ? launch_decode_t<256, true>(a, max_units, num_sms, stream)
               : launch_decode_t<256, false>(a, max_units, num_sms, stream);
  return fp8 ? launch_decode_t<128, true>(a, max_units, num_sms, stream)
             : launch_decode_t<128, false>(a, max_units, num_sms, stream);
}

}  // namespace rpa
