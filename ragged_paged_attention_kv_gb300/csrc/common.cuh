// Shared device helpers for the ragged paged attention kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rpa.h"

namespace rpa {

// ------------------------------------------------------------------ layout
// Workspace: a 256-byte header of int32 words, then the arrays below at
// offsets computed by WorkspaceLayout (host and device agree through it).
enum HeaderWord {
  kHdrStatus = 0,       // RPA_STATUS_* bits, cleared by the planner
  kHdrNumDecode = 1,    // decode work units planned
  kHdrNumPrefill = 2,   // prefill work units planned
  kHdrDecodeChunk = 3,  // keys per decode split
  kHdrDecodeNext = 4,   // dynamic scheduler counter (decode)
  kHdrPrefillNext = 5,  // dynamic scheduler counter (prefill)
  kHdrDecodeShare = 6,  // 1: the decode kernel leaves part of the SMs to the prefill kernel
  kHdrWords = 64,
};

// Decode unit: one (sequence, kv head, split of the key range).  The units of
// one (seq, head) are contiguous, so split 0 of unit u is unit u - split.  The
// sequence's token row q0 and kv_len ride along, so one load gives a unit
// (16-byte aligned: two vector accesses move one).
struct __align__(16) DecodeUnit {
  int32_t seq, head, k_begin, k_end;  // keys [k_begin, k_end) of this split
  int32_t split, nsplit, q0, kv_len;
};

// Prefill unit: one (sequence, tile of new tokens, kv head); one vector access.
struct __align__(16) PrefillUnit {
  int32_t seq, t_begin, t_end, head;    // new tokens [t_begin, t_end) of seq
};

static_assert(sizeof(DecodeUnit) == 32 && sizeof(PrefillUnit) == 16, "unit sizes");

// The planner splits a decode sequence's keys only when the batch has too
// few (sequence, kv head) pairs to keep the GPU busy: splits aim at about
// this many units in total.  Units are handed out longest first, so the
// pairs need no splitting to balance.
#ifndef RPA_DECODE_UNITS_TARGET
#define RPA_DECODE_UNITS_TARGET 512
#endif
constexpr int kDecodeUnitsTarget = RPA_DECODE_UNITS_TARGET;
constexpr int kDecodeChunkMin = 256;      // smallest split, in keys
constexpr int kDecodeRows = 16;           // q-heads per decode tile (padded group)
constexpr int kPrefillRows = 64;          // packed (token, q-head) rows per prefill tile

struct WorkspaceLayout {
  size_t decode_units_off, counters_off, partial_o_off, partial_ml_off, prefill_units_off;
  size_t total;
  int64_t max_decode_units, max_prefill_units;

  __host__ __device__ static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

  __host__ __device__ explicit WorkspaceLayout(const rpa_params_t& p) {
    const int64_t g = p.num_q_heads / p.num_kv_heads;
    // A decode sequence with K keys spans at most K + 63 keys from the 64-key
    // stage below its first key, so it takes ceil((K + 63) / chunk) <= K /
    // chunk + 63 / chunk + 1 splits per kv head; with chunk >= total keys *
    // Hkv / target and chunk >= 256 the units number at most target +
    // (1 + 63/256) * sequences * Hkv.
    max_decode_units = (int64_t)kDecodeUnitsTarget + 2 * (int64_t)p.max_num_seqs * p.num_kv_heads;
    const int64_t tiles = ((int64_t)p.total_tokens * g + kPrefillRows - 1) / kPrefillRows +
                          p.max_num_seqs;
    max_prefill_units = tiles * p.num_kv_heads;
    size_t off = kHdrWords * sizeof(int32_t);
    decode_units_off = off;
    off = align_up(off + max_decode_units * sizeof(DecodeUnit), 256);
    counters_off = off;
    off = align_up(off + (size_t)p.max_num_seqs * p.num_kv_heads * sizeof(int32_t), 256);
    partial_o_off = off;
    off = align_up(off + (size_t)max_decode_units * g * p.head_dim * sizeof(float), 256);
    partial_ml_off = off;
    off = align_up(off + (size_t)max_decode_units * g * 2 * sizeof(float), 256);
    prefill_units_off = off;
    off = align_up(off + (size_t)max_prefill_units * sizeof(PrefillUnit), 256);
    total = off;
  }
};

// ------------------------------------------------ programmatic launches
// The decode and prefill kernels are launched as programmatic dependents of
// the kernel before them on the stream, so their launch (and the planner's
// successors' set-up) overlaps the kernel ahead.  griddep_wait blocks until
// the preceding kernel has completed and its memory is visible; nothing a
// dependent reads or writes in global memory may be touched before it.
// Without a programmatic predecessor it returns at once.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel on the stream (if launched as a programmatic
// dependent) begin launching before this grid completes.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- status
__device__ __forceinline__ void set_status(int32_t* ws_header, int bits) {
  atomicOr(ws_header + kHdrStatus, bits);
}

// ---------------------------------------------------------- memory (PTX)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The same with fp16 A and B.
__device__ __forceinline__ void mma_f16_16816(float* d, const uint32_t* a, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <bool F16>
__device__ __forceinline__ void mma_p_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if (F16) mma_f16_16816(d, a, b0, b1); else mma_bf16_16816(d, a, b0, b1);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits)
  return *reinterpret_cast<uint32_t*>(&v);
}
// Two fp32 -> fp16 (round to nearest even, subnormals kept), packed low-first.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// The sum of the two values a packed pair holds (bf16 or fp16), in fp32:
// the softmax normaliser is summed from exactly the weights the P V product
// uses, so the output is a weighted mean of the values with weights that sum
// to one (the rounding of P then moves the output by at most ~2^-8 times the
// spread of the values around it, instead of 2^-9 times their magnitude).
__device__ __forceinline__ float pair_sum_bf16(uint32_t u) {
  return __uint_as_float(u << 16) + __uint_as_float(u & 0xFFFF0000u);
}
__device__ __forceinline__ float pair_sum_f16(uint32_t u) {
  __half2 h = *reinterpret_cast<__half2*>(&u);
  const float2 f = __half22float2(h);
  return f.x + f.y;
}
// P (two softmax weights) packed for the P V product: bf16 when the values
// are bf16, fp16 when they came from an e4m3 cache (every e4m3 value is
// exact in fp16, and fp16 carries P with 3 more bits).
template <bool F16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  return F16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}
template <bool F16>
__device__ __forceinline__ float pair_sum(uint32_t u) {
  return F16 ? pair_sum_f16(u) : pair_sum_bf16(u);
}

// Byte offset of 16-byte chunk `c` of row `r` in a tile whose rows are
// `row_bytes` long: chunks are XOR-swizzled by the row's low 3 bits so that
// eight consecutive rows at one logical chunk hit eight different banks.
__device__ __forceinline__ uint32_t swz(int r, int c, int row_bytes) {
  return (uint32_t)(r * row_bytes + ((c ^ (r & 7)) << 4));
}

// -------------------------------------------------------------- fp8 e4m3
// Quantise two fp32 values (x / scale already applied) to e4m3 with round to
// nearest even and saturation to +-448; x0 lands in the low byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float x0, float x1) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
}

// Two e4m3 codes (low byte first) -> two bf16 (exact), packed low-first.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  return pack_bf16(f.x, f.y);
}

// x / s (s > 0) rounded to nearest fp32, from r = RN(1/s): q = RN(x*r), then
// one residual correction q + (x - s*q)*r with fused multiply-adds.  With a
// correctly rounded reciprocal this is the correctly rounded quotient
// (Markstein's theorem) away from overflow and subnormal quotients; both of
// those encode to the same e4m3 code either way (saturation, or +-0).  The
// correction turns -0 into +0, so the sign is taken from x.
__device__ __forceinline__ float div_by(float x, float s, float r) {
  const float q = x * r;
  return copysignf(fmaf(fmaf(-q, s, x), r, q), x);
}

// Quantise 8 bf16 values (one 16-byte chunk) to 8 e4m3 codes: x / scale in
// fp32, correctly rounded, then e4m3.  Returns the 8 codes as a uint2.
__device__ __forceinline__ uint2 quantize8(uint4 src, float scale) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&src);
  const float r = __frcp_rn(scale);
  uint32_t w[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float2 a = __bfloat1622float2(b[2 * i]);
    float2 c = __bfloat1622float2(b[2 * i + 1]);
    uint32_t lo = f32x2_to_e4m3x2(div_by(a.x, scale, r), div_by(a.y, scale, r));
    uint32_t hi = f32x2_to_e4m3x2(div_by(c.x, scale, r), div_by(c.y, scale, r));
    w[i] = lo | (hi << 16);
  }
  return make_uint2(w[0], w[1]);
}

// 8 e4m3 codes -> 8 bf16 values (one 16-byte chunk).
__device__ __forceinline__ uint4 dequant8(uint2 codes) {
  uint4 r;
  r.x = e4m3x2_to_bf16x2((uint16_t)(codes.x & 0xFFFF));
  r.y = e4m3x2_to_bf16x2((uint16_t)(codes.x >> 16));
  r.z = e4m3x2_to_bf16x2((uint16_t)(codes.y & 0xFFFF));
  r.w = e4m3x2_to_bf16x2((uint16_t)(codes.y >> 16));
  return r;
}
// Two e4m3 codes -> two fp16 (exact: e4m3 has 3 mantissa bits and exponents
// 2^-9 .. 2^8, all inside fp16), one conversion instruction.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}
// 8 e4m3 codes -> 8 fp16 values (one 16-byte chunk).
__device__ __forceinline__ uint4 dequant8_f16(uint2 codes) {
  uint4 r;
  r.x = e4m3x2_to_f16x2((uint16_t)(codes.x & 0xFFFF));
  r.y = e4m3x2_to_f16x2((uint16_t)(codes.x >> 16));
  r.z = e4m3x2_to_f16x2((uint16_t)(codes.y & 0xFFFF));
  r.w = e4m3x2_to_f16x2((uint16_t)(codes.y >> 16));
  return r;
}
template <bool F16>
__device__ __forceinline__ uint4 dequant8_as(uint2 codes) {
  return F16 ? dequant8_f16(codes) : dequant8(codes);
}

// ------------------------------------------------------------- reductions
__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
  return x;
}
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

constexpr float kLog2e = 1.4426950408889634f;

// 2^x with the hardware approximation (one MUFU operation; denormal results
// flush to zero, which only affects weights below 2^-126).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 lanes in one 64-bit register pair, for the packed f32x2
// arithmetic of sm_100 and later (one instruction does both lanes).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// lo += the low 16-bit value of pk, hi += the high one: bf16 (or fp16 with
// F16) values converted exactly to fp32 inside a mixed-precision add, one
// instruction each (no separate unpacking).
template <bool F16>
__device__ __forceinline__ void add_halves_f32(float& lo, float& hi, uint32_t pk) {
  if constexpr (F16) {
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n add.rn.f32.f16 %0, l, %0;\n"
        " add.rn.f32.f16 %1, h, %1;\n}"
        : "+f"(lo), "+f"(hi)
        : "r"(pk));
  } else {
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n add.rn.f32.bf16 %0, l, %0;\n"
        " add.rn.f32.bf16 %1, h, %1;\n}"
        : "+f"(lo), "+f"(hi)
        : "r"(pk));
  }
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// tanh(x) = 1 - 2 / (e^(2x) + 1), with the hardware 2^x and reciprocal
// approximations: absolute error of a few 1e-7, and exactly +-1 in the
// limits (e^(2x) = inf gives a reciprocal of 0, e^(2x) = 0 gives 1).
__device__ __forceinline__ float tanh_exp(float x) {
  const float e = fast_exp2(x * (2.f * kLog2e));
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(e + 1.f));
  return fmaf(-2.f, r, 1.f);
}

// Logit transform shared by the kernels: raw dot product -> log2-domain
// logit; with a soft cap, cap * tanh(x / cap) is applied to the
// natural-domain logit x = softmax_scale * k_scale * dot first.  Two numbers
// per kv head: with a soft cap, cap * log2e * tanh(dot * mul) with mul =
// softmax_scale * k_scale / cap; without, dot * mul with mul = softmax_scale
// * k_scale * log2e.
struct LogitXform {
  float mul;
  float cap2;  // cap * log2e, 0 = no cap
  __device__ __forceinline__ float operator()(float dot) const {
    if (cap2 > 0.f) return cap2 * tanh_exp(dot * mul);
    return dot * mul;
  }
};
// The factor the raw q . k dot product carries besides softmax_scale: the
// key scale, times q_scale when the queries are quantised (the dot product
// is then one of e4m3 codes).
__device__ __forceinline__ float qk_scale(const rpa_params_t& p, float k_scale) {
  return p.q_scale > 0.f ? k_scale * p.q_scale : k_scale;
}
// Quantises 8 queries (one 16-byte chunk, in place) to e4m3 with q_scale and
// back to bf16 (exact): the operand then holds the codes' values.
__device__ __forceinline__ void quantize_q8(uint4* chunk, float q_scale) {
  *chunk = dequant8(quantize8(*chunk, q_scale));
}
__device__ __forceinline__ LogitXform make_xform(float softmax_scale, float k_scale, float cap) {
  return cap > 0.f ? LogitXform{softmax_scale * k_scale / cap, cap * kLog2e}
                   : LogitXform{softmax_scale * k_scale * kLog2e, 0.f};
}

}  // namespace rpa
