// common.cuh — device helpers shared by the hs2 kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/hs2.h"

#define HS2_DEVI __device__ __forceinline__

namespace hs2 {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPage = 64;

// ---------------------------------------------------------------------------- element access
template <typename T> struct Elem;
template <> struct Elem<float> {
  static HS2_DEVI float to_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static HS2_DEVI float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
};

HS2_DEVI float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
HS2_DEVI float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

HS2_DEVI uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// d = a * b + c with a and b bfloat16 halves of 32-bit words (fp32 c, d; the product of
// two bfloat16 values is exact in fp32, so this equals widening both and an fp32 FMA).
// LL: low half of a times low half of b; HH: high times high; LH/HL likewise.
#define HS2_FMA_BF16(NAME, SA, SB)                                                          \
  HS2_DEVI float NAME(uint32_t a, uint32_t b, float c) {                                   \
    float d;                                                                               \
    asm("{.reg .b16 a0, a1, b0, b1;\n\t"                                                   \
        "mov.b32 {a0, a1}, %1;\n\t"                                                        \
        "mov.b32 {b0, b1}, %2;\n\t"                                                        \
        "fma.rn.f32.bf16 %0, a" #SA ", b" #SB ", %3;}"                                      \
        : "=f"(d) : "r"(a), "r"(b), "f"(c));                                               \
    return d;                                                                              \
  }
HS2_FMA_BF16(fmab_ll, 0, 0)
HS2_FMA_BF16(fmab_hh, 1, 1)
HS2_FMA_BF16(fmab_lh, 0, 1)
HS2_FMA_BF16(fmab_hl, 1, 0)
#undef HS2_FMA_BF16

// L2 cache policy that keeps lines (evict last): for K/V rows that the same kernel, or
// the next SA layer of the group, reads again while other traffic streams past.
HS2_DEVI uint64_t l2_keep_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 16-byte read-only load with an L2 policy (keep or evict-first)
HS2_DEVI uint4 ldg_nc_v4_keep(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

// L2 cache policy that evicts lines first: for data read exactly once (the FA scan's K/V
// stream), so it does not push out what the next kernel reads.
HS2_DEVI uint64_t l2_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// fp32 store with an L2 cache policy
HS2_DEVI void stg_f32_pol(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

HS2_DEVI void stg_u16_pol(uint16_t* p, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.u16 [%0], %1, %2;" ::"l"(p), "h"((unsigned short)v), "l"(pol) : "memory");
}

HS2_DEVI void flag_error(int32_t* dev_err, int bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

// ---------------------------------------------------------------------------- warp helpers
HS2_DEVI float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
HS2_DEVI float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Weights are computed against a running max that may lag the true one by up to this
// much (base 2), i.e. they are at most 2^8: well inside bf16, f16 and fp32 range.
constexpr float kLazyRescale = 8.f;

// 2^x by the hardware approximation (relative error about 2^-22; results below 2^-126
// flush to zero, -inf gives 0): the softmax weights, which are rounded to 16 bits anyway,
// and the decode selection scores (a head's share under 2^-126 is dropped from the sum).
HS2_DEVI float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Selection logits between the FA scan and the selection: a key's base-2 logit x is kept as
// a 16-bit code below the max m of its group of 16 keys (same query head, groups aligned to
// multiples of 16 positions), code = round((m - x) * 2^11), 65535 for x = -inf or 32 or more
// below m; m itself is kept as a float per group. Decoding recovers x to within 2^-12, so
// a head's term 2^(x - lse) to within a relative 1.7e-4 (an omitted term far below m adds
// less than 2^-32 of the group's largest).
constexpr int kLogitGroup = 16;
constexpr float kLogitCodeUnit = 1.f / 2048.f;
HS2_DEVI uint32_t logit_code(float x, float m) { return __float2uint_rn(fminf((m - x) * 2048.f, 65535.f)); }
// 2^(x - lse2) from x's code and (m - lse2) of its group. The code becomes a float without
// a conversion instruction: 2^23 + code is exact in the mantissa, and subtracting 2^23 is exact.
HS2_DEVI float logit_term(uint32_t code, float m_minus_lse2) {
  const float c = __uint_as_float(0x4B000000u | code) - 8388608.f;
  return ex2_approx(fmaf(-c, kLogitCodeUnit, m_minus_lse2));
}

// Programmatic dependent launch. griddep_wait: returns once the grids this launch depends
// on have completed and their memory is visible (at once when it has no such dependency).
// griddep_launch_dependents: the next launch on the stream, if it allows programmatic
// serialization, may begin once every CTA of this grid has called it or exited.
HS2_DEVI void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
HS2_DEVI void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Barrier `id` (1-15) over the first `nthreads` threads (a multiple of 32) that reach it.
HS2_DEVI void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// exp2 of a (possibly -inf) base-2 logit relative to a (possibly -inf) max:
// a row whose max is still -inf contributes exactly zero.
HS2_DEVI float exp2_rel(float x, float m) { return (m == -INFINITY) ? 0.f : exp2f(x - m); }

// m16n8k16 bf16 MMA with fp32 accumulate (legacy warp-level tensor path; used where
// one warp owns a small contraction: decode FA over 8 query heads)
HS2_DEVI void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte global -> shared copy through the L2 only (cp.async.cg); zero-fills the
// destination without reading global memory when `valid` is false.
HS2_DEVI void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
HS2_DEVI void cp_async16(uint32_t s, const void* gmem, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
HS2_DEVI void cp_async16_keep(uint32_t s, const void* gmem, bool valid, uint64_t pol) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(s), "l"(gmem), "r"(n), "l"(pol)
               : "memory");
}
// 8-byte global -> shared copy (cp.async.ca); zero-fills when `valid` is false.
HS2_DEVI void cp_async8(uint32_t s, const void* gmem, bool valid) {
  const int n = valid ? 8 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
// 4-byte global -> shared copy (cp.async.ca); zero-fills when `valid` is false.
HS2_DEVI void cp_async4(uint32_t s, const void* gmem, bool valid) {
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
HS2_DEVI void st_shared_s32(uint32_t s, int v) { asm volatile("st.shared.s32 [%0], %1;" ::"r"(s), "r"(v) : "memory"); }
HS2_DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
HS2_DEVI void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Final scaling of an SA output from its merged state (max M and sum L of the weights,
// base 2): out = Ov * factor. b2 is the head's sink logit in base 2 (-inf: no sink), i.e.
// one more key with a zero value whose weight 2^(b2 - M) joins the denominator
// ("HySparse2：整体架构、KV 生命周期与 PD 分离", §17.1: per-head learnable sink bias).
HS2_DEVI float sa_norm_factor(float M, float L, float b2) {
  const float M2 = fmaxf(M, b2);
  const float sc = exp2_rel(M, M2);
  const float den = L * sc + exp2_rel(b2, M2);
  return den > 0.f ? sc / den : 0.f;
}
// The SA output's sigmoid gate (same section): out * 1 / (1 + e^-g).
HS2_DEVI float sa_gate(float g) { return 1.f / (1.f + __expf(-g)); }
HS2_DEVI float sink_b2(const float* sink, int head) { return sink ? sink[head] * kLog2e : -INFINITY; }

// FP8 E4M3 pairs to f16 pairs (exact: every E4M3 value is an f16 value); element order kept.
HS2_DEVI uint32_t fp8x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  const uint16_t v = (uint16_t)two_bytes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
// 4 E4M3 bytes to two f16 pairs: bytes (0, 1) -> lo, bytes (2, 3) -> hi, element order kept.
HS2_DEVI void fp8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// 8 E4M3 bytes (uint2) to 8 f16 (uint4), element order kept.
HS2_DEVI uint4 fp8x8_to_f16x8(uint2 b) {
  uint4 r;
  fp8x4_to_f16x4(b.x, r.x, r.y);
  fp8x4_to_f16x4(b.y, r.z, r.w);
  return r;
}
// 8 E2M1 codes (a 32-bit word; channel 2i in the low nibble of byte i) to 8 f16 as 4 pairs,
// order kept (cvt.rn.f16x2.e2m1x2 takes the low nibble to the low half).
HS2_DEVI void fp4x8_to_f16x8(uint32_t w, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm("{\n\t.reg .b8 a, b, c, d;\n\tmov.b32 {a, b, c, d}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, a;\n\tcvt.rn.f16x2.e2m1x2 %1, b;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, c;\n\tcvt.rn.f16x2.e2m1x2 %3, d;\n\t}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(w));
}
// f16 pair product (exact for an E2M1 value times an E4M3 scale: at most 5 significant bits,
// magnitude within [2^-10, 2688])
HS2_DEVI uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// The E4M3 scale byte `lo` (and `hi`) as an f16 pair (lo, hi).
HS2_DEVI uint32_t e4m3_pair(uint32_t lo, uint32_t hi) { return fp8x2_to_f16x2((lo & 0xFFu) | ((hi & 0xFFu) << 8)); }

// (lo, hi) floats to an f16 pair, round to nearest.
HS2_DEVI uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// bf16 pair to f16 pair (queries of an FP8 cache run the f16 MMA).
HS2_DEVI uint32_t bf16x2_to_f16x2(uint32_t x) {
  return pack_f16(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}
// m16n8k16 f16 MMA with fp32 accumulate.
HS2_DEVI void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                            uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

HS2_DEVI uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// ---------------------------------------------------------------------------- query geometry
// Query qi of a call: decode -> sequence qi, t = seq_len[qi];
// prefill -> sequence 0, t = qi + 1 (causal row qi).
struct QueryGeom {
  int b;
  int t;
};
HS2_DEVI QueryGeom query_geom(int qi, int prefill, const int32_t* seq_len) {
  QueryGeom q;
  if (prefill) {
    q.b = 0;
    q.t = qi + 1;
  } else {
    q.b = qi;
    q.t = seq_len[qi];
  }
  return q;
}

}  // namespace hs2
