// Shared device helpers for the qffn kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define QFFN_DEVI __device__ __forceinline__
#define QFFN_DEVI_HOST __host__ __device__ __forceinline__

namespace qffn {

constexpr int kNumSMsHint = 152;

// ----------------------------------------------------------------- bf16 bits
QFFN_DEVI float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
QFFN_DEVI float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
QFFN_DEVI float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// fp32 -> bf16, round to nearest even (the cvt instruction; finite inputs).
QFFN_DEVI uint16_t f32_to_bf16(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}
// Two fp32 -> packed bf16x2 (lo in the low half).
QFFN_DEVI uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Round through bf16 and back.
QFFN_DEVI float round_bf16(float f) { return bf16_to_f32(f32_to_bf16(f)); }

// ----------------------------------------------------------------- e4m3
// Two fp32 -> packed E4M3x2 (lo in the low byte), nearest even, saturating.
QFFN_DEVI uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 4 packed E4M3 codes -> 4 floats (exact), via the e4m3x2 -> f16x2 cvt.
QFFN_DEVI void e4m3x4_to_f32(uint32_t w, float& f0, float& f1, float& f2, float& f3) {
  uint32_t h01, h23;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(uint16_t(w & 0xFFFF)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(uint16_t(w >> 16)));
  __half2 a = *reinterpret_cast<__half2*>(&h01);
  __half2 b = *reinterpret_cast<__half2*>(&h23);
  float2 fa = __half22float2(a), fb = __half22float2(b);
  f0 = fa.x; f1 = fa.y; f2 = fb.x; f3 = fb.y;
}

// ----------------------------------------------------------------- double-float
// A value carried as an unevaluated sum hi + lo of two floats (about 48
// significant bits).  two_sum is Knuth's error-free addition: s = fl(a + b)
// and e = (a + b) - s exactly.
QFFN_DEVI void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
// (hi, lo) += x
QFFN_DEVI void df_add(float& hi, float& lo, float x) {
  float s, e;
  two_sum(hi, x, s, e);
  hi = s;
  lo += e;
}
// (hi, lo) += (bhi, blo), renormalised so |lo| <= ulp(hi) / 2
QFFN_DEVI void df_add_df(float& hi, float& lo, float bhi, float blo) {
  float s, e;
  two_sum(hi, bhi, s, e);
  e += lo + blo;
  hi = s + e;
  lo = e - (hi - s);
}
// (hi, lo) <- fl(hi + lo) and its exact error; needs |hi| >= |lo| (Dekker).
QFFN_DEVI void fast_two_sum(float& hi, float& lo) {
  const float s = hi + lo;
  lo = lo - (s - hi);
  hi = s;
}
// Round the double-float th + tl to bf16, nearest-even, as one rounding.  After
// renormalisation th is the float nearest to th + tl, so th's own bf16
// rounding is the right one unless th sits exactly halfway between two bf16
// values; there the sign of tl (relative to th) picks the side.
QFFN_DEVI uint32_t bf16_round_df(float th, float tl) {
  if (tl != 0.0f) fast_two_sum(th, tl);   // (tl == 0 keeps the sign of a zero th)
  const uint32_t bits = __float_as_uint(th);
  uint32_t b = f32_to_bf16(th);
  if ((bits & 0xFFFFu) == 0x8000u && tl != 0.0f) b = (bits >> 16) + (((tl > 0.0f) == (th > 0.0f)) ? 1u : 0u);
  return b;
}

// ----------------------------------------------------------------- packed fp32 pairs
// Two floats in one 64-bit register, operated on by the f32x2 instructions.
QFFN_DEVI uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
QFFN_DEVI void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
QFFN_DEVI uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
QFFN_DEVI uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
QFFN_DEVI uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
QFFN_DEVI uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// the two bf16 halves of a 32-bit word as a float pair (low half first)
QFFN_DEVI uint64_t bf16x2_to_f2(uint32_t w) { return f2_pack(bf16_lo(w), bf16_hi(w)); }
// (hi, lo) += x lane by lane, two_sum on pairs
QFFN_DEVI void f2_df_add(uint64_t& hi, uint64_t& lo, uint64_t x) {
  const uint64_t s = f2_add(hi, x);
  const uint64_t bb = f2_sub(s, hi);
  const uint64_t e = f2_add(f2_sub(hi, f2_sub(s, bb)), f2_sub(x, bb));
  hi = s;
  lo = f2_add(lo, e);
}

// ----------------------------------------------------------------- SwiGLU
// silu(g) * u in fp32.  silu(g) = g * sigmoid(g); the sigmoid is formed from
// e = exp(-|g|) in (0, 1] so neither branch overflows:
//   g >= 0: 1 / (1 + e);   g < 0: e / (1 + e).
QFFN_DEVI float silu_mul_f32(float g, float u) {
  float e = __expf(-fabsf(g));
  float r = __fdividef(1.0f, 1.0f + e);
  float sig = g >= 0.0f ? r : e * r;
  return (g * sig) * u;
}

// Gradient of silu(g) * u: dg = dh * u * silu'(g), du = dh * silu(g), in fp32
// (each rounded once to bf16 by the caller).  silu'(g) = s * (1 + g * (1 - s))
// with s = sigmoid(g) formed from e = exp(-|g|) as in silu_mul_f32.
QFFN_DEVI void swiglu_grad(float g, float u, float dh, float& dg, float& du) {
  const float e = __expf(-fabsf(g));
  const float r = __fdividef(1.0f, 1.0f + e);
  const float s = g >= 0.0f ? r : e * r;
  dg = (dh * u) * (s * (1.0f + g * (1.0f - s)));
  du = dh * (g * s);
}

// h = bf16(silu(g) * u) for the 8 bf16 pairs of two 16-byte vectors.
QFFN_DEVI uint4 swiglu8(uint4 g, uint4 u) {
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    o[j] = pack_bf16x2(silu_mul_f32(bf16_lo(gw[j]), bf16_lo(uw[j])),
                       silu_mul_f32(bf16_hi(gw[j]), bf16_hi(uw[j])));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// ----------------------------------------------------------------- abs-max
// Non-negative floats order like their bit patterns as unsigned integers, so
// a tensor abs-max is an atomicMax on the bits.
QFFN_DEVI void atomic_max_nonneg(float* addr, float v) {
  atomicMax(reinterpret_cast<unsigned int*>(addr), __float_as_uint(v));
}

QFFN_DEVI float warp_max(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

QFFN_DEVI float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 16-byte global loads / stores.
// ld16_ro: data that no thread writes during the kernel (weights, gain).
// ld16_once: plain coherent load (activations that a call may overwrite in
// place afterwards; a plain load keeps the compiler's aliasing order).
QFFN_DEVI uint4 ld16_ro(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
QFFN_DEVI uint4 ld16_ro_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
QFFN_DEVI uint4 ld16_once(const void* p) { return *reinterpret_cast<const uint4*>(p); }
QFFN_DEVI void stg16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Programmatic dependent launch: wait for the preceding kernel's results /
// let the next kernel start launching.  Both are no-ops without the launch
// attribute.
QFFN_DEVI void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
QFFN_DEVI void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace qffn
