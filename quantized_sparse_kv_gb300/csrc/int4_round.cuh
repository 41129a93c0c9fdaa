// Exact int4 codes without a division per element (the bf16 kv_pack path).
//
// The grouped int4 rule of the residual-window page ("KV殘差窗口", section
// 固定預算) as this library states it: scale = fl(amax / 7), code =
// clamp(rint(fl(x / scale)), -7, 7), the divisions correctly rounded in fp32
// and rint to nearest, ties to even. Here the quotient comes from the
// correctly rounded reciprocal r = fl(1 / s) and one correction step
// (Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = fl(x r), the
// residual e = x - q0 s exact through an fma, q = fl(q0 + e r). Adding
// 1.5 * 2^23 + 8 then rounds q to an integer, ties to even, and leaves
// code + 8 in bits 0-3 (bits 4-7 zero). The scale is formed the same way from
// fl(1 / 7). The clamp never binds: |x| <= amax puts fl(x / s) below 7.5.
//
// Every function is host and device code with the same arithmetic on both
// (the device intrinsics are the IEEE operations the host performs), so the
// CPU tests compile this file and check it, on every bf16 pair (amax, x)
// with |x| <= amax, against the correctly rounded division: equal wherever
// recip_ok(amax) holds, which is what the kernels test before taking it.
#pragma once

#include <stdint.h>
#include <string.h>

#include <cmath>

namespace kvq {

__host__ __device__ __forceinline__ float mul_rn(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fmul_rn(a, b);
#else
  return a * b;
#endif
}
__host__ __device__ __forceinline__ float add_rn(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fadd_rn(a, b);
#else
  return a + b;
#endif
}
__host__ __device__ __forceinline__ float fma_rn(float a, float b, float c) {
#ifdef __CUDA_ARCH__
  return __fmaf_rn(a, b, c);
#else
  return std::fma(a, b, c);
#endif
}
__host__ __device__ __forceinline__ float rcp_rn(float s) {  // fl(1 / s)
#ifdef __CUDA_ARCH__
  return __frcp_rn(s);
#else
  return 1.0f / s;
#endif
}
__host__ __device__ __forceinline__ uint32_t bits_of(float f) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(f);
#else
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
#endif
}

// A group maximum the reciprocal path handles: zero, or finite and at least
// 2^-100 (below about 2^-119.6 the residual of a near-tie is no longer exact).
__host__ __device__ __forceinline__ bool recip_ok(float amax) {
  return amax == 0.0f || (amax >= 0x1p-100f && amax <= 3.40282347e38f);
}

// fl(amax / 7) for amax with recip_ok(amax).
__host__ __device__ __forceinline__ float scale_recip(float amax) {
  constexpr float r7 = 1.0f / 7.0f;
  const float q0 = mul_rn(amax, r7);
  return fma_rn(fma_rn(-q0, 7.0f, amax), r7, q0);
}

// The reciprocal the codes use (0 for a zero scale, whose codes are all 0).
__host__ __device__ __forceinline__ float recip_of(float s) {
  return s == 0.0f ? 0.0f : rcp_rn(s);
}

// code + 8 in bits 0-3 of the result (bits 4-7 zero), for |x| <= amax.
__host__ __device__ __forceinline__ uint32_t code8_recip(float x, float s, float r) {
  const float q0 = mul_rn(x, r);
  const float q = fma_rn(fma_rn(-q0, s, x), r, q0);
  return bits_of(add_rn(q, 12582920.0f));  // 1.5 * 2^23 + 8
}

// One code byte from a pair of bf16 values (the low half of w in the low
// nibble), each with its own scale: on the device the four operations run
// on both halves at once as packed f32x2 instructions (per half the same
// IEEE operations); ns = -s.
__host__ __device__ __forceinline__ uint32_t code_byte_recip(uint32_t w, float ns_lo, float ns_hi,
                                                             float r_lo, float r_hi) {
  uint32_t lo_bits = w << 16, hi_bits = w & 0xffff0000u;
#ifdef __CUDA_ARCH__
  uint64_t x, ns, r, q0, e, q, y;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(lo_bits), "r"(hi_bits));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ns) : "f"(ns_lo), "f"(ns_hi));
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(r_lo), "f"(r_hi));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(x), "l"(r));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q0), "l"(ns), "l"(x));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(e), "l"(r), "l"(q0));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(q), "l"(0x4B4000084B400008ull));
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo_bits), "=r"(hi_bits) : "l"(y));
  return hi_bits * 16u + lo_bits;
#else
  float lo, hi;
  memcpy(&lo, &lo_bits, 4);
  memcpy(&hi, &hi_bits, 4);
  return (code8_recip(hi, -ns_hi, r_hi) * 16u + code8_recip(lo, -ns_lo, r_lo)) & 0xffu;
#endif
}

}  // namespace kvq
