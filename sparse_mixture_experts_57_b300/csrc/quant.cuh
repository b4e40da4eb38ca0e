// quant.cuh: packed fp32 arithmetic for the quantisers (FP8 and NVFP4), sm_100 and later.
//
// Both quantisers divide every value by a scale with a correctly rounded quotient, by
// Markstein's method (P. Markstein, IBM J. Res. Dev. 34(1), 1990): y = RN(1/d), q = RN(v y),
// r = v - q d (exact in one fma), RN(q + r y) = RN(v / d), valid for 2^-100 < d < 2^100 and
// |v / d| < 2^100. Here it runs on pairs with the f32x2 forms of mul and fma, which round
// each lane exactly as the scalar instructions do, so the quotients are the same bits at
// half the instruction count.
#pragma once
#include <cstdint>

namespace moe {

__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// The two bf16 values of a 32-bit word (low half first) divided by d: y2 = (RN(1/d), RN(1/d)),
// nd2 = (-d, -d). fma(q, -d, v) is the same rounded value as fma(-q, d, v).
__device__ __forceinline__ void div2_markstein_bf16(uint32_t w, uint64_t y2, uint64_t nd2,
                                                    float& lo, float& hi) {
  const uint64_t v = f32x2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  uint64_t q, r, o;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q) : "l"(v), "l"(y2));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q), "l"(nd2), "l"(v));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(o) : "l"(r), "l"(y2), "l"(q));
  f32x2_unpack(o, lo, hi);
}

}  // namespace moe
