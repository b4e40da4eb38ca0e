// fixed.cuh: the combine fused into the down-projection epilogue.
//
// "Nemotron 3 Nano" summary (shd-paper.top), 技术框架: the combination layer forms the
// gate-weighted sum of the chosen experts' outputs,
//   y[t, :] = sum_j gates[t, j] * out_j[t, :].
// Fused into the epilogue, the k terms of a token come from k tiles that run on different
// SMs in no fixed order. Each term g * v is therefore rounded once to a multiple of 2^-32
// and added to a 64-bit integer accumulator acc[t, :]: integer addition does not depend on
// the order, so the sum is the same on every run. A conversion pass then writes
// y = bf16(acc * 2^-32).
#pragma once

#include <cstdint>

#include "internal.h"

namespace moe {

constexpr float kFixedOne = 4294967296.f;  // 2^32: one unit of output in accumulator units
// Terms must stay below 2^26 in magnitude: 32 of them (the largest k) then sum to below
// 2^31 and the accumulator (2^63 / 2^32 = 2^31 units of output) cannot overflow.
constexpr float kFixedTermLimit = 67108864.f;

// acc[i] += round(term * 2^32); a term outside the range (or NaN) is not added and is
// reported as MOE_ERR_UNSUPPORTED on the status word.
__device__ __forceinline__ void fixed_add(unsigned long long* acc, float term, int* status) {
  if (!(fabsf(term) < kFixedTermLimit)) {
    atomicCAS(status, 0, MOE_ERR_UNSUPPORTED);
    return;
  }
  const long long q = __float2ll_rn(term * kFixedOne);  // the scaling by 2^32 is exact
  atomicAdd(acc, static_cast<unsigned long long>(q));   // two's complement: signed sum
}

// The bf16 nearest to q * 2^-32 (ties to even), from the integer itself: one rounding, in
// integer arithmetic (B300's FP64 rate is a small fraction of its FP32 rate). |q * 2^-32|
// lies in [2^-32, 2^31], always a normal bf16.
__host__ __device__ inline uint16_t fixed_to_bf16(long long q) {
  if (q == 0) return 0;
  const uint16_t sign = q < 0 ? 0x8000u : 0u;
  const unsigned long long m =
      q < 0 ? 0ull - static_cast<unsigned long long>(q) : static_cast<unsigned long long>(q);
#ifdef __CUDA_ARCH__
  const int msb = 63 - __clzll(static_cast<long long>(m));  // m != 0
#else
  const int msb = 63 - __builtin_clzll(m);
#endif
  int e = msb - 32;                    // m * 2^-32 = 1.f * 2^e
  unsigned long long sig;              // 8 significant bits, the leading one included
  if (msb > 7) {
    const int sh = msb - 7;
    sig = m >> sh;
    const unsigned long long rem = m & ((1ull << sh) - 1ull);
    const unsigned long long half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (sig & 1ull))) {
      if (++sig == 256ull) {
        sig = 128ull;
        ++e;
      }
    }
  } else {
    sig = m << (7 - msb);
  }
  return static_cast<uint16_t>(sign | (static_cast<unsigned>(e + 127) << 7) |
                               static_cast<unsigned>(sig & 0x7full));
}

// Token and gate of permuted row r: token[r], and the gate of the slot j of that token whose
// permuted row is r. Inconsistent maps give t = -1 and MOE_ERR_INVALID_ARG.
__device__ __forceinline__ void fixed_row_gate(const int32_t* token, const int32_t* slot_row,
                                               const float* gates, int k, int T, long long r,
                                               int* status, int& t, float& g) {
  t = -1;
  g = 0.f;
  const int tt = __ldg(token + r);
  if (tt < 0 || tt >= T) {
    atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
    return;
  }
  for (int j = 0; j < k; ++j) {
    if (__ldg(slot_row + static_cast<long long>(tt) * k + j) == r) {
      t = tt;
      g = __ldg(gates + static_cast<long long>(tt) * k + j);
      return;
    }
  }
  atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
}

}  // namespace moe
