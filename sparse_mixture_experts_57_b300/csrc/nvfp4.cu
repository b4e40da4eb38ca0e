// nvfp4.cu: NVFP4 quantisation of expert weights and routed activations.
//
// "NVIDIA Nemotron 3: Efficient and Open Intelligence" notes, §2.4: NVFP4 holds E2M1
// elements in 16-element micro-blocks, each block with an E4M3 scale, plus a second-level
// FP32 scale per tensor. For one tensor with global scale g = amax / (6 * 448):
//   block scale  sb = E4M3(amax(block) / (6 g))            (nearest, ties to even, saturating)
//   element code q  = E2M1(v / (sb g))                      (nearest, ties to the even code,
//                                                            saturating at 6)
//   value           = q * sb * g
// Blocks run along the contraction axis K. Every decision is taken in fp32 with correctly
// rounded division, so the codes and scales depend only on the input bits (and match an
// fp32 evaluation of the same formulas exactly).
//
// Layouts (shared with the block-scaled grouped GEMM): codes [rows, K/2], element 2i in the
// low nibble (weights: rows K/2 bytes apart; routed activations: fp4_act_pitch(K) apart); scales as 512-byte atoms, one per (128-row block, 64-element K step): row
// 128 rb + 32 r1 + r0, block kb of the step at byte r0 * 16 + r1 * 4 + kb. One thread
// quantises one row's 64-element K step: 128 bytes in, 32 code bytes and one 32-bit word of
// four scales out (for routed activations the warp loads its 32 steps cooperatively).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "quant.cuh"
#include "scan.cuh"

namespace moe {
namespace {

// Eight values rounded to E2M1 (nearest, ties to the even code, saturating at +-6) and
// packed two per byte, element 2i in the low nibble: the hardware's round-to-nearest-even
// conversion of fp32 to E2M1 pairs (the first source operand goes to the high nibble).
__device__ __forceinline__ uint32_t e2m1x8(const float (&q)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]),
        "f"(q[7]));
  return r;
}

// v / d correctly rounded, for a divisor d with 2^-100 < d < 2^100 and |v / d| < 2^100:
// Markstein's division by fused multiply-add (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// y = RN(1/d) and q = RN(v y), the remainder r = v - q d is exact in one fma, and
// RN(q + r y) = RN(v / d).
__device__ __forceinline__ float div_markstein(float v, float d, float y) {
  const float q = __fmul_rn(v, y);
  const float r = fmaf(-q, d, v);
  return fmaf(r, y, q);
}

// Value of a non-negative E4M3 byte: exponent bias 7, 3 mantissa bits, subnormals below 2^-6.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  if (e == 0u) return static_cast<float>(m) * (1.0f / 512.0f);
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

__device__ __forceinline__ float global_scale(const uint32_t* amax) {
  return __fdiv_rn(__uint_as_float(*amax), kNvfp4GlobalDiv);
}

// Quantise 64 consecutive bf16 values, eight 16-byte vectors that load(m) returns for
// m = 0..7 (each fetched when its block is quantised). Writes 32 code bytes and returns the
// four block-scale bytes packed little-endian (block 0 in the low byte).
template <class Load>
__device__ __forceinline__ uint32_t quant64_from(Load load, float g, uint4* dst) {
  uint32_t sf = 0u;
  uint32_t q[8];
  const float six_g = __fmul_rn(6.0f, g);
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) {
    const uint4 a = load(2 * blk), b = load(2 * blk + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
    float bmax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
    uint32_t sb = 0u;
    float denom = 0.f;
    if (g > 0.f) {
      sb = static_cast<uint32_t>(
          __nv_cvt_float_to_fp8(__fdiv_rn(bmax, six_g), __NV_SATFINITE, __NV_E4M3));
      denom = __fmul_rn(e4m3_value(sb), g);
    }
    float s[16];
    if (denom > 0x1p-100f && denom < 0x1p100f) {
      const float y = __frcp_rn(denom);
      const uint64_t y2 = f32x2_pack(y, y), nd2 = f32x2_pack(-denom, -denom);
#pragma unroll
      for (int i = 0; i < 8; ++i) div2_markstein_bf16(w[i], y2, nd2, s[2 * i], s[2 * i + 1]);
    } else if (denom > 0.f) {  // outside the range of the fast division
#pragma unroll
      for (int i = 0; i < 16; ++i) s[i] = __fdiv_rn(v[i], denom);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) s[i] = 0.f;
    }
    const float lo[8] = {s[0], s[1], s[2], s[3], s[4], s[5], s[6], s[7]};
    const float hi[8] = {s[8], s[9], s[10], s[11], s[12], s[13], s[14], s[15]};
    q[2 * blk] = e2m1x8(lo);
    q[2 * blk + 1] = e2m1x8(hi);
    sf |= sb << (8 * blk);
  }
  dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
  dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
  return sf;
}

// The same from global memory (src 16-byte aligned).
__device__ __forceinline__ uint32_t quant64(const uint4* __restrict__ src, float g, uint4* dst) {
  return quant64_from([src](int m) { return __ldg(src + m); }, g, dst);
}

// Codes of 16 values with block divisor denom = sb * g (0 gives zero codes): two words,
// element 2i in the low nibble of its byte.
__device__ __forceinline__ void code16(const float (&v)[16], float denom, uint32_t& w0,
                                       uint32_t& w1) {
  float s[16];
  if (denom > 0x1p-100f && denom < 0x1p100f) {
    const float y = __frcp_rn(denom);
#pragma unroll
    for (int i = 0; i < 16; ++i) s[i] = div_markstein(v[i], denom, y);
  } else if (denom > 0.f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) s[i] = __fdiv_rn(v[i], denom);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) s[i] = 0.f;
  }
  const float lo[8] = {s[0], s[1], s[2], s[3], s[4], s[5], s[6], s[7]};
  const float hi[8] = {s[8], s[9], s[10], s[11], s[12], s[13], s[14], s[15]};
  w0 = e2m1x8(lo);
  w1 = e2m1x8(hi);
}

__device__ __forceinline__ uint32_t* sf_word(uint8_t* sf, long long row, int j, int KS) {
  const long long rb = row >> 7;
  const int r = static_cast<int>(row & 127);
  return reinterpret_cast<uint32_t*>(sf + (rb * KS + j) * 512 + (r & 31) * 16 + (r >> 5) * 4);
}

__global__ void k_amax_bf16(const uint16_t* __restrict__ src, long long per_matrix,
                            uint32_t* __restrict__ amax) {
  griddep_wait();
  griddep_launch_dependents();
  const int g = blockIdx.y;
  const uint4* p = reinterpret_cast<const uint4*>(src + static_cast<long long>(g) * per_matrix);
  const long long nvec = per_matrix / 8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  uint32_t m = 0u;
  auto fold = [&m](const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7fffu, (w[k] >> 16) & 0x7fffu));
  };
  long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  // four independent 16-byte loads in flight per thread
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    const uint4 v0 = __ldg(p + i), v1 = __ldg(p + i + stride), v2 = __ldg(p + i + 2 * stride),
                v3 = __ldg(p + i + 3 * stride);
    fold(v0);
    fold(v1);
    fold(v2);
    fold(v3);
  }
  for (; i < nvec; i += stride) fold(__ldg(p + i));
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
  // |bf16| bit patterns order like their values; as fp32 bits they keep that order.
  if ((threadIdx.x & 31) == 0 && m) atomicMax(amax + g, m << 16);
}

__global__ void k_quant_weights(const uint16_t* __restrict__ w, int G, int N, int K,
                                const uint32_t* __restrict__ amax, uint8_t* __restrict__ codes,
                                uint8_t* __restrict__ sf) {
  griddep_wait();
  griddep_launch_dependents();
  const int KS = K / 64;
  const long long rows_pad = static_cast<long long>((N + 127) / 128) * 128;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= G * rows_pad * KS) return;
  const long long ar = i / KS;  // row in the padded stack of G matrices
  const int j = static_cast<int>(i - ar * KS);
  const int g = static_cast<int>(ar / rows_pad);
  const int n = static_cast<int>(ar - g * rows_pad);
  uint32_t* word = sf_word(sf, ar, j, KS);
  if (n >= N) {  // rows past N in the last 128-row block: zero scales
    *word = 0u;
    return;
  }
  const long long row = static_cast<long long>(g) * N + n;
  uint4 out[2];
  *word = quant64(reinterpret_cast<const uint4*>(w + row * K + j * 64), global_scale(amax + g),
                  out);
  uint4* dst = reinterpret_cast<uint4*>(codes + row * (K / 2) + j * 32);
  dst[0] = out[0];
  dst[1] = out[1];
}

// 2-D weight blocks: one thread per (matrix, 16-row group, 16-element K block). The block
// scale comes from the amax of the whole 16 x 16 block and is written for each of its rows;
// rows past N in the last 128-row scale block get zero scales.
__global__ void k_quant_weights_2d(const uint16_t* __restrict__ w, int G, int N, int K,
                                   const uint32_t* __restrict__ amax, uint8_t* __restrict__ codes,
                                   uint8_t* __restrict__ sf) {
  griddep_wait();
  griddep_launch_dependents();
  const int KS = K / 64, NB = K / 16;
  const long long rows_pad = static_cast<long long>((N + 127) / 128) * 128;
  const long long groups = rows_pad / 16;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= G * groups * NB) return;
  const long long gi = i / NB;            // 16-row group in the padded stack
  const int b = static_cast<int>(i - gi * NB);
  const int g = static_cast<int>(gi / groups);
  const int r0 = static_cast<int>(gi - g * groups) * 16;
  const int nrows = max(0, min(16, N - r0));
  const float gs = global_scale(amax + g);
  float bmax = 0.f;
  for (int r = 0; r < nrows; ++r) {
    const uint16_t* p = w + (static_cast<long long>(g) * N + r0 + r) * K + b * 16;
    for (int c = 0; c < 16; ++c) bmax = fmaxf(bmax, fabsf(__uint_as_float(static_cast<uint32_t>(p[c]) << 16)));
  }
  uint32_t sb = 0u;
  float denom = 0.f;
  if (gs > 0.f) {
    sb = static_cast<uint32_t>(
        __nv_cvt_float_to_fp8(__fdiv_rn(bmax, __fmul_rn(6.0f, gs)), __NV_SATFINITE, __NV_E4M3));
    denom = __fmul_rn(e4m3_value(sb), gs);
  }
  for (int r = 0; r < 16; ++r) {
    const long long ar = static_cast<long long>(g) * rows_pad + r0 + r;  // padded stack row
    uint8_t* sfb = reinterpret_cast<uint8_t*>(sf_word(sf, ar, b >> 2, KS)) + (b & 3);
    if (r >= nrows) {
      *sfb = 0;
      continue;
    }
    *sfb = static_cast<uint8_t>(sb);
    const long long row = static_cast<long long>(g) * N + r0 + r;
    const uint16_t* p = w + row * K + b * 16;
    float v[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) v[c] = __uint_as_float(static_cast<uint32_t>(p[c]) << 16);
    uint32_t w0, w1;
    code16(v, denom, w0, w1);
    *reinterpret_cast<uint2*>(codes + row * (K / 2) + b * 8) = make_uint2(w0, w1);
  }
}

__global__ void k_finalize_gscale(float* g, int G) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < G) g[i] = __fdiv_rn(g[i], kNvfp4GlobalDiv);  // g[i] holds amax as fp32 bits
}

__global__ void k_pad_offsets(const int32_t* __restrict__ offsets, int E,
                              int32_t* __restrict__ poff, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int warp_sums[33];
  const int e = threadIdx.x;
  int c = 0;
  if (e < E) {
    c = offsets[e + 1] - offsets[e];
    if (c < 0) {
      atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
      c = 0;
    }
    c = (c + 127) & ~127;
  }
  int total;
  const int excl = block_exclusive_scan(c, warp_sums, &total);
  if (e < E) poff[e] = excl;
  if (e == 0) poff[E] = total;
}

constexpr int kQuantThreads = 256;

// Routed activations: one thread per (row, 64-element K step), as for weights, but the warp
// first loads its 32 x 128 bytes cooperatively: in each of eight rounds, eight consecutive
// lanes read one thread's 128-byte step (its row comes by shuffle), so every load covers
// four whole 128-byte lines, and the vectors go through a per-warp shared-memory buffer,
// XOR-swizzled so that neither the stores nor the per-thread reads conflict on banks.
// (Each thread reading its own 128 bytes directly costs eight L1 wavefronts per line.)
__global__ void __launch_bounds__(kQuantThreads, 4)
    k_quant_act(const uint16_t* __restrict__ src, long long ld, long long src_rows,
                const int32_t* __restrict__ row_token, const int32_t* __restrict__ offsets,
                const int32_t* __restrict__ poff, int E, int K, int P_max,
                const uint32_t* __restrict__ amax, uint8_t* __restrict__ codes,
                uint8_t* __restrict__ sf, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint4 s_dyn[];  // [8 warps][256 vectors], then poff[E+1]
  const int lane = threadIdx.x & 31;
  uint4* stage = s_dyn + (threadIdx.x >> 5) * 256;
  int* s_poff = reinterpret_cast<int*>(s_dyn + (kQuantThreads / 32) * 256);
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_poff[i] = poff[i];
  __syncthreads();
  const int KS = K / 64;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long p = i / KS;
  const int j = static_cast<int>(i - p * KS);
  const bool valid = p < s_poff[E] && p < P_max;
  long long srow = -1;  // -1: no source row (past the end, or a padding row of a segment)
  if (valid) {
    srow = p;
    if (offsets) {
      int lo = 0, hi = E - 1;  // expert e with s_poff[e] <= p < s_poff[e+1]
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_poff[mid + 1] > p)
          hi = mid;
        else
          lo = mid + 1;
      }
      const int local = static_cast<int>(p - s_poff[lo]);
      const int base = offsets[lo];
      if (local < offsets[lo + 1] - base) {
        srow = row_token ? row_token[base + local] : base + local;
        if (srow < 0) srow = src_rows;  // a negative token id is as invalid as a large one
      } else {
        srow = -1;  // padding row of the segment
      }
    }
    if (srow >= src_rows) {  // offsets or row_token outside the source tensor
      if (j == 0) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
      srow = -1;
    }
  }
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int owner = 4 * it + (lane >> 3);  // the thread whose step these 8 lanes load
    const long long so = __shfl_sync(0xffffffffu, srow, owner);
    const int jo = __shfl_sync(0xffffffffu, j, owner);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (so >= 0)
      v = __ldg(reinterpret_cast<const uint4*>(src + so * ld + jo * 64 + (lane & 7) * 8));
    const int c = 32 * it + lane;  // vector c & 7 of thread c >> 3
    stage[(c & ~7) | ((c & 7) ^ ((c >> 3) & 7))] = v;
  }
  __syncwarp();
  if (!valid) return;
  uint32_t* word = sf_word(sf, p, j, KS);
  uint4* dst = reinterpret_cast<uint4*>(codes + p * fp4_act_pitch(K) + j * 32);
  if (srow < 0) {  // padding row of a segment
    *word = 0u;
    dst[0] = make_uint4(0u, 0u, 0u, 0u);
    dst[1] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  uint4 out[2];
  const uint4* mine = stage + 8 * lane;
  const int sw = lane & 7;
  *word = quant64_from([mine, sw](int m) { return mine[m ^ sw]; }, global_scale(amax), out);
  dst[0] = out[0];
  dst[1] = out[1];
}

// Routed tokens, each quantised once and written to every one of its k rows of the padded
// expert order: slot j of token t goes to row poff[e] + (slot_row[t k + j] - offsets[e]) with
// e = topk_idx[t k + j]. A token's codes and block scales are the same in all its copies (the
// global scale is that of the whole token tensor), so this gives the bytes that quantising
// each gathered row (k_quant_act) gives, with a sixth of the arithmetic and of the reads at
// top-6. One thread per (token, 64-element K step); a warp loads its 32 steps cooperatively
// as k_quant_act does. The padding rows of each segment are written by k_zero_padding_rows.
__global__ void __launch_bounds__(kQuantThreads, 4)
    k_quant_tokens(const uint16_t* __restrict__ src, long long ld, int T, int k,
                   const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot_row,
                   const int32_t* __restrict__ offsets, const int32_t* __restrict__ poff, int E,
                   int K, int P_max, const uint32_t* __restrict__ amax,
                   uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint4 s_dyn[];  // [8 warps][256 vectors]
  const int lane = threadIdx.x & 31;
  uint4* stage = s_dyn + (threadIdx.x >> 5) * 256;
  const int KS = K / 64;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long t = i / KS;
  const int j = static_cast<int>(i - t * KS);
  const bool valid = t < T;
  const long long srow = valid ? t : -1;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int owner = 4 * it + (lane >> 3);  // the thread whose step these 8 lanes load
    const long long so = __shfl_sync(0xffffffffu, srow, owner);
    const int jo = __shfl_sync(0xffffffffu, j, owner);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (so >= 0)
      v = __ldg(reinterpret_cast<const uint4*>(src + so * ld + jo * 64 + (lane & 7) * 8));
    const int c = 32 * it + lane;  // vector c & 7 of thread c >> 3
    stage[(c & ~7) | ((c & 7) ^ ((c >> 3) & 7))] = v;
  }
  __syncwarp();
  if (!valid) return;
  uint4 out[2];
  const uint4* mine = stage + 8 * lane;
  const int sw = lane & 7;
  const uint32_t word = quant64_from([mine, sw](int m) { return mine[m ^ sw]; },
                                     global_scale(amax), out);
  for (int s = 0; s < k; ++s) {
    const int e = __ldg(topk_idx + t * k + s);
    const int r = __ldg(slot_row + t * k + s);
    bool ok = e >= 0 && e < E;
    long long p = -1;
    if (ok) {
      const int o0 = __ldg(offsets + e), o1 = __ldg(offsets + e + 1);
      ok = r >= o0 && r < o1;
      if (ok) p = static_cast<long long>(__ldg(poff + e)) + (r - o0);
      ok = ok && p < P_max;
    }
    if (!ok) {
      if (j == 0) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
      continue;
    }
    *sf_word(sf, p, j, KS) = word;
    uint4* dst = reinterpret_cast<uint4*>(codes + p * fp4_act_pitch(K) + j * 32);
    dst[0] = out[0];
    dst[1] = out[1];
  }
}

// The padding rows of every expert segment (rows past the expert's count up to the next
// 128-row boundary): zero codes and zero block scales. One block per expert.
__global__ void k_zero_padding_rows(const int32_t* __restrict__ offsets,
                                    const int32_t* __restrict__ poff, int E, int K, int P_max,
                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  griddep_wait();
  griddep_launch_dependents();
  const int e = blockIdx.x;
  if (e >= E) return;
  const int KS = K / 64;
  const long long p0 = static_cast<long long>(__ldg(poff + e)) +
                       (__ldg(offsets + e + 1) - __ldg(offsets + e));
  const long long p1 = min(static_cast<long long>(__ldg(poff + e + 1)), static_cast<long long>(P_max));
  const long long n = (p1 - p0) * KS;
  for (long long q = threadIdx.x; q < n; q += blockDim.x) {
    const long long p = p0 + q / KS;
    const int j = static_cast<int>(q % KS);
    *sf_word(sf, p, j, KS) = 0u;
    uint4* dst = reinterpret_cast<uint4*>(codes + p * fp4_act_pitch(K) + j * 32);
    dst[0] = make_uint4(0u, 0u, 0u, 0u);
    dst[1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace

int launch_amax_bf16(const uint16_t* src, long long elems_per_matrix, int G, uint32_t* amax,
                     cudaStream_t s) {
  if (G <= 0 || elems_per_matrix <= 0) return MOE_OK;
  const long long nvec = elems_per_matrix / 8;
  long long blocks = (nvec + 255) / 256;
  // one matrix: eight 256-thread blocks per SM; more matrices (grid.y) fill the GPU sooner
  const long long cap = (G == 1 ? 8LL : 4LL) * sm_count();
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(k_amax_bf16, dim3(static_cast<unsigned>(blocks), G), dim3(256), 0, s, src,
                    elems_per_matrix, amax);
}

int launch_quant_weights(const uint16_t* w, int G, int N, int K, const uint32_t* amax,
                         uint8_t* codes, uint8_t* sf, cudaStream_t s) {
  const long long n = static_cast<long long>(G) * ((N + 127) / 128) * 128 * (K / 64);
  if (n <= 0) return MOE_OK;
  return launch_pdl(k_quant_weights, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                    s, w, G, N, K, amax, codes, sf);
}

int launch_quant_weights_2d(const uint16_t* w, int G, int N, int K, const uint32_t* amax,
                            uint8_t* codes, uint8_t* sf, cudaStream_t s) {
  const long long n = static_cast<long long>(G) * ((N + 127) / 128) * 8 * (K / 16);
  if (n <= 0) return MOE_OK;
  return launch_pdl(k_quant_weights_2d, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256),
                    0, s, w, G, N, K, amax, codes, sf);
}

int launch_finalize_gscale(float* g, int G, cudaStream_t s) {
  return launch_pdl(k_finalize_gscale, dim3((G + 255) / 256), dim3(256), 0, s, g, G);
}

int launch_pad_offsets(const int32_t* offsets, int E, int32_t* poff, cudaStream_t s) {
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  return launch_pdl(k_pad_offsets, dim3(1), dim3(1024), 0, s, offsets, E, poff, status);
}

int launch_quant_act(const uint16_t* src, long long ld, long long src_rows,
                     const int32_t* row_token, const int32_t* offsets, const int32_t* poff,
                     int E, int K, int P_max, const uint32_t* amax, uint8_t* codes, uint8_t* sf,
                     cudaStream_t s) {
  const long long n = static_cast<long long>(P_max) * (K / 64);
  if (n <= 0) return MOE_OK;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  const size_t smem = (kQuantThreads / 32) * 256 * sizeof(uint4) + static_cast<size_t>(E + 1) * 4;
  return launch_pdl(k_quant_act, dim3(static_cast<unsigned>((n + kQuantThreads - 1) / kQuantThreads)),
                    dim3(kQuantThreads), smem, s, src, ld, src_rows,
                    row_token, offsets, poff, E, K, P_max, amax, codes, sf, status);
}

int launch_quant_tokens(const uint16_t* src, long long ld, int T, int k, const int32_t* topk_idx,
                        const int32_t* slot_row, const int32_t* offsets, const int32_t* poff,
                        int E, int K, int P_max, const uint32_t* amax, uint8_t* codes,
                        uint8_t* sf, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  const long long n = static_cast<long long>(T) * (K / 64);
  const size_t smem = (kQuantThreads / 32) * 256 * sizeof(uint4);
  int st = launch_pdl(k_quant_tokens,
                      dim3(static_cast<unsigned>((n + kQuantThreads - 1) / kQuantThreads)),
                      dim3(kQuantThreads), smem, s, src, ld, T, k, topk_idx, slot_row, offsets,
                      poff, E, K, P_max, amax, codes, sf, status);
  if (st) return st;
  return launch_pdl(k_zero_padding_rows, dim3(E), dim3(256), 0, s, offsets, poff, E, K, P_max,
                    codes, sf);
}

}  // namespace moe
