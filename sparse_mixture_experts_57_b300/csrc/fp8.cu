// fp8.cu: per-tensor E4M3 quantisation of expert weights and routed activations.
//
// "Nemotron 3 Nano" summary (papers.lianghsun.dev), §4: FP8 post-training quantisation with
// selective precision; BF16 and FP8 weights are released. The pages give no scaling
// granularity; this library's reading is one FP32 scale per tensor:
//   s = amax / 448,   q = E4M3(v / s)   (nearest, ties to even, saturating at +-448)
// with each expert matrix, the whole routed-token tensor and the whole h as the tensors.
// The division is correctly rounded (Markstein's FMA correction after a correctly rounded
// reciprocal, on value pairs: quant.cuh), so the codes are those of an fp32 evaluation of
// the rule.
#include "internal.h"
#include "quant.cuh"

namespace moe {
namespace {

// Two E4M3 bytes, lo in the low byte (the conversion puts its first source in the high
// byte): nearest, ties to even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

constexpr int kFp8SegVec = 128;  // 16-byte vectors (8 values) per warp segment

// One warp per (row, 1024-value segment): lane t converts the vectors t, t+32, t+64, t+96
// of the segment, so each 16-byte load and each 8-byte code store of the warp is contiguous.
// The quantisation is elementwise, so no lane needs its neighbours' values. Output rows are
// ldo bytes apart.
__global__ void k_quant_fp8(const uint16_t* __restrict__ src, long long ld,
                            const int32_t* __restrict__ row_map, long long rows, int K,
                            long long rows_per_scale, const uint32_t* __restrict__ amax,
                            uint8_t* __restrict__ out, long long ldo) {
  griddep_wait();
  griddep_launch_dependents();
  const int nvec = K / 8;
  const int segs = (nvec + kFp8SegVec - 1) / kFp8SegVec;
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= rows * segs) return;  // whole warps
  const long long r = wid / segs;
  const int seg = static_cast<int>(wid - r * segs);
  const long long srow = row_map ? row_map[r] : r;
  const uint32_t* am = amax + (rows_per_scale > 0 ? r / rows_per_scale : 0);
  const float s = __fdiv_rn(__uint_as_float(*am), kFp8Div);
  const bool fast = s > 0x1p-100f && s < 0x1p100f;
  const float y = fast ? __frcp_rn(s) : 0.f;
  const uint64_t y2 = f32x2_pack(y, y), ns2 = f32x2_pack(-s, -s);
  const uint4* row = reinterpret_cast<const uint4*>(src + srow * ld);
#pragma unroll
  for (int m = 0; m < kFp8SegVec / 32; ++m) {
    const int v = seg * kFp8SegVec + m * 32 + lane;
    if (v >= nvec) break;
    const uint4 a = __ldg(row + v);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t o[2] = {0u, 0u};
    if (fast) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float lo, hi;
        div2_markstein_bf16(w[k], y2, ns2, lo, hi);
        o[k >> 1] |= e4m3x2(lo, hi) << (16 * (k & 1));
      }
    } else if (s > 0.f) {  // outside the range of the fast division
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
        o[k >> 1] |= e4m3x2(__fdiv_rn(lo, s), __fdiv_rn(hi, s)) << (16 * (k & 1));
      }
    }
    *reinterpret_cast<uint2*>(out + r * ldo + static_cast<long long>(v) * 8) = make_uint2(o[0], o[1]);
  }
}

// Routed tokens, each quantised once and written to every one of its k permuted rows
// slot_row[t k + j] (E4M3 bytes [rows, K], rows ldo bytes apart). A token's codes are the
// same in all its copies (one scale for the whole token tensor), so this gives the bytes that
// quantising each gathered row gives, with a sixth of the arithmetic and of the reads at
// top-6. One warp per (token, 1024-value segment), as k_quant_fp8.
__global__ void k_quant_fp8_tokens(const uint16_t* __restrict__ src, long long ld, int T, int k,
                                   const int32_t* __restrict__ slot_row, long long rows, int K,
                                   const uint32_t* __restrict__ amax, uint8_t* __restrict__ out,
                                   long long ldo, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int nvec = K / 8;
  const int segs = (nvec + kFp8SegVec - 1) / kFp8SegVec;
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= static_cast<long long>(T) * segs) return;  // whole warps
  const long long t = wid / segs;
  const int seg = static_cast<int>(wid - t * segs);
  const float s = __fdiv_rn(__uint_as_float(*amax), kFp8Div);
  const bool fast = s > 0x1p-100f && s < 0x1p100f;
  const float y = fast ? __frcp_rn(s) : 0.f;
  const uint64_t y2 = f32x2_pack(y, y), ns2 = f32x2_pack(-s, -s);
  const uint4* row = reinterpret_cast<const uint4*>(src + t * ld);
  uint2 code[kFp8SegVec / 32];
#pragma unroll
  for (int m = 0; m < kFp8SegVec / 32; ++m) {
    const int v = seg * kFp8SegVec + m * 32 + lane;
    uint32_t o[2] = {0u, 0u};
    if (v < nvec) {
      const uint4 a = __ldg(row + v);
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
      if (fast) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float lo, hi;
          div2_markstein_bf16(w[q], y2, ns2, lo, hi);
          o[q >> 1] |= e4m3x2(lo, hi) << (16 * (q & 1));
        }
      } else if (s > 0.f) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = __uint_as_float(w[q] << 16), hi = __uint_as_float(w[q] & 0xffff0000u);
          o[q >> 1] |= e4m3x2(__fdiv_rn(lo, s), __fdiv_rn(hi, s)) << (16 * (q & 1));
        }
      }
    }
    code[m] = make_uint2(o[0], o[1]);
  }
  for (int j = 0; j < k; ++j) {
    const long long r = __ldg(slot_row + t * k + j);
    if (r < 0 || r >= rows) {
      if (lane == 0 && seg == 0) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
      continue;
    }
#pragma unroll
    for (int m = 0; m < kFp8SegVec / 32; ++m) {
      const int v = seg * kFp8SegVec + m * 32 + lane;
      if (v < nvec) *reinterpret_cast<uint2*>(out + r * ldo + static_cast<long long>(v) * 8) = code[m];
    }
  }
}

__global__ void k_finalize_fp8_scale(float* s, int G) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < G) s[i] = __fdiv_rn(s[i], kFp8Div);  // s[i] holds amax as fp32 bits
}

}  // namespace

int launch_quant_fp8(const uint16_t* src, long long ld, const int32_t* row_map, long long rows,
                     int K, long long rows_per_scale, const uint32_t* amax, uint8_t* out,
                     long long ldo, cudaStream_t s) {
  const long long n = rows * ((K / 8 + kFp8SegVec - 1) / kFp8SegVec) * 32;  // one warp per segment
  if (n <= 0) return MOE_OK;
  return launch_pdl(k_quant_fp8, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, s,
                    src, ld, row_map, rows, K, rows_per_scale, amax, out, ldo);
}

int launch_quant_fp8_tokens(const uint16_t* src, long long ld, int T, int k,
                            const int32_t* slot_row, long long rows, int K, const uint32_t* amax,
                            uint8_t* out, long long ldo, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  const long long n = static_cast<long long>(T) * ((K / 8 + kFp8SegVec - 1) / kFp8SegVec) * 32;
  return launch_pdl(k_quant_fp8_tokens, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                    s, src, ld, T, k, slot_row, rows, K, amax, out, ldo, status);
}

int launch_finalize_fp8_scale(float* s, int G, cudaStream_t stream) {
  return launch_pdl(k_finalize_fp8_scale, dim3((G + 255) / 256), dim3(256), 0, stream, s, G);
}

}  // namespace moe
