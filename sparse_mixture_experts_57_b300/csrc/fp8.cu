// fp8.cu: per-tensor E4M3 quantisation of expert weights and routed activations.
//
// "Nemotron 3 Nano" summary (papers.lianghsun.dev), §4: FP8 post-training quantisation with
// selective precision; BF16 and FP8 weights are released. The pages give no scaling
// granularity; this library's reading is one FP32 scale per tensor:
//   s = amax / 448,   q = E4M3(v / s)   (nearest, ties to even, saturating at +-448)
// with each expert matrix, the whole routed-token tensor and the whole h as the tensors.
// The division is correctly rounded (Markstein's FMA correction after a correctly rounded
// reciprocal, as in nvfp4.cu), so the codes are those of an fp32 evaluation of the rule.
#include <cuda_fp8.h>

#include "internal.h"

namespace moe {
namespace {

// v / s correctly rounded for 2^-100 < s < 2^100 and |v / s| < 2^100 (Markstein, IBM J. Res.
// Dev. 34(1), 1990): y = RN(1/s), q = RN(v y), r = v - q s exact in one fma, RN(q + r y).
__device__ __forceinline__ float div_markstein(float v, float s, float y) {
  const float q = __fmul_rn(v, y);
  const float r = fmaf(-q, s, v);
  return fmaf(r, y, q);
}

__device__ __forceinline__ uint32_t e4m3_byte(float v) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// One thread per 16 elements of a row: 32 bytes of bf16 in, 16 bytes of E4M3 out.
__global__ void k_quant_fp8(const uint16_t* __restrict__ src, long long ld,
                            const int32_t* __restrict__ row_map, long long rows, int K,
                            long long rows_per_scale, const uint32_t* __restrict__ amax,
                            uint8_t* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int per_row = K / 16;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * per_row) return;
  const long long r = i / per_row;
  const int c = static_cast<int>(i - r * per_row);
  const long long srow = row_map ? row_map[r] : r;
  const uint32_t* am = amax + (rows_per_scale > 0 ? r / rows_per_scale : 0);
  const float s = __fdiv_rn(__uint_as_float(*am), kFp8Div);
  const uint4* p = reinterpret_cast<const uint4*>(src + srow * ld + c * 16);
  const uint4 a = __ldg(p), b = __ldg(p + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t o[4] = {0u, 0u, 0u, 0u};
  if (s > 0x1p-100f && s < 0x1p100f) {
    const float y = __frcp_rn(s);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
      const uint32_t pair = e4m3_byte(div_markstein(lo, s, y)) |
                            (e4m3_byte(div_markstein(hi, s, y)) << 8);
      o[k >> 1] |= pair << (16 * (k & 1));
    }
  } else if (s > 0.f) {  // outside the range of the fast division
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
      const uint32_t pair = e4m3_byte(__fdiv_rn(lo, s)) | (e4m3_byte(__fdiv_rn(hi, s)) << 8);
      o[k >> 1] |= pair << (16 * (k & 1));
    }
  }
  *reinterpret_cast<uint4*>(out + r * K + c * 16) = make_uint4(o[0], o[1], o[2], o[3]);
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
                     cudaStream_t s) {
  const long long n = rows * (K / 16);
  if (n <= 0) return MOE_OK;
  return launch_pdl(k_quant_fp8, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, s,
                    src, ld, row_map, rows, K, rows_per_scale, amax, out);
}

int launch_finalize_fp8_scale(float* s, int G, cudaStream_t stream) {
  return launch_pdl(k_finalize_fp8_scale, dim3((G + 255) / 256), dim3(256), 0, stream, s, G);
}

}  // namespace moe
