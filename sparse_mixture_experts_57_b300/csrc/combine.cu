// combine.cu: the combination layer, a gate-weighted gather-reduce back to token order.
//
// "Nemotron 3 Nano" summary (shd-paper.top), 技术框架: a combination layer forms the
// weighted combination of the chosen experts' outputs.
//   y[t, :] = addend[t, :] + sum_j gates[t, j] * y_perm[slot_row[t, j], :]
// (addend: the shared expert's output, or nothing)
// Deterministic (no atomics), fp32 accumulation, 16-byte loads and stores.
#include <cuda_bf16.h>

#include "fixed.cuh"
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void acc8(float (&a)[8], const uint4& v, float g) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] = fmaf(g, __uint_as_float(w[i] << 16), a[2 * i]);
    a[2 * i + 1] = fmaf(g, __uint_as_float(w[i] & 0xffff0000u), a[2 * i + 1]);
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One thread per (token, 8-element column block): every thread issues its k row loads
// back to back, so even a 64-token decode batch keeps thousands of loads in flight.
__global__ void k_combine(const uint16_t* __restrict__ y_perm, int rows,
                          const int32_t* __restrict__ slot_row, const float* __restrict__ gates,
                          int T, int H, int k, const uint16_t* __restrict__ addend,
                          uint16_t* __restrict__ y, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int nvec = H / 8;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(T) * nvec) return;
  const long long t = i / nvec;
  const int v = static_cast<int>(i - t * nvec);
  const int32_t* sr = slot_row + t * k;
  const float* gg = gates + t * k;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (addend)  // the shared expert's output joins the fp32 sum
    acc8(a, __ldg(reinterpret_cast<const uint4*>(addend + t * H) + v), 1.f);
#pragma unroll 4
  for (int j = 0; j < k; ++j) {
    const int r = __ldg(sr + j);
    const float g = __ldg(gg + j);
    if (r < 0 || r >= rows) {  // skipped; the MOE_DEBUG build also reports it
      if constexpr (kDebugBuild) {
        if (v == 0) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
      }
      continue;
    }
    const uint4 yv =
        __ldg(reinterpret_cast<const uint4*>(y_perm + static_cast<long long>(r) * H) + v);
    acc8(a, yv, g);
  }
  reinterpret_cast<uint4*>(y + t * H)[v] =
      make_uint4(pack2(a[0], a[1]), pack2(a[2], a[3]), pack2(a[4], a[5]), pack2(a[6], a[7]));
}

// The fused combine's accumulator starts at zero: consecutive threads store consecutive 16
// bytes, grid-stride.
__global__ void k_zero_fixed(longlong2* __restrict__ acc, long long n2) {
  griddep_wait();
  griddep_launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n2;
       i += stride)
    acc[i] = make_longlong2(0, 0);
}

// y[t, c] = bf16(acc[t, c] * 2^-32), one thread per 8 columns.
__global__ void k_combine_fixed(const longlong2* __restrict__ acc, long long n8,
                                uint4* __restrict__ y) {
  griddep_wait();
  griddep_launch_dependents();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  uint32_t o[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const longlong2 q = __ldg(acc + i * 4 + u);
    o[u] = static_cast<uint32_t>(fixed_to_bf16(q.x)) |
           (static_cast<uint32_t>(fixed_to_bf16(q.y)) << 16);
  }
  y[i] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

int launch_zero_fixed(int64_t* acc, long long n, cudaStream_t s) {
  if (n <= 0) return MOE_OK;
  const long long n2 = n / 2;  // n is a multiple of 8
  const int threads = 256;
  long long blocks = (n2 + threads - 1) / threads;
  const long long cap = static_cast<long long>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  return launch_pdl(k_zero_fixed, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s,
                    reinterpret_cast<longlong2*>(acc), n2);
}

int launch_combine_fixed(const int64_t* acc, long long n, uint16_t* y, cudaStream_t s) {
  if (n <= 0) return MOE_OK;
  const int threads = 256;
  const long long n8 = n / 8;
  return launch_pdl(k_combine_fixed, dim3(static_cast<unsigned>((n8 + threads - 1) / threads)),
                    dim3(threads), 0, s, reinterpret_cast<const longlong2*>(acc), n8,
                    reinterpret_cast<uint4*>(y));
}

int launch_combine(const uint16_t* y_perm, int rows, const int32_t* slot_row, const float* gates,
                   int T, int H, int k, uint16_t* y, cudaStream_t s, const uint16_t* addend) {
  if (T <= 0) return MOE_OK;
  const int threads = 256;
  const long long n = static_cast<long long>(T) * (H / 8);
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  return launch_pdl(k_combine, dim3(static_cast<unsigned>((n + threads - 1) / threads)),
                    dim3(threads), 0, s, y_perm, rows, slot_row, gates, T, H, k, addend, y,
                    status);
}

}  // namespace moe

extern "C" int moe_fixed_to_bf16(const int64_t* q, long long n, uint16_t* out, int on_device,
                                 cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!q || !out))) return MOE_ERR_INVALID_ARG;
  if (!on_device) {
    for (long long i = 0; i < n; ++i) out[i] = moe::fixed_to_bf16(q[i]);
    return MOE_OK;
  }
  if (n % 8 || !moe::aligned16(q) || !moe::aligned16(out)) return MOE_ERR_UNSUPPORTED;
  return moe::launch_combine_fixed(q, n, out, stream);
}
