// combine.cu: the combination layer, a gate-weighted gather-reduce back to token order.
//
// "Nemotron 3 Nano" summary (shd-paper.top), 技术框架: a combination layer forms the
// weighted combination of the chosen experts' outputs.
//   y[t, :] = sum_j gates[t, j] * y_perm[slot_row[t, j], :]
// Deterministic (no atomics): one warp per token, fp32 accumulation, 16-byte loads/stores.
#include <cuda_bf16.h>

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

__global__ void k_combine(const uint16_t* __restrict__ y_perm, int rows,
                          const int32_t* __restrict__ slot_row, const float* __restrict__ gates,
                          int T, int H, int k, uint16_t* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  // lanes j < k hold slot j's row and gate
  int my_row = -1;
  float my_g = 0.f;
  if (lane < k) {
    my_row = slot_row[t * k + lane];
    my_g = gates[t * k + lane];
    if (my_row < 0 || my_row >= rows) my_row = -1;
  }
  const int nvec = H / 8;
  // The loop bound is warp-uniform so every lane takes part in the shuffles.
  for (int base = 0; base < nvec; base += 32) {
    const int v = base + lane;
    const bool active = v < nvec;
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xffffffffu, my_row, j);
      const float g = __shfl_sync(0xffffffffu, my_g, j);
      if (r < 0 || !active) continue;
      const uint4 yv =
          __ldg(reinterpret_cast<const uint4*>(y_perm + static_cast<long long>(r) * H) + v);
      acc8(a, yv, g);
    }
    if (active)
      reinterpret_cast<uint4*>(y + t * H)[v] =
          make_uint4(pack2(a[0], a[1]), pack2(a[2], a[3]), pack2(a[4], a[5]), pack2(a[6], a[7]));
  }
}

}  // namespace

int launch_combine(const uint16_t* y_perm, int rows, const int32_t* slot_row, const float* gates,
                   int T, int H, int k, uint16_t* y, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  const int threads = 256;
  const long long blocks = (static_cast<long long>(T) * 32 + threads - 1) / threads;
  k_combine<<<static_cast<unsigned>(blocks), threads, 0, s>>>(y_perm, rows, slot_row, gates, T, H,
                                                              k, y);
  MOE_LAUNCHED();
  return MOE_OK;
}

}  // namespace moe
