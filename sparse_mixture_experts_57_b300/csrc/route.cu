// route.cu: the learned router of the routed MoE layer.
//
// News piece "NVIDIA AI发布了Nemotron 3", 混合Mamba Transformer MoE架构: a learned router
// picks a few (6) of 128 routable experts per token. "Nemotron 3 Nano" summary
// (papers.lianghsun.dev) §2.2: DeepSeek's aux-loss-free load balancing, read here as
// sigmoid scores plus a per-expert bias that enters the selection only, with the gates
// renormalised from the unbiased scores of the chosen experts.
//
// Two pieces: router logits (a small-batch CUDA-core kernel here; large batches use the
// tcgen05 grouped GEMM with an fp32 epilogue), then a warp-per-token top-k.
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kTokPerWarp = 4;

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc) {
  acc = fmaf(bf_lo(a.x), bf_lo(b.x), acc);
  acc = fmaf(bf_hi(a.x), bf_hi(b.x), acc);
  acc = fmaf(bf_lo(a.y), bf_lo(b.y), acc);
  acc = fmaf(bf_hi(a.y), bf_hi(b.y), acc);
  acc = fmaf(bf_lo(a.z), bf_lo(b.z), acc);
  acc = fmaf(bf_hi(a.z), bf_hi(b.z), acc);
  acc = fmaf(bf_lo(a.w), bf_lo(b.w), acc);
  acc = fmaf(bf_hi(a.w), bf_hi(b.w), acc);
  return acc;
}

// logits[t, e] = sum_p sum_d x[t, p*D + d] * w[e, d] over `parts` planes: with parts > 1
// the input row holds bf16 planes (hi, mid, lo) whose sum is a wider-precision vector.
// One warp per (expert, group of 4 tokens); lanes stride over D in 8-element vectors,
// four strides unrolled so their loads are in flight together.
__global__ void k_router_logits(const uint16_t* __restrict__ x, long long ldx,
                                const uint16_t* __restrict__ w, int T, int D, int E, int parts,
                                float* __restrict__ logits) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int groups = (T + kTokPerWarp - 1) / kTokPerWarp;
  if (gw >= static_cast<long long>(groups) * E) return;
  const int e = static_cast<int>(gw % E);
  const int t0 = static_cast<int>(gw / E) * kTokPerWarp;
  float acc[kTokPerWarp];
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) acc[i] = 0.f;
  const uint4* wrow = reinterpret_cast<const uint4*>(w + static_cast<long long>(e) * D);
  const int nvec = D / 8;
#pragma unroll 4
  for (int v = lane; v < nvec; v += 32) {
    const uint4 wv = __ldg(wrow + v);
#pragma unroll
    for (int i = 0; i < kTokPerWarp; ++i) {
      if (t0 + i < T) {
        const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(t0 + i) * ldx);
        for (int p = 0; p < parts; ++p) acc[i] = dot8(__ldg(xr + p * nvec + v), wv, acc[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kTokPerWarp; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kTokPerWarp; ++i)
      if (t0 + i < T) logits[static_cast<long long>(t0 + i) * E + e] = acc[i];
  }
}

// Warp per token. Each lane holds experts e = lane + 32*i. The k best biased scores are
// extracted by k (+1 for the gap) rounds of a warp-wide arg-max; ties go to the lower index.
template <int VPL>
__global__ void k_topk(const float* __restrict__ logits, const float* __restrict__ bias, int T,
                       int E, int k, int32_t* __restrict__ idx, float* __restrict__ gates,
                       uint8_t* __restrict__ tie) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  float s[VPL], u[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float z = logits[t * E + e];
      s[i] = 1.f / (1.f + expf(-z));
      const float ui = s[i] + bias[e];
      u[i] = (ui == ui) ? ui : -INFINITY;  // NaN never wins
    } else {
      s[i] = 0.f;
      u[i] = -INFINITY;
    }
  }
  uint32_t taken = 0;
  float my_s = 0.f;
  int my_e = 0;
  float uk = 0.f, uk1 = -INFINITY;
  const int rounds = k < E ? k + 1 : k;
  for (int j = 0; j < rounds; ++j) {
    float bu = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (u[i] > bu || (u[i] == bu && e < be))) {
        bu = u[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ou = __shfl_xor_sync(0xffffffffu, bu, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ou > bu || (ou == bu && oe < be)) {
        bu = ou;
        be = oe;
      }
    }
    if (j == k) {
      uk1 = bu;
      break;
    }
    const int owner = be & 31, slot = be >> 5;
    float sv = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (i == slot) sv = s[i];
    if (lane == owner) taken |= 1u << slot;
    sv = __shfl_sync(0xffffffffu, sv, owner);
    if (lane == j) {
      my_s = sv;
      my_e = be;
    }
    if (j == k - 1) uk = bu;
  }
  float sum = lane < k ? my_s : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    idx[t * k + lane] = my_e;
    gates[t * k + lane] = my_s / sum;
  }
  if (tie && lane == 0) tie[t] = (k < E && (uk - uk1) < 1e-5f) ? 1 : 0;
}

}  // namespace

int launch_router_logits(const uint16_t* x, int64_t ldx, const uint16_t* w_router, int T, int D,
                         int E, int parts, float* logits, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  const long long warps = static_cast<long long>((T + kTokPerWarp - 1) / kTokPerWarp) * E;
  const int threads = 256;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  return launch_pdl(k_router_logits, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s,
                    x, static_cast<long long>(ldx), w_router, T, D, E, parts, logits);
}

int launch_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* idx,
                float* gates, uint8_t* tie, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  const int threads = 256;
  const long long blocks = (static_cast<long long>(T) * 32 + threads - 1) / threads;
  const dim3 b(static_cast<unsigned>(blocks)), th(threads);
  if (E <= 32) return launch_pdl(k_topk<1>, b, th, 0, s, logits, bias, T, E, k, idx, gates, tie);
  if (E <= 64) return launch_pdl(k_topk<2>, b, th, 0, s, logits, bias, T, E, k, idx, gates, tie);
  if (E <= 128) return launch_pdl(k_topk<4>, b, th, 0, s, logits, bias, T, E, k, idx, gates, tie);
  if (E <= 256) return launch_pdl(k_topk<8>, b, th, 0, s, logits, bias, T, E, k, idx, gates, tie);
  if (E <= 512) return launch_pdl(k_topk<16>, b, th, 0, s, logits, bias, T, E, k, idx, gates, tie);
  return launch_pdl(k_topk<32>, b, th, 0, s, logits, bias, T, E, k, idx, gates, tie);
}

}  // namespace moe
