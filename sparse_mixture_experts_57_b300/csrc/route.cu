// route.cu: the learned router of the routed MoE layer.
//
// News piece "NVIDIA AI发布了Nemotron 3", 混合Mamba Transformer MoE架构: a learned router
// picks a few (6) of 128 routable experts per token. "Nemotron 3 Nano" summary
// (papers.lianghsun.dev) §2.2: DeepSeek's aux-loss-free load balancing, read here as
// sigmoid scores plus a per-expert bias that enters the selection only, with the gates
// renormalised from the unbiased scores of the chosen experts.
//
// Two pieces: router logits (small-batch CUDA-core kernels here; large batches use the
// tcgen05 grouped GEMM with an fp32 epilogue), then a warp-per-token top-k.
#include <cuda_bf16.h>

#include <algorithm>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "scan.cuh"
#include "tc2.cuh"

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

// Small batches: one CTA per (8 tokens, 8 experts). The CTA stages its 8 token rows (all
// `parts` planes) in shared memory once; warp w then streams expert e0 + w's router row
// from global memory and dots it with the 8 staged rows. Each router row is read once per
// 8-token group and each token row once per 8-expert group, instead of once per warp.
constexpr int kSmallTok = 8, kSmallExp = 8;
constexpr int kSmallMaxElems = 6144;  // staged elements per token row (all planes)

// Router logits of 8 staged token rows against expert e, by one warp: each lane takes every
// 32nd 16-byte vector of the expert's row, in ascending order. The row is streamed through
// a ring of kAhead registers refilled one vector per iteration, so kAhead loads stay in
// flight while the loop body stays small (these kernels run once per layer with a cold
// instruction cache: unrolling the 8-token x kAhead-vector product multiplies the code that
// every SM must fetch). Returns the logit of token t on lane t < 8.
template <int PARTS>
__device__ __forceinline__ float logits_warp(const uint4* sx, const uint16_t* __restrict__ w,
                                             int D, int e) {
  constexpr int kAhead = 8;
  const int nvec = D / 8, rowv = PARTS * nvec;
  const int lane = threadIdx.x & 31;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const uint4* wrow = reinterpret_cast<const uint4*>(w + static_cast<long long>(e) * D);
  uint4 ring[kAhead];
#pragma unroll
  for (int j = 0; j < kAhead; ++j) ring[j] = lane + 32 * j < nvec ? __ldg(wrow + lane + 32 * j) : zero;
  float acc[kSmallTok];
#pragma unroll
  for (int t = 0; t < kSmallTok; ++t) acc[t] = 0.f;
#pragma unroll 1
  for (int v = lane; v < nvec; v += 32) {
    const uint4 wv = ring[0];
#pragma unroll
    for (int j = 0; j + 1 < kAhead; ++j) ring[j] = ring[j + 1];
    const int vn = v + 32 * kAhead;
    ring[kAhead - 1] = vn < nvec ? __ldg(wrow + vn) : zero;
#pragma unroll
    for (int t = 0; t < kSmallTok; ++t) {
#pragma unroll
      for (int p = 0; p < PARTS; ++p) acc[t] = dot8(sx[t * rowv + p * nvec + v], wv, acc[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < kSmallTok; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
  }
  float v = acc[0];
#pragma unroll
  for (int t = 1; t < kSmallTok; ++t)
    if (lane == t) v = acc[t];
  return v;
}

// Router logits of the 8 tokens t0.. against expert e (one warp per expert): the tokens are
// staged in shared memory (sx) with plain loads, then logits_warp. Every thread of the CTA
// must call this.
template <int PARTS>
__device__ __forceinline__ void logits_tile(const uint16_t* __restrict__ x, long long ldx,
                                            const uint16_t* __restrict__ w, int T, int D, int E,
                                            int t0, uint4* sx, float* __restrict__ logits) {
  const int nvec = D / 8, rowv = PARTS * nvec, n = kSmallTok * rowv;
  const int nt = blockDim.x;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  auto xload = [&](int i) {
    const int t = i / rowv, v = i - t * rowv;
    return t0 + t < T ? __ldg(reinterpret_cast<const uint4*>(x + (t0 + t) * ldx) + v) : zero;
  };
  int i = threadIdx.x;
#pragma unroll 1
  for (; i + 3 * nt < n; i += 4 * nt) {
    const uint4 a = xload(i), b = xload(i + nt), c = xload(i + 2 * nt), d = xload(i + 3 * nt);
    sx[i] = a;
    sx[i + nt] = b;
    sx[i + 2 * nt] = c;
    sx[i + 3 * nt] = d;
  }
#pragma unroll 1
  for (; i < n; i += nt) sx[i] = xload(i);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.y * kSmallExp + (threadIdx.x >> 5);
  if (e >= E) return;
  const float v = logits_warp<PARTS>(sx, w, D, e);
  if (lane < kSmallTok && t0 + lane < T) logits[static_cast<long long>(t0 + lane) * E + e] = v;
}

template <int PARTS>
__global__ void __launch_bounds__(256)
    k_router_logits_small(const uint16_t* __restrict__ x, long long ldx,
                          const uint16_t* __restrict__ w, int T, int D, int E,
                          float* __restrict__ logits) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint4 sx[];  // [kSmallTok][PARTS * D / 8]
  logits_tile<PARTS>(x, ldx, w, T, D, E, blockIdx.x * kSmallTok, sx, logits);
}

// Top-k of one token, by one warp. Each lane holds experts e = lane + 32*i. The k best
// biased scores are extracted by k (+1 for the gap) rounds of a warp-wide arg-max; ties go to
// the lower index. `row` points at the token's E logits; with CG the logits are read from L2
// (they were written by other CTAs of the same kernel).
template <int VPL, bool CG>
__device__ __forceinline__ void topk_token(const float* __restrict__ row,
                                           const float* __restrict__ bias, long long t, int E,
                                           int k, int32_t* __restrict__ idx,
                                           float* __restrict__ gates, uint8_t* __restrict__ tie) {
  const int lane = threadIdx.x & 31;
  float s[VPL], u[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float z = CG ? __ldcg(row + e) : row[e];
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

// Order-preserving map of a float (not NaN, not -0) to uint32 and back.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The same selection as topk_token (order by biased score descending, lower index first on
// equal scores; identical outputs) for many experts per lane: instead of k + 1 arg-max
// rounds over all E scores, the k-th largest score is found bit by bit on order-preserving
// keys (32 rounds of a per-lane count and a warp sum), the k winners are compacted into
// lanes 0..k-1 in index order, ranked among themselves, and moved to lane = rank.
template <int VPL, bool CG>
__device__ __forceinline__ void topk_token_select(const float* __restrict__ row,
                                                  const float* __restrict__ bias, long long t,
                                                  int E, int k, int32_t* __restrict__ idx,
                                                  float* __restrict__ gates,
                                                  uint8_t* __restrict__ tie) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  float s[VPL];
  uint32_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float z = CG ? __ldcg(row + e) : row[e];
      s[i] = 1.f / (1.f + expf(-z));
      const float ui = s[i] + bias[e];
      // NaN never wins; -0 cannot arise (s > 0) but would compare equal to +0: fold it
      key[i] = order_key((ui == ui) ? ui + 0.f : -INFINITY);
    } else {
      s[i] = 0.f;
      key[i] = 0u;  // below every valid key (the key of -inf is 0x007fffff)
    }
  }
  // 1. kth = the k-th largest key, found bit by bit from the top. Once exactly k keys are at
  //    or above the candidate prefix, they are the k largest and the k-th is their minimum:
  //    the search stops there instead of resolving the remaining low bits.
  uint32_t kth = 0u;
#pragma unroll 1
  for (int b = 31; b >= 0; --b) {
    const uint32_t cand = kth | (1u << b);
    uint32_t c = 0u;
#pragma unroll
    for (int i = 0; i < VPL; ++i) c += key[i] >= cand ? 1u : 0u;
    const uint32_t total = __reduce_add_sync(0xffffffffu, c);
    if (total == static_cast<uint32_t>(k)) {
      uint32_t m = 0xffffffffu;
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (key[i] >= cand) m = min(m, key[i]);
      kth = __reduce_min_sync(0xffffffffu, m);
      break;
    }
    if (total > static_cast<uint32_t>(k)) kth = cand;
  }
  uint32_t gt = 0u, eq = 0u, below = 0u;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    gt += key[i] > kth ? 1u : 0u;
    eq += key[i] == kth ? 1u : 0u;
    if (key[i] < kth) below = max(below, key[i]);
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  below = __reduce_max_sync(0xffffffffu, below);
  const uint32_t need_eq = static_cast<uint32_t>(k) - gt;  // >= 1 equal keys are taken
  const float uk = key_float(kth);
  const float uk1 = eq > need_eq ? uk : key_float(below);
  // 2. compact the winners into lanes 0..k-1 in index order (e = lane + 32 i: i major)
  uint32_t my_key = 0u, base = 0u, eq_seen = 0u;
  int my_e = 0;
  float my_s = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const uint32_t eqm = __ballot_sync(0xffffffffu, key[i] == kth);
    const bool win = key[i] > kth ||
                     (key[i] == kth && eq_seen + __popc(eqm & lt_mask) < need_eq);
    eq_seen += __popc(eqm);
    const uint32_t m = __ballot_sync(0xffffffffu, win);
    const uint32_t n = __popc(m);
    const bool mine = lane >= static_cast<int>(base) && lane < static_cast<int>(base + n);
    const int src = mine ? static_cast<int>(__fns(m, 0u, lane - static_cast<int>(base) + 1)) : lane;
    const uint32_t kv = __shfl_sync(0xffffffffu, key[i], src);
    const float sv = __shfl_sync(0xffffffffu, s[i], src);
    if (mine) {
      my_key = kv;
      my_e = src + 32 * i;
      my_s = sv;
    }
    base += n;
  }
  // 3. rank among the k winners: higher key first, then lower index
  int rank = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t kj = __shfl_sync(0xffffffffu, my_key, j);
    const int ej = __shfl_sync(0xffffffffu, my_e, j);
    rank += (kj > my_key || (kj == my_key && ej < my_e)) ? 1 : 0;
  }
  // 4. lane r takes the winner of rank r
  int from = 0;
  for (int j = 0; j < k; ++j) {
    const int rj = __shfl_sync(0xffffffffu, rank, j);
    if (rj == lane) from = j;
  }
  my_e = __shfl_sync(0xffffffffu, my_e, from);
  my_s = __shfl_sync(0xffffffffu, my_s, from);
  float sum = lane < k ? my_s : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    idx[t * k + lane] = my_e;
    gates[t * k + lane] = my_s / sum;
  }
  if (tie && lane == 0) tie[t] = (k < E && (uk - uk1) < 1e-5f) ? 1 : 0;
}

// k + 1 arg-max rounds cost about (k + 1)(5 VPL + 40) instructions per token, the bitwise
// selection about 32 (2 VPL + 8) + 15 VPL + 5 k + 100.
template <int VPL>
__device__ __forceinline__ bool use_select(int k) {
  return (k + 1) * (5 * VPL + 40) > 32 * (2 * VPL + 8) + 15 * VPL + 5 * k + 100;
}

// One token per warp; each warp's work is a dependent chain (k-th-key rounds or arg-max
// rounds), so the kernel runs on latency and residency: the register cap keeps four
// 256-thread CTAs per SM (two for 32 experts per lane, whose scores would not fit).
template <int VPL>
__global__ void __launch_bounds__(256, VPL >= 32 ? 2 : 4)
    k_topk(const float* __restrict__ logits, const float* __restrict__ bias, int T,
                       int E, int k, int32_t* __restrict__ idx, float* __restrict__ gates,
                       uint8_t* __restrict__ tie) {
  griddep_wait();
  griddep_launch_dependents();
  const long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  if (use_select<VPL>(k))
    topk_token_select<VPL, false>(logits + t * E, bias, t, E, k, idx, gates, tie);
  else
    topk_token<VPL, false>(logits + t * E, bias, t, E, k, idx, gates, tie);
}

// Small batches, routing and dispatch maps in one kernel. Grid (token groups of 8, expert
// groups of 8), 256 threads:
//  1. every CTA computes its 8 x 8 tile of router logits (as k_router_logits_small);
//  2. the last CTA to finish a token group (an atomic count per group) runs the top-k of its
//     8 tokens, one warp per token;
//  3. with perm set, the last token group to finish builds the dispatch maps for all tokens
//     in shared memory: per-expert counts and offsets, then row_token / slot_row with rows of
//     one expert in ascending token order (a token-word x expert bit matrix, as moe_permute).
// Which CTA takes steps 2 and 3 depends on timing; what they compute does not.
// "Last" is decided by flags rather than counters: each CTA stores the launch's generation
// tag `gen` (a new nonzero 64-bit value per launch) into its own flag word, fences, and reads
// its peers' flags; the SC fences guarantee that at least one CTA sees every flag set. Two
// CTAs may both see it; both then compute and store the same values. Flags holding another
// tag count as unset, so the scratch needs no clearing before a launch; the CTAs that finish
// a step store 0 into its flags again (a captured graph that replays one tag finds them clear).
constexpr int kFusedMaxT = 256, kFusedMaxE = 256;
constexpr int kFusedGroups = kFusedMaxT / kSmallTok;    // token groups (grid.x) at most
constexpr int kFusedExpGroups = kFusedMaxE / kSmallExp;  // expert groups (grid.y) at most

// Warp-wide: store this CTA's flag (slot `mine` of `flags`), then true on every lane if all
// n flags hold gen.
__device__ __forceinline__ bool flag_all_set(unsigned long long* flags, int mine, int n,
                                             unsigned long long gen) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) __stcg(flags + mine, gen);
  __threadfence();
  const bool set = lane >= n || lane == mine || __ldcg(flags + lane) == gen;
  return __all_sync(0xffffffffu, set);
}

// Dispatch maps of all T tokens, built by one CTA (every thread calls this) from their
// top-k (idx, written by other CTAs of the kernel and read through L2): per-expert counts
// and offsets, then row_token / slot_row, the rows of one expert in ascending token order (a
// token-word x expert bit matrix, as moe_permute). scratch: W * E * 8 bytes of shared
// memory, W = ceil(T / 32); warp_sums: 33 ints of shared memory.
__device__ __noinline__ void dispatch_maps(const int32_t* __restrict__ idx, int T, int E, int k,
                                           int32_t* __restrict__ counts,
                                           int32_t* __restrict__ offsets,
                                           int32_t* __restrict__ row_token,
                                           int32_t* __restrict__ slot_row, uint32_t* scratch,
                                           int* warp_sums, int* status) {
  __shared__ int s_off[kFusedMaxE];
  const int tid = threadIdx.x;
  const int W = (T + 31) / 32;
  uint32_t* bits = scratch;                           // [W][E]
  int* wpref = reinterpret_cast<int*>(bits + W * E);  // [W][E]
  for (int i = tid; i < W * E; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  bool bad = false;
  for (int i = tid; i < T * k; i += blockDim.x) {
    const int t = i / k;
    const int e = __ldcg(idx + i);
    if (e < 0 || e >= E) {
      bad = true;
      continue;
    }
    const uint32_t bit = 1u << (t & 31);
    if (atomicOr(&bits[(t >> 5) * E + e], bit) & bit) bad = true;
  }
  if (__syncthreads_or(bad) && tid == 0) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
  int c = 0;
  if (tid < E) {
    for (int wd = 0; wd < W; ++wd) {
      wpref[wd * E + tid] = c;
      c += __popc(bits[wd * E + tid]);
    }
    counts[tid] = c;
  }
  int total;
  const int excl = block_exclusive_scan(c, warp_sums, &total);
  if (tid < E) {
    offsets[tid] = excl;
    s_off[tid] = excl;
  }
  if (tid == 0) offsets[E] = total;
  __syncthreads();
  for (int i = tid; i < T * k; i += blockDim.x) {
    const int t = i / k;
    const int e = __ldcg(idx + i);
    if (e < 0 || e >= E) {
      slot_row[i] = -1;
      continue;
    }
    const int o = (t >> 5) * E + e;
    const int row = s_off[e] + wpref[o] + __popc(bits[o] & ((1u << (t & 31)) - 1u));
    row_token[row] = t;
    slot_row[i] = row;
  }
}

template <int VPL, int PARTS>
__global__ void __launch_bounds__(256)
    k_route_small(const uint16_t* __restrict__ x, long long ldx, const uint16_t* __restrict__ w,
                  const float* __restrict__ bias, int T, int D, int E, int k,
                  float* __restrict__ logits, int32_t* __restrict__ idx,
                  float* __restrict__ gates, uint8_t* __restrict__ tie, int perm,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ row_token, int32_t* __restrict__ slot_row,
                  unsigned long long* __restrict__ sync, unsigned long long gen, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint4 sx[];
  __shared__ int s_flag;
  __shared__ int warp_sums[33];
  __shared__ float s_bias[kFusedMaxE];  // fetched now: only the last CTA of a group uses it
  const int tid = threadIdx.x, warp = tid >> 5;
  const int t0 = blockIdx.x * kSmallTok;
  for (int e = tid; e < E; e += blockDim.x) s_bias[e] = __ldg(bias + e);
  // 1. logits tile
  logits_tile<PARTS>(x, ldx, w, T, D, E, t0, sx, logits);
  // 2. the last CTA of this token group: top-k of its tokens
  unsigned long long* gflags = sync + blockIdx.x * kFusedExpGroups;  // [grid.y] per group
  unsigned long long* tflags = sync + kFusedGroups * kFusedExpGroups;  // [grid.x]
  __threadfence();  // this thread's logits before the CTA's flag
  __syncthreads();
  if (warp == 0) {
    const bool all = flag_all_set(gflags, blockIdx.y, gridDim.y, gen);
    if (tid == 0) s_flag = all;
  }
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  if (warp < kSmallTok && t0 + warp < T) {
    const float* row = logits + static_cast<long long>(t0 + warp) * E;
    if (use_select<VPL>(k))
      topk_token_select<VPL, true>(row, s_bias, t0 + warp, E, k, idx, gates, tie);
    else
      topk_token<VPL, true>(row, s_bias, t0 + warp, E, k, idx, gates, tie);
  }
  if (tid < static_cast<int>(gridDim.y)) __stcg(gflags + tid, 0ull);
  if (!perm) return;
  // 3. the last token group: dispatch maps for all tokens
  __threadfence();  // this thread's top-k results before the group's flag
  __syncthreads();
  if (warp == 0) {
    const bool all = flag_all_set(tflags, blockIdx.x, gridDim.x, gen);
    if (tid == 0) s_flag = all;
  }
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  dispatch_maps(idx, T, E, k, counts, offsets, row_token, slot_row,
                reinterpret_cast<uint32_t*>(sx), warp_sums, status);
  if (tid < static_cast<int>(gridDim.x)) __stcg(tflags + tid, 0ull);
}

// Small batches with E <= 128, the same three steps with a cluster per token group. Grid
// (token groups of 8, C = ceil(E / 8) expert groups), cluster (1, C, 1), 256 threads:
//  0. the CTA's 8 router-weight rows are prefetched into L2 before the kernel waits for its
//     predecessor (they are layer parameters that no earlier kernel writes); the group's
//     token rows are staged with one bulk copy each;
//  1. every CTA computes its 8 x 8 tile of logits and stores each token's values straight
//     into the shared memory of the CTA that ranks that token (token t: rank t % C);
//  2. after a cluster barrier, each CTA runs the top-k of its tokens from shared memory,
//     one warp per token;
//  3. after a second cluster barrier, rank 0 of each group stores the group's flag, and the
//     last group to finish builds the dispatch maps (dispatch_maps).
// Compared with k_route_small, the logits never go through L2 and no CTA waits on flags of
// its own group: the exchange is a hardware cluster barrier.
constexpr int kClusterMaxE = 128;

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <int VPL, int PARTS>
__global__ void __launch_bounds__(256)
    k_route_cluster(const uint16_t* __restrict__ x, long long ldx,
                    const uint16_t* __restrict__ w, const float* __restrict__ bias, int T, int D,
                    int E, int k, int32_t* __restrict__ idx, float* __restrict__ gates,
                    uint8_t* __restrict__ tie, int perm, int32_t* __restrict__ counts,
                    int32_t* __restrict__ offsets, int32_t* __restrict__ row_token,
                    int32_t* __restrict__ slot_row, unsigned long long* __restrict__ sync,
                    unsigned long long gen, int* status) {
  extern __shared__ uint4 sx[];  // [8][PARTS * D / 8] token rows; later the dispatch scratch
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ float s_lg[kSmallTok][kClusterMaxE];  // logits of the tokens this CTA ranks
  __shared__ float s_bias[kClusterMaxE];
  __shared__ int s_flag;
  __shared__ int s_abort;
  __shared__ int warp_sums[33];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = static_cast<int>(gridDim.y);
  const uint32_t rank = cluster_ctarank();
  const int t0 = blockIdx.x * kSmallTok;
  const int nt = min(kSmallTok, T - t0);
  const int e = blockIdx.y * kSmallExp + warp;
  const int rowv = PARTS * (D / 8);
  if (lane == 0 && e < E)
    prefetch_l2(w + static_cast<long long>(e) * D, static_cast<uint32_t>(D) * 2u);
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  cluster_arrive_relaxed();  // this CTA has started: peers may write its shared memory
  griddep_wait();
  griddep_launch_dependents();
  for (int i = tid; i < E; i += blockDim.x) s_bias[i] = __ldg(bias + i);
  __syncthreads();
  if (tid == 0) {
    const uint32_t row_bytes = static_cast<uint32_t>(rowv) * 16u;
    mbar_arrive_expect_tx(&s_bar, row_bytes * static_cast<uint32_t>(nt));
    const uint64_t pol = policy_evict_first();
    for (int t = 0; t < nt; ++t)
      bulk_load(sx + t * rowv, x + static_cast<long long>(t0 + t) * ldx, row_bytes, &s_bar, pol);
  }
  for (int i = nt * rowv + tid; i < kSmallTok * rowv; i += blockDim.x)
    sx[i] = make_uint4(0u, 0u, 0u, 0u);  // rows past T
  if (!mbar_wait(&s_bar, 0, &s_abort)) {
    if (tid == 0) atomicCAS(status, 0, MOE_ERR_TIMEOUT);
    mbar_wait(&s_bar, 0, &s_abort, kDrainLimitNs);  // no copy may land after the CTA exits
  }
  __syncthreads();
  float v = 0.f;
  if (e < E) v = logits_warp<PARTS>(sx, w, D, e);
  cluster_wait();  // every CTA of the cluster has started
  if (e < E && lane < nt)
    st_cluster_f32(mapa_shared(&s_lg[lane][e], static_cast<uint32_t>(lane % C)), v);
  cluster_sync();  // all logits of the group delivered
  const int t = static_cast<int>(rank) + C * warp;
  if (t < nt) {
    if (use_select<VPL>(k))
      topk_token_select<VPL, false>(s_lg[t], s_bias, t0 + t, E, k, idx, gates, tie);
    else
      topk_token<VPL, false>(s_lg[t], s_bias, t0 + t, E, k, idx, gates, tie);
  }
  __threadfence();  // this thread's top-k results before the group's flag
  cluster_sync();   // every top-k of the group is written; no CTA reads peers' memory after
  if (!perm || rank != 0) return;
  unsigned long long* tflags = sync + kFusedGroups * kFusedExpGroups;  // [grid.x]
  if (warp == 0) {
    const bool all = flag_all_set(tflags, blockIdx.x, gridDim.x, gen);
    if (tid == 0) s_flag = all;
  }
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  dispatch_maps(idx, T, E, k, counts, offsets, row_token, slot_row,
                reinterpret_cast<uint32_t*>(sx), warp_sums, status);
  if (tid < static_cast<int>(gridDim.x)) __stcg(tflags + tid, 0ull);
}

// x_perm[r, :] = x[row_token[r], :], one warp per row (16-byte vectors).
__global__ void k_gather_rows(const int32_t* __restrict__ row_token, const uint16_t* __restrict__ x,
                              long long ldx, int rows, int H, uint16_t* __restrict__ x_perm,
                              int src_rows, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (r >= rows) return;
  const int t = row_token[r];
  if constexpr (kDebugBuild) {  // the routing kernel wrote row_token: check it in debug builds
    if (t < 0 || t >= src_rows) {
      if (lane == 0) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
      return;
    }
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<long long>(t) * ldx);
  uint4* dst = reinterpret_cast<uint4*>(x_perm + r * H);
#pragma unroll 4
  for (int v = lane; v < H / 8; v += 32) dst[v] = __ldg(src + v);
}

// Launch set-up state per kernel and device. Kernels of one signature share one
// instantiation of a generic lambda, so this state cannot live in the lambda's statics: it
// is kept per kernel address.
struct KernelSetup {
  const void* fn = nullptr;
  int dev = -1;
  int usable = 0;
};

KernelSetup& kernel_setup(const void* fn) {
  constexpr int kSlots = 64;  // this file launches fewer than 20 kernels
  static std::mutex m;
  static KernelSetup table[kSlots];
  static int n = 0;
  std::lock_guard<std::mutex> lock(m);
  for (int i = 0; i < n; ++i)
    if (table[i].fn == fn) return table[i];
  if (n == kSlots) {  // not reached; a fresh state means the kernel is set up again
    static KernelSetup spare;
    spare = KernelSetup{fn, -1, 0};
    return spare;
  }
  table[n].fn = fn;
  return table[n++];
}

}  // namespace

int launch_router_logits(const uint16_t* x, int64_t ldx, const uint16_t* w_router, int T, int D,
                         int E, int parts, float* logits, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  if ((parts == 1 || parts == 3) && static_cast<long long>(parts) * D <= kSmallMaxElems) {
    const dim3 grid((T + kSmallTok - 1) / kSmallTok, (E + kSmallExp - 1) / kSmallExp);
    const size_t smem = static_cast<size_t>(kSmallTok) * parts * D * 2;
    auto go = [&](auto kern) -> int {
      KernelSetup& su = kernel_setup(reinterpret_cast<const void*>(kern));
      int dev = 0;
      MOE_CUDA(cudaGetDevice(&dev));
      if (su.dev != dev) {
        MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kSmallTok * kSmallMaxElems * 2));
        su.dev = dev;
      }
      return launch_pdl(kern, grid, dim3(32 * kSmallExp), smem, s, x,
                        static_cast<long long>(ldx), w_router, T, D, E, logits);
    };
    return parts == 1 ? go(k_router_logits_small<1>) : go(k_router_logits_small<3>);
  }
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

// The CUDA error of the last refused cluster launch of the small-batch routing (0: none).
int& cluster_launch_error() {
  static int e = 0;
  return e;
}

bool route_fused_ok(int T, int D, int E, int k, int parts) {
  return T >= 1 && T <= kFusedMaxT && E >= 1 && E <= kFusedMaxE && k <= 32 &&
         (parts == 1 || parts == 3) &&
         static_cast<long long>(parts) * D <= kSmallMaxElems && D % 8 == 0;
}

// 64-bit flag words (per token group: one per expert group; one per token group), as pairs
// of ints
size_t route_fused_sync_ints(int) {
  return 2 * static_cast<size_t>(kFusedGroups * kFusedExpGroups + kFusedGroups);
}

int launch_route_fused(const uint16_t* x, int64_t ldx, const uint16_t* w_router,
                       const float* bias, int T, int D, int E, int k, int parts, float* logits,
                       int32_t* idx, float* gates, uint8_t* tie, int32_t* counts,
                       int32_t* offsets, int32_t* row_token, int32_t* slot_row, int* sync,
                       cudaStream_t s) {
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  if (reinterpret_cast<uintptr_t>(sync) % 8) return MOE_ERR_UNSUPPORTED;
  static std::atomic<unsigned long long> launches{0};
  const unsigned long long gen = (launches.fetch_add(1) % ((1ull << 48) - 1)) + 1;  // never 0
  const dim3 grid((T + kSmallTok - 1) / kSmallTok, (E + kSmallExp - 1) / kSmallExp);
  const int W = (T + 31) / 32;
  const size_t smem = std::max(static_cast<size_t>(kSmallTok) * parts * D * 2,
                               static_cast<size_t>(W) * E * 8);
  const int perm = row_token != nullptr;
  auto go = [&](auto kern) -> int {
    KernelSetup& su = kernel_setup(reinterpret_cast<const void*>(kern));
    int dev = 0;
    MOE_CUDA(cudaGetDevice(&dev));
    if (su.dev != dev) {
      MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmallTok * kSmallMaxElems * 2));
      su.dev = dev;
    }
    return launch_pdl(kern, grid, dim3(256), smem, s, x, static_cast<long long>(ldx), w_router,
                      bias, T, D, E, k, logits, idx, gates, tie, perm, counts, offsets,
                      row_token, slot_row, reinterpret_cast<unsigned long long*>(sync), gen,
                      status);
  };
  // The cluster form: one cluster of C = ceil(E / 8) CTAs per token group (C <= 16; more
  // than 8 is a non-portable cluster size). Returns 1 when it cannot run here (the caller
  // then launches k_route_small).
  auto go_cluster = [&](auto kern) -> int {
    KernelSetup& su = kernel_setup(reinterpret_cast<const void*>(kern));
    int dev = 0;
    MOE_CUDA(cudaGetDevice(&dev));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = grid.y;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (su.dev != dev) {
      MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmallTok * kSmallMaxElems * 2));
      MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
      // the largest cluster (16 CTAs) with the largest staging buffer must fit at least once
      cudaLaunchConfig_t probe = cfg;
      cudaLaunchAttribute pattr = attr[0];
      pattr.val.clusterDim.y = kClusterMaxE / kSmallExp;
      probe.gridDim = dim3(1, pattr.val.clusterDim.y);
      probe.dynamicSmemBytes = kSmallTok * kSmallMaxElems * 2;
      probe.attrs = &pattr;
      int n = 0;
      su.usable = cudaOccupancyMaxActiveClusters(&n, kern, &probe) == cudaSuccess && n > 0;
      cudaGetLastError();  // a refused query is not an error of this call
      su.dev = dev;
    }
    if (!su.usable) return 1;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, x, static_cast<long long>(ldx),
                                             w_router, bias, T, D, E, k, idx, gates, tie, perm,
                                             counts, offsets, row_token, slot_row,
                                             reinterpret_cast<unsigned long long*>(sync), gen,
                                             status);
    if (e == cudaSuccess) return MOE_OK;
    // a configuration this device refuses (nothing was launched): use k_route_small from now
    cluster_launch_error() = static_cast<int>(e);
    cudaGetLastError();
    su.usable = 0;
    return 1;
  };
  if (E <= kClusterMaxE && ldx % 8 == 0 && aligned16(x)) {
    int st = 1;
    if (parts == 3)
      st = E <= 32 ? go_cluster(k_route_cluster<1, 3>)
         : E <= 64 ? go_cluster(k_route_cluster<2, 3>) : go_cluster(k_route_cluster<4, 3>);
    else
      st = E <= 32 ? go_cluster(k_route_cluster<1, 1>)
         : E <= 64 ? go_cluster(k_route_cluster<2, 1>) : go_cluster(k_route_cluster<4, 1>);
    if (st != 1) return st;
  }
  if (parts == 3) {
    if (E <= 32) return go(k_route_small<1, 3>);
    if (E <= 64) return go(k_route_small<2, 3>);
    if (E <= 128) return go(k_route_small<4, 3>);
    return go(k_route_small<8, 3>);
  }
  if (E <= 32) return go(k_route_small<1, 1>);
  if (E <= 64) return go(k_route_small<2, 1>);
  if (E <= 128) return go(k_route_small<4, 1>);
  return go(k_route_small<8, 1>);
}

int launch_gather_rows(const int32_t* row_token, const uint16_t* x, int64_t ldx, int src_rows,
                       int rows, int H, uint16_t* x_perm, cudaStream_t s) {
  if (rows <= 0) return MOE_OK;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  const long long threads = static_cast<long long>(rows) * 32;
  return launch_pdl(k_gather_rows, dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256),
                    0, s, row_token, x, static_cast<long long>(ldx), rows, H, x_perm, src_rows,
                    status);
}

}  // namespace moe

extern "C" int moe_route_cluster_refusal(void) { return moe::cluster_launch_error(); }
