// permute.cu: dispatch of routed (token, slot) pairs into expert-contiguous order.
//
// "Nemotron 3 Nano" summary (shd-paper.top), 技术框架: the chosen experts process their
// tokens in parallel. "NVIDIA Nemotron 3" notes §2.2: tokens are dispatched to experts.
//
// A deterministic counting sort that keeps tokens in ascending order inside each expert
// segment:
//   mark    : one warp per 32 tokens builds, for every expert, the 32-bit mask of which of
//             those tokens chose it -> bits[w][e]
//   count   : per expert, exclusive popcount prefix over the token words -> wpref[w][e],
//             and counts[e]
//   offsets : exclusive scan of counts
//   gather  : rank of (t, e) = wpref[t/32][e] + popc(bits[t/32][e] below t's bit);
//             row = offsets[e] + rank; copy the token row into x_perm with 16-byte moves.
// Small problems run mark, count and offsets as one single-block kernel (k_perm_small).
#include <cuda_runtime.h>

#include "internal.h"
#include "scan.cuh"

namespace moe {
namespace {

constexpr int kMarkWarps = 4;

__global__ void k_perm_mark(const int32_t* __restrict__ idx, int T, int E, int k,
                            uint32_t* __restrict__ bits, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint32_t smask[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int W = (T + 31) / 32;
  const int w = blockIdx.x * kMarkWarps + wib;
  if (w >= W) return;
  uint32_t* m = smask + wib * E;
  for (int e = lane; e < E; e += 32) m[e] = 0u;
  __syncwarp();
  const int t = w * 32 + lane;
  bool bad = false;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[static_cast<long long>(t) * k + j];
      if (e < 0 || e >= E) {
        bad = true;
        continue;
      }
      const uint32_t old = atomicOr(&m[e], 1u << lane);
      if (old & (1u << lane)) bad = true;  // the same expert twice for one token
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(status, 0, MOE_ERR_INVALID_ARG);
  __syncwarp();
  uint32_t* out = bits + static_cast<long long>(w) * E;
  for (int e = lane; e < E; e += 32) out[e] = m[e];
}

// Block (32 x 32): 32 experts per block along x, 32 chunks of token words along y.
__global__ void k_perm_count(const uint32_t* __restrict__ bits, int W, int E,
                             int32_t* __restrict__ wpref, int32_t* __restrict__ counts) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int part[32][33];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int e = blockIdx.x * 32 + tx;
  const int chunk = (W + 31) / 32;
  const int w0 = min(W, ty * chunk), w1 = min(W, w0 + chunk);
  int sum = 0;
  if (e < E)
    for (int w = w0; w < w1; ++w) sum += __popc(bits[static_cast<long long>(w) * E + e]);
  part[ty][tx] = sum;
  __syncthreads();
  int pre = 0;
  for (int i = 0; i < ty; ++i) pre += part[i][tx];
  if (e < E) {
    int run = pre;
    for (int w = w0; w < w1; ++w) {
      const long long o = static_cast<long long>(w) * E + e;
      wpref[o] = run;
      run += __popc(bits[o]);
    }
    if (ty == 31) counts[e] = run;
  }
}

// Single block, 1024 threads: offsets = exclusive scan of counts (E <= 1024).
__global__ void k_perm_offsets(const int32_t* __restrict__ counts, int E,
                               int32_t* __restrict__ offsets) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int warp_sums[33];
  const int i = threadIdx.x;
  const int c = i < E ? counts[i] : 0;
  int total;
  const int excl = block_exclusive_scan(c, warp_sums, &total);
  if (i < E) offsets[i] = excl;
  if (i == 0) offsets[E] = total;
}

// Small problems (few token words): one 1024-thread block marks, counts and scans in
// shared memory, replacing the mark, count and offsets kernels.
constexpr int kSmallMaxWords = 8192;  // ceil(T/32) * E bit-matrix words held in shared memory
constexpr int kSmallMaxTokenWords = 64;

__global__ void __launch_bounds__(1024)
    k_perm_small(const int32_t* __restrict__ idx, int T, int E, int k,
                 uint32_t* __restrict__ bits_g, int32_t* __restrict__ wpref_g,
                 int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint32_t bits[];  // [W][E]
  __shared__ int warp_sums[33];
  const int W = (T + 31) / 32;
  const int tid = threadIdx.x;
  for (int i = tid; i < W * E; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  bool bad = false;
  const long long n = static_cast<long long>(T) * k;
  for (long long i = tid; i < n; i += blockDim.x) {
    const int t = static_cast<int>(i / k);
    const int e = idx[i];
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
    for (int w = 0; w < W; ++w) {
      const uint32_t b = bits[w * E + tid];
      wpref_g[w * E + tid] = c;
      bits_g[w * E + tid] = b;
      c += __popc(b);
    }
    counts[tid] = c;
  }
  int total;
  const int excl = block_exclusive_scan(c, warp_sums, &total);
  if (tid < E) offsets[tid] = excl;
  if (tid == 0) offsets[E] = total;
}

// One warp per (token, slot).
__global__ void k_perm_gather(const int32_t* __restrict__ idx, const uint16_t* __restrict__ x,
                              long long ldx, int T, int H, int E, int k,
                              const uint32_t* __restrict__ bits,
                              const int32_t* __restrict__ wpref,
                              const int32_t* __restrict__ offsets,
                              int32_t* __restrict__ row_token, int32_t* __restrict__ slot_row,
                              uint16_t* __restrict__ x_perm) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long gid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (gid >= static_cast<long long>(T) * k) return;
  const int t = static_cast<int>(gid / k);
  const int e = idx[gid];
  if (e < 0 || e >= E) {
    if (lane == 0) slot_row[gid] = -1;
    return;
  }
  const long long o = static_cast<long long>(t >> 5) * E + e;
  const uint32_t below = bits[o] & ((1u << (t & 31)) - 1u);
  const int row = offsets[e] + wpref[o] + __popc(below);
  if (lane == 0) {
    row_token[row] = t;
    slot_row[gid] = row;
  }
  if (x_perm == nullptr) return;  // index-only permutation (the NVFP4 path gathers itself)
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<long long>(t) * ldx);
  uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<long long>(row) * H);
  const int nvec = H / 8;
  for (int v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
}

}  // namespace

size_t permute_scratch_bytes(int T, int E) {
  const size_t W = (static_cast<size_t>(T) + 31) / 32;
  return align_up(W * E * 4, 256) * 2;
}

int launch_permute(const int32_t* idx, const uint16_t* x, int64_t ldx, int T, int H, int E, int k,
                   int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* slot_row,
                   uint16_t* x_perm, void* scratch, cudaStream_t s) {
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  if (T <= 0) {
    MOE_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s));
    MOE_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s));
    return MOE_OK;
  }
  const int W = (T + 31) / 32;
  uint32_t* bits = static_cast<uint32_t*>(scratch);
  int32_t* wpref = reinterpret_cast<int32_t*>(static_cast<char*>(scratch) +
                                              align_up(static_cast<size_t>(W) * E * 4, 256));
  int st;
  if (W <= kSmallMaxTokenWords && static_cast<long long>(W) * E <= kSmallMaxWords) {
    st = launch_pdl(k_perm_small, dim3(1), dim3(1024), static_cast<size_t>(W) * E * 4, s, idx, T,
                    E, k, bits, wpref, counts, offsets, status);
    if (st) return st;
  } else {
    const size_t mark_smem = static_cast<size_t>(kMarkWarps) * E * 4;
    st = launch_pdl(k_perm_mark, dim3((W + kMarkWarps - 1) / kMarkWarps), dim3(kMarkWarps * 32),
                    mark_smem, s, idx, T, E, k, bits, status);
    if (st) return st;
    st = launch_pdl(k_perm_count, dim3((E + 31) / 32), dim3(32, 32), 0, s,
                    static_cast<const uint32_t*>(bits), W, E, wpref, counts);
    if (st) return st;
    st = launch_pdl(k_perm_offsets, dim3(1), dim3(1024), 0, s, static_cast<const int32_t*>(counts),
                    E, offsets);
    if (st) return st;
  }
  const long long warps = static_cast<long long>(T) * k;
  const int threads = 256;
  st = launch_pdl(k_perm_gather, dim3(static_cast<unsigned>((warps * 32 + threads - 1) / threads)),
                  dim3(threads), 0, s, idx, x, static_cast<long long>(ldx), T, H, E, k,
                  static_cast<const uint32_t*>(bits), static_cast<const int32_t*>(wpref),
                  static_cast<const int32_t*>(offsets), row_token, slot_row, x_perm);
  if (st) return st;
  return MOE_OK;
}

}  // namespace moe
