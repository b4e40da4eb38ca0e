// scan.cuh: block-wide exclusive prefix sum shared by the permutation kernels.
#pragma once

namespace moe {

// Exclusive scan of one value per thread over a block of up to 1024 threads.
// Returns this thread's exclusive prefix; *total receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int c, int* warp_sums, int* total) {
  const int i = threadIdx.x, lane = i & 31, wid = i >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int ws = lane < nw ? warp_sums[lane] : 0;
    int wincl = ws;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wincl, d);
      if (lane >= d) wincl += v;
    }
    warp_sums[lane] = wincl - ws;
    if (lane == 31) warp_sums[32] = wincl;
  }
  __syncthreads();
  *total = warp_sums[32];
  return warp_sums[wid] + incl - c;
}

}  // namespace moe
