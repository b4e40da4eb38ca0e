// selftest.cu: a self-test of the failure path that every tcgen05 pipeline kernel of this
// library shares, run on a live GPU without faulting or hanging it.
//
// The grouped GEMMs split each CTA into roles (a TMA producer, an MMA issuer, epilogue
// warps) that hand shared-memory stages and TMEM accumulators to one another through
// mbarriers. Every wait is bounded (mbar_wait). When a wait gives up, the waiting role
// records MOE_ERR_TIMEOUT on the device status word and raises the CTA's abort flag; the
// other roles see the flag and leave their own waits; the producer waits (again bounded)
// for the copies it still has in flight to land (drain_stages); TMEM is released; the CTA
// returns. This kernel builds exactly that situation with the same primitives: one bulk
// copy in flight, a producer wait on a barrier that nothing ever arrives on (with a short
// limit), and MMA and epilogue roles waiting on a barrier that nothing arrives on either
// (with the normal limit, so they can only leave early through the abort flag).
#include "internal.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kSelftestThreads = 128;
constexpr uint32_t kSelftestCopyBytes = 4096;
constexpr int kSelftestReportInts = 8;

__device__ __forceinline__ void record_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

// report[8 * blockIdx.x + i]: 0 producer wait gave up, 1 MMA role left through the abort flag,
// 2 epilogue role left through the abort flag, 3 the copy in flight landed before exit,
// 4 microseconds from the first wait to the release of TMEM.
__global__ void __launch_bounds__(kSelftestThreads)
    k_wait_selftest(const uint8_t* __restrict__ src, unsigned long long short_ns, int* status,
                    int* report) {
  __shared__ __align__(128) uint8_t stage[kSelftestCopyBytes];
  __shared__ uint64_t full, empty, tfull;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int flags[4];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&full, 1);
    mbar_init(&empty, 1);
    mbar_init(&tfull, 1);
    abort_flag = 0;
    for (int i = 0; i < 4; ++i) flags[i] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  griddep_launch_dependents();
  volatile int* ab = &abort_flag;
  const unsigned long long t0 = global_timer_ns();
  if (warp == 0) {
    if (lane == 0) {
      // producer: one stage armed and its copy issued, then a wait for a free stage that
      // never comes
      mbar_arrive_expect_tx(&full, kSelftestCopyBytes);
      bulk_load(stage, src, kSelftestCopyBytes, &full, policy_evict_first());
      if (!mbar_wait(&empty, 0u, ab, short_ns)) {
        *ab = 1;
        record_status(status, MOE_ERR_TIMEOUT);
        flags[0] = 1;
      }
      // next slot: stage 0 of the following phase, after one arming
      if (drain_stages(&full, 1, 0, 1u, 1))
        flags[3] = 1;
      else
        record_status(status, MOE_ERR_TIMEOUT);
    }
  } else if (warp == 1) {
    if (lane == 0 && !mbar_wait(&tfull, 0u, ab)) flags[1] = *ab;  // MMA issuer
  } else {
    const bool ok = mbar_wait(&tfull, 0u, ab);                    // epilogue warps
    if (warp == 2 && lane == 0 && !ok) flags[2] = *ab;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_slot, 32);
  }
  if (threadIdx.x == 0) {
    int* rep = report + static_cast<long long>(blockIdx.x) * kSelftestReportInts;
    for (int i = 0; i < 4; ++i) rep[i] = flags[i];
    rep[4] = static_cast<int>((global_timer_ns() - t0) / 1000ull);
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_selftest_wait_timeout(const void* src, int limit_us, int blocks, int* report,
                                         cudaStream_t stream) {
  using namespace moe;
  if (!src || !report || limit_us < 1 || limit_us > 1000000 || blocks < 1 || blocks > 1024)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(src)) return MOE_ERR_UNSUPPORTED;
  int* status = status_word();
  if (!status) return MOE_ERR_CUDA;
  return launch_pdl(k_wait_selftest, dim3(blocks), dim3(kSelftestThreads), 0, stream,
                    static_cast<const uint8_t*>(src), 1000ull * limit_us, status, report);
}
