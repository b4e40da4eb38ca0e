// debug.cu: the MOE_DEBUG build's workspace guards.
//
// In that build every workspace slice is followed by a 256-byte guard region (Carver). An
// entry point fills its guards with a fixed pattern before its first kernel and checks them
// after its last one, all on the caller's stream; a damaged guard means some kernel wrote
// past its slice, and the check records MOE_ERR_WORKSPACE on the device status word. The
// release build compiles none of this (the guards and WsGuard are empty there).
#include "internal.h"

#ifdef MOE_DEBUG
namespace moe {
namespace {

struct GuardList {
  uint32_t* p[kMaxWsGuards];
  int n;
};

__device__ __forceinline__ uint32_t guard_word(int g, int i) {
  return 0xA5C3E100u ^ (static_cast<uint32_t>(g) << 8) ^ static_cast<uint32_t>(i);
}

constexpr int kGuardWords = static_cast<int>(kWsGuardBytes / 4);

__global__ void k_guard_fill(GuardList l) {
  griddep_wait();
  griddep_launch_dependents();
  const int g = blockIdx.x, i = threadIdx.x;
  if (g < l.n && i < kGuardWords) l.p[g][i] = guard_word(g, i);
}

__global__ void k_guard_check(GuardList l, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int g = blockIdx.x, i = threadIdx.x;
  if (g < l.n && i < kGuardWords && l.p[g][i] != guard_word(g, i))
    atomicCAS(status, 0, MOE_ERR_WORKSPACE);
}

GuardList guard_list(const Carver& c) {
  GuardList l;
  l.n = c.nguards;
  for (int i = 0; i < c.nguards; ++i) l.p[i] = reinterpret_cast<uint32_t*>(c.guards[i]);
  return l;
}

}  // namespace

WsGuard::WsGuard(const Carver& c, cudaStream_t s) : c_(c), s_(s) {
  if (c_.nguards > 0)
    launch_pdl(k_guard_fill, dim3(c_.nguards), dim3(kGuardWords), 0, s_, guard_list(c_));
}

WsGuard::~WsGuard() {
  int* status = status_word();
  if (c_.nguards > 0 && status)
    launch_pdl(k_guard_check, dim3(c_.nguards), dim3(kGuardWords), 0, s_, guard_list(c_),
               status);
}

}  // namespace moe

// Host-side check of the detector itself (MOE_DEBUG build only): carves two slices of
// `workspace`, fills the guards, overwrites one byte of the first guard with cudaMemsetAsync
// (a host API call; no kernel writes out of bounds), then runs the check, which must record
// MOE_ERR_WORKSPACE on the status word.
#endif

// Host-side check of the detector itself: carves two slices of `workspace`, fills the
// guards, overwrites one byte of the first guard with cudaMemsetAsync (a host API call; no
// kernel writes out of bounds), then runs the check, which must record MOE_ERR_WORKSPACE on
// the status word. The release build has no guards and returns MOE_ERR_UNSUPPORTED.
extern "C" int moe_debug_guard_selftest(void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
#ifdef MOE_DEBUG
  using namespace moe;
  Carver c(workspace, workspace_bytes);
  c.take<uint32_t>(100);
  c.take<uint32_t>(300);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  {
    const WsGuard guard(c, stream);
    MOE_CUDA(cudaMemsetAsync(c.guards[0] + 17, 0x5A, 1, stream));
  }
  return MOE_OK;
#else
  (void)workspace;
  (void)workspace_bytes;
  (void)stream;
  return MOE_ERR_UNSUPPORTED;
#endif
}

extern "C" int moe_debug_build(void) { return moe::kDebugBuild ? 1 : 0; }
