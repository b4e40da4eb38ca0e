// permute_noalloc.cu: moe_permute_noalloc, the expert permutation without a workspace.
//
// moe_permute needs scratch (a token-word x expert bit matrix and its popcount prefix) and
// takes it from a caller-provided workspace. Some callers cannot provide one. For example,
// a host runtime that owns all device memory through its own pool may forbid any other
// allocation, and a serving loop may run on a fixed memory plan with no room for
// per-call buffers. This entry point keeps that scratch in a fixed-size array that lives in
// the library's own device image. The caller passes only inputs and outputs, and no call
// here allocates or frees anything.
//
// Every GPU that loads the library holds kNoAllocScratchBytes for this array until the
// process exits. All calls on a device share the same array, so two calls that overlap on
// the GPU (different streams, no ordering between them) race on it and give wrong results.
// Calls ordered on one stream are fine.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace moe {
namespace {

// 2 MiB: enough for ceil(T/32) * E <= 262144, e.g. T = 16384 tokens with E = 512 experts.
constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;

static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_permute_scratch on the current device. In host code the symbol name
// stands for a host-side shadow, not a device address, so the address is looked up once
// per device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress((void**)&p, g_permute_scratch);
    if (e != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_permute_noalloc_max_scratch_bytes(void) {
  return moe::kNoAllocScratchBytes;
}

extern "C" int moe_permute_noalloc(const int32_t* topk_idx, const uint16_t* x, int T, int H,
                                   int E, int k, int32_t* counts, int32_t* offsets,
                                   int32_t* row_token, int32_t* slot_row, uint16_t* x_perm,
                                   cudaStream_t stream) {
  using namespace moe;
  if (!dims_ok(T, H, E, k)) return MOE_ERR_INVALID_ARG;  // the limits moe_permute applies
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !x || !row_token || !slot_row || !x_perm))
    return MOE_ERR_INVALID_ARG;
  if (H % 8 || !aligned16(x) || !aligned16(x_perm)) return MOE_ERR_UNSUPPORTED;
  // The scratch must fit in the fixed array; larger problems need moe_permute.
  if (permute_scratch_bytes(T, E) > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  // Nothing in the scratch has to start at zero: the mark kernel writes every bit-matrix
  // word and the count kernel every prefix word before either is read, so the previous
  // call's contents never leak into this one.
  return launch_permute(topk_idx, x, H, T, H, E, k, counts, offsets, row_token, slot_row, x_perm,
                        scratch, stream);
}
