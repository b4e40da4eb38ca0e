// internal.h: declarations shared by the translation units of libmoe (host side).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

// Device status word of the current device (see moe_get_device_status).
int* status_word();

// Streaming-multiprocessor count of the current device.
int sm_count();

// Record the first failing CUDA call and map it to a status code.
int cuda_status(cudaError_t e);
#define MOE_CUDA(call)                                \
  do {                                                \
    cudaError_t e__ = (call);                         \
    if (e__ != cudaSuccess) return ::moe::cuda_status(e__); \
  } while (0)
#define MOE_LAUNCHED() MOE_CUDA(cudaGetLastError())

// Kernel launch with programmatic dependent launch: the kernel may be scheduled while its
// predecessor on the stream is still running. Every kernel of this library calls
// griddep_wait() before its first global-memory access, which waits for the predecessor
// to complete and its writes to become visible, so stream order is kept. Only launch
// latency and the kernels' set-up (barrier init, TMEM allocation) overlap.
template <typename... Params, typename... Args>
inline int launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
  return e == cudaSuccess ? 0 : cuda_status(e);
}

#ifdef __CUDACC__
// Wait until the preceding kernel of the stream has completed and its memory is visible.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next kernel of the stream to be scheduled (it still waits in griddep_wait).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bump allocator over a caller-provided workspace (256-byte aligned slices).
struct Carver {
  char* base;
  size_t cap;
  size_t used = 0;
  Carver(void* b, size_t c) : base(static_cast<char*>(b)), cap(c) {}
  // Slices start on 256-byte device addresses whatever the alignment of `base`; the
  // workspace-size queries therefore add 256 bytes of slack.
  template <class T>
  T* take(size_t count) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    used = align_up(b + used, 256) - b;
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += count * sizeof(T);
    return p;
  }
  bool ok() const { return base != nullptr && used <= cap; }
};

// Epilogues of the grouped GEMM.
enum Epilogue : int {
  EPI_BF16 = 0,         // out = bf16(acc)
  EPI_SQRELU_BF16 = 1,  // out = bf16(max(acc, 0)^2)
  EPI_F32 = 2,          // out = acc (fp32)
  EPI_SPLIT_BF16 = 3,   // acc = hi + mid + lo, three bf16 planes at out, out + lo_offset,
                        // out + 2 * lo_offset (about fp32 accuracy for the router input)
};

// One grouped GEMM: for every group e and every row r in [offsets[e], offsets[e+1]):
//   out[r, n] = epi( sum_k act[r, k] * w[e, n, kw(k)] ),  n < N
// kw(k) = k mod k_wrap when k_wrap > 0 (the weights are re-read for a split input).
struct GroupedGemm {
  const void* act;       // [rows, K] bf16, row stride act_ld elements
  int64_t act_ld;
  int rows;
  const void* w;         // [E, N, Kw] bf16 (Kw = k_wrap ? k_wrap : K)
  int E;
  int N;
  int K;
  int k_wrap;
  const int* offsets;    // [E+1] device, or nullptr for one dense group of `rows`
  void* out;             // [rows, ldo] bf16 or fp32
  int64_t ldo;
  int64_t lo_offset;     // EPI_SPLIT_BF16 only: element distance between the planes
  int epi;
  int force_mode;        // 0 auto, 1 rows-as-M, 2 weights-as-M (swap)
  int precise;           // 1: fp32 partial sums every 256 of K (for routing inputs)
};
int launch_grouped_gemm(const GroupedGemm& g, cudaStream_t s);

// Router pieces.
int launch_router_logits(const uint16_t* x, int64_t ldx, const uint16_t* w_router, int T,
                         int D, int E, int parts, float* logits, cudaStream_t s);
int launch_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* idx,
                float* gates, uint8_t* tie, cudaStream_t s);

// Permutation pieces.
size_t permute_scratch_bytes(int T, int E);
int launch_permute(const int32_t* idx, const uint16_t* x, int64_t ldx, int T, int H, int E,
                   int k, int32_t* counts, int32_t* offsets, int32_t* row_token,
                   int32_t* slot_row, uint16_t* x_perm, void* scratch, cudaStream_t s);

int launch_combine(const uint16_t* y_perm, int rows, const int32_t* slot_row,
                   const float* gates, int T, int H, int k, uint16_t* y, cudaStream_t s);

}  // namespace moe
