// internal.h: declarations shared by the translation units of libmoe (host side).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

// Device status word of the current device (see moe_get_device_status).
int* status_word();

// Streaming-multiprocessor count of the current device.
int sm_count();

// Sizes every routed-layer call accepts: T >= 0 tokens of width D > 0, 1 <= E <= 1024
// experts, 1 <= k <= min(32, E) of them per token, T * k rows addressable by int32.
bool dims_ok(int T, int D, int E, int k);

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
// In the MOE_DEBUG build every slice is followed by a 256-byte guard region; the entry
// points fill the guards with a pattern before their first kernel and check them after the
// last one (WsGuard), so a kernel that writes past its slice is reported on the status word
// as MOE_ERR_WORKSPACE. The workspace-size queries carve the same way, so they include the
// guards.
constexpr int kMaxWsGuards = 64;
constexpr size_t kWsGuardBytes = 256;
struct Carver {
  char* base;
  size_t cap;
  size_t used = 0;
#ifdef MOE_DEBUG
  char* guards[kMaxWsGuards];
  int nguards = 0;
#endif
  Carver(void* b, size_t c) : base(static_cast<char*>(b)), cap(c) {}
  // Slices start on 256-byte device addresses whatever the alignment of `base`; the
  // workspace-size queries therefore add 256 bytes of slack.
  template <class T>
  T* take(size_t count) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    used = align_up(b + used, 256) - b;
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += count * sizeof(T);
#ifdef MOE_DEBUG
    used = align_up(b + used, 256) - b;
    if (base && nguards < kMaxWsGuards) guards[nguards++] = base + used;
    used += kWsGuardBytes;
#endif
    return p;
  }
  bool ok() const { return base != nullptr && used <= cap; }
};

// MOE_DEBUG build: fills the workspace guards of `c` (stream-ordered) when constructed and
// checks them when destroyed, i.e. after the entry point has enqueued its last kernel. The
// release build compiles this to nothing.
struct WsGuard {
#ifdef MOE_DEBUG
  WsGuard(const Carver& c, cudaStream_t s);
  ~WsGuard();
  const Carver& c_;
  cudaStream_t s_;
#else
  WsGuard(const Carver&, cudaStream_t) {}
#endif
};

// Whether this library was built with MOE_DEBUG (extra device-side checks, workspace guards).
constexpr bool kDebugBuild =
#ifdef MOE_DEBUG
    true;
#else
    false;
#endif

// Epilogues of the grouped GEMM.
enum Epilogue : int {
  EPI_BF16 = 0,         // out = bf16(acc)
  EPI_SQRELU_BF16 = 1,  // out = bf16(max(acc, 0)^2)
  EPI_F32 = 2,          // out = acc (fp32)
  EPI_SPLIT_BF16 = 3,   // acc = hi + mid + lo, three bf16 planes at out, out + lo_offset,
                        // out + 2 * lo_offset (about fp32 accuracy for the router input)
  EPI_ADD_BF16 = 4,     // out = bf16(acc + add[row, col]) (add: bf16, row stride ld_add)
  EPI_COMBINE_I64 = 5,  // combine fused into the epilogue: out is an int64 [T, ldo] sum,
                        // out[token(row), col] += round(gate(row) * acc * 2^32) (fixed.cuh)
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
  // E4M3 operands (act and w hold one byte per element): the epilogue multiplies by
  // (a_amax / 448) * w_scale[e]; with EPI_SQRELU_BF16, out_amax (if set) receives the max
  // of the stored values (fp32 bits).
  // Gathered activations (bf16, rows-as-M): row r of group e reads act row
  // row_token[offsets[e] + r] (act has src_rows rows); x_perm is never materialised.
  const int32_t* row_token = nullptr;
  int src_rows = 0;
  const uint16_t* add = nullptr;  // EPI_ADD_BF16 only
  int64_t ld_add = 0;
  int fp8 = 0;
  const uint32_t* a_amax = nullptr;
  const float* w_scale = nullptr;
  uint32_t* out_amax = nullptr;
  int64_t w_ld = 0;  // bytes between weight rows (0: Kw times the element size)
  // EPI_COMBINE_I64 only: row r belongs to token comb_token[r] (< comb_T); its gate is
  // comb_gates[t k + j] for the slot j with comb_slot_row[t k + j] == r (k = comb_k).
  const int32_t* comb_token = nullptr;
  const int32_t* comb_slot_row = nullptr;
  const float* comb_gates = nullptr;
  int comb_k = 0;
  int comb_T = 0;
};
int launch_grouped_gemm(const GroupedGemm& g, cudaStream_t s);
// The rows-as-M GEMM on CTA pairs (cta_group::2, 256 x 256 pair tiles): used by
// launch_grouped_gemm for bf16/E4M3 GEMMs with at least 256 rows per group on average.
bool grouped_gemm_2sm_ok(const GroupedGemm& g);
int launch_grouped_gemm_2sm(const GroupedGemm& g, cudaStream_t s);
// Whether a grouped GEMM of `rows` routed rows over E groups runs with the rows on the MMA's
// M side (and can then gather its activation rows itself).
bool grouped_gemm_rows_as_m(int rows, int E);

// Tiled TMA descriptor (rank 2 or 3), zero fill out of bounds, 128-byte swizzle unless
// another is given. dims and box are innermost first; strides_bytes holds the rank - 1 outer
// strides.
bool encode_tmap(CUtensorMap* m, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// ------------------------------------------------------------------------------ NVFP4 ----
// NVFP4 matrix [R, K]: E2M1 codes, two per byte (element 2i in bits 0-3), [R, K/2]; one
// E4M3 scale per 16 elements of K stored as 512-byte atoms, atom (R/128 block rb, K/64
// step j) at (rb * (K/64) + j) * 512 with row 128 rb + 32 r1 + r0, block kb at byte
// r0 * 16 + r1 * 4 + kb; and an fp32 global scale g = amax / (6 * 448).
constexpr float kNvfp4GlobalDiv = 2688.0f;  // 6 (E2M1 max) * 448 (E4M3 max)

inline size_t nvfp4_sf_bytes(long long rows, int K) {
  return static_cast<size_t>((rows + 127) / 128) * (K / 64) * 512;
}

// amax[g] = max |src| over matrix g (bf16 bits; amax kept as fp32 bits). amax must be zeroed.
int launch_amax_bf16(const uint16_t* src, long long elems_per_matrix, int G, uint32_t* amax,
                     cudaStream_t s);
// Quantise G weight matrices [N, K] with per-matrix global scales from amax[g].
int launch_quant_weights(const uint16_t* w, int G, int N, int K, const uint32_t* amax,
                         uint8_t* codes, uint8_t* sf, cudaStream_t s);
// The same with 2-D (16 rows x 16 K) weight blocks: the block scale is repeated per row.
int launch_quant_weights_2d(const uint16_t* w, int G, int N, int K, const uint32_t* amax,
                            uint8_t* codes, uint8_t* sf, cudaStream_t s);
// g[i] = amax[i] / 2688 in place (amax held as fp32 bits in the same words).
int launch_finalize_gscale(float* g, int G, cudaStream_t s);
// poff = exclusive scan of round_up(offsets[e+1] - offsets[e], 128): expert segments padded
// to whole 128-row tiles.
int launch_pad_offsets(const int32_t* offsets, int E, int32_t* poff, cudaStream_t s);
// Quantise activation rows into the padded layout. Row p of expert e (local = p - poff[e]):
// gather mode (offsets != null): source row row_token[offsets[e] + local] (or
// offsets[e] + local when row_token is null) if local < count[e], else a zero row;
// identity mode (offsets == null): source row p. Global scale from *amax. A source row at or
// past src_rows is read as zeros and reported on the status word.
int launch_quant_act(const uint16_t* src, long long ld, long long src_rows,
                     const int32_t* row_token, const int32_t* offsets, const int32_t* poff,
                     int E, int K, int P_max, const uint32_t* amax, uint8_t* codes, uint8_t* sf,
                     cudaStream_t s);

// ------------------------------------------------------------------------------- FP8 ----
// Routed tokens in the padded layout, each token quantised once (global scale from *amax)
// and written to its k rows: slot s of token t goes to row poff[e] + slot_row[t k + s] -
// offsets[e], e = topk_idx[t k + s]; padding rows get zero codes and scales. The same bytes
// as launch_quant_act in gather mode. Out-of-range maps are skipped and reported.
int launch_quant_tokens(const uint16_t* src, long long ld, int T, int k, const int32_t* topk_idx,
                        const int32_t* slot_row, const int32_t* offsets, const int32_t* poff,
                        int E, int K, int P_max, const uint32_t* amax, uint8_t* codes,
                        uint8_t* sf, cudaStream_t s);

// Per-tensor E4M3: s = amax / 448, q = E4M3(v / s). Codes are one byte per element.
constexpr float kFp8Div = 448.0f;
// Quantise rows of src (bf16, row stride ld) into out [rows, K] E4M3 bytes. Row r reads src
// row row_map[r] when row_map is set, else row r. Matrix r / rows_per_scale uses the scale
// of amax[r / rows_per_scale] (rows_per_scale = 0: one scale for all rows).
int launch_quant_fp8(const uint16_t* src, long long ld, const int32_t* row_map, long long rows,
                     int K, long long rows_per_scale, const uint32_t* amax, uint8_t* out,
                     long long ldo, cudaStream_t s);
// Routed tokens quantised once each and written to their k permuted rows slot_row[t k + j]
// of out [rows, K] (rows ldo bytes apart); the same bytes as launch_quant_fp8 with
// row_map = row_token.
int launch_quant_fp8_tokens(const uint16_t* src, long long ld, int T, int k,
                            const int32_t* slot_row, long long rows, int K, const uint32_t* amax,
                            uint8_t* out, long long ldo, cudaStream_t s);
// Row pitch in bytes of the E4M3 tensors the grouped GEMMs read (activations and weight
// codes): K rounded up to 128 bytes, so that every row's 128-byte K-slices start on a
// 128-byte boundary.
#ifdef __CUDACC__
#define MOE_HD __host__ __device__
#else
#define MOE_HD
#endif
MOE_HD inline long long fp8_act_pitch(int K) {
  return (static_cast<long long>(K) + 127) / 128 * 128;
}
// s[i] = amax[i] / 448 in place.
int launch_finalize_fp8_scale(float* s, int G, cudaStream_t stream);

// Row pitch in bytes of the NVFP4 activation codes the block-scaled GEMMs read: K/2 rounded
// up to 128 bytes (the weight codes keep K/2).
MOE_HD inline long long fp4_act_pitch(int K) {
  return (static_cast<long long>(K / 2) + 127) / 128 * 128;
}

struct Fp4Gemm {
  const uint8_t* a_codes;  // [P, K/2], rows a_ld bytes apart, padded per group (poff)
  long long a_ld;
  const uint8_t* a_sf;     // atoms of the padded rows
  const uint32_t* a_amax;  // activation amax (fp32 bits); g_a = amax / 2688
  int P;                   // allocated padded rows (bound for poff[E])
  const int32_t* poff;     // [E+1] padded group offsets (multiples of 128)
  const uint8_t* w_codes;  // [E, N, K/2]
  const uint8_t* w_sf;     // [E][ceil(N/128)][K/64] atoms
  const float* w_gscale;   // [E]
  int E, N, K;
  const int32_t* out_off;  // [E+1] output row offsets (store only local < count), or null:
                           // output row = padded row (every row stored)
  int out_rows;            // rows of `out`
  void* out;               // bf16 [out_rows, ldo]
  long long ldo;
  int epi;                 // EPI_SQRELU_BF16 or EPI_BF16
  uint32_t* out_amax;      // EPI_SQRELU_BF16: max of the stored values (fp32 bits), or null
};
int launch_fp4_gemm(const Fp4Gemm& g, cudaStream_t s);

// Router pieces.
int launch_router_logits(const uint16_t* x, int64_t ldx, const uint16_t* w_router, int T,
                         int D, int E, int parts, float* logits, cudaStream_t s);
int launch_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* idx,
                float* gates, uint8_t* tie, cudaStream_t s);

// Small batches (T <= 256, E <= 256): router logits, top-k and, when row_token is set, the
// dispatch maps (counts, offsets, row_token, slot_row) in one kernel. `sync` holds
// route_fused_sync_ints(T) ints of 8-byte aligned scratch; its contents at entry do not
// matter (generation-tagged counters).
bool route_fused_ok(int T, int D, int E, int k, int parts);
size_t route_fused_sync_ints(int T);
int launch_route_fused(const uint16_t* x, int64_t ldx, const uint16_t* w_router,
                       const float* bias, int T, int D, int E, int k, int parts, float* logits,
                       int32_t* idx, float* gates, uint8_t* tie, int32_t* counts,
                       int32_t* offsets, int32_t* row_token, int32_t* slot_row, int* sync,
                       cudaStream_t s);
// x_perm[r] = x[row_token[r]] for r < rows (x has src_rows rows; the MOE_DEBUG build checks
// every row_token against it and reports MOE_ERR_INVALID_ARG on the status word).
int launch_gather_rows(const int32_t* row_token, const uint16_t* x, int64_t ldx, int src_rows,
                       int rows, int H, uint16_t* x_perm, cudaStream_t s);

// Permutation pieces.
size_t permute_scratch_bytes(int T, int E);
int launch_permute(const int32_t* idx, const uint16_t* x, int64_t ldx, int T, int H, int E,
                   int k, int32_t* counts, int32_t* offsets, int32_t* row_token,
                   int32_t* slot_row, uint16_t* x_perm, void* scratch, cudaStream_t s);

// y = addend + gate-weighted sum of the rows (addend [T, H] bf16, or null).
int launch_combine(const uint16_t* y_perm, int rows, const int32_t* slot_row,
                   const float* gates, int T, int H, int k, uint16_t* y, cudaStream_t s,
                   const uint16_t* addend = nullptr);
// The fused combine's two passes: zero the n int64 sums, and after the down-projection's
// EPI_COMBINE_I64 epilogue write y = bf16(acc * 2^-32) (n a multiple of 8).
int launch_zero_fixed(int64_t* acc, long long n, cudaStream_t s);
int launch_combine_fixed(const int64_t* acc, long long n, uint16_t* y, cudaStream_t s);

}  // namespace moe
