// capi.cu: the extern "C" entry points of libmoe. Argument checks, workspace layout and
// stream-ordered orchestration of the kernels. No call allocates device memory.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace moe {

__device__ int g_status_word = 0;

namespace {
constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::mutex g_mu;

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}
}  // namespace

int* status_word() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[d] = static_cast<int*>(p);
  }
  return g_status_ptr[d];
}

int sm_count() {
  const int d = current_device();
  if (d < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sm_count[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0)
      n = 1;
    g_sm_count[d] = n;
  }
  return g_sm_count[d];
}

int cuda_status(cudaError_t) { return MOE_ERR_CUDA; }

bool dims_ok(int T, int D, int E, int k) {
  if (T < 0 || D <= 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return false;
  if (static_cast<long long>(T) * k > 0x7fffffffLL) return false;
  return true;
}

namespace {

// Workspace of one routed MoE layer of width D: routing, permutation, FFN buffers.
struct LayerWs {
  float* logits;
  int32_t* idx;
  float* gates;
  uint8_t* tie;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_token;
  int32_t* slot_row;
  int* sync;  // counters of the fused small-batch routing kernel
  void* perm_scratch;
  uint16_t* x_perm;
  uint16_t* h;
  uint16_t* y_perm;  // [rows, D] expert outputs, or null with the fused combine
  int64_t* acc;      // fused combine: [T, D] fixed-point sums, else null
};

// fused_combine: the down-projection adds into acc (fixed.cuh) instead of writing y_perm.
LayerWs carve_layer(Carver& c, int T, int D, int E, int k, int F, bool fused_combine = false) {
  const size_t rows = static_cast<size_t>(T) * k;
  LayerWs w;
  w.logits = c.take<float>(static_cast<size_t>(T) * E);
  w.idx = c.take<int32_t>(rows);
  w.gates = c.take<float>(rows);
  w.tie = c.take<uint8_t>(T > 0 ? T : 1);
  w.counts = c.take<int32_t>(E);
  w.offsets = c.take<int32_t>(E + 1);
  w.row_token = c.take<int32_t>(rows);
  w.slot_row = c.take<int32_t>(rows);
  w.sync = c.take<int>(route_fused_sync_ints(T));
  w.perm_scratch = c.take<char>(permute_scratch_bytes(T, E));
  w.x_perm = c.take<uint16_t>(rows * D);
  w.h = c.take<uint16_t>(rows * F);
  w.y_perm = fused_combine ? nullptr : c.take<uint16_t>(rows * D);
  w.acc = fused_combine ? c.take<int64_t>(static_cast<size_t>(T) * D) : nullptr;
  return w;
}

// Router logits: CUDA cores for small batches, tcgen05 GEMM (fp32 epilogue) otherwise.
// `parts` bf16 planes per input row (1, or 3 for a hi/mid/lo split of an fp32 vector).
int router_logits(const uint16_t* x, int64_t ldx, const uint16_t* w_router, int T, int D, int E,
                  int parts, float* logits, cudaStream_t s) {
  if (T > 512 && E % 16 == 0 && D % 64 == 0) {
    GroupedGemm g{};
    g.act = x;
    g.act_ld = ldx;
    g.rows = T;
    g.w = w_router;
    g.E = 1;
    g.N = E;
    g.K = parts * D;
    g.k_wrap = parts > 1 ? D : 0;
    g.offsets = nullptr;
    g.out = logits;
    g.ldo = E;
    g.lo_offset = 0;
    g.epi = EPI_F32;
    g.force_mode = 1;
    g.precise = 1;
    return launch_grouped_gemm(g, s);
  }
  return launch_router_logits(x, ldx, w_router, T, D, E, parts, logits, s);
}

// Expert FFNs. The up-projection reads x_perm [rows, D], or, when row_token is given, gathers
// the rows from x_src (src_rows rows, row stride ld_src) by token: x_perm is never written.
// Profiling hook (moe_set_profile_events): events recorded around the expert GEMMs of the
// layer calls made on this thread.
struct ProfileEvents {
  cudaEvent_t ev[4];
  bool on = false;
};
thread_local ProfileEvents g_profile;

// Mark i: 0 before the up-projection GEMM, 1 after it, 2 before the down-projection GEMM,
// 3 after it.
int profile_mark(int i, cudaStream_t s) {
  if (!g_profile.on) return MOE_OK;
  MOE_CUDA(cudaEventRecord(g_profile.ev[i], s));
  return MOE_OK;
}

// With `fc`, the down-projection's epilogue adds each row's gated output into its token's
// fixed-point sum fc->acc (EPI_COMBINE_I64) and y_perm is not written.
struct FusedCombine {
  int64_t* acc;
  const int32_t* row_token;
  const int32_t* slot_row;
  const float* gates;
  int T, k;
};

int ffn(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_up,
        const uint16_t* w_down, int rows, int D, int F, int E, uint16_t* h, uint16_t* y_perm,
        cudaStream_t s, const int32_t* row_token = nullptr, const uint16_t* x_src = nullptr,
        int64_t ld_src = 0, int src_rows = 0, const FusedCombine* fc = nullptr) {
  GroupedGemm up{};
  up.act = row_token ? x_src : x_perm;
  up.act_ld = row_token ? ld_src : D;
  up.rows = rows;
  up.row_token = row_token;
  up.src_rows = src_rows;
  up.w = w_up;
  up.E = E;
  up.N = F;
  up.K = D;
  up.offsets = offsets;
  up.out = h;
  up.ldo = F;
  up.epi = EPI_SQRELU_BF16;
  int st = profile_mark(0, s);
  if (st) return st;
  st = launch_grouped_gemm(up, s);
  if (st) return st;
  st = profile_mark(1, s);
  if (st) return st;
  GroupedGemm dn{};
  dn.act = h;
  dn.act_ld = F;
  dn.rows = rows;
  dn.w = w_down;
  dn.E = E;
  dn.N = D;
  dn.K = F;
  dn.offsets = offsets;
  dn.out = y_perm;
  dn.ldo = D;
  dn.epi = EPI_BF16;
  if (fc) {
    dn.out = fc->acc;
    dn.epi = EPI_COMBINE_I64;
    dn.comb_token = fc->row_token;
    dn.comb_slot_row = fc->slot_row;
    dn.comb_gates = fc->gates;
    dn.comb_k = fc->k;
    dn.comb_T = fc->T;
  }
  st = profile_mark(2, s);
  if (st) return st;
  st = launch_grouped_gemm(dn, s);
  if (st) return st;
  return profile_mark(3, s);
}

// route -> permute -> grouped FFN -> combine for rows of width D read from x (row stride ldx).
// Routing reads xr (row stride ldr, width Dr, in `parts` bf16 planes).
int layer(const uint16_t* x, int64_t ldx, const uint16_t* xr, int64_t ldr, int Dr, int parts,
          const uint16_t* w_router, const float* bias, const uint16_t* w_up,
          const uint16_t* w_down, int T, int D, int E, int k, int F, uint16_t* y,
          int32_t* idx_out, float* gates_out, const LayerWs& w, cudaStream_t s,
          const uint16_t* addend = nullptr, bool gather_tokens = false) {
  if (w.acc && addend) return MOE_ERR_UNSUPPORTED;  // no fused-combine call takes an addend
  int32_t* idx = idx_out ? idx_out : w.idx;
  float* gates = gates_out ? gates_out : w.gates;
  // gather_tokens: with the rows on the MMA's M side the up-projection gathers its token
  // rows itself (TMA gather4), so the permutation only builds the maps (no x_perm copy).
  const int rows = T * k;
  // gather_tokens (moe_forward_gathered): the up-projection gathers its token rows itself
  // with TMA gather4 (32 copies per K-slice with the rows on the MMA's M side, BN / 4 with
  // the weights there), so x_perm is never written. Both forms measured slower than reading
  // a materialised x_perm on B300, so moe_forward does not gather.
  const bool gather = gather_tokens;
  int st;
  if (route_fused_ok(T, Dr, E, k, parts)) {
    // small batches: logits, top-k and the dispatch maps in one kernel, then the row copy
    st = launch_route_fused(xr, ldr, w_router, bias, T, Dr, E, k, parts, w.logits, idx, gates,
                            w.tie, w.counts, w.offsets, w.row_token, w.slot_row, w.sync, s);
    if (st) return st;
    if (!gather) {
      st = launch_gather_rows(w.row_token, x, ldx, T, rows, D, w.x_perm, s);
      if (st) return st;
    }
  } else {
    st = router_logits(xr, ldr, w_router, T, Dr, E, parts, w.logits, s);
    if (st) return st;
    st = launch_topk(w.logits, bias, T, E, k, idx, gates, w.tie, s);
    if (st) return st;
    st = launch_permute(idx, x, ldx, T, D, E, k, w.counts, w.offsets, w.row_token, w.slot_row,
                        gather ? nullptr : w.x_perm, w.perm_scratch, s);
    if (st) return st;
  }
  if (w.acc) {  // combine fused into the down-projection (carve_layer with fused_combine)
    st = launch_zero_fixed(w.acc, static_cast<long long>(T) * D, s);
    if (st) return st;
    const FusedCombine fc{w.acc, w.row_token, w.slot_row, gates, T, k};
    st = gather ? ffn(nullptr, w.offsets, w_up, w_down, rows, D, F, E, w.h, nullptr, s,
                      w.row_token, x, ldx, T, &fc)
                : ffn(w.x_perm, w.offsets, w_up, w_down, rows, D, F, E, w.h, nullptr, s,
                      nullptr, nullptr, 0, 0, &fc);
    if (st) return st;
    return launch_combine_fixed(w.acc, static_cast<long long>(T) * D, y, s);
  }
  if (gather)
    st = ffn(nullptr, w.offsets, w_up, w_down, rows, D, F, E, w.h, w.y_perm, s, w.row_token, x,
             ldx, T);
  else
    st = ffn(w.x_perm, w.offsets, w_up, w_down, rows, D, F, E, w.h, w.y_perm, s);
  if (st) return st;
  return launch_combine(w.y_perm, rows, w.slot_row, gates, T, D, k, y, s, addend);
}

// The shared expert on every token: h_s = max(0, x . w_up_s^T)^2, then
// out = h_s . w_down_s^T (+ add when given: EPI_ADD_BF16 with add [T, N_out] bf16).
int shared_expert(const uint16_t* x, int64_t ldx, int T, int H, int Fs, const uint16_t* w_up_s,
                  const uint16_t* w_down_s, uint16_t* h_s, uint16_t* out,
                  cudaStream_t s) {
  GroupedGemm up{};
  up.act = x;
  up.act_ld = ldx;
  up.rows = T;
  up.w = w_up_s;
  up.E = 1;
  up.N = Fs;
  up.K = H;
  up.out = h_s;
  up.ldo = Fs;
  up.epi = EPI_SQRELU_BF16;
  int st = launch_grouped_gemm(up, s);
  if (st) return st;
  GroupedGemm dn{};
  dn.act = h_s;
  dn.act_ld = Fs;
  dn.rows = T;
  dn.w = w_down_s;
  dn.E = 1;
  dn.N = H;
  dn.K = Fs;
  dn.out = out;
  dn.ldo = H;
  dn.epi = EPI_BF16;
  return launch_grouped_gemm(dn, s);
}

// NVFP4 expert FFN buffers. P bounds the padded rows: every group rounded up to whole
// 128-row tiles adds at most 127 rows.
struct Fp4Ws {
  int P;
  int32_t* poff;
  uint32_t* amax;  // [0] activations entering the up-projection, [1] hidden activations
  uint8_t* xq;
  uint8_t* xsf;
  uint16_t* h;
  uint8_t* hq;
  uint8_t* hsf;
};

int fp4_rows_bound(int rows, int E) {
  const long long p = static_cast<long long>(rows) + 127LL * E;
  return static_cast<int>(align_up(static_cast<size_t>(p), 128));
}

Fp4Ws carve_fp4(Carver& c, int rows, int H, int F, int E) {
  Fp4Ws w;
  w.P = fp4_rows_bound(rows, E);
  const size_t P = static_cast<size_t>(w.P);
  w.poff = c.take<int32_t>(E + 1);
  w.amax = c.take<uint32_t>(2);
  w.xq = c.take<uint8_t>(P * fp4_act_pitch(H));
  w.xsf = c.take<uint8_t>(nvfp4_sf_bytes(w.P, H));
  w.h = c.take<uint16_t>(P * F);
  w.hq = c.take<uint8_t>(P * fp4_act_pitch(F));
  w.hsf = c.take<uint8_t>(nvfp4_sf_bytes(w.P, F));
  return w;
}

struct Nvfp4Weights {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* gscale;
};

// The routing of the tokens whose rows enter the experts (layer calls): token t's slot j
// is expert topk_idx[t k + j], permuted row slot_row[t k + j].
struct TokenSlots {
  const int32_t* topk_idx;
  const int32_t* slot_row;
  int T, k;
};

// NVFP4 expert FFNs. The rows entering the experts are rows offsets[e] + r of `src` (row
// stride ld), or, with `slots`, the routed tokens of src: each token is quantised once and
// written to its k rows. amax_rows rows of src make up the activation tensor whose amax sets
// its global scale.
int ffn_nvfp4(const uint16_t* src, long long ld, long long amax_rows, const TokenSlots* slots,
              const int32_t* offsets, const Nvfp4Weights& up, const Nvfp4Weights& down, int rows,
              int H, int F, int E, uint16_t* y_perm, const Fp4Ws& w, cudaStream_t s) {
  MOE_CUDA(cudaMemsetAsync(w.amax, 0, 2 * sizeof(uint32_t), s));
  int st = launch_amax_bf16(src, amax_rows * ld, 1, w.amax, s);
  if (st) return st;
  st = launch_pad_offsets(offsets, E, w.poff, s);
  if (st) return st;
  if (slots)
    st = launch_quant_tokens(src, ld, slots->T, slots->k, slots->topk_idx, slots->slot_row,
                             offsets, w.poff, E, H, w.P, w.amax, w.xq, w.xsf, s);
  else
    st = launch_quant_act(src, ld, amax_rows, nullptr, offsets, w.poff, E, H, w.P, w.amax, w.xq,
                          w.xsf, s);
  if (st) return st;
  Fp4Gemm g{};
  g.a_codes = w.xq;
  g.a_ld = fp4_act_pitch(H);
  g.a_sf = w.xsf;
  g.a_amax = w.amax;
  g.P = w.P;
  g.poff = w.poff;
  g.w_codes = up.codes;
  g.w_sf = up.scales;
  g.w_gscale = up.gscale;
  g.E = E;
  g.N = F;
  g.K = H;
  g.out_off = nullptr;
  g.out_rows = w.P;
  g.out = w.h;
  g.ldo = F;
  g.epi = EPI_SQRELU_BF16;
  g.out_amax = w.amax + 1;
  st = profile_mark(0, s);
  if (st) return st;
  st = launch_fp4_gemm(g, s);
  if (st) return st;
  st = profile_mark(1, s);
  if (st) return st;
  st = launch_quant_act(w.h, F, w.P, nullptr, nullptr, w.poff, E, F, w.P, w.amax + 1, w.hq,
                        w.hsf, s);
  if (st) return st;
  Fp4Gemm d{};
  d.a_codes = w.hq;
  d.a_ld = fp4_act_pitch(F);
  d.a_sf = w.hsf;
  d.a_amax = w.amax + 1;
  d.P = w.P;
  d.poff = w.poff;
  d.w_codes = down.codes;
  d.w_sf = down.scales;
  d.w_gscale = down.gscale;
  d.E = E;
  d.N = H;
  d.K = F;
  d.out_off = offsets;
  d.out_rows = rows;
  d.out = y_perm;
  d.ldo = H;
  d.epi = EPI_BF16;
  st = profile_mark(2, s);
  if (st) return st;
  st = launch_fp4_gemm(d, s);
  if (st) return st;
  return profile_mark(3, s);
}

// FP8 expert FFN buffers (unpadded: the E4M3 GEMM needs no scale atoms).
struct Fp8Ws {
  uint32_t* amax;  // [0] activations entering the up-projection, [1] hidden activations
  uint8_t* xq;
  uint16_t* h;
  uint8_t* hq;
};

// xq and hq rows are fp8_act_pitch(H) and fp8_act_pitch(F) bytes apart.
Fp8Ws carve_fp8(Carver& c, int rows, int H, int F) {
  Fp8Ws w;
  w.amax = c.take<uint32_t>(2);
  w.xq = c.take<uint8_t>(static_cast<size_t>(rows) * fp8_act_pitch(H));
  w.h = c.take<uint16_t>(static_cast<size_t>(rows) * F);
  w.hq = c.take<uint8_t>(static_cast<size_t>(rows) * fp8_act_pitch(F));
  return w;
}

// FP8 expert FFNs. The rows entering the experts are src rows r, or, with `slots`, the
// routed tokens of src (each quantised once and written to its k permuted rows); amax_rows
// rows of src make up the activation tensor of the scale.
int ffn_fp8(const uint16_t* src, long long ld, long long amax_rows, const TokenSlots* slots,
            const int32_t* offsets, const uint8_t* up, const float* up_scale, const uint8_t* down,
            const float* down_scale, int rows, int H, int F, int E, uint16_t* y_perm,
            const Fp8Ws& w, cudaStream_t s) {
  MOE_CUDA(cudaMemsetAsync(w.amax, 0, 2 * sizeof(uint32_t), s));
  int st = launch_amax_bf16(src, amax_rows * ld, 1, w.amax, s);
  if (st) return st;
  if (slots)
    st = launch_quant_fp8_tokens(src, ld, slots->T, slots->k, slots->slot_row, rows, H, w.amax,
                                 w.xq, fp8_act_pitch(H), s);
  else
    st = launch_quant_fp8(src, ld, nullptr, rows, H, 0, w.amax, w.xq, fp8_act_pitch(H), s);
  if (st) return st;
  GroupedGemm g{};
  g.act = w.xq;
  g.act_ld = fp8_act_pitch(H);
  g.rows = rows;
  g.w = up;
  g.w_ld = fp8_act_pitch(H);
  g.E = E;
  g.N = F;
  g.K = H;
  g.offsets = offsets;
  g.out = w.h;
  g.ldo = F;
  g.epi = EPI_SQRELU_BF16;
  g.fp8 = 1;
  g.a_amax = w.amax;
  g.w_scale = up_scale;
  g.out_amax = w.amax + 1;
  st = profile_mark(0, s);
  if (st) return st;
  st = launch_grouped_gemm(g, s);
  if (st) return st;
  st = profile_mark(1, s);
  if (st) return st;
  st = launch_quant_fp8(w.h, F, nullptr, rows, F, 0, w.amax + 1, w.hq, fp8_act_pitch(F), s);
  if (st) return st;
  GroupedGemm d{};
  d.act = w.hq;
  d.act_ld = fp8_act_pitch(F);
  d.rows = rows;
  d.w = down;
  d.w_ld = fp8_act_pitch(F);
  d.E = E;
  d.N = H;
  d.K = F;
  d.offsets = offsets;
  d.out = y_perm;
  d.ldo = H;
  d.epi = EPI_BF16;
  d.fp8 = 1;
  d.a_amax = w.amax + 1;
  d.w_scale = down_scale;
  st = profile_mark(2, s);
  if (st) return st;
  st = launch_grouped_gemm(d, s);
  if (st) return st;
  return profile_mark(3, s);
}

// Routing and dispatch buffers at the head of the moe_forward_nvfp4 / moe_forward_fp8
// workspaces, followed by y_perm.
struct QuantFwdWs {
  float* logits;
  int32_t* idx;
  float* gates;
  uint8_t* tie;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_token;
  int32_t* slot_row;
  int* sync;
  void* perm_scratch;
  uint16_t* y_perm;
};

QuantFwdWs carve_quant_fwd(Carver& c, int T, int H, int E, int k) {
  QuantFwdWs w;
  const size_t rows = static_cast<size_t>(T) * k;
  w.logits = c.take<float>(static_cast<size_t>(T) * E);
  w.idx = c.take<int32_t>(rows);
  w.gates = c.take<float>(rows);
  w.tie = c.take<uint8_t>(T > 0 ? T : 1);
  w.counts = c.take<int32_t>(E);
  w.offsets = c.take<int32_t>(E + 1);
  w.row_token = c.take<int32_t>(rows);
  w.slot_row = c.take<int32_t>(rows);
  w.sync = c.take<int>(route_fused_sync_ints(T));
  w.perm_scratch = c.take<char>(permute_scratch_bytes(T, E));
  w.y_perm = c.take<uint16_t>(rows * H);
  return w;
}

// Routing, dispatch maps and permutation of the quantised layers (no bf16 x_perm).
int quant_fwd_route(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int H,
                    int E, int k, const QuantFwdWs& w, int32_t* idx, float* gates,
                    cudaStream_t stream) {
  int st;
  if (route_fused_ok(T, H, E, k, 1)) {  // small batches: routing and maps in one kernel
    return launch_route_fused(x, H, w_router, bias, T, H, E, k, 1, w.logits, idx, gates, w.tie,
                              w.counts, w.offsets, w.row_token, w.slot_row, w.sync, stream);
  }
  st = router_logits(x, H, w_router, T, H, E, 1, w.logits, stream);
  if (st) return st;
  st = launch_topk(w.logits, bias, T, E, k, idx, gates, w.tie, stream);
  if (st) return st;
  return launch_permute(idx, x, H, T, H, E, k, w.counts, w.offsets, w.row_token, w.slot_row,
                        nullptr, w.perm_scratch, stream);
}

bool nvfp4_weights_ok(const uint8_t* codes, const uint8_t* scales, const float* g) {
  return codes && scales && g && aligned16(codes) && aligned16(scales);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_set_profile_events(const cudaEvent_t* events, int n) {
  if (n == 0) {
    g_profile.on = false;
    return MOE_OK;
  }
  if (n != 4 || !events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return MOE_ERR_INVALID_ARG;
    g_profile.ev[i] = events[i];
  }
  g_profile.on = true;
  return MOE_OK;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or alignment";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    default: return "unknown status";
  }
}

int moe_get_device_status(cudaStream_t stream, int* status_out) {
  if (!status_out) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(cudaStreamSynchronize(stream));
  int* p = status_word();
  if (!p) return MOE_ERR_CUDA;
  int v = 0;
  MOE_CUDA(cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost));
  const int zero = 0;
  MOE_CUDA(cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice));
  *status_out = v;
  return MOE_OK;
}

size_t moe_route_workspace_size(int T, int D, int E, int k) {
  (void)D;
  (void)k;
  if (T < 0 || E < 1) return 0;
  Carver c(nullptr, 0);
  c.take<float>(static_cast<size_t>(T) * E);
  c.take<int>(route_fused_sync_ints(T));
  return c.used + 256;
}

int moe_route(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int D, int E,
              int k, int32_t* topk_idx, float* gates, uint8_t* tie_flag, void* workspace,
              size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(T, D, E, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !bias || !topk_idx || !gates) return MOE_ERR_INVALID_ARG;
  if (D % 8 || !aligned16(x) || !aligned16(w_router)) return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  float* logits = c.take<float>(static_cast<size_t>(T) * E);
  int* sync = c.take<int>(route_fused_sync_ints(T));
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  if (route_fused_ok(T, D, E, k, 1))  // small batches: logits and top-k in one kernel
    return launch_route_fused(x, D, w_router, bias, T, D, E, k, 1, logits, topk_idx, gates,
                              tie_flag, nullptr, nullptr, nullptr, nullptr, sync, stream);
  int st = router_logits(x, D, w_router, T, D, E, 1, logits, stream);
  if (st) return st;
  return launch_topk(logits, bias, T, E, k, topk_idx, gates, tie_flag, stream);
}

size_t moe_route_dispatch_workspace_size(int T, int D, int E, int k) {
  if (!dims_ok(T, D, E, k)) return 0;
  Carver c(nullptr, 0);
  c.take<float>(static_cast<size_t>(T) * E);
  c.take<int>(route_fused_sync_ints(T));
  c.take<char>(permute_scratch_bytes(T, E));
  return c.used + 256;
}

int moe_route_dispatch(const uint16_t* x, const uint16_t* w_router, const float* bias, int T,
                       int D, int E, int k, int32_t* topk_idx, float* gates, uint8_t* tie_flag,
                       int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* slot_row,
                       uint16_t* x_perm, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
  if (!dims_ok(T, D, E, k)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T == 0) {
    MOE_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream));
    MOE_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), stream));
    return MOE_OK;
  }
  if (!x || !w_router || !bias || !topk_idx || !gates || !row_token || !slot_row || !x_perm)
    return MOE_ERR_INVALID_ARG;
  if (D % 8 || !aligned16(x) || !aligned16(w_router) || !aligned16(x_perm))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  float* logits = c.take<float>(static_cast<size_t>(T) * E);
  int* sync = c.take<int>(route_fused_sync_ints(T));
  void* scratch = c.take<char>(permute_scratch_bytes(T, E));
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  if (route_fused_ok(T, D, E, k, 1)) {
    // small batches: logits, top-k and the dispatch maps in one kernel, then the row copy
    const int st = launch_route_fused(x, D, w_router, bias, T, D, E, k, 1, logits, topk_idx,
                                      gates, tie_flag, counts, offsets, row_token, slot_row,
                                      sync, stream);
    if (st) return st;
    return launch_gather_rows(row_token, x, D, T, T * k, D, x_perm, stream);
  }
  int st = router_logits(x, D, w_router, T, D, E, 1, logits, stream);
  if (st) return st;
  st = launch_topk(logits, bias, T, E, k, topk_idx, gates, tie_flag, stream);
  if (st) return st;
  return launch_permute(topk_idx, x, D, T, D, E, k, counts, offsets, row_token, slot_row, x_perm,
                        scratch, stream);
}

size_t moe_permute_workspace_size(int T, int E, int k) {
  (void)k;
  if (T < 0 || E < 1) return 0;
  Carver c(nullptr, 0);
  c.take<char>(permute_scratch_bytes(T, E));
  return c.used + 256;
}

int moe_permute(const int32_t* topk_idx, const uint16_t* x, int T, int H, int E, int k,
                int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* slot_row,
                uint16_t* x_perm, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(T, H, E, k)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !x || !row_token || !slot_row || !x_perm))
    return MOE_ERR_INVALID_ARG;
  if (H % 8 || !aligned16(x) || !aligned16(x_perm)) return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  void* scratch = c.take<char>(permute_scratch_bytes(T, E));
  if (T > 0 && !c.ok()) return MOE_ERR_WORKSPACE;
  if (T == 0)
    return launch_permute(topk_idx, x, H, T, H, E, k, counts, offsets, row_token, slot_row,
                          x_perm, scratch, stream);
  const WsGuard guard(c, stream);
  return launch_permute(topk_idx, x, H, T, H, E, k, counts, offsets, row_token, slot_row, x_perm,
                        scratch, stream);
}

size_t moe_grouped_ffn_workspace_size(int rows, int H, int F, int E) {
  (void)H;
  (void)E;
  if (rows < 0 || F < 0) return 0;
  Carver c(nullptr, 0);
  c.take<uint16_t>(static_cast<size_t>(rows) * F);
  return c.used + 256;
}

int moe_grouped_ffn(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_up,
                    const uint16_t* w_down, int rows, int H, int F, int E, uint16_t* y_perm,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (rows < 0 || H <= 0 || F <= 0 || E < 1 || E > 1024) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x_perm || !offsets || !w_up || !w_down || !y_perm) return MOE_ERR_INVALID_ARG;
  if (H % 64 || F % 64 || !aligned16(x_perm) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(y_perm))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  uint16_t* h = c.take<uint16_t>(static_cast<size_t>(rows) * F);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  return ffn(x_perm, offsets, w_up, w_down, rows, H, F, E, h, y_perm, stream);
}

int moe_combine(const uint16_t* y_perm, int rows, const int32_t* slot_row, const float* gates,
                int T, int H, int k, uint16_t* y, cudaStream_t stream) {
  if (T < 0 || rows < 0 || H <= 0 || k < 1 || k > 32) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y_perm || !slot_row || !gates || !y) return MOE_ERR_INVALID_ARG;
  if (H % 8 || !aligned16(y_perm) || !aligned16(y)) return MOE_ERR_UNSUPPORTED;
  return launch_combine(y_perm, rows, slot_row, gates, T, H, k, y, stream);
}

int moe_linear(const uint16_t* x, const uint16_t* w, int T, int K, int N, uint16_t* y,
               cudaStream_t stream) {
  if (T < 0 || K <= 0 || N <= 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w || !y) return MOE_ERR_INVALID_ARG;
  if (K % 64 || N % 64 || !aligned16(x) || !aligned16(w) || !aligned16(y))
    return MOE_ERR_UNSUPPORTED;
  GroupedGemm g{};
  g.act = x;
  g.act_ld = K;
  g.rows = T;
  g.w = w;
  g.E = 1;
  g.N = N;
  g.K = K;
  g.out = y;
  g.ldo = N;
  g.epi = EPI_BF16;
  return launch_grouped_gemm(g, stream);
}

size_t moe_forward_workspace_size(int T, int H, int E, int k, int F) {
  if (!dims_ok(T, H, E, k) || F <= 0) return 0;
  Carver c(nullptr, 0);
  carve_layer(c, T, H, E, k, F);
  return c.used + 256;
}

int moe_forward(const uint16_t* x, const uint16_t* w_router, const float* bias,
                const uint16_t* w_up, const uint16_t* w_down, int T, int H, int E, int k, int F,
                uint16_t* y, int32_t* topk_idx_out, float* gates_out, void* workspace,
                size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(T, H, E, k) || F <= 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !bias || !w_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
  if (H % 64 || F % 64 || !aligned16(x) || !aligned16(w_router) || !aligned16(w_up) ||
      !aligned16(w_down) || !aligned16(y))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const LayerWs w = carve_layer(c, T, H, E, k, F);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  return layer(x, H, x, H, H, 1, w_router, bias, w_up, w_down, T, H, E, k, F, y, topk_idx_out,
               gates_out, w, stream);
}

int moe_forward_gathered(const uint16_t* x, const uint16_t* w_router, const float* bias,
                         const uint16_t* w_up, const uint16_t* w_down, int T, int H, int E, int k,
                         int F, uint16_t* y, int32_t* topk_idx_out, float* gates_out,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(T, H, E, k) || F <= 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !bias || !w_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
  if (H % 64 || F % 64 || !aligned16(x) || !aligned16(w_router) || !aligned16(w_up) ||
      !aligned16(w_down) || !aligned16(y))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const LayerWs w = carve_layer(c, T, H, E, k, F);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  return layer(x, H, x, H, H, 1, w_router, bias, w_up, w_down, T, H, E, k, F, y, topk_idx_out,
               gates_out, w, stream, nullptr, true);
}

size_t moe_forward_fused_combine_workspace_size(int T, int H, int E, int k, int F) {
  if (!dims_ok(T, H, E, k) || F <= 0) return 0;
  Carver c(nullptr, 0);
  carve_layer(c, T, H, E, k, F, true);
  return c.used + 256;
}

int moe_forward_fused_combine(const uint16_t* x, const uint16_t* w_router, const float* bias,
                              const uint16_t* w_up, const uint16_t* w_down, int T, int H, int E,
                              int k, int F, uint16_t* y, int32_t* topk_idx_out,
                              float* gates_out, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
  if (!dims_ok(T, H, E, k) || F <= 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !bias || !w_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
  if (H % 64 || F % 64 || !aligned16(x) || !aligned16(w_router) || !aligned16(w_up) ||
      !aligned16(w_down) || !aligned16(y))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const LayerWs w = carve_layer(c, T, H, E, k, F, true);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  return layer(x, H, x, H, H, 1, w_router, bias, w_up, w_down, T, H, E, k, F, y, topk_idx_out,
               gates_out, w, stream);
}

size_t latent_moe_workspace_size(int T, int H, int L, int Ep, int kp, int F,
                                 int router_on_latent) {
  if (!dims_ok(T, L, Ep, kp) || H <= 0 || F <= 0) return 0;
  Carver c(nullptr, 0);
  c.take<uint16_t>(static_cast<size_t>(T) * L * (router_on_latent ? 3 : 1));  // x_lat planes
  c.take<uint16_t>(static_cast<size_t>(T) * L);                               // y_lat
  carve_layer(c, T, L, Ep, kp, F);
  return c.used + 256;
}

int latent_moe(const uint16_t* x, const uint16_t* w_in, const uint16_t* w_out,
               const uint16_t* w_router, const float* bias, int router_on_latent,
               const uint16_t* w_up, const uint16_t* w_down, int T, int H, int L, int Ep, int kp,
               int F, uint16_t* y, int32_t* topk_idx_out, float* gates_out, void* workspace,
               size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(T, L, Ep, kp) || H <= 0 || F <= 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_in || !w_out || !w_router || !bias || !w_up || !w_down || !y)
    return MOE_ERR_INVALID_ARG;
  if (H % 64 || L % 64 || F % 64 || !aligned16(x) || !aligned16(w_in) || !aligned16(w_out) ||
      !aligned16(w_router) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(y))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const int lat_ld = router_on_latent ? 3 * L : L;
  uint16_t* x_lat = c.take<uint16_t>(static_cast<size_t>(T) * lat_ld);
  uint16_t* y_lat = c.take<uint16_t>(static_cast<size_t>(T) * L);
  const LayerWs w = carve_layer(c, T, L, Ep, kp, F);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);

  // x_lat = x . w_in^T  (H -> L). With routing on the latent vector, the epilogue writes
  // x_lat as three bf16 planes hi | mid | lo (sum within about 2^-24 of the fp32 value):
  // the experts read hi, the router reads all three.
  GroupedGemm g{};
  g.act = x;
  g.act_ld = H;
  g.rows = T;
  g.w = w_in;
  g.E = 1;
  g.N = L;
  g.K = H;
  g.out = x_lat;
  g.ldo = lat_ld;
  g.lo_offset = L;
  g.epi = router_on_latent ? EPI_SPLIT_BF16 : EPI_BF16;
  g.precise = router_on_latent;  // x_lat decides the routing: keep it near fp32 accuracy
  int st = launch_grouped_gemm(g, stream);
  if (st) return st;

  if (router_on_latent)
    st = layer(x_lat, lat_ld, x_lat, lat_ld, L, 3, w_router, bias, w_up, w_down, T, L, Ep, kp, F,
               y_lat, topk_idx_out, gates_out, w, stream);
  else
    st = layer(x_lat, lat_ld, x, H, H, 1, w_router, bias, w_up, w_down, T, L, Ep, kp, F, y_lat,
               topk_idx_out, gates_out, w, stream);
  if (st) return st;

  // y = y_lat . w_out^T  (L -> H), applied once after the combine.
  GroupedGemm o{};
  o.act = y_lat;
  o.act_ld = L;
  o.rows = T;
  o.w = w_out;
  o.E = 1;
  o.N = H;
  o.K = L;
  o.out = y;
  o.ldo = H;
  o.epi = EPI_BF16;
  return launch_grouped_gemm(o, stream);
}

size_t moe_nvfp4_codes_bytes(int G, int N, int K) {
  if (G < 1 || N < 1 || K < 64 || K % 64) return 0;
  return static_cast<size_t>(G) * N * (K / 2);
}

size_t moe_nvfp4_scales_bytes(int G, int N, int K) {
  if (G < 1 || N < 1 || K < 64 || K % 64) return 0;
  return static_cast<size_t>(G) * nvfp4_sf_bytes(N, K);
}

int moe_quantize_nvfp4_weights(const uint16_t* w, int G, int N, int K, uint8_t* codes,
                               uint8_t* scales, float* global_scale, cudaStream_t stream) {
  if (G < 1 || G > 1024 || N < 1 || K < 64) return MOE_ERR_INVALID_ARG;
  if (!w || !codes || !scales || !global_scale) return MOE_ERR_INVALID_ARG;
  if (K % 64 || !aligned16(w) || !aligned16(codes) || !aligned16(scales))
    return MOE_ERR_UNSUPPORTED;
  // global_scale first accumulates each matrix's amax (as fp32 bits), then holds amax / 2688.
  MOE_CUDA(cudaMemsetAsync(global_scale, 0, sizeof(float) * G, stream));
  uint32_t* amax = reinterpret_cast<uint32_t*>(global_scale);
  int st = launch_amax_bf16(w, static_cast<long long>(N) * K, G, amax, stream);
  if (st) return st;
  st = launch_quant_weights(w, G, N, K, amax, codes, scales, stream);
  if (st) return st;
  return launch_finalize_gscale(global_scale, G, stream);
}

int moe_quantize_nvfp4_weights_2d(const uint16_t* w, int G, int N, int K, uint8_t* codes,
                                  uint8_t* scales, float* global_scale, cudaStream_t stream) {
  if (G < 1 || G > 1024 || N < 1 || K < 64) return MOE_ERR_INVALID_ARG;
  if (!w || !codes || !scales || !global_scale) return MOE_ERR_INVALID_ARG;
  if (K % 64 || !aligned16(w) || !aligned16(codes) || !aligned16(scales))
    return MOE_ERR_UNSUPPORTED;
  MOE_CUDA(cudaMemsetAsync(global_scale, 0, sizeof(float) * G, stream));
  uint32_t* amax = reinterpret_cast<uint32_t*>(global_scale);
  int st = launch_amax_bf16(w, static_cast<long long>(N) * K, G, amax, stream);
  if (st) return st;
  st = launch_quant_weights_2d(w, G, N, K, amax, codes, scales, stream);
  if (st) return st;
  return launch_finalize_gscale(global_scale, G, stream);
}

size_t moe_grouped_ffn_nvfp4_workspace_size(int rows, int H, int F, int E) {
  if (rows < 0 || H <= 0 || F <= 0 || E < 1 || E > 1024) return 0;
  Carver c(nullptr, 0);
  carve_fp4(c, rows, H, F, E);
  return c.used + 256;
}

int moe_grouped_ffn_nvfp4(const uint16_t* x_perm, const int32_t* offsets,
                          const uint8_t* up_codes, const uint8_t* up_scales,
                          const float* up_gscale, const uint8_t* down_codes,
                          const uint8_t* down_scales, const float* down_gscale, int rows, int H,
                          int F, int E, uint16_t* y_perm, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  if (rows < 0 || H <= 0 || F <= 0 || E < 1 || E > 1024) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(rows) + 127LL * E + 127 > 0x7fffffffLL) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x_perm || !offsets || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!nvfp4_weights_ok(up_codes, up_scales, up_gscale) ||
      !nvfp4_weights_ok(down_codes, down_scales, down_gscale))
    return MOE_ERR_INVALID_ARG;
  if (H % 64 || F % 64 || !aligned16(x_perm) || !aligned16(y_perm)) return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const Fp4Ws w = carve_fp4(c, rows, H, F, E);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  return ffn_nvfp4(x_perm, H, rows, nullptr, offsets, {up_codes, up_scales, up_gscale},
                   {down_codes, down_scales, down_gscale}, rows, H, F, E, y_perm, w, stream);
}

size_t moe_forward_nvfp4_workspace_size(int T, int H, int E, int k, int F) {
  if (!dims_ok(T, H, E, k) || F <= 0) return 0;
  Carver c(nullptr, 0);
  carve_quant_fwd(c, T, H, E, k);
  carve_fp4(c, T * k, H, F, E);
  return c.used + 256;
}

int moe_forward_nvfp4(const uint16_t* x, const uint16_t* w_router, const float* bias,
                      const uint8_t* up_codes, const uint8_t* up_scales, const float* up_gscale,
                      const uint8_t* down_codes, const uint8_t* down_scales,
                      const float* down_gscale, int T, int H, int E, int k, int F, uint16_t* y,
                      int32_t* topk_idx_out, float* gates_out, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(T, H, E, k) || F <= 0) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * k + 127LL * E + 127 > 0x7fffffffLL) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !bias || !y) return MOE_ERR_INVALID_ARG;
  if (!nvfp4_weights_ok(up_codes, up_scales, up_gscale) ||
      !nvfp4_weights_ok(down_codes, down_scales, down_gscale))
    return MOE_ERR_INVALID_ARG;
  if (H % 64 || F % 64 || !aligned16(x) || !aligned16(w_router) || !aligned16(y))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const int rows = T * k;
  const QuantFwdWs f = carve_quant_fwd(c, T, H, E, k);
  const Fp4Ws w = carve_fp4(c, rows, H, F, E);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  int32_t* idx = topk_idx_out ? topk_idx_out : f.idx;
  float* gates = gates_out ? gates_out : f.gates;
  // routing and dispatch stay in bf16/fp32; the expert FFNs run in NVFP4
  int st = quant_fwd_route(x, w_router, bias, T, H, E, k, f, idx, gates, stream);
  if (st) return st;
  const TokenSlots slots{idx, f.slot_row, T, k};
  st = ffn_nvfp4(x, H, T, &slots, f.offsets, {up_codes, up_scales, up_gscale},
                 {down_codes, down_scales, down_gscale}, rows, H, F, E, f.y_perm, w, stream);
  if (st) return st;
  return launch_combine(f.y_perm, rows, f.slot_row, gates, T, H, k, y, stream);
}

size_t moe_fp8_codes_bytes(int G, int N, int K) {
  if (G < 1 || N < 1 || K < 1) return 0;
  return static_cast<size_t>(G) * N * static_cast<size_t>(fp8_act_pitch(K));
}

int moe_quantize_fp8_weights(const uint16_t* w, int G, int N, int K, uint8_t* codes,
                             float* scale, cudaStream_t stream) {
  if (G < 1 || N < 1 || K < 16) return MOE_ERR_INVALID_ARG;
  if (!w || !codes || !scale) return MOE_ERR_INVALID_ARG;
  if (K % 16 || !aligned16(w) || !aligned16(codes)) return MOE_ERR_UNSUPPORTED;
  // scale first accumulates each matrix's amax (as fp32 bits), then holds amax / 448.
  MOE_CUDA(cudaMemsetAsync(scale, 0, sizeof(float) * G, stream));
  uint32_t* amax = reinterpret_cast<uint32_t*>(scale);
  int st = launch_amax_bf16(w, static_cast<long long>(N) * K, G, amax, stream);
  if (st) return st;
  st = launch_quant_fp8(w, K, nullptr, static_cast<long long>(G) * N, K, N, amax, codes,
                        fp8_act_pitch(K), stream);
  if (st) return st;
  return launch_finalize_fp8_scale(scale, G, stream);
}

size_t moe_grouped_ffn_fp8_workspace_size(int rows, int H, int F, int E) {
  (void)E;
  if (rows < 0 || H <= 0 || F <= 0) return 0;
  Carver c(nullptr, 0);
  carve_fp8(c, rows, H, F);
  return c.used + 256;
}

int moe_grouped_ffn_fp8(const uint16_t* x_perm, const int32_t* offsets, const uint8_t* up_codes,
                        const float* up_scale, const uint8_t* down_codes, const float* down_scale,
                        int rows, int H, int F, int E, uint16_t* y_perm, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  if (rows < 0 || H <= 0 || F <= 0 || E < 1 || E > 1024) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x_perm || !offsets || !up_codes || !up_scale || !down_codes || !down_scale || !y_perm)
    return MOE_ERR_INVALID_ARG;
  if (H % 64 || F % 64 || !aligned16(x_perm) || !aligned16(y_perm) || !aligned16(up_codes) ||
      !aligned16(down_codes))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const Fp8Ws w = carve_fp8(c, rows, H, F);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  return ffn_fp8(x_perm, H, rows, nullptr, offsets, up_codes, up_scale, down_codes, down_scale,
                 rows, H, F, E, y_perm, w, stream);
}

size_t moe_forward_fp8_workspace_size(int T, int H, int E, int k, int F) {
  if (!dims_ok(T, H, E, k) || F <= 0) return 0;
  Carver c(nullptr, 0);
  carve_quant_fwd(c, T, H, E, k);
  carve_fp8(c, T * k, H, F);
  return c.used + 256;
}

int moe_forward_fp8(const uint16_t* x, const uint16_t* w_router, const float* bias,
                    const uint8_t* up_codes, const float* up_scale, const uint8_t* down_codes,
                    const float* down_scale, int T, int H, int E, int k, int F, uint16_t* y,
                    int32_t* topk_idx_out, float* gates_out, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(T, H, E, k) || F <= 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !bias || !y || !up_codes || !up_scale || !down_codes || !down_scale)
    return MOE_ERR_INVALID_ARG;
  if (H % 64 || F % 64 || !aligned16(x) || !aligned16(w_router) || !aligned16(y) ||
      !aligned16(up_codes) || !aligned16(down_codes))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const int rows = T * k;
  const QuantFwdWs f = carve_quant_fwd(c, T, H, E, k);
  const Fp8Ws w = carve_fp8(c, rows, H, F);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  int32_t* idx = topk_idx_out ? topk_idx_out : f.idx;
  float* gates = gates_out ? gates_out : f.gates;
  int st = quant_fwd_route(x, w_router, bias, T, H, E, k, f, idx, gates, stream);
  if (st) return st;
  // the tokens are quantised straight from x in expert order (row_token), no bf16 x_perm
  const TokenSlots slots{idx, f.slot_row, T, k};
  st = ffn_fp8(x, H, T, &slots, f.offsets, up_codes, up_scale, down_codes, down_scale, rows, H,
               F, E, f.y_perm, w, stream);
  if (st) return st;
  return launch_combine(f.y_perm, rows, f.slot_row, gates, T, H, k, y, stream);
}

size_t moe_forward_shared_workspace_size(int T, int H, int E, int k, int F, int Fs) {
  if (!dims_ok(T, H, E, k) || F <= 0 || Fs <= 0) return 0;
  Carver c(nullptr, 0);
  carve_layer(c, T, H, E, k, F);
  c.take<uint16_t>(static_cast<size_t>(T) * Fs);  // h of the shared expert
  c.take<uint16_t>(static_cast<size_t>(T) * H);   // its output
  return c.used + 256;
}

int moe_forward_shared(const uint16_t* x, const uint16_t* w_router, const float* bias,
                       const uint16_t* w_up, const uint16_t* w_down, const uint16_t* w_up_shared,
                       const uint16_t* w_down_shared, int T, int H, int E, int k, int F, int Fs,
                       uint16_t* y, int32_t* topk_idx_out, float* gates_out, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(T, H, E, k) || F <= 0 || Fs <= 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !bias || !w_up || !w_down || !w_up_shared || !w_down_shared || !y)
    return MOE_ERR_INVALID_ARG;
  if (H % 64 || F % 64 || Fs % 64 || !aligned16(x) || !aligned16(w_router) || !aligned16(w_up) ||
      !aligned16(w_down) || !aligned16(w_up_shared) || !aligned16(w_down_shared) || !aligned16(y))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const LayerWs w = carve_layer(c, T, H, E, k, F);
  uint16_t* h_s = c.take<uint16_t>(static_cast<size_t>(T) * Fs);
  uint16_t* y_s = c.take<uint16_t>(static_cast<size_t>(T) * H);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);
  int st = shared_expert(x, H, T, H, Fs, w_up_shared, w_down_shared, h_s, y_s, stream);
  if (st) return st;
  // the combine adds the shared expert's output into its fp32 sum
  return layer(x, H, x, H, H, 1, w_router, bias, w_up, w_down, T, H, E, k, F, y, topk_idx_out,
               gates_out, w, stream, y_s);
}

size_t latent_moe_shared_workspace_size(int T, int H, int L, int Ep, int kp, int F, int Fs,
                                        int router_on_latent) {
  if (!dims_ok(T, L, Ep, kp) || H <= 0 || F <= 0 || Fs <= 0) return 0;
  Carver c(nullptr, 0);
  c.take<uint16_t>(static_cast<size_t>(T) * L * (router_on_latent ? 3 : 1));  // x_lat planes
  c.take<uint16_t>(static_cast<size_t>(T) * L);                               // y_lat
  carve_layer(c, T, L, Ep, kp, F);
  c.take<uint16_t>(static_cast<size_t>(T) * Fs);  // h of the shared expert
  c.take<uint16_t>(static_cast<size_t>(T) * H);   // its output
  return c.used + 256;
}

int latent_moe_shared(const uint16_t* x, const uint16_t* w_in, const uint16_t* w_out,
                      const uint16_t* w_router, const float* bias, int router_on_latent,
                      const uint16_t* w_up, const uint16_t* w_down, const uint16_t* w_up_shared,
                      const uint16_t* w_down_shared, int T, int H, int L, int Ep, int kp, int F,
                      int Fs, uint16_t* y, int32_t* topk_idx_out, float* gates_out,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(T, L, Ep, kp) || H <= 0 || F <= 0 || Fs <= 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_in || !w_out || !w_router || !bias || !w_up || !w_down || !w_up_shared ||
      !w_down_shared || !y)
    return MOE_ERR_INVALID_ARG;
  if (H % 64 || L % 64 || F % 64 || Fs % 64 || !aligned16(x) || !aligned16(w_in) ||
      !aligned16(w_out) || !aligned16(w_router) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(w_up_shared) || !aligned16(w_down_shared) || !aligned16(y))
    return MOE_ERR_UNSUPPORTED;
  Carver c(workspace, workspace_bytes);
  const int lat_ld = router_on_latent ? 3 * L : L;
  uint16_t* x_lat = c.take<uint16_t>(static_cast<size_t>(T) * lat_ld);
  uint16_t* y_lat = c.take<uint16_t>(static_cast<size_t>(T) * L);
  const LayerWs w = carve_layer(c, T, L, Ep, kp, F);
  uint16_t* h_s = c.take<uint16_t>(static_cast<size_t>(T) * Fs);
  uint16_t* y_s = c.take<uint16_t>(static_cast<size_t>(T) * H);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  const WsGuard guard(c, stream);

  // shared expert in H on the token itself (Nemotron 3 notes §2.2)
  int st = shared_expert(x, H, T, H, Fs, w_up_shared, w_down_shared, h_s, y_s, stream);
  if (st) return st;
  GroupedGemm g{};
  g.act = x;
  g.act_ld = H;
  g.rows = T;
  g.w = w_in;
  g.E = 1;
  g.N = L;
  g.K = H;
  g.out = x_lat;
  g.ldo = lat_ld;
  g.lo_offset = L;
  g.epi = router_on_latent ? EPI_SPLIT_BF16 : EPI_BF16;
  g.precise = router_on_latent;
  st = launch_grouped_gemm(g, stream);
  if (st) return st;
  if (router_on_latent)
    st = layer(x_lat, lat_ld, x_lat, lat_ld, L, 3, w_router, bias, w_up, w_down, T, L, Ep, kp, F,
               y_lat, topk_idx_out, gates_out, w, stream);
  else
    st = layer(x_lat, lat_ld, x, H, H, 1, w_router, bias, w_up, w_down, T, L, Ep, kp, F, y_lat,
               topk_idx_out, gates_out, w, stream);
  if (st) return st;
  // y = y_lat . w_out^T + shared expert output (added in the GEMM's fp32 epilogue)
  GroupedGemm o{};
  o.act = y_lat;
  o.act_ld = L;
  o.rows = T;
  o.w = w_out;
  o.E = 1;
  o.N = H;
  o.K = L;
  o.out = y;
  o.ldo = H;
  o.epi = EPI_ADD_BF16;
  o.add = y_s;
  o.ld_add = H;
  return launch_grouped_gemm(o, stream);
}

// ------------------------------------------------------------ quantised activation views ----

int moe_grouped_ffn_nvfp4_view(int rows, int H, int F, int E, const void* workspace,
                               size_t workspace_bytes, moe_quant_view* out) {
  if (rows < 0 || H <= 0 || F <= 0 || E < 1 || E > 1024 || !out) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(rows) + 127LL * E + 127 > 0x7fffffffLL) return MOE_ERR_INVALID_ARG;
  Carver c(const_cast<void*>(workspace), workspace_bytes);
  const Fp4Ws w = carve_fp4(c, rows, H, F, E);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  *out = moe_quant_view{};
  out->padded_offsets = w.poff;
  out->amax = w.amax;
  out->x_codes = w.xq;
  out->x_scales = w.xsf;
  out->h = w.h;
  out->h_codes = w.hq;
  out->h_scales = w.hsf;
  out->buffer_rows = w.P;
  out->x_codes_ld = fp4_act_pitch(H);
  out->h_codes_ld = fp4_act_pitch(F);
  return MOE_OK;
}

int moe_forward_nvfp4_view(int T, int H, int E, int k, int F, const void* workspace,
                           size_t workspace_bytes, moe_quant_view* out) {
  if (!dims_ok(T, H, E, k) || F <= 0 || !out) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * k + 127LL * E + 127 > 0x7fffffffLL) return MOE_ERR_INVALID_ARG;
  Carver c(const_cast<void*>(workspace), workspace_bytes);
  const QuantFwdWs f = carve_quant_fwd(c, T, H, E, k);
  const Fp4Ws w = carve_fp4(c, T * k, H, F, E);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  *out = moe_quant_view{};
  out->offsets = f.offsets;
  out->row_token = f.row_token;
  out->padded_offsets = w.poff;
  out->amax = w.amax;
  out->x_codes = w.xq;
  out->x_scales = w.xsf;
  out->h = w.h;
  out->h_codes = w.hq;
  out->h_scales = w.hsf;
  out->buffer_rows = w.P;
  out->x_codes_ld = fp4_act_pitch(H);
  out->h_codes_ld = fp4_act_pitch(F);
  return MOE_OK;
}

int moe_grouped_ffn_fp8_view(int rows, int H, int F, int E, const void* workspace,
                             size_t workspace_bytes, moe_quant_view* out) {
  if (rows < 0 || H <= 0 || F <= 0 || E < 1 || E > 1024 || !out) return MOE_ERR_INVALID_ARG;
  Carver c(const_cast<void*>(workspace), workspace_bytes);
  const Fp8Ws w = carve_fp8(c, rows, H, F);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  *out = moe_quant_view{};
  out->amax = w.amax;
  out->x_codes = w.xq;
  out->h = w.h;
  out->h_codes = w.hq;
  out->buffer_rows = rows;
  out->x_codes_ld = fp8_act_pitch(H);
  out->h_codes_ld = fp8_act_pitch(F);
  return MOE_OK;
}

int moe_forward_fp8_view(int T, int H, int E, int k, int F, const void* workspace,
                         size_t workspace_bytes, moe_quant_view* out) {
  if (!dims_ok(T, H, E, k) || F <= 0 || !out) return MOE_ERR_INVALID_ARG;
  Carver c(const_cast<void*>(workspace), workspace_bytes);
  const QuantFwdWs f = carve_quant_fwd(c, T, H, E, k);
  const Fp8Ws w = carve_fp8(c, T * k, H, F);
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  *out = moe_quant_view{};
  out->offsets = f.offsets;
  out->row_token = f.row_token;
  out->amax = w.amax;
  out->x_codes = w.xq;
  out->h = w.h;
  out->h_codes = w.hq;
  out->buffer_rows = T * k;
  out->x_codes_ld = fp8_act_pitch(H);
  out->h_codes_ld = fp8_act_pitch(F);
  return MOE_OK;
}

}  // extern "C"
