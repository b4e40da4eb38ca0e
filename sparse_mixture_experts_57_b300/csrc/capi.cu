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

namespace {

bool dims_ok(int T, int D, int E, int k) {
  if (T < 0 || D <= 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return false;
  if (static_cast<long long>(T) * k > 0x7fffffffLL) return false;
  return true;
}

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
  void* perm_scratch;
  uint16_t* x_perm;
  uint16_t* h;
  uint16_t* y_perm;
};

LayerWs carve_layer(Carver& c, int T, int D, int E, int k, int F) {
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
  w.perm_scratch = c.take<char>(permute_scratch_bytes(T, E));
  w.x_perm = c.take<uint16_t>(rows * D);
  w.h = c.take<uint16_t>(rows * F);
  w.y_perm = c.take<uint16_t>(rows * D);
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

int ffn(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_up,
        const uint16_t* w_down, int rows, int D, int F, int E, uint16_t* h, uint16_t* y_perm,
        cudaStream_t s) {
  GroupedGemm up{};
  up.act = x_perm;
  up.act_ld = D;
  up.rows = rows;
  up.w = w_up;
  up.E = E;
  up.N = F;
  up.K = D;
  up.offsets = offsets;
  up.out = h;
  up.ldo = F;
  up.epi = EPI_SQRELU_BF16;
  int st = launch_grouped_gemm(up, s);
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
  return launch_grouped_gemm(dn, s);
}

// route -> permute -> grouped FFN -> combine for rows of width D read from x (row stride ldx).
// Routing reads xr (row stride ldr, width Dr, in `parts` bf16 planes).
int layer(const uint16_t* x, int64_t ldx, const uint16_t* xr, int64_t ldr, int Dr, int parts,
          const uint16_t* w_router, const float* bias, const uint16_t* w_up,
          const uint16_t* w_down, int T, int D, int E, int k, int F, uint16_t* y,
          int32_t* idx_out, float* gates_out, const LayerWs& w, cudaStream_t s) {
  int st = router_logits(xr, ldr, w_router, T, Dr, E, parts, w.logits, s);
  if (st) return st;
  int32_t* idx = idx_out ? idx_out : w.idx;
  float* gates = gates_out ? gates_out : w.gates;
  st = launch_topk(w.logits, bias, T, E, k, idx, gates, w.tie, s);
  if (st) return st;
  st = launch_permute(idx, x, ldx, T, D, E, k, w.counts, w.offsets, w.row_token, w.slot_row,
                      w.x_perm, w.perm_scratch, s);
  if (st) return st;
  const int rows = T * k;
  st = ffn(w.x_perm, w.offsets, w_up, w_down, rows, D, F, E, w.h, w.y_perm, s);
  if (st) return st;
  return launch_combine(w.y_perm, rows, w.slot_row, gates, T, D, k, y, s);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

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
  return align_up(static_cast<size_t>(T) * E * sizeof(float), 256) + 256;
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
  if (!c.ok()) return MOE_ERR_WORKSPACE;
  int st = router_logits(x, D, w_router, T, D, E, 1, logits, stream);
  if (st) return st;
  return launch_topk(logits, bias, T, E, k, topk_idx, gates, tie_flag, stream);
}

size_t moe_permute_workspace_size(int T, int E, int k) {
  (void)k;
  if (T < 0 || E < 1) return 0;
  return permute_scratch_bytes(T, E) + 256;
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
  return launch_permute(topk_idx, x, H, T, H, E, k, counts, offsets, row_token, slot_row, x_perm,
                        scratch, stream);
}

size_t moe_grouped_ffn_workspace_size(int rows, int H, int F, int E) {
  (void)H;
  (void)E;
  if (rows < 0 || F < 0) return 0;
  return align_up(static_cast<size_t>(rows) * F * 2, 256) + 256;
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

}  // extern "C"
