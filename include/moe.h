/*
 * moe.h: C ABI of the B300 (sm_103a) routed Mixture-of-Experts layer forward pass.
 *
 * The layer follows "NVIDIA Nemotron 3: Efficient and Open Intelligence" (papercache
 * notes) §2.1-§2.2 with Fig. 3b, the two "Nemotron 3 Nano" summaries (papers.lianghsun.dev
 * §2.2, aux-loss-free balancing; shd-paper.top 技术框架, route -> experts -> weighted
 * combination), and the news piece "NVIDIA AI发布了Nemotron 3" (混合Mamba Transformer
 * MoE架构: a learned router picks 6 of 128 routable experts).
 *
 * Conventions shared by every call:
 *  - bfloat16 tensors are passed as uint16_t bit patterns. All matrices are row-major.
 *    Weights are stored [out_features, in_features], so the contraction axis is the
 *    contiguous one.
 *  - All tensor pointers are DEVICE pointers, owned by the caller. No call allocates or
 *    frees device memory. Scratch comes from a caller-provided workspace of at least the
 *    size that the matching *_workspace_size() reports. Outputs and workspace must not
 *    overlap the inputs.
 *  - Calls are asynchronous on `stream`. A call returns after its kernels are enqueued.
 *    The return code covers argument checks and launch errors only.
 *  - Faults found on the device (an expert index out of range, a duplicate expert in one
 *    token's list, a pipeline wait that ran out of time) set a device status word. Read
 *    it with moe_get_device_status().
 *  - Sizes: H, F and the latent size L must be multiples of 64. Tensor pointers must be
 *    16-byte aligned. 1 <= E <= 1024 and 1 <= k <= min(E, 32). T*k must fit in int32.
 *    T == 0 is allowed and does nothing.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, negative or inconsistent size, bad index   */
  MOE_ERR_UNSUPPORTED = 2,  /* size or alignment outside what the kernels handle        */
  MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than *_workspace_size()     */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed              */
  MOE_ERR_TIMEOUT = 5       /* a device pipeline wait exceeded its limit (device word)  */
};

/* Text for a status code. The string is static and must not be freed. */
const char* moe_status_string(int status);

/* Synchronise `stream`, then read and clear the current device's status word. The word
 * holds MOE_OK or the first error that a kernel recorded since it was last cleared. */
int moe_get_device_status(cudaStream_t stream, int* status_out);

/* moe_set_profile_events: a profiling hook with no counterpart in the pages. With n = 4, the
 * layer and grouped-FFN calls made afterwards on the calling thread record events[0] and
 * events[1] on their stream just before and just after the expert up-projection GEMM, and
 * events[2] and events[3] around the down-projection GEMM (for the NVFP4 and FP8 calls the
 * activation quantisers fall outside both brackets). The events belong to the caller
 * (cudaEventCreate); the library keeps the four handles and only records them. n = 0 turns
 * the hook off. MOE_ERR_INVALID_ARG for another n or a NULL handle. A failed record makes
 * the layer call return MOE_ERR_CUDA. */
int moe_set_profile_events(const cudaEvent_t* events, int n);

/* moe_route_cluster_refusal: a diagnostic with no counterpart in the pages. Small batches
 * (T <= 256, E <= 128) route with one thread-block cluster per group of 8 tokens (up to 16
 * CTAs, a non-portable cluster size). If the device refuses that launch configuration, the
 * library falls back to its cluster-free routing kernel (same results) for the rest of the
 * process; this returns the cudaError_t of the refusal, or 0 if none happened. */
int moe_route_cluster_refusal(void);

/* ---------------------------------------------------------------------------------------
 * moe_route: the learned router with aux-loss-free, bias-corrected top-k.
 *   z[t,e] = sum_d x[t,d] * w_router[e,d]   (bf16 inputs, fp32 accumulation)
 *   s = sigmoid(z); u = s + bias[e] (bias for SELECTION only)
 *   topk_idx[t,:] = the k experts with the largest u, in descending u; the lower expert
 *                   index wins exact ties
 *   gates[t,j]    = s[t,topk_idx[t,j]] / sum_j' s[t,topk_idx[t,j']]
 *   tie_flag[t]   = 1 when u_(k) - u_(k+1) < 1e-5 (a near-tie diagnostic; may be NULL)
 * Pages: Nemotron 3 Nano summary §2.2 (aux-loss-free balancing), news piece (learned
 * router, top-6 of 128). The sigmoid/bias/renormalisation details are this library's
 * reading of the aux-loss-free scheme.
 * Layout: x [T,D] bf16, w_router [E,D] bf16, bias [E] fp32; topk_idx [T,k] int32,
 * gates [T,k] fp32, tie_flag [T] uint8. Workspace: moe_route_workspace_size(); its contents
 * at entry do not matter, and two calls in flight at once must not share it.
 * ------------------------------------------------------------------------------------- */
size_t moe_route_workspace_size(int T, int D, int E, int k);
int moe_route(const uint16_t* x, const uint16_t* w_router, const float* bias,
              int T, int D, int E, int k,
              int32_t* topk_idx, float* gates, uint8_t* tie_flag,
              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * moe_permute: dispatch of the routed (token, slot) pairs into expert-contiguous order.
 *   counts[e]        rows routed to expert e
 *   offsets[e]       exclusive prefix sum of counts; offsets[E] = T*k
 *   row_token[r]     token of permuted row r (rows of one expert in ascending token order)
 *   slot_row[t*k+j]  permuted row that holds (token t, slot j); -1 if topk_idx was invalid
 *   x_perm[r,:]      = x[row_token[r],:]
 * Pages: shd-paper.top summary 技术框架 (the selected experts process their tokens in
 * parallel); NVIDIA Nemotron 3 notes §2.2 (token dispatch to experts).
 * Layout: topk_idx [T,k] int32, x [T,H] bf16; outputs as above, x_perm [T*k,H] bf16.
 * Invalid or duplicate expert indices are reported on the device status word
 * (MOE_ERR_INVALID_ARG). Workspace: moe_permute_workspace_size().
 * ------------------------------------------------------------------------------------- */
size_t moe_permute_workspace_size(int T, int E, int k);
int moe_permute(const int32_t* topk_idx, const uint16_t* x, int T, int H, int E, int k,
                int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* slot_row,
                uint16_t* x_perm, void* workspace, size_t workspace_bytes,
                cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * moe_route_dispatch: moe_route followed by moe_permute, with the same outputs as the two
 * calls (topk_idx, gates, tie_flag; counts, offsets, row_token, slot_row, x_perm; D plays
 * the role of H). For small batches (T <= 256, E <= 256, D <= 6144) the router logits, the
 * top-k and the dispatch maps run as one kernel, followed by the row copy.
 * Workspace: moe_route_dispatch_workspace_size(). Its contents at entry do not matter (the
 * fused kernel's CTAs signal one another through flag words tagged with a per-launch
 * value). Two calls in flight at once must not share a workspace.
 * ------------------------------------------------------------------------------------- */
size_t moe_route_dispatch_workspace_size(int T, int D, int E, int k);
int moe_route_dispatch(const uint16_t* x, const uint16_t* w_router, const float* bias, int T,
                       int D, int E, int k, int32_t* topk_idx, float* gates, uint8_t* tie_flag,
                       int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* slot_row,
                       uint16_t* x_perm, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * moe_permute_noalloc: moe_permute for callers that cannot provide a workspace.
 * The pages have no counterpart to this call; it exists for integration only. Some callers
 * cannot hand the library device memory for scratch, for example a host runtime whose own
 * pool owns all device memory and forbids other allocations, or a serving loop that runs
 * on a fixed memory plan. This call takes the same inputs and outputs as moe_permute and
 * gives the same results. Its scratch lives in a fixed array inside the library's device
 * image: moe_permute_noalloc_max_scratch_bytes() bytes (2 MiB), held on every GPU that
 * loads the library until the process exits. No call allocates or frees memory.
 * Limits and rules:
 *  - ceil(T/32) * E * 8 bytes (rounded up to 256-byte slices) must fit in that array, e.g.
 *    T = 16384 with E = 512; larger problems return MOE_ERR_UNSUPPORTED (use moe_permute).
 *  - All calls on one device share the array. Calls that overlap on the GPU (unordered
 *    streams) race on it; calls ordered on one stream do not. Nothing in the array has to
 *    start at zero: each call overwrites every word it reads.
 *  - The first call on each device looks up the array's device address with that device
 *    current. Make that first call before any stream capture.
 *  - The library caches that address, and the device status word's, per device for the
 *    life of the process. Do not keep using the library on a device after
 *    cudaDeviceReset() there: the cached addresses belong to the destroyed context.
 * Arguments, layouts and device-side error reporting are those of moe_permute.
 * ------------------------------------------------------------------------------------- */
size_t moe_permute_noalloc_max_scratch_bytes(void);
int moe_permute_noalloc(const int32_t* topk_idx, const uint16_t* x, int T, int H, int E, int k,
                        int32_t* counts, int32_t* offsets, int32_t* row_token,
                        int32_t* slot_row, uint16_t* x_perm, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * moe_grouped_ffn: every expert's FFN on its segment of permuted rows.
 *   for rows r in [offsets[e], offsets[e+1]):
 *     h[r,:]      = max(0, x_perm[r,:] . w_up[e]^T)^2     (squared ReLU, stored bf16)
 *     y_perm[r,:] = h[r,:] . w_down[e]^T
 * Pages: NVIDIA Nemotron 3 notes §2.2 (each expert matrix is H x C; decode-sized batches
 * are bound by reading expert weights). The activation is this library's reading.
 * Layout: x_perm [rows,H] bf16, offsets [E+1] int32 (device), w_up [E,F,H] bf16,
 * w_down [E,H,F] bf16, y_perm [rows,H] bf16. fp32 accumulation on tcgen05 tensor cores.
 * Workspace: moe_grouped_ffn_workspace_size() (holds h).
 * ------------------------------------------------------------------------------------- */
size_t moe_grouped_ffn_workspace_size(int rows, int H, int F, int E);
int moe_grouped_ffn(const uint16_t* x_perm, const int32_t* offsets,
                    const uint16_t* w_up, const uint16_t* w_down,
                    int rows, int H, int F, int E, uint16_t* y_perm,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * moe_combine: the combination layer, the gate-weighted sum back in token order.
 *   y[t,:] = sum_j gates[t*k+j] * y_perm[slot_row[t*k+j],:]   (fp32 accumulation)
 * Pages: shd-paper.top summary 技术框架 (weighted combination of the experts' outputs).
 * Rows with slot_row outside [0, rows) are skipped.
 * Layout: y_perm [rows,H] bf16, slot_row [T*k] int32, gates [T*k] fp32, y [T,H] bf16.
 * ------------------------------------------------------------------------------------- */
int moe_combine(const uint16_t* y_perm, int rows, const int32_t* slot_row,
                const float* gates, int T, int H, int k, uint16_t* y,
                cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * moe_linear: y[t,:] = x[t,:] . w^T (bf16 in, fp32 accumulation, bf16 out).
 * Used for the LatentMoE projections, which the pages keep in BF16 (NVIDIA Nemotron 3
 * notes §2.4). Layout: x [T,K] bf16, w [N,K] bf16, y [T,N] bf16. K and N multiples of 64.
 * ------------------------------------------------------------------------------------- */
int moe_linear(const uint16_t* x, const uint16_t* w, int T, int K, int N, uint16_t* y,
               cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * moe_forward: route + permute + grouped FFN + combine, the whole routed MoE layer.
 * Layout: x [T,H], w_router [E,H], bias [E] fp32, w_up [E,F,H], w_down [E,H,F], y [T,H].
 * topk_idx_out [T,k] and gates_out [T,k] are optional copies of the routing (NULL to skip).
 * Workspace: moe_forward_workspace_size().
 * ------------------------------------------------------------------------------------- */
size_t moe_forward_workspace_size(int T, int H, int E, int k, int F);
int moe_forward(const uint16_t* x, const uint16_t* w_router, const float* bias,
                const uint16_t* w_up, const uint16_t* w_down,
                int T, int H, int E, int k, int F, uint16_t* y,
                int32_t* topk_idx_out, float* gates_out,
                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* moe_forward_gathered: moe_forward whose up-projection gathers the routed token rows
 * straight from x with TMA tile::gather4, so the permuted copy x_perm is never written.
 * With more than 48 rows per expert on average the rows sit on the MMA's M side and a
 * 128-row K-slice takes 32 gather4 copies; with fewer, the weights sit on M and a slice of
 * BN token rows takes BN / 4. Same results as moe_forward, bit for bit (the same operands in
 * the same order), same arguments and workspace (moe_forward_workspace_size()). On B300 both
 * forms are slower than reading a materialised x_perm, so moe_forward does not use them. */
int moe_forward_gathered(const uint16_t* x, const uint16_t* w_router, const float* bias,
                         const uint16_t* w_up, const uint16_t* w_down, int T, int H, int E, int k,
                         int F, uint16_t* y, int32_t* topk_idx_out, float* gates_out,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* moe_forward_fused_combine: moe_forward with the combine (shd-paper.top summary 技术框架,
 * the weighted combination of the chosen experts' outputs) fused into the down-projection's
 * epilogue. Each routed row's output, times its gate, is rounded once to a multiple of 2^-32
 * and added with 64-bit integer atomics to its token's accumulator [T,H] in the workspace;
 * integer addition does not depend on the order in which the tiles finish, so the result
 * is the same on every run. A last pass writes y = bf16(sum * 2^-32). y_perm is never
 * written. Differences from moe_forward: the expert outputs are not rounded to bf16 before
 * the combine (so y can differ from moe_forward's in the last bf16 place), and a term with
 * |gate * output| >= 2^26 (or NaN) is not added and sets MOE_ERR_UNSUPPORTED on the device
 * status word. Same arguments as moe_forward; workspace from
 * moe_forward_fused_combine_workspace_size() (moe_forward's minus y_perm, plus 8*T*H bytes). */
size_t moe_forward_fused_combine_workspace_size(int T, int H, int E, int k, int F);
/* moe_fixed_to_bf16: the last pass of moe_forward_fused_combine on its own, for testing:
 * out[i] = the bf16 nearest to q[i] * 2^-32 (ties to even; bit patterns as uint16), rounded
 * once from the integer. on_device = 0: host pointers, computed on the calling thread (no
 * CUDA call). on_device = 1: device pointers, the library's conversion kernel on `stream`
 * (n a multiple of 8, both pointers 16-byte aligned, else MOE_ERR_UNSUPPORTED). The pages
 * have no counterpart: the fixed-point sum is this library's way of making the fused
 * combine independent of the order of its additions. MOE_ERR_INVALID_ARG for n < 0 or a
 * NULL pointer with n > 0. */
int moe_fixed_to_bf16(const int64_t* q, long long n, uint16_t* out, int on_device,
                      cudaStream_t stream);
int moe_forward_fused_combine(const uint16_t* x, const uint16_t* w_router, const float* bias,
                              const uint16_t* w_up, const uint16_t* w_down, int T, int H, int E,
                              int k, int F, uint16_t* y, int32_t* topk_idx_out,
                              float* gates_out, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * latent_moe: the LatentMoE layer (NVIDIA Nemotron 3 notes §2.2, Fig. 3b).
 *   x_lat = x . w_in^T                      (H -> L, bf16 projection)
 *   route x_lat (router_on_latent = 1, w_router [Ep,L]) or x (router_on_latent = 0,
 *   w_router [Ep,H]) to Ep experts with kp active, run the experts in L
 *   (w_up [Ep,F,L], w_down [Ep,L,F]), combine in L,
 *   y = y_lat . w_out^T                     (L -> H, bf16 projection, applied once)
 * The pages scale experts as Ep = E*H/L and kp = k*H/L; both are free parameters here.
 * For routing on the latent vector, x_lat is kept to about fp32 accuracy (three bf16
 * planes hi + mid + lo), so the selection does not depend on the bf16 rounding of x_lat.
 * The experts read the bf16 x_lat (hi).
 * topk_idx_out / gates_out [T,kp] are optional. Workspace: latent_moe_workspace_size().
 * ------------------------------------------------------------------------------------- */
size_t latent_moe_workspace_size(int T, int H, int L, int Ep, int kp, int F,
                                 int router_on_latent);
int latent_moe(const uint16_t* x, const uint16_t* w_in, const uint16_t* w_out,
               const uint16_t* w_router, const float* bias, int router_on_latent,
               const uint16_t* w_up, const uint16_t* w_down,
               int T, int H, int L, int Ep, int kp, int F, uint16_t* y,
               int32_t* topk_idx_out, float* gates_out,
               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * Shared expert (NVIDIA Nemotron 3 notes §2.2: the shared-expert computation, like the routing
 * gate, stays in the hidden size H). This library's reading: an FFN of the routed experts'
 * form applied to every token with weight 1 and added to the routed output,
 *   y = routed(x) + max(0, x . w_up_shared^T)^2 . w_down_shared^T,
 * with w_up_shared [Fs, H] and w_down_shared [H, Fs] bf16. Several shared experts are one
 * FFN whose intermediate size Fs is their total (stack their matrices along Fs).
 * moe_forward_shared: moe_forward plus the shared expert (its output joins the combine's fp32
 *   sum). latent_moe_shared: latent_moe plus the shared expert on x in H (added in the
 *   epilogue of the L -> H projection). Fs must be a multiple of 64. Workspace: the
 *   matching *_workspace_size().
 * ------------------------------------------------------------------------------------- */
size_t moe_forward_shared_workspace_size(int T, int H, int E, int k, int F, int Fs);
int moe_forward_shared(const uint16_t* x, const uint16_t* w_router, const float* bias,
                       const uint16_t* w_up, const uint16_t* w_down, const uint16_t* w_up_shared,
                       const uint16_t* w_down_shared, int T, int H, int E, int k, int F, int Fs,
                       uint16_t* y, int32_t* topk_idx_out, float* gates_out, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream);
size_t latent_moe_shared_workspace_size(int T, int H, int L, int Ep, int kp, int F, int Fs,
                                        int router_on_latent);
int latent_moe_shared(const uint16_t* x, const uint16_t* w_in, const uint16_t* w_out,
                      const uint16_t* w_router, const float* bias, int router_on_latent,
                      const uint16_t* w_up, const uint16_t* w_down, const uint16_t* w_up_shared,
                      const uint16_t* w_down_shared, int T, int H, int L, int Ep, int kp, int F,
                      int Fs, uint16_t* y, int32_t* topk_idx_out, float* gates_out,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * NVFP4 expert FFNs (NVIDIA Nemotron 3 notes §2.4: E2M1 elements in 16-element micro-blocks,
 * an E4M3 scale per block, a second-level FP32 scale per tensor). For a tensor with
 * amax A the global scale is g = A / (6 * 448); each block of 16 consecutive K elements gets
 * sb = E4M3(amax(block) / (6 g)) and each element q = E2M1(v / (sb g)), both rounded to
 * nearest with ties to even and saturating; the value is q * sb * g. Decisions are taken in
 * fp32 with correctly rounded division. Routing, dispatch and the combine stay bf16/fp32.
 *
 * NVFP4 matrix formats used by these calls, for G matrices of [N, K] (K a multiple of 64):
 *  - codes  [G, N, K/2] bytes: E2M1 codes (sign in bit 3), element 2i in the low nibble.
 *  - scales E4M3 bytes in the tensor cores' tile order: per matrix, one 512-byte atom per
 *    (128-row block rb, 64-element K step j), atoms ordered by rb then j
 *    (ceil(N/128) * K/64 atoms per matrix); inside an atom, row 128 rb + 32 r1 + r0 and
 *    K block kb (0..3 within the step) sit at byte r0 * 16 + r1 * 4 + kb. Rows past N in
 *    the last block hold zero scales.
 *  - global_scale [G] fp32: g of each matrix (each expert matrix is its own tensor).
 * ------------------------------------------------------------------------------------- */
size_t moe_nvfp4_codes_bytes(int G, int N, int K);
size_t moe_nvfp4_scales_bytes(int G, int N, int K);

/* moe_quantize_nvfp4_weights: quantise G bf16 weight matrices w [G, N, K] into the formats
 * above (a set-up step, done once per weight set). K must be a multiple of 64; w, codes
 * and scales 16-byte aligned; G <= 1024. (The NVFP4 FFN calls need N a multiple of 64.) No workspace: global_scale doubles as the
 * per-matrix amax accumulator. Asynchronous on `stream`. */
int moe_quantize_nvfp4_weights(const uint16_t* w, int G, int N, int K, uint8_t* codes,
                               uint8_t* scales, float* global_scale, cudaStream_t stream);

/* moe_grouped_ffn_nvfp4: moe_grouped_ffn with NVFP4 operands.
 *   x_perm rows are quantised in the call with one global scale over the whole x_perm
 *   tensor; h = max(0, x_q . w_up_q[e]^T)^2 (fp32 accumulation, then bf16) is quantised with
 *   one global scale over all of h; y_perm = h_q . w_down_q[e]^T, stored bf16.
 * Each expert's row segment is padded internally to whole 128-row tiles (at most 127 extra
 * rows per expert). Layout: x_perm [rows, H] bf16, offsets [E+1] int32, y_perm [rows, H] bf16;
 * up weights quantised from [E, F, H], down weights from [E, H, F].
 * Workspace: moe_grouped_ffn_nvfp4_workspace_size(). */
/* moe_quantize_nvfp4_weights_2d: as moe_quantize_nvfp4_weights, with 2-D weight blocks
 * (NVIDIA Nemotron 3 notes §2.4: 2-D block scaling for weights): one block scale per 16 rows
 * x 16 K elements, sb = E4M3(amax(16x16 block) / (6 g)); the last row block may have fewer
 * rows. The output formats are the 1-D ones (each row holds its block's scale), so the NVFP4
 * FFN calls take these weights unchanged. */
int moe_quantize_nvfp4_weights_2d(const uint16_t* w, int G, int N, int K, uint8_t* codes,
                                  uint8_t* scales, float* global_scale, cudaStream_t stream);

size_t moe_grouped_ffn_nvfp4_workspace_size(int rows, int H, int F, int E);
int moe_grouped_ffn_nvfp4(const uint16_t* x_perm, const int32_t* offsets,
                          const uint8_t* up_codes, const uint8_t* up_scales,
                          const float* up_gscale, const uint8_t* down_codes,
                          const uint8_t* down_scales, const float* down_gscale, int rows, int H,
                          int F, int E, uint16_t* y_perm, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/* moe_forward_nvfp4: the routed MoE layer with NVFP4 expert FFNs: moe_route (bf16 inputs,
 * fp32 scores), the permutation, moe_grouped_ffn_nvfp4 on the routed tokens (the tokens are
 * quantised straight from x, with the global scale of the whole x, and gathered into the
 * padded expert order in one pass; no bf16 x_perm is written) and moe_combine.
 * Layout: as moe_forward, with the NVFP4 weights above. Workspace:
 * moe_forward_nvfp4_workspace_size(). */
size_t moe_forward_nvfp4_workspace_size(int T, int H, int E, int k, int F);
int moe_forward_nvfp4(const uint16_t* x, const uint16_t* w_router, const float* bias,
                      const uint8_t* up_codes, const uint8_t* up_scales, const float* up_gscale,
                      const uint8_t* down_codes, const uint8_t* down_scales,
                      const float* down_gscale, int T, int H, int E, int k, int F, uint16_t* y,
                      int32_t* topk_idx_out, float* gates_out, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * FP8 expert FFNs (Nemotron 3 Nano summary §4: FP8 post-training quantisation; BF16 and FP8
 * weights are released). The pages give no scaling granularity; this library reads it as
 * per-tensor E4M3: s = amax / 448 and q = E4M3(v / s), nearest with ties to even and
 * saturating at +-448; the value is q * s. Tensors: each expert matrix, the whole routed
 * token tensor, and the whole h. Decisions in fp32 with correctly rounded division. The GEMMs
 * run on tcgen05 kind::f8f6f4 (E4M3 x E4M3, fp32 accumulation); routing, dispatch and the
 * combine stay bf16/fp32.
 * Formats: codes [G, N, ldk] bytes (E4M3; row n of matrix g at (g N + n) ldk, K codes then
 * padding), ldk = K rounded up to a multiple of 128 so that every 128-byte K-slice the GEMMs
 * load starts on a 128-byte boundary; scale [G] fp32 (s of each matrix).
 * ------------------------------------------------------------------------------------- */

/* moe_quantize_fp8_weights: quantise G bf16 matrices w [G, N, K] (K a multiple of 16; w and
 * codes 16-byte aligned) into codes ([G, N, ldk], moe_fp8_codes_bytes() bytes; the padding
 * bytes of each row are left as they are) and per-matrix scales. A set-up step; no
 * workspace (scale doubles as the amax accumulator). Asynchronous on `stream`. */
size_t moe_fp8_codes_bytes(int G, int N, int K);
int moe_quantize_fp8_weights(const uint16_t* w, int G, int N, int K, uint8_t* codes,
                             float* scale, cudaStream_t stream);

/* moe_grouped_ffn_fp8: moe_grouped_ffn with E4M3 operands. x_perm rows are quantised in the
 * call with the scale of the whole x_perm; h = max(0, x_q . w_up_q[e]^T)^2 is stored bf16 and
 * quantised with the scale of the whole h; y_perm = h_q . w_down_q[e]^T (bf16).
 * Layout: x_perm [rows, H] bf16, offsets [E+1], up codes from [E, F, H], down codes from
 * [E, H, F], y_perm [rows, H] bf16. Workspace: moe_grouped_ffn_fp8_workspace_size(). */
size_t moe_grouped_ffn_fp8_workspace_size(int rows, int H, int F, int E);
int moe_grouped_ffn_fp8(const uint16_t* x_perm, const int32_t* offsets, const uint8_t* up_codes,
                        const float* up_scale, const uint8_t* down_codes, const float* down_scale,
                        int rows, int H, int F, int E, uint16_t* y_perm, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/* moe_forward_fp8: the routed MoE layer with FP8 expert FFNs: moe_route, the permutation,
 * the FP8 FFNs on the routed tokens (quantised straight from x in expert order, with the
 * scale of the whole x) and moe_combine. Layout as moe_forward. Workspace:
 * moe_forward_fp8_workspace_size(). */
size_t moe_forward_fp8_workspace_size(int T, int H, int E, int k, int F);
int moe_forward_fp8(const uint16_t* x, const uint16_t* w_router, const float* bias,
                    const uint8_t* up_codes, const float* up_scale, const uint8_t* down_codes,
                    const float* down_scale, int T, int H, int E, int k, int F, uint16_t* y,
                    int32_t* topk_idx_out, float* gates_out, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * Quantised activation views. The NVFP4 and FP8 FFN calls quantise their activations into
 * the caller's workspace: the routed tokens entering the up-projection (x) and the hidden
 * activations h entering the down-projection, each with one global scale over the whole
 * tensor (NVIDIA Nemotron 3 notes §2.4 for NVFP4; per-tensor E4M3 for FP8). These calls
 * return where those buffers sit inside a workspace laid out by the named call with the
 * same sizes, so a caller can read what the call actually fed the tensor cores.
 * They make no CUDA call and touch no memory: they only compute addresses. The contents
 * are those of the last call that used the workspace, valid once that call has completed
 * on its stream and until the workspace is used again.
 *
 * Fields (NULL where the call has no such buffer):
 *  - offsets [E+1], row_token [rows]: the forward calls' dispatch maps (moe_permute's).
 *  - padded_offsets [E+1] (NVFP4): start row of each expert's segment in the padded
 *    buffers; every segment is rounded up to whole 128-row tiles, rows past the expert's
 *    count are padding (zero codes and zero scales).
 *  - amax [2]: fp32 bit patterns of amax(|x|) over the whole token tensor (all of x for the
 *    forward calls, all of x_perm for the grouped-FFN calls) and of amax(|h|) over the
 *    stored bf16 h. Global scales: g = amax / (6 * 448) (NVFP4), s = amax / 448 (FP8).
 *  - x_codes, x_scales: the quantised routed tokens. NVFP4: codes [buffer_rows, H/2] and
 *    scale atoms of [buffer_rows, H] (the formats above), padded segment order; row
 *    padded_offsets[e] + r holds permuted row offsets[e] + r. FP8: E4M3 bytes
 *    [buffer_rows, H] in permuted row order; x_scales is NULL. Code rows are x_codes_ld
 *    bytes apart: H/2 (NVFP4) or H (FP8) rounded up to a multiple of 128, so every
 *    128-byte K-slice the GEMM loads starts on a 128-byte boundary.
 *  - h [buffer_rows, F] bf16: max(0, x_q . w_up_q[e]^T)^2 as stored by the up-projection
 *    (NVFP4: padded order, padding rows zero).
 *  - h_codes, h_scales: h quantised for the down-projection, as x_codes / x_scales, code
 *    rows h_codes_ld bytes apart (F/2 or F rounded up to a multiple of 128).
 *  - buffer_rows: rows of the x / h buffers (NVFP4: the padded-row bound
 *    rows + 127 E rounded up to 128; FP8: rows).
 * Return: MOE_ERR_INVALID_ARG for sizes the named call rejects or a NULL out;
 * MOE_ERR_WORKSPACE if the workspace is smaller than the call needs.
 * ------------------------------------------------------------------------------------- */
typedef struct moe_quant_view {
  const int32_t* offsets;
  const int32_t* row_token;
  const int32_t* padded_offsets;
  const uint32_t* amax;
  const uint8_t* x_codes;
  const uint8_t* x_scales;
  const uint16_t* h;
  const uint8_t* h_codes;
  const uint8_t* h_scales;
  long long buffer_rows;
  long long x_codes_ld;
  long long h_codes_ld;
} moe_quant_view;

int moe_grouped_ffn_nvfp4_view(int rows, int H, int F, int E, const void* workspace,
                               size_t workspace_bytes, moe_quant_view* out);
int moe_forward_nvfp4_view(int T, int H, int E, int k, int F, const void* workspace,
                           size_t workspace_bytes, moe_quant_view* out);
int moe_grouped_ffn_fp8_view(int rows, int H, int F, int E, const void* workspace,
                             size_t workspace_bytes, moe_quant_view* out);
int moe_forward_fp8_view(int T, int H, int E, int k, int F, const void* workspace,
                         size_t workspace_bytes, moe_quant_view* out);

/* ---------------------------------------------------------------------------------------
 * moe_selftest_wait_timeout: runs the failure path that every tensor-core pipeline kernel of
 * this library shares, on purpose, so a caller can check it on a live GPU. Every wait of a
 * kernel pipeline is bounded; when one gives up the kernel records MOE_ERR_TIMEOUT on the
 * device status word, stops its other roles through a per-CTA abort flag, waits (bounded)
 * for its copies in flight to land, releases its tensor memory and returns, so the GPU
 * stays usable. Each of the `blocks` CTAs here allocates tensor memory, issues one 4 KB bulk
 * copy from `src`, and then waits on barriers that nothing arrives on: the producer role
 * with a limit of limit_us microseconds, the other roles with the pipelines' normal limit,
 * which only the abort flag can cut short.
 *   src     device, 16-byte aligned, at least 4096 bytes (read only);
 *   report  device int [blocks * 8], written per CTA: [0] 1 if the producer's wait gave
 *           up, [1] and [2] 1 if the MMA and epilogue roles left through the abort flag,
 *           [3] 1 if the copy in flight landed before the CTA exited, [4] microseconds from
 *           the first wait to the release of tensor memory; [5..7] unused.
 * By design the call leaves MOE_ERR_TIMEOUT on the device status word (read and clear it
 * with moe_get_device_status). Returns MOE_ERR_INVALID_ARG for a null pointer, limit_us
 * outside [1, 10^6] or blocks outside [1, 1024]; MOE_ERR_UNSUPPORTED for an unaligned src.
 * Asynchronous on `stream`.
 * ------------------------------------------------------------------------------------- */
int moe_selftest_wait_timeout(const void* src, int limit_us, int blocks, int* report,
                              cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * Debug build. The library also builds as libmoe_debug.so (compiled with MOE_DEBUG), with
 * the same entry points and results plus checks that the release build leaves out:
 *  - every workspace slice is followed by a 256-byte guard region (the *_workspace_size
 *    queries of that build include them); each call fills its guards before its first kernel
 *    and checks them after its last one, and a damaged guard (a kernel that wrote past its
 *    slice) is reported as MOE_ERR_WORKSPACE on the device status word;
 *  - device-side range checks of indices the library itself produced (row_token in the row
 *    copy, slot_row in the combine), reported as MOE_ERR_INVALID_ARG on the status word.
 * moe_debug_build() returns 1 in that build and 0 in the release build.
 * moe_debug_guard_selftest() checks the guard detector: it carves two slices of `workspace`
 * (at least 8 KiB, device), fills their guards, overwrites one guard byte with
 * cudaMemsetAsync and runs the check, which must leave MOE_ERR_WORKSPACE on the status word.
 * The release build returns MOE_ERR_UNSUPPORTED from it.
 * ------------------------------------------------------------------------------------- */
int moe_debug_build(void);
int moe_debug_guard_selftest(void* workspace, size_t workspace_bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
