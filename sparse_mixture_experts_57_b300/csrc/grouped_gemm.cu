// grouped_gemm.cu: persistent, warp-specialised grouped GEMM on tcgen05 tensor cores.
//
// This is the expert FFN contraction of the routed MoE layer ("NVIDIA Nemotron 3: Efficient
// and Open Intelligence" notes, §2.2: each expert is an H x C matrix pair). It is also used
// for the LatentMoE projections (§2.2, Fig. 3b) and for the router logits of large batches.
//
//   out[r, n] = epi( sum_k act[r, k] * w[e, n, k] )   for r in group e's row segment
//
// Design (one CTA per SM, 192 threads):
//   warp 0 lane 0  TMA producer: K-slices of the activation rows and of the expert's
//                  weight rows into a STAGES-deep shared-memory ring (128-byte swizzle).
//   warp 1 lane 0  MMA issuer: tcgen05.mma (M=128, N=BN, K=16) into a double-buffered
//                  fp32 accumulator in tensor memory; tcgen05.commit frees ring slots.
//   warps 2..5     epilogue: tcgen05.ld of the accumulator, activation, bf16/fp32 stores.
// The work list is flattened over (group, row tile, column tile), so a skewed expert load
// (one expert holding every token) spreads over all SMs.
// Two operand orders:
//   rows-as-M (prefill): M = 128 routed rows, N = BN output features.
//   weights-as-M (decode, few rows per expert): M = 128 weight rows (output features),
//   N = BN routed rows. Tensor cores then do no more than a few x the needed work, and
//   the kernel becomes a weight stream from HBM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "fixed.cuh"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128;  // MMA M
constexpr int BK = 64;   // K per pipeline stage: one 128-byte swizzle row of bf16
constexpr int UK = 16;   // K per tcgen05.mma for 16-bit inputs
constexpr int MAX_GROUPS = 1024;
constexpr int NUM_THREADS = 192;          // producer, MMA issuer, 4 epilogue warps
constexpr int NUM_THREADS_CHUNKED = 320;  // producer, MMA issuer, 8 epilogue warps
__host__ __device__ constexpr int kernel_threads(bool chunked) {
  return chunked ? NUM_THREADS_CHUNKED : NUM_THREADS;
}

struct KArgs {
  const int* offsets;
  int dense_rows;
  int E;
  int N;
  int K;
  int k_wrap;
  int rows_total;
  void* out;
  long long ldo;
  long long lo_offset;
  int epi;
  int kchunk;  // CHUNKED kernels: K-blocks (of 64) accumulated per TMEM partial sum
  int* status;
  const int* row_token;    // GATHER kernels: token of each routed row
  int src_rows;            // GATHER kernels: rows of the gathered activation tensor
  const uint16_t* add;     // EPI_ADD_BF16: bf16 addend, row stride ld_add
  long long ld_add;
  const uint32_t* a_amax;  // E4M3 kernels: activation amax (fp32 bits)
  const float* w_scale;    // E4M3 kernels: per-group weight scale
  uint32_t* out_amax;      // max of the stored (bf16) squared-ReLU outputs, or null
  const int32_t* comb_token;     // EPI_COMBINE_I64: token of each routed row,
  const int32_t* comb_slot_row;  // the permuted rows of each token's k slots,
  const float* comb_gates;       // and their gates
  int comb_k, comb_T;
};

template <int BN>
__host__ __device__ constexpr uint32_t tmem_cols() {
  uint32_t need = 2u * BN, c = 32;
  while (c < need) c <<= 1;
  return c;
}

template <int BN, int STAGES>
constexpr size_t smem_bytes() {
  return 1024 + size_t(STAGES) * (BM * BK * 2 + BN * BK * 2) + (2 * STAGES + 4) * 8 + 16 +
         3 * (MAX_GROUPS + 1) * 4 + BM * 4;
}

__device__ __forceinline__ void record(int* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ void decode_tile(int tile, int n_ct, const int* pref, int E, int& e,
                                            int& rt, int& ct) {
  const int rtg = tile / n_ct;
  ct = tile - rtg * n_ct;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid + 1] > rtg)
      hi = mid;
    else
      lo = mid + 1;
  }
  e = lo;
  rt = rtg - pref[lo];
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16 consecutive output columns of one row (rows-as-M epilogue).
__device__ __forceinline__ void store_row16(const KArgs& a, long long row, int col,
                                            const float* acc) {
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = acc[i];
  if (a.epi == EPI_F32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(a.out) + row * a.ldo + col);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    return;
  }
  if (a.epi == EPI_SQRELU_BF16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float t = fmaxf(v[i], 0.f);
      v[i] = t * t;
    }
  }
  if (a.epi == EPI_ADD_BF16) {
    const uint4* ap = reinterpret_cast<const uint4*>(a.add + row * a.ld_add + col);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = __ldg(ap + h);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * h + 2 * i] += __uint_as_float(w[i] << 16);
        v[8 * h + 2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
      }
    }
  }
  uint32_t hi[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) hi[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
  __nv_bfloat16* base = static_cast<__nv_bfloat16*>(a.out) + row * a.ldo + col;
  uint4* p = reinterpret_cast<uint4*>(base);
  p[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  p[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
  if (a.epi == EPI_SPLIT_BF16) {
    // v = hi + mid + lo to about 2^-24 relative: three bf16 planes lo_offset apart
    uint32_t mid[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float r[2], m2[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float x = v[2 * i + h];
        r[h] = x - __bfloat162float(__float2bfloat16_rn(x));
        m2[h] = r[h] - __bfloat162float(__float2bfloat16_rn(r[h]));
      }
      mid[i] = pack_bf16(r[0], r[1]);
      lo[i] = pack_bf16(m2[0], m2[1]);
    }
    uint4* q = reinterpret_cast<uint4*>(base + a.lo_offset);
    q[0] = make_uint4(mid[0], mid[1], mid[2], mid[3]);
    q[1] = make_uint4(mid[4], mid[5], mid[6], mid[7]);
    uint4* z = reinterpret_cast<uint4*>(base + 2 * a.lo_offset);
    z[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    z[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  }
}

// EPI_COMBINE_I64, rows-as-M: 16 consecutive columns of one row added to its token's sum.
__device__ __forceinline__ void combine_row16(const KArgs& a, int t, float g, int col,
                                              const float* v) {
  unsigned long long* p = static_cast<unsigned long long*>(a.out) + static_cast<long long>(t) * a.ldo + col;
#pragma unroll
  for (int i = 0; i < 16; ++i) fixed_add(p + i, g * v[i], a.status);
}

// One output element (weights-as-M epilogue: lanes hold consecutive features of a row).
__device__ __forceinline__ void store_one(const KArgs& a, long long row, int col, float v) {
  if (a.epi == EPI_F32) {
    static_cast<float*>(a.out)[row * a.ldo + col] = v;
    return;
  }
  if (a.epi == EPI_SQRELU_BF16) {
    const float t = fmaxf(v, 0.f);
    v = t * t;
  }
  if (a.epi == EPI_ADD_BF16) v += __uint_as_float(static_cast<uint32_t>(a.add[row * a.ld_add + col]) << 16);
  __nv_bfloat16* base = static_cast<__nv_bfloat16*>(a.out) + row * a.ldo + col;
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  *base = h;
  if (a.epi == EPI_SPLIT_BF16) {
    const float r = v - __bfloat162float(h);
    const __nv_bfloat16 m = __float2bfloat16_rn(r);
    base[a.lo_offset] = m;
    base[2 * a.lo_offset] = __float2bfloat16_rn(r - __bfloat162float(m));
  }
}

// CHUNKED (rows-as-M only): the accumulator restarts every kchunk K-blocks and the epilogue
// sums the partial tiles in fp32 registers. tcgen05's fp32 accumulation error grows about
// linearly with the number of accumulated products, so short chunks keep the result close
// to an fp32 dot product. Used for the GEMMs that feed the router's top-k decision.
// F8: E4M3 operands (kind::f8f6f4, K = 32 per MMA): a 128-byte K-slice holds 128 elements,
// the last slice may run past K (TMA fills zeros), and the epilogue applies the per-tensor
// scales (a_amax / 448) * w_scale[group].
// GATHER (rows-as-M, bf16): the activation rows of a tile are gathered from the token
// tensor by row_token with TMA gather4 (32 per K-slice), so the permuted copy of the tokens
// is never written. The whole producer warp loads a tile's 128 token ids into shared memory;
// lane 0 issues the copies. Rows past the group's end gather an out-of-range row (zeros).
template <int BN, int STAGES, bool SWAP, bool CHUNKED = false, bool F8 = false,
          bool GATHER = false>
__global__ void __launch_bounds__(kernel_threads(CHUNKED), 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tm_act,
                   const __grid_constant__ CUtensorMap tm_w, const KArgs a) {
  constexpr uint32_t A_BYTES = BM * BK * 2;
  constexpr uint32_t B_BYTES = BN * BK * 2;
  constexpr int BKE = F8 ? 2 * BK : BK;  // K elements per 128-byte slice
  constexpr int RT = SWAP ? BN : BM;  // routed rows per tile
  constexpr int CT = SWAP ? BM : BN;  // output features per tile
  constexpr uint32_t TMEM_COLS = tmem_cols<BN>();
  constexpr uint32_t ACC_STRIDE = TMEM_COLS / 2;
  constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN);
  static_assert(!(F8 && CHUNKED), "E4M3 kernels have no chunked variant");
  static_assert(!GATHER || (!CHUNKED && !F8), "gathered rows: bf16 only");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
  static_assert(!CHUNKED || (!SWAP && BN % 128 == 0),
                "chunked accumulation: rows-as-M, BN 128 or 256");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_pref = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_off = s_pref + (MAX_GROUPS + 1);
  int* s_cnt = s_off + (MAX_GROUPS + 1);
  int* s_tok = s_cnt + (MAX_GROUPS + 1);  // GATHER: token ids of the producer's current tile

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = a.E;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kernel_threads(CHUNKED) - 64);  // every epilogue thread
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_act);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  // On-chip set-up above overlaps the previous kernel; global memory is touched only after
  // it has completed.
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 2) {
    // Row segments of the groups and the exclusive prefix of their row-tile counts.
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int local = 0;
    bool bad = false;
    for (int e = e0; e < e1; ++e) {
      const int lo = a.offsets ? a.offsets[e] : 0;
      const int hi = a.offsets ? a.offsets[e + 1] : a.dense_rows;
      int cnt = hi - lo;
      if (lo < 0 || cnt < 0 || hi > a.rows_total) {
        bad = true;
        cnt = 0;
      }
      s_off[e] = lo;
      s_cnt[e] = cnt;
      local += (cnt + RT - 1) / RT;
    }
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e1; ++e) {
      s_pref[e] = run;
      run += (s_cnt[e] + RT - 1) / RT;
    }
    if (lane == 31) s_pref[E] = incl;
    if (__any_sync(0xffffffffu, bad) && lane == 0) record(a.status, MOE_ERR_INVALID_ARG);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int n_ct = (a.N + CT - 1) / CT;
  const int total = s_pref[E] * n_ct;
  const int KB = (a.K + BKE - 1) / BKE;

  if (warp == 0 && GATHER) {
    // ------------------------------------------------------- TMA producer (gathered rows)
    const uint64_t pol_w = SWAP ? policy_evict_first() : policy_evict_last();
    const uint64_t pol_a = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    long long armed = 0;
    bool ok = true;
    // token ids of a tile's rows (rows past the group's end: an out-of-range row, read as
    // zeros), one per lane and register; the next tile's ids load while lane 0 issues the
    // current tile's copies
    constexpr int TJ = (RT + 31) / 32;
    int tok[TJ];
    auto fetch_ids = [&](int tile) {
      if (tile >= total) return;
      int e, rt, ct;
      decode_tile(tile, n_ct, s_pref, E, e, rt, ct);
      const int rbeg = rt * RT;
      const int valid_rows = min(RT, s_cnt[e] - rbeg);
#pragma unroll
      for (int j = 0; j < TJ; ++j) {
        const int i = lane + 32 * j;
        tok[j] = i < valid_rows ? __ldg(a.row_token + s_off[e] + rbeg + i) : a.src_rows;
      }
    };
    fetch_ids(blockIdx.x);
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      int e, rt, ct;
      decode_tile(tile, n_ct, s_pref, E, e, rt, ct);
      const int col0 = ct * CT;
#pragma unroll
      for (int j = 0; j < TJ; ++j) {
        const int i = lane + 32 * j;
        if (i < RT) s_tok[i] = tok[j];
      }
      __syncwarp();
      fetch_ids(tile + static_cast<int>(gridDim.x));
      if (lane == 0) {
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES);
          ++armed;
          const int kc = kb * BKE;
          // the activation rows: the A operand (rows-as-M) or the B operand (weights-as-M)
          uint8_t* dst = SWAP ? sB + stage * B_BYTES : sA + stage * A_BYTES;
          if (SWAP) tma_load_3d(sA + stage * A_BYTES, &tm_w, &full[stage], kc, col0, e, pol_w);
#pragma unroll 4
          for (int g4 = 0; g4 < RT / 4; ++g4)
            tma_gather4(dst + g4 * 512, &tm_act, &full[stage], kc, s_tok[4 * g4],
                        s_tok[4 * g4 + 1], s_tok[4 * g4 + 2], s_tok[4 * g4 + 3], pol_a);
          if (!SWAP) tma_load_3d(sB + stage * B_BYTES, &tm_w, &full[stage], kc, col0, e, pol_w);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);  // s_tok is rewritten only after lane 0 is done
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      record(a.status, MOE_ERR_TIMEOUT);
    }
    if (lane == 0 && !drain_stages(full, STAGES, stage, phase, armed))
      record(a.status, MOE_ERR_TIMEOUT);
  } else if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer
      const uint64_t pol_w = SWAP ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_a = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long armed = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, rt, ct;
        decode_tile(tile, n_ct, s_pref, E, e, rt, ct);
        const int row0 = s_off[e] + rt * RT;
        const int col0 = ct * CT;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES);
          ++armed;
          const int kc = kb * BKE;
          const int kw = a.k_wrap ? (kc % a.k_wrap) : kc;
          if (!SWAP) {
            tma_load_2d(sA + stage * A_BYTES, &tm_act, &full[stage], kc, row0, pol_a);
            tma_load_3d(sB + stage * B_BYTES, &tm_w, &full[stage], kw, col0, e, pol_w);
          } else {
            tma_load_3d(sA + stage * A_BYTES, &tm_w, &full[stage], kw, col0, e, pol_w);
            tma_load_2d(sB + stage * B_BYTES, &tm_act, &full[stage], kc, row0, pol_a);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record(a.status, MOE_ERR_TIMEOUT);
      }
      if (!drain_stages(full, STAGES, stage, phase, armed)) record(a.status, MOE_ERR_TIMEOUT);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const int kc = CHUNKED ? a.kchunk : KB;
        uint32_t d_tmem = 0;
        for (int kb = 0; kb < KB; ++kb) {
          const int kin = CHUNKED ? (kb % kc) : kb;   // position inside the current chunk
          if (kin == 0) {
            if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d_tmem = tmem_base + acc * ACC_STRIDE;
          }
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_k_sw128(smem_u32(sA + stage * A_BYTES));
          const uint64_t bdesc = sdesc_k_sw128(smem_u32(sB + stage * B_BYTES));
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            if constexpr (F8)
              umma_e4m3(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, IDESC, (kin | kk) != 0);
            else
              umma_bf16(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, IDESC, (kin | kk) != 0);
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (kin == kc - 1 || kb == KB - 1) {
            umma_commit(&tfull[acc]);
            if (++acc == 2) {
              acc = 0;
              acc_phase ^= 1u;
            }
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        *abort_flag = 1;
        record(a.status, MOE_ERR_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int m = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    float vmax = 0.f;  // E4M3 squared-ReLU kernels: max of the stored outputs
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, rt, ct;
      decode_tile(tile, n_ct, s_pref, E, e, rt, ct);
      const int rbeg = rt * RT;
      const int valid_rows = min(RT, s_cnt[e] - rbeg);
      const long long row0 = static_cast<long long>(s_off[e]) + rbeg;
      const int col0 = ct * CT;
      if constexpr (CHUNKED) {
        // eight epilogue warps: two per TMEM lane quadrant, each summing half the columns
        constexpr int HB = BN / 2;
        const int hc0 = ((warp - 2) >> 2) * HB;  // this warp's first column in the tile
        const int ncols = min(BN, a.N - col0) - hc0;
        const int nchunks = (KB + a.kchunk - 1) / a.kchunk;
        float sum[HB];
#pragma unroll
        for (int i = 0; i < HB; ++i) sum[i] = 0.f;
        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
          if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tb =
              tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_STRIDE;
          // two loads in flight per wait. Columns past ncols (inside the accumulator) are
          // summed too and never stored.
#pragma unroll
          for (int jb = 0; jb < HB / 32; ++jb) {
            uint32_t r[2][16];
#pragma unroll
            for (int u = 0; u < 2; ++u) tmem_ld16(tb + hc0 + jb * 32 + u * 16, r[u]);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
              for (int i = 0; i < 16; ++i) sum[jb * 32 + u * 16 + i] += __uint_as_float(r[u][i]);
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        if (!ok) {
          *abort_flag = 1;
          record(a.status, MOE_ERR_TIMEOUT);
          break;
        }
        if (m < valid_rows) {
#pragma unroll
          for (int j = 0; j < HB / 16; ++j)
            if (j * 16 < ncols) store_row16(a, row0 + m, col0 + hc0 + j * 16, sum + j * 16);
        }
        continue;
      }
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) {
        *abort_flag = 1;
        record(a.status, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_STRIDE;
      float scale = 1.f;
      if constexpr (F8) scale = __fdiv_rn(__uint_as_float(*a.a_amax), kFp8Div) * a.w_scale[e];
      if (!SWAP) {
        const int ncols = min(BN, a.N - col0);
        int ctok = -1;  // EPI_COMBINE_I64: this row's token and gate
        float cgate = 0.f;
        if (a.epi == EPI_COMBINE_I64 && m < valid_rows)
          fixed_row_gate(a.comb_token, a.comb_slot_row, a.comb_gates, a.comb_k, a.comb_T,
                         row0 + m, a.status, ctok, cgate);
        for (int n0 = 0; n0 < ncols; n0 += 16) {
          uint32_t r[16];
          tmem_ld16(tb + n0, r);
          tmem_ld_wait();
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]) * scale;
          if (m < valid_rows) {
            if (F8 && a.out_amax) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float t = fmaxf(v[i], 0.f);
                vmax = fmaxf(vmax, t * t);
              }
            }
            if (a.epi == EPI_COMBINE_I64) {
              if (ctok >= 0) combine_row16(a, ctok, cgate, col0 + n0, v);
            } else {
              store_row16(a, row0 + m, col0 + n0, v);
            }
          }
        }
      } else {
        const int f = col0 + m;
        for (int n0 = 0; n0 < valid_rows; n0 += 16) {
          uint32_t r[16];
          tmem_ld16(tb + n0, r);
          tmem_ld_wait();
          if (a.epi == EPI_COMBINE_I64) {
            // lanes 0..15 look up rows n0..n0+15; each row's token and gate are then
            // broadcast, and the warp adds 32 consecutive features of that token's sum
            int ctok = -1;
            float cgate = 0.f;
            if (lane < 16 && n0 + lane < valid_rows)
              fixed_row_gate(a.comb_token, a.comb_slot_row, a.comb_gates, a.comb_k, a.comb_T,
                             row0 + n0 + lane, a.status, ctok, cgate);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int t = __shfl_sync(0xffffffffu, ctok, i);
              const float g = __shfl_sync(0xffffffffu, cgate, i);
              if (f < a.N && t >= 0)
                fixed_add(static_cast<unsigned long long*>(a.out) + static_cast<long long>(t) * a.ldo + f,
                          g * (__uint_as_float(r[i]) * scale), a.status);
            }
            continue;
          }
          if (f < a.N) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (n0 + i < valid_rows) {
                const float v = __uint_as_float(r[i]) * scale;
                if (F8 && a.out_amax) {
                  const float t = fmaxf(v, 0.f);
                  vmax = fmaxf(vmax, t * t);
                }
                store_one(a, row0 + n0 + i, f, v);
              }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (F8 && a.out_amax) {
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, d));
      if (lane == 0) record_stored_amax(a.out_amax, vmax);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------ host side ----

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 map over [outer, inner] with a row stride in elements; box {64, box_rows}.
bool map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
            uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over [E, N, K] (K contiguous); box {64, box_rows, 1}.
bool map_3d(CUtensorMap* m, const void* base, uint64_t K, uint64_t N, uint64_t E,
            uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {K, N, E};
  cuuint64_t strides[2] = {K * 2, N * K * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int STAGES, bool SWAP, bool CHUNKED = false, bool F8 = false,
          bool GATHER = false>
int launch_variant(const GroupedGemm& g, const KArgs& ka, cudaStream_t s) {
  CUtensorMap tm_act, tm_w;
  const int act_box = SWAP ? BN : BM;
  const int w_box = SWAP ? BM : BN;
  const int Kw = g.k_wrap ? g.k_wrap : g.K;
  if constexpr (F8) {
    // one byte per element: 128-element K slices
    const uint64_t ad[2] = {static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.rows)};
    const uint64_t as[1] = {static_cast<uint64_t>(g.act_ld)};
    const uint32_t ab[2] = {2 * BK, static_cast<uint32_t>(act_box)};
    if (!encode_tmap(&tm_act, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, g.act, ad, as, ab))
      return MOE_ERR_CUDA;
    const uint64_t wld = g.w_ld ? static_cast<uint64_t>(g.w_ld) : static_cast<uint64_t>(g.K);
    const uint64_t wd[3] = {static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.N),
                            static_cast<uint64_t>(g.E)};
    const uint64_t ws[2] = {wld, static_cast<uint64_t>(g.N) * wld};
    const uint32_t wb[3] = {2 * BK, static_cast<uint32_t>(w_box), 1};
    if (!encode_tmap(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, g.w, wd, ws, wb))
      return MOE_ERR_CUDA;
  } else {
    // gathered rows: a one-row box over the whole token tensor
    if (!map_2d(&tm_act, g.act, g.K, GATHER ? g.src_rows : g.rows, g.act_ld,
                GATHER ? 1 : act_box))
      return MOE_ERR_CUDA;
    if (!map_3d(&tm_w, g.w, Kw, g.N, g.E, w_box)) return MOE_ERR_CUDA;
  }
  constexpr size_t smem = smem_bytes<BN, STAGES>();
  static_assert(smem <= 232448, "shared memory per CTA");
  auto kern = k_grouped_gemm<BN, STAGES, SWAP, CHUNKED, F8, GATHER>;
  static int configured_device = -1;
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (configured_device != dev) {
    MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem)));
    configured_device = dev;
  }
  // Upper bound on the tile count; CTAs without work exit at once.
  const int RT = SWAP ? BN : BM, CT = SWAP ? BM : BN;
  const long long row_tiles = g.offsets ? (static_cast<long long>(g.rows) / RT + g.E)
                                        : (static_cast<long long>(g.rows) + RT - 1) / RT;
  const long long tiles = row_tiles * ((g.N + CT - 1) / CT);
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  if (grid <= 0) return MOE_OK;
  return launch_pdl(kern, dim3(grid), dim3(kernel_threads(CHUNKED)), smem, s, tm_act, tm_w, ka);
}

int pick_bn_rows_as_m(int N) {
  const int cands[4] = {256, 224, 192, 128};
  int best = cands[0];
  long long best_pad = -1;
  for (int c : cands) {
    const long long pad = static_cast<long long>((N + c - 1) / c) * c;
    if (best_pad < 0 || pad < best_pad) {
      best_pad = pad;
      best = c;
    }
  }
  return best;
}

}  // namespace

bool encode_tmap(CUtensorMap* m, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn || rank < 2 || rank > 3) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides_bytes[i];
  return fn(m, dtype, rank, const_cast<void*>(base), d, st, b, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool grouped_gemm_rows_as_m(int rows, int E) {
  return static_cast<double>(rows) / (E > 0 ? E : 1) > 48.0;
}

int launch_grouped_gemm(const GroupedGemm& g, cudaStream_t s) {
  if (g.rows <= 0) return MOE_OK;
  if (g.K % BK || g.N % 16 || (g.k_wrap && (g.k_wrap % BK || g.K % g.k_wrap)) || g.E < 1 ||
      g.E > MAX_GROUPS)
    return MOE_ERR_UNSUPPORTED;
  if (g.fp8 && (g.k_wrap || g.precise || !g.a_amax || !g.w_scale || g.act_ld % 16 ||
                (g.w_ld && (g.w_ld < g.K || g.w_ld % 16))))
    return MOE_ERR_UNSUPPORTED;
  if (!g.fp8 && g.w_ld) return MOE_ERR_UNSUPPORTED;
  if (g.epi == EPI_ADD_BF16 && (!g.add || g.ld_add % 8 || g.precise)) return MOE_ERR_UNSUPPORTED;
  if (g.epi == EPI_COMBINE_I64 &&
      (g.precise || g.fp8 || g.row_token || g.k_wrap || !g.offsets || !g.comb_token ||
       !g.comb_slot_row || !g.comb_gates || g.comb_k < 1 || g.comb_T < 1 || g.ldo % 2))
    return MOE_ERR_UNSUPPORTED;
  if (g.row_token && (g.fp8 || g.precise || g.k_wrap || !g.offsets || g.src_rows <= 0))
    return MOE_ERR_UNSUPPORTED;
  KArgs ka;
  ka.offsets = g.offsets;
  ka.dense_rows = g.rows;
  ka.E = g.offsets ? g.E : 1;
  ka.N = g.N;
  ka.K = g.K;
  ka.k_wrap = g.k_wrap;
  ka.rows_total = g.rows;
  ka.out = g.out;
  ka.ldo = g.ldo;
  ka.lo_offset = g.lo_offset;
  ka.epi = g.epi;
  ka.kchunk = 4;  // 256-deep partial sums in the chunked variant
  ka.add = g.add;
  ka.ld_add = g.ld_add;
  ka.row_token = g.row_token;
  ka.src_rows = g.src_rows;
  ka.a_amax = g.a_amax;
  ka.w_scale = g.w_scale;
  ka.out_amax = g.epi == EPI_SQRELU_BF16 ? g.out_amax : nullptr;
  ka.comb_token = g.comb_token;
  ka.comb_slot_row = g.comb_slot_row;
  ka.comb_gates = g.comb_gates;
  ka.comb_k = g.comb_k;
  ka.comb_T = g.comb_T;
  ka.status = status_word();
  if (!ka.status) return MOE_ERR_CUDA;
  GroupedGemm gg = g;
  if (!g.offsets) gg.E = 1;

  // Chunked (routing) GEMMs: 256-wide tiles halve the operand bytes per MMA cycle of 128-wide
  // ones when N > 128. For N <= 128 the 128-wide tile is the faster one: measured on the
  // prefill router (T = 16384, N = 128), routing took 53.3 us with it against 57.3 us with a
  // half-empty 256-wide tile.
  if (g.precise)
    return g.N > 128 ? launch_variant<256, 4, false, true>(gg, ka, s)
                     : launch_variant<128, 6, false, true>(gg, ka, s);
  if (g.row_token) {  // gathered activation rows
    const double rows_per_group = static_cast<double>(g.rows) / gg.E;
    if (g.force_mode == 2 || (g.force_mode == 0 && rows_per_group <= 48.0)) {
      // weights on M: each K-slice gathers BN / 4 groups of four token rows for the B operand
      if (rows_per_group <= 16.0) return launch_variant<16, 10, true, false, false, true>(gg, ka, s);
      if (rows_per_group <= 32.0) return launch_variant<32, 8, true, false, false, true>(gg, ka, s);
      return launch_variant<64, 8, true, false, false, true>(gg, ka, s);
    }
    switch (pick_bn_rows_as_m(g.N)) {
      case 256: return launch_variant<256, 4, false, false, false, true>(gg, ka, s);
      case 224: return launch_variant<224, 4, false, false, false, true>(gg, ka, s);
      case 192: return launch_variant<192, 5, false, false, false, true>(gg, ka, s);
      default: return launch_variant<128, 6, false, false, false, true>(gg, ka, s);
    }
  }
  // Few rows per group: put the weights on the MMA's M side and the rows on N.
  const double avg_rows = static_cast<double>(g.rows) / gg.E;
  bool swap = g.force_mode == 2 || (g.force_mode == 0 && avg_rows <= 48.0);
  // Many rows per group: 256 x 256 tiles on CTA pairs.
  if (!swap && grouped_gemm_2sm_ok(g)) return launch_grouped_gemm_2sm(g, s);
  if (g.fp8) {
    if (swap) {
      if (avg_rows <= 16.0) return launch_variant<16, 10, true, false, true>(gg, ka, s);
      if (avg_rows <= 32.0) return launch_variant<32, 8, true, false, true>(gg, ka, s);
      return launch_variant<64, 8, true, false, true>(gg, ka, s);
    }
    switch (pick_bn_rows_as_m(g.N)) {
      case 256: return launch_variant<256, 4, false, false, true>(gg, ka, s);
      case 224: return launch_variant<224, 4, false, false, true>(gg, ka, s);
      case 192: return launch_variant<192, 5, false, false, true>(gg, ka, s);
      default: return launch_variant<128, 6, false, false, true>(gg, ka, s);
    }
  }
  if (swap) {
    if (avg_rows <= 16.0) return launch_variant<16, 10, true>(gg, ka, s);
    if (avg_rows <= 32.0) return launch_variant<32, 8, true>(gg, ka, s);
    return launch_variant<64, 8, true>(gg, ka, s);
  }
  switch (pick_bn_rows_as_m(g.N)) {
    case 256: return launch_variant<256, 4, false>(gg, ka, s);
    case 224: return launch_variant<224, 4, false>(gg, ka, s);
    case 192: return launch_variant<192, 5, false>(gg, ka, s);
    default: return launch_variant<128, 6, false>(gg, ka, s);
  }
}

}  // namespace moe
