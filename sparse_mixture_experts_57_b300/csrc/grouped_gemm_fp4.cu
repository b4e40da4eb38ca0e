// grouped_gemm_fp4.cu: block-scaled NVFP4 grouped GEMM on tcgen05 tensor cores.
//
// The expert FFN contraction of the routed MoE layer ("NVIDIA Nemotron 3: Efficient and
// Open Intelligence" notes, §2.2) with both operands in NVFP4 (§2.4: E2M1 elements, an E4M3
// scale per 16 elements, an FP32 scale per tensor):
//
//   out[r, n] = epi( g_a * g_w[e] * sum_k (qa[r,k] sa[r,k/16]) (qw[e,n,k] sw[e,n,k/16]) )
//
// for the rows r of group e. Activation rows are laid out with every group padded to whole
// 128-row tiles, so each row tile starts on a scale-atom boundary.
//
// One CTA per SM, 448 threads, tiles of 256 activation rows (two 128-row halves) by 192
// output columns:
//   warp 0 lane 0  TMA producer: per stage four tensor copies, 256 K-elements (128 bytes)
//                  of the tile's 256 activation rows and of its 192 weight rows (128-byte
//                  swizzle), and the matching scale atoms of both activation halves and of
//                  both weight row blocks the tile touches (two 2 KB rows each). The scale
//                  copies go first and complete on their own barrier.
//   warps 10..13   scale writers, one per TMEM lane quadrant: once a stage's scale atoms
//                  have landed (its operand codes may still be arriving), read them from
//                  shared memory and write them into a two-slot ring of TMEM scale columns
//                  (tcgen05.st), in the layout the block-scaled MMA reads (see below).
//   warp 1 lane 0  MMA issuer: per K step two tcgen05.mma kind::mxf4nvf4 (M=128, N=192,
//                  K=64) with block scales, one per activation half, both on the same weight
//                  tile, into two fp32 accumulators of 192 TMEM columns.
//   warps 2..9     epilogue, one warp per (accumulator, lane quadrant): tcgen05.ld of its
//                  192 columns into registers, 32 columns per tcgen05.wait::ld (global
//                  scales, activation, packed to bf16), then the accumulators are released
//                  to the next tile's MMAs before the stores go out. A warp's 32-row band
//                  goes out as 32x16 pieces staged in swizzled shared memory and written by
//                  TMA stores; only the partial last band of an expert is stored row by row.
//                  The accumulators are single-buffered (two of 192 columns fill TMEM with
//                  the scale ring), so the time this read takes lies between one tile's
//                  MMAs and the next.
//
// Why two accumulators on one weight tile: with block-scaled FP4 MMAs the tensor cores
// consume operand bytes 4x faster than with bf16, and every byte must first be written into
// shared memory by the TMA, whose delivery into one SM (not the L2's output) is the limit:
// three 64 KB stages in flight against about two microseconds of L2 latency under load.
// A tile of M x N outputs moves 32 (M + N) bytes per 64-element K step for M N / 16384
// cycles of MMA work: 96 bytes per MMA cycle at 128 x 256, 75 at 256 x 192.
//
// TMEM (512 columns): accumulator 0 in [0, 192), scale slot 0 in [192, 256), accumulator 1
// in [256, 448), scale slot 1 in [448, 512). Scale columns read by one MMA with scale
// addresses (a, b): A row m at lane m, column a + m / 32; B row n at lane 32 q + n % 32,
// column b + n / 32, for the lane quadrant q of every output row block (so the B scales are
// written to all four quadrants). MMA j of a stage reads, in its slot, the A scales of half h
// at +16 h + 4 j and the B scales at +32 + 8 j (addresses on 4-column boundaries). The slot
// of stage i is i mod 2: its scale writers wait until the MMAs of stage i - 2 have completed.
// Writing the scales with warp stores keeps the tensor pipe's own queue free of copies.
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128;         // rows of one activation half (one MMA's M)
constexpr int BM2 = 2 * BM;     // activation rows of a tile
constexpr int BN = 192;
constexpr int BKB = 128;        // K bytes per stage and row: 256 E2M1 elements
constexpr int KSTEP = 64;       // K elements per MMA
constexpr int STEPS_PER_STAGE = 4;
constexpr int STAGES = 3;
constexpr int MAXG = 1024;
constexpr int NUM_THREADS = 448;
constexpr int EPI_WARP0 = 2, SFW_WARP0 = 10;
constexpr uint32_t A_HALF = BM * BKB;
constexpr uint32_t A_BYTES = 2 * A_HALF;
constexpr uint32_t B_BYTES = BN * BKB;
constexpr uint32_t ATOM = 512;
constexpr uint32_t SF_ONE = STEPS_PER_STAGE * ATOM;  // one 128-row block, 4 K steps
constexpr uint32_t SFA_STAGE = 2 * SF_ONE;           // the two activation halves
constexpr uint32_t SFB_STAGE = 2 * SF_ONE;           // the two 128-row weight blocks touched
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_STRIDE = 256;  // accumulator h at column 256 h
constexpr uint32_t SF_COL0 = BN;      // scale slot s at column 192 + 256 s
constexpr uint32_t SF_B_OFF = 32;
constexpr uint32_t STG_BYTES = 1024;  // one 32 x 16 bf16 output piece
constexpr int NUM_EPI_WARPS = 8;
static_assert(SF_COL0 + 64 <= ACC_STRIDE && ACC_STRIDE + SF_COL0 + 64 <= TMEM_COLS,
              "TMEM budget");
static_assert(BN % 64 == 0 && BN <= 256, "weight tiles start on 64-row boundaries");
constexpr uint32_t IDESC = idesc_nvfp4_f32(BM, BN);
// Bytes landing per stage: every box is copied whole (rows outside a tensor read as zeros).
constexpr uint32_t STAGE_TX = A_BYTES + B_BYTES + SFA_STAGE + SFB_STAGE;
constexpr uint32_t SF_TX = SFA_STAGE + SFB_STAGE;  // the scale boxes, on their own barrier

struct KArgs {
  const int* poff;
  const int* out_off;
  int E, N, K, P;
  const uint8_t* a_sf;
  const uint8_t* w_sf;
  const uint32_t* a_amax;
  const float* w_gscale;
  void* out;
  long long ldo;
  int out_rows;
  int epi;
  uint32_t* out_amax;
  int* status;
};

constexpr size_t smem_bytes() {
  return 1024 + size_t(STAGES) * STAGE_TX + size_t(NUM_EPI_WARPS) * 2 * STG_BYTES + (4 * STAGES + 2) * 8 + 16 + (MAXG + 1) * 4;
}

__device__ __forceinline__ void record(int* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_fp4_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
               const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfw,
               const __grid_constant__ CUtensorMap tm_out, const KArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * A_BYTES;
  uint8_t* sSFA = sB + STAGES * B_BYTES;
  uint8_t* sSFB = sSFA + STAGES * SFA_STAGE;
  uint8_t* sStage = sSFB + STAGES * SFB_STAGE;  // per epilogue warp: two 1 KB pieces
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + NUM_EPI_WARPS * 2 * STG_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* sfull = empty + STAGES;  // the stage's scales are in TMEM
  uint64_t* tfull = sfull + STAGES;  // the accumulators hold a finished tile
  uint64_t* tempty = tfull + 1;      // the epilogue has read the accumulators
  uint64_t* sffull = tempty + 1;     // the stage's scale atoms have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sffull + STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_pref = reinterpret_cast<int*>(tmem_slot + 4);  // row-tile prefix per group

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = a.E;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&sfull[i], 4);
      mbar_init(&sffull[i], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 32 * (SFW_WARP0 - EPI_WARP0));
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_sfa);
    prefetch_tmap(&tm_sfw);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 2) {
    // Row-tile prefix over the groups' padded segments (whole 128-row blocks, 256-row
    // tiles). A group whose offsets are inconsistent is reported and gets no tiles, so no
    // role ever reads it.
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int local = 0;
    bool bad = false;
    for (int e = e0; e < e1; ++e) {
      const int lo = a.poff[e], hi = a.poff[e + 1];
      int tiles = (hi - lo + BM2 - 1) / BM2;
      if (lo < 0 || hi < lo || hi > a.P || ((lo | hi) & (BM - 1))) {
        bad = true;
        tiles = 0;
      } else if (a.out_off) {
        const int olo = a.out_off[e], ocnt = a.out_off[e + 1] - olo;
        if (olo < 0 || ocnt < 0 || olo + ocnt > a.out_rows || ocnt > hi - lo) {
          bad = true;
          tiles = 0;
        }
      } else if (hi > a.out_rows) {
        bad = true;
        tiles = 0;
      }
      s_pref[e] = tiles;  // temporarily the tile count
      local += tiles;
    }
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e1; ++e) {
      const int t = s_pref[e];
      s_pref[e] = run;
      run += t;
    }
    if (lane == 31) s_pref[E] = incl;
    if (__any_sync(0xffffffffu, bad) && lane == 0) record(a.status, MOE_ERR_INVALID_ARG);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int n_ct = (a.N + BN - 1) / BN;
  const int total = s_pref[E] * n_ct;
  const int KS = a.K / KSTEP;                                      // MMA steps along K
  const int NST = (KS + STEPS_PER_STAGE - 1) / STEPS_PER_STAGE;    // pipeline stages along K

  auto decode = [&](int tile, int& e, int& rt, int& ct) {
    const int rtg = tile / n_ct;
    ct = tile - rtg * n_ct;
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_pref[mid + 1] > rtg)
        hi = mid;
      else
        lo = mid + 1;
    }
    e = lo;
    rt = rtg - s_pref[lo];
  };
  // Whether the tile's second activation half lies inside the group's padded segment.
  auto second_half = [&](int e, int rt) {
    return rt * BM2 + BM < __ldg(a.poff + e + 1) - __ldg(a.poff + e);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer
      const uint64_t pol = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long armed = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, rt, ct;
        decode(tile, e, rt, ct);
        const int row0 = __ldg(a.poff + e) + rt * BM2;
        const int col0 = ct * BN;
        for (int kb = 0; kb < NST; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          // The scale atoms first, on their own barrier: the scale writers can put them into
          // TMEM while the operand codes are still arriving. 8-byte elements, 256 per row
          // block and stage.
          mbar_arrive_expect_tx(&sffull[stage], SF_TX);
          tma_load_2d(sSFA + stage * SFA_STAGE, &tm_sfa, &sffull[stage], kb * 256, row0 / BM, pol);
          tma_load_3d(sSFB + stage * SFB_STAGE, &tm_sfw, &sffull[stage], kb * 256, col0 / 128, e,
                      pol);
          mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES);
          ++armed;
          // Rows past a group's segment (a half tile) are loaded and not used; rows past the
          // end of a tensor read as zeros.
          tma_load_2d(sA + stage * A_BYTES, &tm_a, &full[stage], kb * BKB, row0, pol);
          tma_load_3d(sB + stage * B_BYTES, &tm_w, &full[stage], kb * BKB, col0, e, pol);
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
      if (!drain_stages(sffull, STAGES, stage, phase, armed)) record(a.status, MOE_ERR_TIMEOUT);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      uint32_t slot = 0;  // scale slot of the stage: the stage count mod 2
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, rt, ct;
        decode(tile, e, rt, ct);
        const bool two_a = second_half(e, rt);
        if (!mbar_wait(tempty, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < NST; ++kb) {
          const int nsteps = min(STEPS_PER_STAGE, KS - kb * STEPS_PER_STAGE);
          // the stage's scales are in TMEM and its operand codes have landed
          if (!mbar_wait(&sfull[stage], phase, abort_flag) ||
              !mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf = tmem_base + SF_COL0 + slot * ACC_STRIDE;
          const uint64_t adesc = sdesc_k_sw128(smem_u32(sA + stage * A_BYTES));
          const uint64_t adesc1 = sdesc_k_sw128(smem_u32(sA + stage * A_BYTES + A_HALF));
          const uint64_t bdesc = sdesc_k_sw128(smem_u32(sB + stage * B_BYTES));
          for (int j = 0; j < nsteps; ++j) {
            const uint32_t acc = (kb | j) != 0;
            umma_nvfp4(tmem_base, adesc + 2u * j, bdesc + 2u * j, IDESC, sf + 4 * j,
                       sf + SF_B_OFF + 8 * j, acc);
            if (two_a)
              umma_nvfp4(tmem_base + ACC_STRIDE, adesc1 + 2u * j, bdesc + 2u * j, IDESC,
                         sf + 16 + 4 * j, sf + SF_B_OFF + 8 * j, acc);
          }
          umma_commit(&empty[stage]);
          slot ^= 1u;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull);
        acc_phase ^= 1u;
      }
      if (!ok) {
        *abort_flag = 1;
        record(a.status, MOE_ERR_TIMEOUT);
      }
    }
  } else if (warp >= SFW_WARP0) {
    // -------------------------------------------------------------------- scale writers
    // Quadrant q of TMEM, lane r0 = this lane. The smem atoms hold row 32 r1 + r0 of step j
    // at byte j * 512 + r0 * 16 + r1 * 4 (four E4M3 scales, one per 16 K elements). The A
    // stage holds the first activation half's atoms, then the second's; the B stage the
    // atoms of the weight row block holding the tile's first row and of the next block
    // (zeros past the last), the tile's 192 rows starting at row 0 or 64 of the first.
    const int q = warp & 3;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;  // stages so far: the scale slot is it mod 2
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      int e, rt, ct;
      decode(tile, e, rt, ct);
      const bool mid = ((ct * BN) & 127) != 0;  // the tile starts at row 64 of its first block
      for (int kb = 0; kb < NST; ++kb, ++it) {
        const int nsteps = min(STEPS_PER_STAGE, KS - kb * STEPS_PER_STAGE);
        if (!mbar_wait(&sffull[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        // The slot was last read by the MMAs of stage it - 2 (committed to empty[] of that
        // stage, whose completion parity is its use count mod 2).
        if (it >= 2 && !mbar_wait(&empty[(it - 2) % STAGES], ((it - 2) / STAGES) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* sa = sSFA + stage * SFA_STAGE;
        const uint8_t* sb = sSFB + stage * SFB_STAGE;
        uint32_t wa0[STEPS_PER_STAGE], wa1[STEPS_PER_STAGE];
        uint32_t wb[2][16];
#pragma unroll
        for (int j = 0; j < STEPS_PER_STAGE; ++j) {
          uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
          wa0[j] = 0u;
          wa1[j] = 0u;
          if (j < nsteps) {
            wa0[j] = *reinterpret_cast<const uint32_t*>(sa + j * ATOM + lane * 16 + q * 4);
            wa1[j] = *reinterpret_cast<const uint32_t*>(sa + SF_ONE + j * ATOM + lane * 16 + q * 4);
            v0 = *reinterpret_cast<const uint4*>(sb + j * ATOM + lane * 16);
            v1 = *reinterpret_cast<const uint4*>(sb + SF_ONE + j * ATOM + lane * 16);
          }
          // column c of MMA j: weight row 32 c + lane of the tile
          uint32_t* w = wb[j >> 1] + 8 * (j & 1);
          w[0] = mid ? v0.z : v0.x;
          w[1] = mid ? v0.w : v0.y;
          w[2] = mid ? v1.x : v0.z;
          w[3] = mid ? v1.y : v0.w;
          w[4] = mid ? v1.z : v1.x;
          w[5] = mid ? v1.w : v1.y;
          w[6] = 0u;
          w[7] = 0u;
        }
        const uint32_t sf = SF_COL0 + static_cast<uint32_t>(it & 1) * ACC_STRIDE;
#pragma unroll
        for (int j = 0; j < STEPS_PER_STAGE; ++j) {
          tmem_st1(lane_base + sf + 4 * j + q, wa0[j]);
          tmem_st1(lane_base + sf + 16 + 4 * j + q, wa1[j]);
        }
        tmem_st16(lane_base + sf + SF_B_OFF, wb[0]);
        tmem_st16(lane_base + sf + SF_B_OFF + 16, wb[1]);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) record(a.status, MOE_ERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int h = (warp - EPI_WARP0) >> 2;  // accumulator: rows [128 h, 128 h + 128) of the tile
    const int m = q * 32 + lane;
    const float ga = __fdiv_rn(__uint_as_float(*a.a_amax), kNvfp4GlobalDiv);
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ACC_STRIDE * h;
    uint8_t* stg = sStage + (warp - EPI_WARP0) * 2 * STG_BYTES;
    float vmax = 0.f;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, rt, ct;
      decode(tile, e, rt, ct);
      const int local = rt * BM2 + h * BM + m;
      int ocnt, obase;
      if (a.out_off) {
        obase = __ldg(a.out_off + e);
        ocnt = __ldg(a.out_off + e + 1) - obase;
      } else {
        obase = __ldg(a.poff + e);
        ocnt = __ldg(a.poff + e + 1) - obase;
      }
      const bool valid = local < ocnt;
      const long long row = static_cast<long long>(obase) + local;
      const int c0 = ct * BN;                       // first column of the tile
      const int ncols = max(0, min(BN, a.N - c0));  // warp-uniform, a multiple of 32
      const float scale = ga * __ldg(a.w_gscale + e);
      if (!mbar_wait(tfull, acc_phase, abort_flag)) {
        *abort_flag = 1;
        record(a.status, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      uint32_t p[BN / 2];  // this row's outputs, packed bf16 pairs
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        if (32 * c < ncols) {
          uint32_t r0[16], r1[16];
          tmem_ld16(tb + 32 * c, r0);
          tmem_ld16(tb + 32 * c + 16, r1);
          tmem_ld_wait();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(hh ? r1[i] : r0[i]) * scale;
            if (a.epi == EPI_SQRELU_BF16) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float t = fmaxf(v[i], 0.f);
                v[i] = t * t;
              }
              if (valid) {
#pragma unroll
                for (int i = 0; i < 16; ++i) vmax = fmaxf(vmax, v[i]);
              }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) p[16 * c + 8 * hh + i] = pack_bf16(v[2 * i], v[2 * i + 1]);
          }
        }
      }
      // The accumulators are in registers: let the next tile's MMAs start.
      tc_fence_before();
      mbar_arrive(tempty);
      acc_phase ^= 1u;
      const int band0 = rt * BM2 + h * BM + q * 32;  // first local row of this warp's band
      if (band0 + 32 <= ocnt) {
        // Whole band valid: 32 x 16 pieces through shared memory (32-byte swizzle: 16-byte
        // chunk i of row r at chunk i ^ ((r >> 2) & 1)), written by TMA.
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) {
          if (16 * c < ncols) {
            uint8_t* buf = stg + (c & 1) * STG_BYTES;
            if (lane == 0) bulk_wait_group_read<1>();  // the store that last used buf is done
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 2; ++i)
              *reinterpret_cast<uint4*>(buf + lane * 32 + ((i ^ ((lane >> 2) & 1)) << 4)) =
                  make_uint4(p[8 * c + 4 * i], p[8 * c + 4 * i + 1], p[8 * c + 4 * i + 2],
                             p[8 * c + 4 * i + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm_out, buf, c0 + 16 * c, obase + band0);
              bulk_commit_group();
            }
          }
        }
      } else if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + row * a.ldo + c0);
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) {
          if (16 * c < ncols) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
              dst[2 * c + i] = make_uint4(p[8 * c + 4 * i], p[8 * c + 4 * i + 1],
                                          p[8 * c + 4 * i + 2], p[8 * c + 4 * i + 3]);
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();  // the staged pieces are written out
    if (a.out_amax) {
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

}  // namespace

int launch_fp4_gemm(const Fp4Gemm& g, cudaStream_t s) {
  if (g.P <= 0) return MOE_OK;
  if (g.K % KSTEP || g.N % 32 || g.E < 1 || g.E > MAXG || g.P % BM || g.ldo % 8 ||
      g.a_ld < g.K / 2 || g.a_ld % 16 ||
      ((reinterpret_cast<uintptr_t>(g.out) | reinterpret_cast<uintptr_t>(g.a_codes) |
        reinterpret_cast<uintptr_t>(g.w_codes) | reinterpret_cast<uintptr_t>(g.a_sf) |
        reinterpret_cast<uintptr_t>(g.w_sf)) & 15))
    return MOE_ERR_UNSUPPORTED;
  if (g.epi != EPI_BF16 && g.epi != EPI_SQRELU_BF16) return MOE_ERR_UNSUPPORTED;
  KArgs ka;
  ka.poff = g.poff;
  ka.out_off = g.out_off;
  ka.E = g.E;
  ka.N = g.N;
  ka.K = g.K;
  ka.P = g.P;
  ka.a_sf = g.a_sf;
  ka.w_sf = g.w_sf;
  ka.a_amax = g.a_amax;
  ka.w_gscale = g.w_gscale;
  ka.out = g.out;
  ka.ldo = g.ldo;
  ka.out_rows = g.out_rows;
  ka.epi = g.epi;
  ka.out_amax = g.epi == EPI_SQRELU_BF16 ? g.out_amax : nullptr;
  ka.status = status_word();
  if (!ka.status) return MOE_ERR_CUDA;

  CUtensorMap tm_a, tm_w;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(g.K / 2), static_cast<uint64_t>(g.P)};
    const uint64_t strides[1] = {static_cast<uint64_t>(g.a_ld)};
    const uint32_t box[2] = {BKB, BM2};
    if (!encode_tmap(&tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, g.a_codes, dims, strides, box))
      return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(g.K / 2), static_cast<uint64_t>(g.N),
                              static_cast<uint64_t>(g.E)};
    const uint64_t strides[2] = {static_cast<uint64_t>(g.K / 2),
                                 static_cast<uint64_t>(g.N) * (g.K / 2)};
    const uint32_t box[3] = {BKB, BN, 1};
    if (!encode_tmap(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, g.w_codes, dims, strides, box))
      return MOE_ERR_CUDA;
  }
  // Scale atoms as rows of 8-byte elements: one row per 128-row block, K/64 atoms of 64
  // elements along it.
  const int KS = g.K / KSTEP;
  CUtensorMap tm_sfa, tm_sfw;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(KS) * (ATOM / 8), static_cast<uint64_t>(g.P / BM)};
    const uint64_t strides[1] = {static_cast<uint64_t>(KS) * ATOM};
    const uint32_t box[2] = {SF_ONE / 8, 2};
    if (!encode_tmap(&tm_sfa, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, g.a_sf, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return MOE_ERR_CUDA;
  }
  {
    const int nbw = (g.N + 127) / 128;
    const uint64_t dims[3] = {static_cast<uint64_t>(KS) * (ATOM / 8), static_cast<uint64_t>(nbw),
                              static_cast<uint64_t>(g.E)};
    const uint64_t strides[2] = {static_cast<uint64_t>(KS) * ATOM,
                                 static_cast<uint64_t>(nbw) * KS * ATOM};
    const uint32_t box[3] = {SF_ONE / 8, 2, 1};
    if (!encode_tmap(&tm_sfw, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, g.w_sf, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return MOE_ERR_CUDA;
  }
  CUtensorMap tm_out;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(g.N), static_cast<uint64_t>(g.out_rows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(g.ldo) * 2};
    const uint32_t box[2] = {16, 32};
    if (!encode_tmap(&tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.out, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_32B))
      return MOE_ERR_CUDA;
  }
  constexpr size_t smem = smem_bytes();
  static_assert(smem <= 232448, "shared memory per CTA");
  static int configured_device = -1;
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (configured_device != dev) {
    MOE_CUDA(cudaFuncSetAttribute(k_fp4_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem)));
    configured_device = dev;
  }
  // at most one tile per 128-row block and column tile (a group's last tile may be half)
  const long long tiles = static_cast<long long>(g.P / BM) * ((g.N + BN - 1) / BN);
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  if (grid <= 0) return MOE_OK;
  return launch_pdl(k_fp4_gemm, dim3(grid), dim3(NUM_THREADS), smem, s, tm_a, tm_w, tm_sfa,
                    tm_sfw, tm_out, ka);
}

}  // namespace moe
