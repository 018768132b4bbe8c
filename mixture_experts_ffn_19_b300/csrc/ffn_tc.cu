// Expert FFNs in bf16 on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// The per-expert Python loop of «为什么MoE有效？稀疏激活的数学直觉与工程实践» §3
// (whose note says production code replaces it with a grouped GEMM) becomes two
// persistent grouped GEMMs over the ragged expert segments produced by dispatch:
//   GEMM-1  H = silu(X Wg^T) * (X Wu^T)     SwiGLU, «大模型MoE架构揭秘» §3.2
//   GEMM-2  Y = H Wd^T
// Shared experts («DeepSeek-V2 ...» summary §2.3) are extra segments whose rows
// are read straight from x.
//
// Tile: 128 rows x 256 accumulator columns x 64-deep K steps, one CTA per SM.
//   warp 0      TMA producer: A tile (128 x 64) and B tile (256 x 64) per stage,
//               128-byte swizzle, 4-stage ring of 48 KB stages
//   warp 1      allocates 512 TMEM columns; one lane issues tcgen05.mma
//               (M=128, N=256, K=16, bf16 x bf16 -> fp32) and commits stages
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, activation, bf16 store
// The two 256-column accumulators in TMEM alternate so the epilogue of one tile
// overlaps the main loop of the next.  In GEMM-1 the B tile stacks 128 gate rows
// over 128 up rows of the same output features, so columns [0,128) of the
// accumulator hold x.Wg and [128,256) hold x.Wu for the same features and the
// SwiGLU product is formed in registers.  Tiles walk segment by segment, row
// tiles fastest, so CTAs running together share one weight tile through L2.
// Every wait is bounded (kWaitLimitNs); on time-out the CTA records
// MOE_ERR_TIMEOUT in the status word, stops issuing work and frees its TMEM.
#include <algorithm>
#include <mutex>

#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

// When the GEMMs let their successor launch: at their start (1), or once a CTA
// has finished its tiles (0), so that the successor's waiting CTAs do not sit
// beside a GEMM that still runs.
#ifndef MOE_GEMM_EARLY_TRIGGER
#define MOE_GEMM_EARLY_TRIGGER 0
#endif

namespace moe {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int NUM_THREADS = 192;
// Below this many tiles per CTA the sum of a CTA's tile times varies too much
// for a fixed deal to finish every CTA together, so CTAs claim tiles as they go.
#ifndef MOE_DYNAMIC_TILES_PER_CTA
#define MOE_DYNAMIC_TILES_PER_CTA 32
#endif
constexpr int kDynamicTilesPerCta = MOE_DYNAMIC_TILES_PER_CTA;
constexpr int QSLOTS = 4;                // tile-index queue from the TMA warp

// Tile width BN (the MMA's N: output columns of a GEMM-2 tile, gate + up
// columns of a GEMM-1 tile) and the depth of the shared-memory ring.
#ifndef MOE_PREFILL_BN
#define MOE_PREFILL_BN 256
#endif
#ifndef MOE_PREFILL_STAGES
#define MOE_PREFILL_STAGES 4
#endif

template <int BN_, int STAGES_>
struct TileCfg {
  static constexpr int BN = BN_, STAGES = STAGES_;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;       // two accumulators
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
  struct Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t qfull[QSLOTS];     // tile index published (dynamic claiming)
    uint64_t qempty[QSLOTS];    // read by the MMA lane and the four epilogue warps
    int q_tile[QSLOTS];
    uint32_t tmem_base;
    int abort;
    int total_mtiles;
    int dyn;
    int mt_prefix[kMaxExperts + 16];
  };
  static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(Ctrl);
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "tmem");
};
using Prefill = TileCfg<MOE_PREFILL_BN, MOE_PREFILL_STAGES>;

struct TcParams {
  int E, S, K, n_out, n_tiles_n, bn_out;  // bn_out: output columns per tile
  const int32_t* offsets;
  __nv_bfloat16* out;
  int* status;
  int* ctr;                              // [2] tile-claim and done counters (zero between launches)
};


struct TileCoord {
  int seg, m, n;
};

template <class CtrlT>
__device__ __forceinline__ TileCoord tile_coord(const CtrlT* c, int nseg, int n_tiles_n, int T) {
  const int q = T / n_tiles_n;
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {   // largest segment whose first row tile is <= q
    const int mid = (lo + hi + 1) >> 1;
    if (c->mt_prefix[mid] <= q) lo = mid; else hi = mid - 1;
  }
  const int mt = c->mt_prefix[lo + 1] - c->mt_prefix[lo];
  const int local = T - c->mt_prefix[lo] * n_tiles_n;
  return {lo, local % mt, local / mt};
}

__device__ __forceinline__ float silu_f(float a) { return a / (1.f + __expf(-a)); }

template <int MODE, class C>
__global__ void __launch_bounds__(NUM_THREADS, 1)
ffn_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
              const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
              TcParams p) {
  griddep_wait();
  if (MOE_GEMM_EARLY_TRIGGER) griddep_launch_dependents();
  constexpr int BN = C::BN, STAGES = C::STAGES, B_BYTES = C::B_BYTES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES, TMEM_COLS = C::TMEM_COLS;
  constexpr uint32_t IDESC = C::IDESC;
  using Ctrl = typename C::Ctrl;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nseg = p.E + p.S;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&ctrl->full[s], 1); mbar_init(&ctrl->empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&ctrl->tfull[b], 1); mbar_init(&ctrl->tempty[b], 128); }
    for (int q = 0; q < QSLOTS; ++q) { mbar_init(&ctrl->qfull[q], 1); mbar_init(&ctrl->qempty[q], 5); }
    ctrl->abort = 0;
    int run = 0;
    for (int s = 0; s < nseg; ++s) {
      ctrl->mt_prefix[s] = run;
      run += (p.offsets[s + 1] - p.offsets[s]) / BM;
    }
    ctrl->mt_prefix[nseg] = run;
    ctrl->total_mtiles = run;
    ctrl->dyn = p.ctr != nullptr && run * p.n_tiles_n < kDynamicTilesPerCta * (int)gridDim.x;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0); tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB0); tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) { tmem_alloc(&ctrl->tmem_base, TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctrl->tmem_base;
  const int total_tiles = ctrl->total_mtiles * p.n_tiles_n;
  const int KB = (p.K + BK - 1) / BK;
  volatile int* abort = &ctrl->abort;

  const bool dyn = ctrl->dyn != 0;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t kc = 0, qi = 0;
      // tiles in the static order T, T + grid, ...; or (dynamic) the first
      // wave in that order, then whatever tile the shared counter hands out,
      // each index published to the MMA and epilogue roles through the queue
      for (int T = blockIdx.x;; ++qi) {
        if (T >= total_tiles || *abort) T = -1;
        if (dyn) {
          const int slot = qi % QSLOTS;
          if (!mbar_wait(&ctrl->qempty[slot], ((qi / QSLOTS) & 1) ^ 1, abort, p.status)) break;
          ctrl->q_tile[slot] = T;
          mbar_arrive(&ctrl->qfull[slot]);
        }
        if (T < 0) break;
        const TileCoord tc = tile_coord(ctrl, nseg, p.n_tiles_n, T);
        const CUtensorMap* amap = &tmA0;
        int a_row = p.offsets[tc.seg] + tc.m * BM;
        if (MODE == 0 && tc.seg >= p.E) { amap = &tmA1; a_row = tc.m * BM; }
        const int b_row = tc.seg * p.n_out + tc.n * (MODE == 0 ? BN / 2 : BN);
        for (int kb = 0; kb < KB; ++kb, ++kc) {
          const int st = kc % STAGES;
          const uint32_t ph = (kc / STAGES) & 1;
          if (!mbar_wait(&ctrl->empty[st], ph ^ 1, abort, p.status)) break;
          uint8_t* a_s = smem + (size_t)st * STAGE_BYTES;
          uint8_t* b_s = a_s + A_BYTES;
          mbar_arrive_expect_tx(&ctrl->full[st], STAGE_BYTES);
          tma_load_2d(a_s, amap, &ctrl->full[st], kb * BK, a_row);
          if (MODE == 0) {
            tma_load_2d(b_s, &tmB0, &ctrl->full[st], kb * BK, b_row);
            tma_load_2d(b_s + B_BYTES / 2, &tmB1, &ctrl->full[st], kb * BK, b_row);
          } else {
            tma_load_2d(b_s, &tmB0, &ctrl->full[st], kb * BK, b_row);
          }
        }
        T = dyn ? (int)gridDim.x + atomicAdd(&p.ctr[0], 1) : T + (int)gridDim.x;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t kc = 0;
      for (uint32_t it = 0;; ++it) {
        int T = blockIdx.x + (int)(it * gridDim.x);
        if (dyn) {
          const int slot = it % QSLOTS;
          if (!mbar_wait(&ctrl->qfull[slot], (it / QSLOTS) & 1, abort, p.status)) break;
          T = ctrl->q_tile[slot];
          mbar_arrive(&ctrl->qempty[slot]);
        }
        if (T < 0 || T >= total_tiles || *abort) break;
        const uint32_t buf = it & 1, use = it >> 1;
        if (!mbar_wait(&ctrl->tempty[buf], (use & 1) ^ 1, abort, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++kc) {
          const int st = kc % STAGES;
          const uint32_t ph = (kc / STAGES) & 1;
          if (!mbar_wait(&ctrl->full[st], ph, abort, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + (size_t)st * STAGE_BYTES);
          const uint64_t adesc = sdesc_kmajor_sw128(a_addr);
          const uint64_t bdesc = sdesc_kmajor_sw128(a_addr + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb | k) != 0);
          umma_commit(&ctrl->empty[st]);
        }
        if (!ok) break;
        umma_commit(&ctrl->tfull[buf]);
      }
    }
  } else {
    // epilogue warps 2..5: TMEM lane quarter = warp % 4
    const int q = warp & 3;
    for (uint32_t it = 0;; ++it) {
      if (__any_sync(0xffffffffu, *abort != 0)) break;
      int T = blockIdx.x + (int)(it * gridDim.x);
      if (dyn) {
        const int slot = it % QSLOTS;
        const bool got = mbar_wait(&ctrl->qfull[slot], (it / QSLOTS) & 1, abort, p.status);
        if (!__all_sync(0xffffffffu, got)) break;
        T = ctrl->q_tile[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctrl->qempty[slot]);
      }
      if (T < 0 || T >= total_tiles) break;
      const TileCoord tc = tile_coord(ctrl, nseg, p.n_tiles_n, T);
      const uint32_t buf = it & 1, use = it >> 1;
      const bool ok = mbar_wait(&ctrl->tfull[buf], use & 1, abort, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;   // tcgen05.ld below is warp-collective
      tc_fence_after();
      const int row = p.offsets[tc.seg] + tc.m * BM + q * 32 + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN;
      __nv_bfloat16* out_row = p.out + (size_t)row * p.n_out;
      const int col0 = tc.n * p.bn_out;
      if (MODE == 0) {
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + BN / 2 + c * 32, u);
          tmem_wait_ld();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h0 = silu_f(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
            const float h1 = silu_f(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
            packed[i] = pack_bf16x2(h0, h1);
          }
          const int cc = col0 + c * 32;
          uint4* dst = reinterpret_cast<uint4*>(out_row + cc);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            if (cc + 8 * v + 8 <= p.n_out)
              dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t a[32];
          tmem_ld32(taddr + c * 32, a);
          tmem_wait_ld();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
          const int cc = col0 + c * 32;
          uint4* dst = reinterpret_cast<uint4*>(out_row + cc);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            if (cc + 8 * v + 8 <= p.n_out)
              dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl->tempty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (!MOE_GEMM_EARLY_TRIGGER) griddep_launch_dependents();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  // the last CTA to finish leaves the counters at zero for the next launch
  if (dyn && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&p.ctr[1], 1) == (int)gridDim.x - 1) {
      atomicExch(&p.ctr[0], 0);
      atomicExch(&p.ctr[1], 0);
    }
  }
}

// ---------------------------------------------------------------- swap-AB variant
//
// For decode-sized batches (a few tokens per expert) the 128-row token tiles
// above are mostly padding.  Here the roles swap: the weights are the MMA's
// M=128 operand and the expert's tokens (in chunks of up to 64) are the N
// operand, N = tokens rounded up to 16.  GEMM-1 stacks 64 gate rows over 64 up
// rows of the same features in one M=128 tile; the epilogue warps holding the
// up rows pass them through shared memory to the warps holding the gate rows,
// which form silu(g)*u and store H.  GEMM-2 takes 128 rows of W_down per tile.
// Tiles walk segment by segment, feature block by feature block, token chunk
// fastest, so a weight tile is read from HBM once.
//
// FP8 weights (W8): the weight tile arrives as E4M3 codes (8 KB per stage, half
// the HBM bytes) in a staging buffer; four converter warps widen it to f16 in
// the 128-byte-swizzled layout the MMA reads (every E4M3 value is exact in
// f16; one conversion per code pair, against three for bf16) and release the
// stage to the MMA warp, which multiplies f16 by f16: the token rows and H are
// f16 copies in this path.  The per-expert-matrix scales multiply the
// accumulators in the epilogue («大模型MoE架构揭秘» §5.4: expert weights in low
// precision with per-expert scales, router in high precision).

namespace swp {

constexpr int BM = 128, TOK = 64, BK = 64;
constexpr int TOKB = 16;                       // token rows per TMA box
constexpr int A_BYTES = BM * BK * 2;
constexpr int BQ_BYTES = TOKB * BK * 2;        // one 16-row token box
constexpr int A8_BYTES = BM * BK;              // E4M3 weight tile (W8 staging)
constexpr int TMEM_COLS = 128;                 // two 64-column accumulators
constexpr int XS = TOK + 1;                    // exchange row (floats), conflict-free
constexpr int MAX_STAGES = 10;
constexpr int CONV_WARPS = 4;                  // W8 converter warps 6..9
constexpr float kF16Max = 65504.f;             // largest finite f16

// bf16 weights: one ring of [A (bf16 weights) | B (tokens)] stages, 64 deep
// in K.  E4M3 weights: stages 128 deep in K, so every weight row is read as
// a whole 128-byte line (64-byte pieces of rows 8 KB apart held the DRAM
// below half its bandwidth): a TMA ring of [B (2 K-chunks) | E4M3 tile]
// stages and a ring of converted stages of two f16 A tiles.
template <bool W8>
struct Shape {
  static constexpr int KSUB = W8 ? 2 : 1;               // 64-deep K-chunks per stage
  static constexpr int TOK = swp::TOK;                   // tokens per chunk
  static constexpr int B_BYTES = TOK * BK * 2;
  static constexpr int STAGE_BYTES = W8 ? KSUB * (B_BYTES + A8_BYTES) : A_BYTES + B_BYTES;
  static constexpr int STAGES = W8 ? 4 : 8;             // TMA ring
  static constexpr int A_STAGES = W8 ? 2 : 0;           // converted ring (KSUB A tiles each)
  static constexpr int THREADS = W8 ? 192 + 32 * CONV_WARPS : 192;
};

struct Ctrl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t conv[4];              // W8: converted f16 tile ready
  uint64_t afree[4];             // W8: converted tile consumed by the MMA
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t xfull;                // up values written to the exchange buffer
  uint64_t xempty;               // exchange buffer consumed
  uint32_t tmem_base;
  int abort;
  int total_chunks;
  int pad;
  int ch_prefix[kMaxExperts + 16];
};

constexpr size_t XCH_BYTES = (size_t)64 * XS * 4;
template <bool W8>
constexpr size_t ring_bytes() {
  return (size_t)Shape<W8>::STAGES * Shape<W8>::STAGE_BYTES +
         (size_t)Shape<W8>::A_STAGES * Shape<W8>::KSUB * A_BYTES;
}
template <bool W8>
constexpr size_t smem_bytes() {
  return 1024 + ring_bytes<W8>() + XCH_BYTES + sizeof(Ctrl);
}
static_assert(smem_bytes<true>() <= 232448 && smem_bytes<false>() <= 232448, "shared memory");

struct Params {
  int E, S, N, K, n_out, n_fb;   // n_fb: feature blocks per segment
  const int32_t* offsets;
  const int32_t* counts;         // [E] valid rows of the routed segments
  __nv_bfloat16* out;
  int* status;
  const float* scale0;           // W8: per-segment scales of the gate (GEMM-1) / down weights
  const float* scale1;           // W8: per-segment scales of the up weights (GEMM-1)
};

// 8 E4M3 codes -> 8 f16 (exact: every E4M3 value, subnormals included, is an
// f16 normal), one conversion-unit instruction per pair.  Widening to bf16
// instead took three per pair (through f32) and kept the converter warps
// 7-9 % of the decode step longer.
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t word = i < 2 ? v.x : v.y;
    const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((word >> (16 * (i & 1))) & 0xFFFFu);
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
    w[i] = *reinterpret_cast<const uint32_t*>(&hr);   // the pair as one register
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ int seg_rows(const Params& p, int s) {
  return s < p.E ? p.counts[s] : p.N;
}

template <int MODE, bool W8>
__global__ void __launch_bounds__(Shape<W8>::THREADS, 1)
ffn_tc_swap_kernel(const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   Params p) {
  griddep_wait();
  if (MOE_GEMM_EARLY_TRIGGER) griddep_launch_dependents();
  // tmB0/tmB1: token rows (x_perm / x for GEMM-1, H for GEMM-2; their f16
  // copies with E4M3 weights); tmA0/tmA1: weights (gate / up for GEMM-1,
  // down for GEMM-2), bf16 or E4M3
  constexpr int STAGES = Shape<W8>::STAGES, STAGE_BYTES = Shape<W8>::STAGE_BYTES;
  constexpr int A_STAGES = Shape<W8>::A_STAGES, KSUB = Shape<W8>::KSUB;
  constexpr int TOK = Shape<W8>::TOK, B_BYTES = Shape<W8>::B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* xch = reinterpret_cast<float*>(smem + ring_bytes<W8>());
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + ring_bytes<W8>() + XCH_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nseg = p.E + p.S;
  // tiles of TMA stage s1 and converted stage s2, K-chunk j (all 1024-byte
  // aligned): W8 stage = [B0 | B1 | E4M3 128 rows x 128 bytes], converted
  // stage = [A0 | A1]
  auto b_tile = [&](int s1, int j) {
    return smem + (size_t)s1 * STAGE_BYTES + (W8 ? j * B_BYTES : A_BYTES);
  };
  auto w8_tile = [&](int s1) { return smem + (size_t)s1 * STAGE_BYTES + KSUB * B_BYTES; };
  auto a_tile = [&](int s1, int s2, int j) {
    return W8 ? smem + (size_t)STAGES * STAGE_BYTES + ((size_t)s2 * KSUB + j) * A_BYTES
              : smem + (size_t)s1 * STAGE_BYTES;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);
    }
    for (int s = 0; s < A_STAGES; ++s) {
      mbar_init(&ctrl->conv[s], 32 * CONV_WARPS);
      mbar_init(&ctrl->afree[s], 1);
    }
    for (int b = 0; b < 2; ++b) { mbar_init(&ctrl->tfull[b], 1); mbar_init(&ctrl->tempty[b], 128); }
    mbar_init(&ctrl->xfull, 64);
    mbar_init(&ctrl->xempty, 64);
    ctrl->abort = 0;
    int run = 0;
    for (int s = 0; s < nseg; ++s) {
      ctrl->ch_prefix[s] = run;
      run += (seg_rows(p, s) + TOK - 1) / TOK;
    }
    ctrl->ch_prefix[nseg] = run;
    ctrl->total_chunks = run;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0); tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB0); tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) { tmem_alloc(&ctrl->tmem_base, TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctrl->tmem_base;
  const int total_tiles = ctrl->total_chunks * p.n_fb;
  // bf16 weights: the tiles are dealt to the fewest CTAs that still need the
  // same number of waves, so every wave is full.  The kernel streams weights
  // from HBM, and a short last wave (DeepSeek-V2 decode: 936 tiles =
  // 6 x 148 + 48) leaves too few SMs to keep HBM busy, while 134 CTAs with 7
  // tiles each do (decode steps 2.7-2.8 % faster).  The E4M3 kernel, bound
  // by its stage hand-offs rather than by HBM, keeps every CTA (it measured
  // 0.6-0.8 % slower dealt that way).
  const int waves = (total_tiles + (int)gridDim.x - 1) / (int)gridDim.x;
  const int stride =
      (!W8 && waves > 0) ? (total_tiles + waves - 1) / waves : (int)gridDim.x;
  const int T0 = (int)blockIdx.x < stride ? (int)blockIdx.x : total_tiles;   // idle CTAs: no tile
  const int KB = (p.K + BK * KSUB - 1) / (BK * KSUB);   // stages per tile
  volatile int* abort = &ctrl->abort;
  const Ctrl* cc = ctrl;
  // tile -> (segment, feature block, token chunk); chunk fastest
  auto coord = [&](int T, int& seg, int& fb, int& ch) {
    const int q = T / p.n_fb;
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cc->ch_prefix[mid] <= q) lo = mid; else hi = mid - 1;
    }
    const int nch = cc->ch_prefix[lo + 1] - cc->ch_prefix[lo];
    const int local = T - cc->ch_prefix[lo] * p.n_fb;
    seg = lo; fb = local / nch; ch = local % nch;
  };

  if (warp == 0) {
    if (lane == 0) {
      uint32_t kc = 0;
      for (int T = T0; T < total_tiles && !*abort; T += stride) {
        int seg, fb, ch;
        coord(T, seg, fb, ch);
        const CUtensorMap* bmap = &tmB0;
        int b_row = p.offsets[seg] + ch * TOK;
        if (MODE == 0 && seg >= p.E) { bmap = &tmB1; b_row = ch * TOK; }
        const int a_row = seg * p.n_out + fb * (MODE == 0 ? BM / 2 : BM);
        // only the 16-row token boxes this chunk uses (decode experts see a few tokens)
        const int nq = (min(TOK, seg_rows(p, seg) - ch * TOK) + TOKB - 1) / TOKB;
        for (int kb = 0; kb < KB; ++kb, ++kc) {
          const int st = kc % STAGES;
          const uint32_t ph = (kc / STAGES) & 1;
          if (!mbar_wait(&ctrl->empty[st], ph ^ 1, abort, p.status)) break;
          // weights: the bf16 A tile, or the E4M3 tile the converters widen
          uint8_t* w_s = W8 ? w8_tile(st) : a_tile(st, 0, 0);
          const int half = W8 ? KSUB * A8_BYTES / 2 : A_BYTES / 2;
          const int k0 = kb * BK * KSUB;
          mbar_arrive_expect_tx(&ctrl->full[st],
                                KSUB * ((W8 ? A8_BYTES : A_BYTES) + nq * BQ_BYTES));
          if (MODE == 0) {
            tma_load_2d(w_s, &tmA0, &ctrl->full[st], k0, a_row);
            tma_load_2d(w_s + half, &tmA1, &ctrl->full[st], k0, a_row);
          } else {
            tma_load_2d(w_s, &tmA0, &ctrl->full[st], k0, a_row);
          }
#pragma unroll
          for (int j = 0; j < KSUB; ++j)
            for (int q = 0; q < nq; ++q)
              tma_load_2d(b_tile(st, j) + q * BQ_BYTES, bmap, &ctrl->full[st], k0 + j * BK,
                          b_row + q * TOKB);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t kc = 0, it = 0;
      for (int T = T0; T < total_tiles && !*abort; T += stride, ++it) {
        int seg, fb, ch;
        coord(T, seg, fb, ch);
        const int nt = min(TOK, seg_rows(p, seg) - ch * TOK);
        const uint32_t idesc = W8 ? idesc_f16_f32(BM, (nt + 15) / 16 * 16)
                                  : idesc_bf16_f32(BM, (nt + 15) / 16 * 16);
        const uint32_t buf = it & 1, use = it >> 1;
        if (!mbar_wait(&ctrl->tempty[buf], (use & 1) ^ 1, abort, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * TOK;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++kc) {
          const int st = kc % STAGES;
          const uint32_t ph = (kc / STAGES) & 1;
          constexpr int AS = A_STAGES > 0 ? A_STAGES : 1;
          const int s2 = W8 ? (int)(kc % AS) : 0;
          const uint32_t ph2 = W8 ? (kc / AS) & 1 : 0;
          // W8: the converted tile (its converters saw this stage's TMA land)
          if (!mbar_wait(W8 ? &ctrl->conv[s2] : &ctrl->full[st], W8 ? ph2 : ph, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < KSUB; ++j) {
            const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(a_tile(st, s2, j)));
            const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(b_tile(st, j)));
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              umma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | j | k) != 0);
          }
          umma_commit(&ctrl->empty[st]);
          if (W8) umma_commit(&ctrl->afree[s2]);
        }
        if (!ok) break;
        umma_commit(&ctrl->tfull[buf]);
      }
    }
  } else if (W8 && warp >= 6 && warp < 6 + CONV_WARPS) {
    // converter warps: E4M3 staging tile (128 rows x 128 codes) -> two f16
    // tiles in the 128-byte swizzled K-major layout (16-byte chunk c of row r
    // at chunk c ^ (r & 7)); 16 threads per row, 2 * CONV_WARPS rows per pass
    constexpr int ROWS_PER_PASS = 2 * CONV_WARPS;
    const int ct = threadIdx.x - 192;
    uint32_t kc = 0;
    for (int T = T0; T < total_tiles && !*abort; T += stride) {
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb, ++kc) {
        const int st = kc % STAGES;
        const uint32_t ph = (kc / STAGES) & 1;
        constexpr int AS = A_STAGES > 0 ? A_STAGES : 1;   // (bf16 weights: no converter)
        const int s2 = kc % AS;
        const uint32_t ph2 = (kc / AS) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&ctrl->full[st], ph, abort, p.status) &&
                                         mbar_wait(&ctrl->afree[s2], ph2 ^ 1, abort, p.status))) {
          ok = false;
          break;
        }
        const uint8_t* w_s = w8_tile(st);
        // 8 codes per thread and pass: chunk c16 of the row's 16, i.e. K-chunk
        // j = c16 / 8, 16-byte chunk c = c16 % 8 of the bf16 row.  All of this
        // thread's codes first (loads in flight together), then conversions
        // and swizzled stores.
        constexpr int PASSES = BM / ROWS_PER_PASS;
        const int c16 = ct & 15, j = c16 >> 3, c = c16 & 7;
        uint8_t* a_s = a_tile(st, s2, j);
        uint2 v[PASSES];
#pragma unroll
        for (int pass = 0; pass < PASSES; ++pass)
          v[pass] = *reinterpret_cast<const uint2*>(w_s + (pass * ROWS_PER_PASS + (ct >> 4)) * (BK * KSUB) +
                                                    c16 * 8);
#pragma unroll
        for (int pass = 0; pass < PASSES; ++pass) {
          const int r = pass * ROWS_PER_PASS + (ct >> 4);
          *reinterpret_cast<uint4*>(a_s + r * 128 + ((c ^ (r & 7)) << 4)) = e4m3x8_to_f16x8(v[pass]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&ctrl->conv[s2]);
      }
      if (!ok) break;
    }
  } else if (warp >= 2 && warp < 6) {
    const int q = warp & 3;                      // TMEM lanes 32q .. 32q+31 = weight rows
    uint32_t it = 0;
    for (int T = T0; T < total_tiles; T += stride, ++it) {
      if (__any_sync(0xffffffffu, *abort != 0)) break;
      int seg, fb, ch;
      coord(T, seg, fb, ch);
      const int nt = min(TOK, seg_rows(p, seg) - ch * TOK);
      const uint32_t buf = it & 1, use = it >> 1;
      const bool ok = mbar_wait(&ctrl->tfull[buf], use & 1, abort, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * TOK;
      const int row0 = p.offsets[seg] + ch * TOK;
      const int ncc = (nt + 31) / 32;
      if (MODE == 0) {
        // rows 64..127 (q = 2, 3) hold x.Wu; rows 0..63 (q = 0, 1) hold x.Wg
        // The hand-over uses two mbarriers (bounded waits), not a named
        // barrier, so a warp that gives up cannot strand the others.
        const int f = (q & 1) * 32 + lane;       // feature inside the 64-wide block
        bool xok = true;
        if (q >= 2) {
          xok = mbar_wait(&ctrl->xempty, (it & 1) ^ 1, abort, p.status);
          if (__all_sync(0xffffffffu, xok)) {
            const float su = W8 ? p.scale1[seg] : 1.f;
            for (int c = 0; c < ncc; ++c) {
              uint32_t u[32];
              tmem_ld32(taddr + c * 32, u);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) xch[f * XS + c * 32 + i] = __uint_as_float(u[i]) * su;
            }
            mbar_arrive(&ctrl->xfull);
          }
        } else {
          xok = mbar_wait(&ctrl->xfull, it & 1, abort, p.status);
        }
        if (!__all_sync(0xffffffffu, xok)) break;
        if (q < 2) {
          const int col = fb * 64 + f;
          const float sg = W8 ? p.scale0[seg] : 1.f;
          for (int c = 0; c < ncc; ++c) {
            uint32_t g[32];
            tmem_ld32(taddr + c * 32, g);
            tmem_wait_ld();
            if (col < p.n_out) {
              bool over = false;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int t = c * 32 + i;
                if (t < nt) {
                  const float h = silu_f(__uint_as_float(g[i]) * sg) * xch[f * XS + t];
                  const size_t o = (size_t)(row0 + t) * p.n_out + col;
                  if (W8) {
                    // H feeds the down GEMM as f16: a value past its range is an error
                    over |= fabsf(h) > kF16Max;
                    reinterpret_cast<__half*>(p.out)[o] = __float2half_rn(h);
                  } else {
                    p.out[o] = __float2bfloat16_rn(h);
                  }
                }
              }
              if (W8 && over) set_status(p.status, kDevBadState);
            }
          }
          mbar_arrive(&ctrl->xempty);            // the next tile may overwrite xch
        }
      } else {
        const int col = fb * BM + q * 32 + lane;
        const float sd = W8 ? p.scale0[seg] : 1.f;
        for (int c = 0; c < ncc; ++c) {
          uint32_t y[32];
          tmem_ld32(taddr + c * 32, y);
          tmem_wait_ld();
          if (col < p.n_out) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int t = c * 32 + i;
              if (t < nt) p.out[(size_t)(row0 + t) * p.n_out + col] = __float2bfloat16_rn(__uint_as_float(y[i]) * sd);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl->tempty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (!MOE_GEMM_EARLY_TRIGGER) griddep_launch_dependents();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace swp

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// 2-D bf16 (or f16) map over a row-major [rows, cols] matrix, box [box_rows, 64], 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D E4M3 map over a row-major [rows, cols] byte matrix, box [box_rows, 128]
// (whole 128-byte lines), no swizzle (the converter warps lay the f16 tiles
// out themselves).
bool make_map8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {2 * BK, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

// E4M3 path: f16 copies of the token rows the gate/up GEMM reads, so that its
// MMAs take f16 on both sides.  Routed rows keep x_perm's row indices
// (segment e's valid rows are offsets[e] .. offsets[e] + counts[e] - 1), and
// the shared experts read an f16 copy of x.  One CTA per row; the valid rows
// are numbered through a prefix sum of counts, so padding rows cost nothing.
// bf16 -> f16 is exact from 2^-14 to 65504; a finite value past 65504 is an
// error (status), as for H.  xp and xp16 may be the same buffer: a thread
// loads all of its vectors of the row, then rewrites the same 16-byte pieces.
// A row outside [0, max_rows) (inconsistent offsets and counts from a caller)
// is skipped and reported.
constexpr int kCvtThreads = 256, kCvtBatch = 4;
__global__ void __launch_bounds__(kCvtThreads)
tokens_f16_kernel(const __nv_bfloat16* xp, __half* xp16, const __nv_bfloat16* x, __half* x16,
                  const int32_t* offsets, const int32_t* counts, int E, int N, int d, int shared,
                  int64_t max_rows, int* status) {
  griddep_wait();
  __shared__ int pre[kMaxExperts + 1];
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) { pre[e] = run; run += min(max(counts[e], 0), N); }
    pre[E] = run;
  }
  __syncthreads();
  const int routed = pre[E];
  const int total = routed + (shared ? N : 0);
  const int nvec = d / 8;
  bool over = false;
  for (int i = blockIdx.x; i < total; i += gridDim.x) {
    const uint4* src;
    uint4* dst;
    if (i < routed) {
      int lo = 0, hi = E - 1;   // the last segment whose first valid row number is <= i
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= i) lo = mid; else hi = mid - 1;
      }
      const int64_t r = (int64_t)offsets[lo] + (i - pre[lo]);
      if (r < 0 || r >= max_rows) {
        if (threadIdx.x == 0) set_status(status, kDevBadState);
        continue;
      }
      src = reinterpret_cast<const uint4*>(xp + (size_t)r * d);
      dst = reinterpret_cast<uint4*>(xp16 + (size_t)r * d);
    } else {
      const size_t row = (size_t)(i - routed);
      src = reinterpret_cast<const uint4*>(x + row * d);
      dst = reinterpret_cast<uint4*>(x16 + row * d);
    }
    for (int v0 = threadIdx.x; v0 < nvec; v0 += kCvtThreads * kCvtBatch) {
      uint4 a[kCvtBatch];
#pragma unroll
      for (int u = 0; u < kCvtBatch; ++u) {
        const int v = v0 + u * kCvtThreads;
        if (v < nvec) a[u] = src[v];
      }
#pragma unroll
      for (int u = 0; u < kCvtBatch; ++u) {
        const int v = v0 + u * kCvtThreads;
        if (v >= nvec) continue;
        const uint32_t in[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&in[j]));
          over |= (isfinite(f.x) && fabsf(f.x) > swp::kF16Max) ||
                  (isfinite(f.y) && fabsf(f.y) > swp::kF16Max);
          const __half2 h = __floats2half2_rn(f.x, f.y);
          out[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        dst[v] = make_uint4(out[0], out[1], out[2], out[3]);
      }
    }
  }
  if (over) set_status(status, kDevBadState);
  griddep_launch_dependents();
}

// Swap-AB (weights as the M operand) when experts see few tokens: decode-sized
// batches, where 128-row token tiles would be mostly padding.  E4M3 weights
// always take this kernel (it handles any number of tokens per expert).
bool use_swap(const FfnParams& p) {
  if (p.w_scales) return true;
  if (!p.counts) return false;
  if ((int64_t)p.N * p.k > 64LL * p.E) return false;
  return p.S == 0 || p.N <= 512;
}

template <bool W8>
cudaError_t launch_swap(const FfnParams& p, cudaStream_t s, cudaEvent_t mid) {
  constexpr size_t SMEM = swp::smem_bytes<W8>();
  constexpr int THREADS = swp::Shape<W8>::THREADS;
  cudaError_t err = cudaFuncSetAttribute(swp::ffn_tc_swap_kernel<0, W8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(swp::ffn_tc_swap_kernel<1, W8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM);
  if (err != cudaSuccess) return err;
  const int ET = p.E + p.S;
  auto wmap = [&](CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box) {
    return W8 ? make_map8(m, base, rows, cols, box) : make_map(m, base, rows, cols, box);
  };
  // E4M3 weights: the MMAs take f16 tokens (f16 copies made here) and f16 H
  const CUtensorMapDataType tdt = W8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const void* tok = W8 ? p.tok16 : p.x_perm;
  const void* xs = W8 ? p.x16 : p.x;
  if (W8) {
    if (!p.tok16 || !p.x16) return cudaErrorInvalidValue;
    const int64_t rows = (int64_t)p.N * p.k + (p.S > 0 ? p.N : 0);
    int grid = (int)std::min<int64_t>(rows, 8LL * p.num_sms);
    if (grid < 1) grid = 1;
    if ((err = launch_chained(tokens_f16_kernel, grid, kCvtThreads, 0, s,
                              static_cast<const __nv_bfloat16*>(p.x_perm), static_cast<__half*>(p.tok16),
                              static_cast<const __nv_bfloat16*>(p.x), static_cast<__half*>(p.x16),
                              p.offsets, p.counts, p.E, p.N, p.d, p.S > 0 ? 1 : 0,
                              p.max_rows, p.status)) !=
        cudaSuccess)
      return err;
    count_launch();
  }
  CUtensorMap b0, b1, a0, a1;
  if (!make_map(&b0, tok, (uint64_t)p.max_rows, p.d, swp::TOKB, tdt) ||
      !make_map(&b1, xs, (uint64_t)p.N, p.d, swp::TOKB, tdt) ||
      !wmap(&a0, p.w_gate, (uint64_t)ET * p.F, p.d, swp::BM / 2) ||
      !wmap(&a1, p.w_up, (uint64_t)ET * p.F, p.d, swp::BM / 2))
    return cudaErrorInvalidValue;
  swp::Params t1{p.E, p.S, p.N, p.d, p.F, (p.F + 63) / 64, p.offsets, p.counts,
                 static_cast<__nv_bfloat16*>(p.h), p.status,
                 W8 ? p.w_scales : nullptr, W8 ? p.w_scales + ET : nullptr};
  if ((err = launch_chained(swp::ffn_tc_swap_kernel<0, W8>, p.num_sms, THREADS, SMEM, s, b0, b1,
                            a0, a1, t1)) != cudaSuccess)
    return err;
  count_launch();
  if (mid) cudaEventRecord(mid, s);
  if (!make_map(&b0, p.h, (uint64_t)p.max_total_rows, p.F, swp::TOKB, tdt) ||
      !wmap(&a0, p.w_down, (uint64_t)ET * p.d, p.F, swp::BM))
    return cudaErrorInvalidValue;
  swp::Params t2{p.E, p.S, p.N, p.F, p.d, (p.d + swp::BM - 1) / swp::BM, p.offsets, p.counts,
                 static_cast<__nv_bfloat16*>(p.y_perm), p.status,
                 W8 ? p.w_scales + 2 * ET : nullptr, nullptr};
  if ((err = launch_chained(swp::ffn_tc_swap_kernel<1, W8>, p.num_sms, THREADS, SMEM, s, b0, b0,
                            a0, a0, t2)) != cudaSuccess)
    return err;
  count_launch();
  return cudaSuccess;
}

}  // namespace

namespace {

template <class C>
cudaError_t launch_prefill(const FfnParams& p, cudaStream_t s, cudaEvent_t mid) {
  constexpr int BN = C::BN;
  cudaError_t err = cudaFuncSetAttribute(ffn_tc_kernel<0, C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(ffn_tc_kernel<1, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const int ET = p.E + p.S;
  CUtensorMap a0, a1, b0, b1;
  // GEMM-1: A = x_perm (routed) / x (shared), B = gate and up weights
  if (!make_map(&a0, p.x_perm, (uint64_t)p.max_rows, p.d, BM) ||
      !make_map(&a1, p.x, (uint64_t)p.N, p.d, BM) ||
      !make_map(&b0, p.w_gate, (uint64_t)ET * p.F, p.d, BN / 2) ||
      !make_map(&b1, p.w_up, (uint64_t)ET * p.F, p.d, BN / 2))
    return cudaErrorInvalidValue;
  TcParams t1{p.E, p.S, p.d, p.F, (p.F + BN / 2 - 1) / (BN / 2), BN / 2, p.offsets,
              static_cast<__nv_bfloat16*>(p.h), p.status, p.tile_ctr};
  if ((err = launch_chained(ffn_tc_kernel<0, C>, p.num_sms, NUM_THREADS, C::SMEM_BYTES, s, a0, a1,
                            b0, b1, t1)) != cudaSuccess)
    return err;
  count_launch();
  if (mid) cudaEventRecord(mid, s);
  // GEMM-2: A = H, B = down weights
  if (!make_map(&a0, p.h, (uint64_t)p.max_total_rows, p.F, BM) ||
      !make_map(&b0, p.w_down, (uint64_t)ET * p.d, p.F, BN))
    return cudaErrorInvalidValue;
  // GEMM-2's tiles cost the same whatever the segment (no SwiGLU, weights
  // shared by every row tile of a segment): the static deal measured faster
  TcParams t2{p.E, p.S, p.F, p.d, (p.d + BN - 1) / BN, BN, p.offsets,
              static_cast<__nv_bfloat16*>(p.y_perm), p.status, nullptr};
  if ((err = launch_chained(ffn_tc_kernel<1, C>, p.num_sms, NUM_THREADS, C::SMEM_BYTES, s, a0, a0,
                            b0, b0, t2)) != cudaSuccess)
    return err;
  count_launch();
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_ffn_tc(const FfnParams& p, cudaStream_t s, cudaEvent_t mid) {
  cudaError_t err = get_encoder();
  if (err != cudaSuccess) return err;
  if (p.w_scales) return launch_swap<true>(p, s, mid);
  if (use_swap(p)) return launch_swap<false>(p, s, mid);
  return launch_prefill<Prefill>(p, s, mid);
}

}  // namespace moe
