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
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int BM = 128, BK = 64, BN = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem_base;
  int abort;
  int total_mtiles;
  int pad;
  int mt_prefix[kMaxExperts + 16];
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(Ctrl);

struct TcParams {
  int E, S, K, n_out, n_tiles_n, bn_out;  // bn_out: output columns per tile (128 or 256)
  const int32_t* offsets;
  __nv_bfloat16* out;
  int* status;
};

struct TileCoord {
  int seg, m, n;
};

__device__ __forceinline__ TileCoord tile_coord(const Ctrl* c, int nseg, int n_tiles_n, int T) {
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

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
ffn_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
              const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
              TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nseg = p.E + p.S;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&ctrl->full[s], 1); mbar_init(&ctrl->empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&ctrl->tfull[b], 1); mbar_init(&ctrl->tempty[b], 128); }
    ctrl->abort = 0;
    int run = 0;
    for (int s = 0; s < nseg; ++s) {
      ctrl->mt_prefix[s] = run;
      run += (p.offsets[s + 1] - p.offsets[s]) / BM;
    }
    ctrl->mt_prefix[nseg] = run;
    ctrl->total_mtiles = run;
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

  if (warp == 0) {
    if (lane == 0) {
      uint32_t kc = 0;
      for (int T = blockIdx.x; T < total_tiles && !*abort; T += gridDim.x) {
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
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t kc = 0, it = 0;
      for (int T = blockIdx.x; T < total_tiles && !*abort; T += gridDim.x, ++it) {
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
    uint32_t it = 0;
    for (int T = blockIdx.x; T < total_tiles; T += gridDim.x, ++it) {
      if (__any_sync(0xffffffffu, *abort != 0)) break;
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
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + 128 + c * 32, u);
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
        for (int c = 0; c < 8; ++c) {
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
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

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

// 2-D bf16 map over a row-major [rows, cols] matrix, box [box_rows, 64], 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_ffn_tc(const FfnParams& p, cudaStream_t s, cudaEvent_t mid) {
  cudaError_t err = get_encoder();
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(ffn_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(ffn_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
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
              static_cast<__nv_bfloat16*>(p.h), p.status};
  ffn_tc_kernel<0><<<p.num_sms, NUM_THREADS, SMEM_BYTES, s>>>(a0, a1, b0, b1, t1);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (mid) cudaEventRecord(mid, s);
  // GEMM-2: A = H, B = down weights
  if (!make_map(&a0, p.h, (uint64_t)p.max_total_rows, p.F, BM) ||
      !make_map(&b0, p.w_down, (uint64_t)ET * p.d, p.F, BN))
    return cudaErrorInvalidValue;
  TcParams t2{p.E, p.S, p.F, p.d, (p.d + BN - 1) / BN, BN, p.offsets,
              static_cast<__nv_bfloat16*>(p.y_perm), p.status};
  ffn_tc_kernel<1><<<p.num_sms, NUM_THREADS, SMEM_BYTES, s>>>(a0, a0, b0, b0, t2);
  return cudaGetLastError();
}

}  // namespace moe
