// Router contraction for bf16 on the tensor cores: partial logits
//   part[ks][t][e] = sum_{j in K-slice ks} x[t,j] * W_r[e,j]
// («为什么MoE有效？稀疏激活的数学直觉与工程实践» §2.2: the router is a bias-free
// linear map d_model -> n_experts).
//
// One CTA per (128-token tile, K slice): TMA streams 128x64 tiles of x and
// E_pad x 64 tiles of W_r (E padded to a multiple of 16, rows past E read as
// zeros) through a 4-stage ring; one thread issues tcgen05.mma (M=128,
// N=E_pad, K=16); successive 64-deep K blocks rotate over up to 8 TMEM
// accumulators so each fp32 accumulation stays a few MMAs long; four epilogue
// warps add the accumulators (compensated fp32) and store fp32 partials.  Splitting K
// keeps >= 2 CTAs per SM busy even for decode-sized batches; the reduce kernel
// sums the slices (compensated fp32, in slice order), so the logits stay within ~1e-7
// of the exact value and the top-k matches an exact evaluation except on
// genuine near-ties.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int BM = 128, BK = 64, STAGES = 4, NUM_THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full;
  uint64_t staged;               // the four epilogue warps have written their rows
  uint32_t tmem_base;
  int abort;
};

size_t smem_bytes(int e_pad) { return 1024 + (size_t)STAGES * (A_BYTES + e_pad * BK * 2) + sizeof(Ctrl); }

struct Params {
  int N, E, d, e_pad, k_slice, tmem_cols, acc_cols, nacc;
  float* part;
  int* status;
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
route_logits_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                Params p) {
  griddep_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int b_bytes = p.e_pad * BK * 2;
  const int stage_bytes = A_BYTES + b_bytes;           // a multiple of 1024 (e_pad % 16 == 0)
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + (size_t)STAGES * stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * BM;
  const int ks = blockIdx.y;
  const int k_begin = ks * p.k_slice;
  const int k_end = min(p.d, k_begin + p.k_slice);
  const int KB = (k_end - k_begin + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&ctrl->full[s], 1); mbar_init(&ctrl->empty[s], 1); }
    mbar_init(&ctrl->acc_full, 1);
    mbar_init(&ctrl->staged, 128);
    ctrl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) { tma_prefetch_desc(&tmX); tma_prefetch_desc(&tmW); }
  if (warp == 1) { tmem_alloc(&ctrl->tmem_base, p.tmem_cols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  volatile int* abort = &ctrl->abort;

  if (warp == 0) {
    if (lane == 0) {
      for (int kb = 0; kb < KB; ++kb) {
        const int st = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        if (!mbar_wait(&ctrl->empty[st], ph ^ 1, abort, p.status)) break;
        uint8_t* a_s = smem + (size_t)st * stage_bytes;
        mbar_arrive_expect_tx(&ctrl->full[st], stage_bytes);
        tma_load_2d(a_s, &tmX, &ctrl->full[st], k_begin + kb * BK, t0);
        tma_load_2d(a_s + A_BYTES, &tmW, &ctrl->full[st], k_begin + kb * BK, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, p.e_pad);
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        const int st = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        if (!mbar_wait(&ctrl->full[st], ph, abort, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + (size_t)st * stage_bytes);
        const uint64_t adesc = sdesc_kmajor_sw128(a_addr);
        const uint64_t bdesc = sdesc_kmajor_sw128(a_addr + A_BYTES);
        // K blocks rotate over nacc accumulators: each fp32 accumulation stays short
        const uint32_t d = tmem + (uint32_t)((kb % p.nacc) * p.acc_cols);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          umma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, (kb >= p.nacc) || k != 0);
        umma_commit(&ctrl->empty[st]);
      }
      if (ok) umma_commit(&ctrl->acc_full);
    }
  } else {
    const int q = warp & 3;
    const bool ok = mbar_wait(&ctrl->acc_full, 0, abort, p.status);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      // the tile's logits go through shared memory (the ring is idle once the
      // last MMA has completed): a thread per token row writes its row there,
      // then the four warps store the tile's contiguous rows coalesced
      // (scattered 4-byte stores of each row cost about 4 us per tile)
      const int ES = p.E + 1;
      float* stage = reinterpret_cast<float*>(smem);   // [128][E + 1]
      const int row = q * 32 + lane;
      const int used = KB < p.nacc ? KB : p.nacc;
      for (int c = 0; c < p.acc_cols / 32; ++c) {
        KahanF acc[32];
        for (int a = 0; a < used; ++a) {
          uint32_t r[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * p.acc_cols + c * 32), r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i].add(__uint_as_float(r[i]));
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c * 32 + i < p.E) stage[row * ES + c * 32 + i] = acc[i].s;
      }
      // a bounded hand-off (an mbarrier, not a named barrier): a warp that
      // gave up earlier cannot leave the others waiting for ever
      mbar_arrive(&ctrl->staged);
      const bool staged = mbar_wait(&ctrl->staged, 0, abort, p.status);
      const int rows = staged ? min(BM, p.N - t0) : 0, n_all = rows * p.E;
      float* dst = p.part + ((size_t)ks * p.N + t0) * p.E;
      const int et = threadIdx.x - 64;                 // 0 .. 127
      const int de = 128 % p.E, dr = 128 / p.E;
      int cc = et % p.E, rr = et / p.E;
      for (int i = et; i < n_all; i += 128) {
        dst[i] = stage[rr * ES + cc];
        cc += de;
        rr += dr;
        if (cc >= p.E) { cc -= p.E; ++rr; }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

bool encode(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  std::call_once(g_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_route_logits_tc(const RouteSplit& s, const void* x, const void* w_router,
                                   int N, int E, int d, float* part, int* status,
                                   cudaStream_t stream) {
  CUtensorMap mx, mw;
  const int e_pad = (E + 15) / 16 * 16;
  if (!encode(&mx, x, (uint64_t)N, (uint64_t)d, BM) ||
      !encode(&mw, w_router, (uint64_t)E, (uint64_t)d, (uint32_t)e_pad))
    return cudaErrorInvalidValue;
  // at most 256 TMEM columns per CTA, so two CTAs can share an SM
  const int acc_cols = (e_pad + 31) / 32 * 32;
  const int nacc = 256 / acc_cols < 1 ? 1 : (256 / acc_cols < 8 ? 256 / acc_cols : 8);
  int cols = 32;
  while (cols < nacc * acc_cols) cols <<= 1;
  Params p{N, E, d, e_pad, s.k_slice, cols, acc_cols, nacc, part, status};
  const size_t smem = smem_bytes(e_pad);
  cudaError_t err = cudaFuncSetAttribute(route_logits_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((N + BM - 1) / BM, s.ks);
  if ((err = launch_chained(route_logits_tc, grid, NUM_THREADS, smem, stream, mx, mw, p)) !=
      cudaSuccess)
    return err;
  count_launch();
  return cudaSuccess;
}

}  // namespace moe
