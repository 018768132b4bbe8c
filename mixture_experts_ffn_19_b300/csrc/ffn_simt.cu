// Expert FFNs in fp32 on the CUDA cores (dtype MOE_F32).
//
// Experts as in «为什么MoE有效？稀疏激活的数学直觉与工程实践» §3 code
// (Linear(d, d_ff) -> GELU -> Linear(d_ff, d), with biases) or the SwiGLU form
// of «大模型MoE架构揭秘：如何用2%参数实现万亿级算力调度» §3.2.
//
// fp32 is kept end to end (no TF32): the tensor cores' TF32 mode carries a
// 10-bit mantissa, too coarse for a 1e-4 relative tolerance.  Each CTA owns a
// 64 x 64 output tile of one segment (segments are 128-row aligned, so a tile
// never straddles two experts); the segment is found from `offsets` on the
// device, so the host never needs the routed counts.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kBM = 64, kBN = 64, kBK = 32, kPad = 4;

__device__ __forceinline__ float gelu_erf(float a) {
  return 0.5f * a * (1.f + erff(a * 0.70710678118654752f));
}
__device__ __forceinline__ float silu(float a) { return a / (1.f + expf(-a)); }

// Find the segment containing row r (offsets ascending, nseg+1 entries).
__device__ int find_segment(const int32_t* offsets, int nseg, int r) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// STAGE 1: H = act(A W1^T + b1)   (or silu(A Wg^T) * (A Wu^T))
// STAGE 2: Y = H W2^T + b2
template <int STAGE, bool SWIGLU>
__global__ void __launch_bounds__(256) ffn_simt_kernel(FfnParams p) {
  griddep_begin();
  __shared__ __align__(16) float As[kBK][kBM + kPad];
  __shared__ __align__(16) float Bs[kBK][kBN + kPad];
  __shared__ __align__(16) float Us[SWIGLU && STAGE == 1 ? kBK : 1][kBN + kPad];
  __shared__ int s_seg;
  const int nseg = p.E + p.S;
  const int row0 = blockIdx.x * kBM;
  if (threadIdx.x == 0) s_seg = (row0 < p.offsets[nseg]) ? find_segment(p.offsets, nseg, row0) : -1;
  __syncthreads();
  const int seg = s_seg;
  if (seg < 0) return;
  const int n0 = blockIdx.y * kBN;
  const int K = (STAGE == 1) ? p.d : p.F;
  const int NO = (STAGE == 1) ? p.F : p.d;   // output width
  const float* W = static_cast<const float*>(STAGE == 1 ? p.w_gate : p.w_down) + (size_t)seg * NO * K;
  const float* U = SWIGLU && STAGE == 1 ? static_cast<const float*>(p.w_up) + (size_t)seg * NO * K : nullptr;
  // A rows: routed -> x_perm, shared -> x (token = row - segment start), H for stage 2
  const bool shared = seg >= p.E;
  const float* A;
  int a_row0, a_rows;
  if (STAGE == 2) { A = static_cast<const float*>(p.h); a_row0 = row0; a_rows = INT32_MAX; }
  else if (shared) { A = static_cast<const float*>(p.x); a_row0 = row0 - p.offsets[seg]; a_rows = p.N; }
  else { A = static_cast<const float*>(p.x_perm); a_row0 = row0; a_rows = INT32_MAX; }

  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  float acc[4][4], accu[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = accu[i][j] = 0.f;

  // loader: rows lr and lr + 32, k offset lk (4 floats); the next K step's
  // tiles are loaded into registers while the current one is computed
  const int lr = tid >> 3, lk = (tid & 7) * 4;
  float4 ra[2], rb[2], ru[2];
  auto load = [&](int k0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = lr + 32 * h, ar = a_row0 + r;
      const bool kin = k0 + lk < K;
      ra[h] = (ar < a_rows && kin) ? *reinterpret_cast<const float4*>(A + (size_t)ar * K + k0 + lk)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
      rb[h] = (n0 + r < NO && kin) ? *reinterpret_cast<const float4*>(W + (size_t)(n0 + r) * K + k0 + lk)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
      if (SWIGLU && STAGE == 1)
        ru[h] = (n0 + r < NO && kin) ? *reinterpret_cast<const float4*>(U + (size_t)(n0 + r) * K + k0 + lk)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load(0);
  for (int k0 = 0; k0 < K; k0 += kBK) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = lr + 32 * h;
      As[lk + 0][r] = ra[h].x; As[lk + 1][r] = ra[h].y; As[lk + 2][r] = ra[h].z; As[lk + 3][r] = ra[h].w;
      Bs[lk + 0][r] = rb[h].x; Bs[lk + 1][r] = rb[h].y; Bs[lk + 2][r] = rb[h].z; Bs[lk + 3][r] = rb[h].w;
      if (SWIGLU && STAGE == 1) {
        Us[lk + 0][r] = ru[h].x; Us[lk + 1][r] = ru[h].y; Us[lk + 2][r] = ru[h].z; Us[lk + 3][r] = ru[h].w;
      }
    }
    __syncthreads();
    if (k0 + kBK < K) load(k0 + kBK);
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      if (SWIGLU && STAGE == 1) {
        const float4 u = *reinterpret_cast<const float4*>(&Us[kk][tx * 4]);
        const float uv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) accu[i][j] = fmaf(av[i], uv[j], accu[i][j]);
      }
    }
    __syncthreads();
  }
  const float* bias = nullptr;
  if (STAGE == 1 && p.b1) bias = static_cast<const float*>(p.b1) + (size_t)seg * NO;
  if (STAGE == 2 && p.b2) bias = static_cast<const float*>(p.b2) + (size_t)seg * NO;
  float* out = static_cast<float*>(STAGE == 1 ? p.h : p.y_perm);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + tx * 4 + j;
      if (c >= NO) continue;
      float v = acc[i][j] + (bias ? bias[c] : 0.f);
      if (STAGE == 1) v = SWIGLU ? silu(acc[i][j]) * accu[i][j] : gelu_erf(v);
      out[(size_t)r * NO + c] = v;
    }
  }
}

}  // namespace

cudaError_t launch_ffn_simt(const FfnParams& p, cudaStream_t s, cudaEvent_t mid) {
  const int mt = (int)((p.max_total_rows + kBM - 1) / kBM);
  dim3 g1(mt, (p.F + kBN - 1) / kBN), g2(mt, (p.d + kBN - 1) / kBN);
  cudaError_t err = p.act == 1 ? launch_chained(ffn_simt_kernel<1, true>, g1, 256, 0, s, p)
                                : launch_chained(ffn_simt_kernel<1, false>, g1, 256, 0, s, p);
  if (err != cudaSuccess) return err;
  count_launch();
  if (mid) cudaEventRecord(mid, s);
  if ((err = launch_chained(ffn_simt_kernel<2, false>, g2, 256, 0, s, p)) != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

}  // namespace moe
