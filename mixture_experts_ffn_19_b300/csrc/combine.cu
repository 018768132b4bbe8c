// Combine: y[t] = sum_s shared_s(x_t) + sum_j g_tj * expert_{e_tj}(x_t).
//
// «为什么MoE有效？稀疏激活的数学直觉与工程实践» §2.1 (y = sum_i g_i(x) Expert_i(x))
// and §3 code (output[token_indices] += w * expert_output); «DeepSeek-V2 ...»
// summary §2.3 (layer output = shared-expert output + gated routed output).
//
// A gather, not a scatter: each token reads its own k + S rows of y_perm and
// sums them in fp32 in a fixed order (shared experts, then slots 0..k-1), so
// the result is deterministic without atomics.  One CTA per token, 16-byte
// vectors across d.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

template <typename T>
struct Vec;  // 16 bytes of T as fp32 lanes

template <>
struct Vec<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void load(const uint4& u, float (&f)[8]) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
  }
  __device__ static uint4 store(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
};

template <>
struct Vec<float> {
  static constexpr int n = 4;
  __device__ static void load(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 store(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// VPT 16-byte vectors per thread, loaded for RG rows at a time before any
// FMA.  With short rows and few rows per token (the 64-expert layer: 256
// vectors, 2 rows) two vectors per thread halve the CTA, so twice the tokens,
// and their row bytes, are in flight per SM: 53 -> 41 us there.  With long
// rows or many rows per token (8 rows of 640 vectors) the CTA already keeps
// enough in flight and the smaller row groups only add latency.
//
// SPLIT (small batches): gridDim.y CTAs share a token's row, CTA y taking the
// y-th range of its vectors in one pass, so a few tokens still keep enough row
// bytes in flight (DeepSeek-V2 decode: 32 tokens of 8 rows x 640 vectors,
// 12.2 -> 8.1 us).
template <typename T, int VPT, bool SPLIT>
__global__ void __launch_bounds__(256) combine_kernel(CombineParams p) {
  griddep_begin();
  constexpr int VN = Vec<T>::n, RG = VPT >= 4 ? 2 : 4 / VPT;
  const int t = blockIdx.x;
  __shared__ int rows[kMaxTopk + 8];
  __shared__ float gates[kMaxTopk + 8];
  __shared__ int nrows;
  if (threadIdx.x < 32) {
    // lane i < S + k fetches contribution i (shared experts, then slots in
    // order) in parallel; the kept ones are packed in that order
    const int lane = threadIdx.x, nr = p.S + p.k;
    int row = -1;
    float g = 0.f;
    if (lane < p.S) {
      row = p.offsets[p.E + lane] + t;
      g = 1.f;
    } else if (lane < nr) {
      const size_t a = (size_t)t * p.k + (lane - p.S);
      if (p.final_idx[a] >= 0) { row = p.pos[a]; g = p.topk_w[a]; }
    }
    const unsigned kept = __ballot_sync(0xffffffffu, row >= 0);
    if (row >= 0) {
      const int at = __popc(kept & lanemask_lt());
      rows[at] = row;
      gates[at] = g;
    }
    if (lane == 0) nrows = __popc(kept);
  }
  __syncthreads();
  const int nvec = p.d / VN, nt = blockDim.x;
  const uint4* src = static_cast<const uint4*>(p.y_perm);
  uint4* dst = static_cast<uint4*>(p.y);
  const int n = nrows;
  const int per = SPLIT ? (nvec + gridDim.y - 1) / gridDim.y : nvec;
  const int vb = SPLIT ? blockIdx.y * per : 0;
  const int ve = SPLIT ? min(nvec, vb + per) : nvec;
  for (int v0 = vb + threadIdx.x; v0 < ve; v0 += nt * VPT) {
    float acc[VPT][VN];
#pragma unroll
    for (int b = 0; b < VPT; ++b)
#pragma unroll
      for (int q = 0; q < VN; ++q) acc[b][q] = 0.f;
    // rows in groups of RG: the loads of a group (all VPT vectors) are issued
    // before its FMAs
    for (int r0 = 0; r0 < n; r0 += RG) {
      uint4 u[RG][VPT];
#pragma unroll
      for (int i = 0; i < RG; ++i)
#pragma unroll
        for (int b = 0; b < VPT; ++b)
          if (r0 + i < n && v0 + b * nt < ve) u[i][b] = src[(size_t)rows[r0 + i] * nvec + v0 + b * nt];
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        if (r0 + i < n) {
          const float g = gates[r0 + i];
#pragma unroll
          for (int b = 0; b < VPT; ++b) {
            if (v0 + b * nt < ve) {
              float f[VN];
              Vec<T>::load(u[i][b], f);
#pragma unroll
              for (int q = 0; q < VN; ++q) acc[b][q] = fmaf(g, f[q], acc[b][q]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < VPT; ++b)
      if (v0 + b * nt < ve) dst[(size_t)t * nvec + v0 + b * nt] = Vec<T>::store(acc[b]);
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, bool bf16, cudaStream_t s) {
  const int vn = bf16 ? 8 : 4;
  const int nvec = p.d / vn;
  const int vpt = (nvec >= 128 && nvec <= 256 && p.S + p.k <= 4) ? 2 : 1;
  const int per = (nvec + vpt - 1) / vpt;
  const int threads = per < 256 ? ((per + 31) / 32) * 32 : 256;
  const int split = p.N < 1024 ? (nvec + threads * vpt - 1) / (threads * vpt) : 1;
  cudaError_t err;
  if (split > 1) {
    const dim3 grid(p.N, split);
    err = bf16 ? launch_chained(combine_kernel<__nv_bfloat16, 1, true>, grid, threads, 0, s, p)
               : launch_chained(combine_kernel<float, 1, true>, grid, threads, 0, s, p);
  } else if (vpt == 2) {
    err = bf16 ? launch_chained(combine_kernel<__nv_bfloat16, 2, false>, p.N, threads, 0, s, p)
               : launch_chained(combine_kernel<float, 2, false>, p.N, threads, 0, s, p);
  } else {
    err = bf16 ? launch_chained(combine_kernel<__nv_bfloat16, 1, false>, p.N, threads, 0, s, p)
               : launch_chained(combine_kernel<float, 1, false>, p.N, threads, 0, s, p);
  }
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

}  // namespace moe
