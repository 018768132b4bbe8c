// FP8 E4M3 expert weights: the quantiser behind moe_quantize_fp8.
//
// «大模型MoE架构揭秘：如何用2%参数实现万亿级算力调度» §5.4 and «GPT-4 Has 1.8
// Trillion Parameters...» §4.4: expert weights kept in low precision with
// per-expert scales while the router stays in high precision.  One fp32 scale
// per expert matrix: scale = amax / 448 (the largest finite E4M3 value; 1 for
// an all-zero matrix); code = round-to-nearest-even of the fp32 quotient
// w / scale, saturated to +-448.
//
// Three launches: |w| maximum per matrix (exact, so the atomics are
// order-independent), the codes, then amax -> scale in place.
#include <algorithm>

#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kQThreads = 256;

__global__ void __launch_bounds__(kQThreads) amax_kernel(const uint4* w, int64_t nvec, unsigned* amax_bits) {
  const int m = blockIdx.y;
  const uint4* src = w + (size_t)m * nvec;
  float mx = 0.f;
  for (int64_t i = (int64_t)blockIdx.x * kQThreads + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * kQThreads) {
    const uint4 u = src[i];
    const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(v[j])), fabsf(bf16_hi(v[j]))));
  }
  mx = warp_max(mx);
  __shared__ float red[kQThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < kQThreads / 32; ++i) mx = fmaxf(mx, red[i]);
    // non-negative floats order like their bit patterns
    atomicMax(&amax_bits[m], __float_as_uint(mx));
  }
}

__device__ __forceinline__ float scale_of(unsigned amax_bits) {
  const float amax = __uint_as_float(amax_bits);
  return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

__global__ void __launch_bounds__(kQThreads) quantize_kernel(const uint4* w, int64_t nvec,
                                                            const unsigned* amax_bits, uint2* q) {
  const int m = blockIdx.y;
  const float scale = scale_of(amax_bits[m]);
  const uint4* src = w + (size_t)m * nvec;
  uint2* dst = q + (size_t)m * nvec;
  for (int64_t i = (int64_t)blockIdx.x * kQThreads + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * kQThreads) {
    const uint4 u = src[i];
    const uint32_t v[4] = {u.x, u.y, u.z, u.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = make_float2(__fdiv_rn(bf16_lo(v[j]), scale), __fdiv_rn(bf16_hi(v[j]), scale));
      const uint32_t pair = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      out[j >> 1] |= pair << (16 * (j & 1));
    }
    dst[i] = make_uint2(out[0], out[1]);
  }
}

__global__ void scale_kernel(float* scales, int n_mat) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m < n_mat) scales[m] = scale_of(__float_as_uint(scales[m]));
}

}  // namespace

cudaError_t launch_quantize_fp8(const void* w, int n_mat, int64_t per_mat, uint8_t* q, float* scales,
                                int num_sms, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(scales, 0, sizeof(float) * (size_t)n_mat, s);
  if (err != cudaSuccess) return err;
  const int64_t nvec = per_mat / 8;
  const int64_t want = (nvec + kQThreads - 1) / kQThreads;
  // about 8 CTAs per SM over all matrices
  const int bx = (int)std::max<int64_t>(1, std::min<int64_t>(want, (8LL * num_sms + n_mat - 1) / n_mat));
  const dim3 grid(bx, n_mat);
  unsigned* amax_bits = reinterpret_cast<unsigned*>(scales);
  amax_kernel<<<grid, kQThreads, 0, s>>>(static_cast<const uint4*>(w), nvec, amax_bits);
  count_launch();
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  quantize_kernel<<<grid, kQThreads, 0, s>>>(static_cast<const uint4*>(w), nvec, amax_bits,
                                             reinterpret_cast<uint2*>(q));
  count_launch();
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  scale_kernel<<<(n_mat + 255) / 256, 256, 0, s>>>(scales, n_mat);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
