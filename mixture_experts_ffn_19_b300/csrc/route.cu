// Router: logits z = x W_r^T (+ b), fp32 softmax, top-k with renormalised
// gates, and the per-CTA partial sums of the load-balance statistics.
//
// «为什么MoE有效？稀疏激活的数学直觉与工程实践» §2.2 (router = bias-free linear
// map, softmax, torch.topk, renormalise); «DeepSeek-V2 ...» summary §2.2
// (expert_bias added to the logits before the softmax; load_balance_loss).
//
// One CTA owns 32 tokens.  The contraction is tiled through shared memory
// (64-wide K chunks, fp32 FMA, each K chunk summed separately and folded into
// the running sum with Kahan compensation so the logits stay within ~1e-7 of
// the exact value: top-k decisions then only differ from an exact evaluation
// on genuine near-ties).  The epilogue is warp-per-token: softmax with warp
// shuffles, then k rounds of a shuffle arg-max (ties to the lower expert).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kTM = kRouteTM;   // tokens per CTA
constexpr int kKC = 64;         // K chunk
constexpr int kXS = kKC + 4;    // padded smem row (floats), 16-byte aligned rows
constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ void load8(const T* src, float (&v)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* src, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(src);
  v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}
template <>
__device__ __forceinline__ void load8<float>(const float* src, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(src)[0];
  const float4 b = reinterpret_cast<const float4*>(src)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// EJ = experts per thread column group = ceil(E / 32).
template <typename T, int EJ>
__global__ void __launch_bounds__(kThreads) route_kernel(RouteParams p) {
  extern __shared__ __align__(16) float sm[];
  const int E = p.E, d = p.d, k = p.k, N = p.N;
  const int EP = EJ * 32;                        // padded expert rows
  float* xs = sm;                                // [kTM][kXS]
  float* ws = xs + kTM * kXS;                    // [EP][kXS]
  float* lg = ws + EP * kXS;                     // [kTM][EP+1] logits, then probabilities
  int* picks_s = reinterpret_cast<int*>(lg + kTM * (EP + 1));   // [EP]

  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kTM;
  const T* x = static_cast<const T*>(p.x);
  const T* wr = static_cast<const T*>(p.w_router);

  const int tx = tid & 7;      // tokens tx, tx+8, tx+16, tx+24
  const int ty = tid >> 3;     // experts ty, ty+32, ...

  float sum[4][EJ], cmp[4][EJ];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EJ; ++j) sum[i][j] = cmp[i][j] = 0.f;

  for (int k0 = 0; k0 < d; k0 += kKC) {
    // stage x tile [kTM][kKC] and W tile [EP][kKC] as fp32 (zero outside)
    for (int v = tid; v < kTM * (kKC / 8); v += kThreads) {
      const int r = v / (kKC / 8), c = (v % (kKC / 8)) * 8;
      float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (t0 + r < N && k0 + c < d) load8<T>(x + (size_t)(t0 + r) * d + k0 + c, f);
#pragma unroll
      for (int q = 0; q < 8; ++q) xs[r * kXS + c + q] = f[q];
    }
    for (int v = tid; v < EP * (kKC / 8); v += kThreads) {
      const int r = v / (kKC / 8), c = (v % (kKC / 8)) * 8;
      float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (r < E && k0 + c < d) load8<T>(wr + (size_t)r * d + k0 + c, f);
#pragma unroll
      for (int q = 0; q < 8; ++q) ws[r * kXS + c + q] = f[q];
    }
    __syncthreads();
    float acc[4][EJ];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < EJ; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < kKC; kk += 4) {
      float4 xv[4], wv[EJ];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        xv[i] = *reinterpret_cast<const float4*>(&xs[(tx + 8 * i) * kXS + kk]);
#pragma unroll
      for (int j = 0; j < EJ; ++j)
        wv[j] = *reinterpret_cast<const float4*>(&ws[(ty + 32 * j) * kXS + kk]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < EJ; ++j) {
          float a = acc[i][j];
          a = fmaf(xv[i].x, wv[j].x, a);
          a = fmaf(xv[i].y, wv[j].y, a);
          a = fmaf(xv[i].z, wv[j].z, a);
          a = fmaf(xv[i].w, wv[j].w, a);
          acc[i][j] = a;
        }
    }
    // fold the chunk into the running sum with Kahan compensation
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < EJ; ++j) {
        const float y = acc[i][j] - cmp[i][j];
        const float t = sum[i][j] + y;
        cmp[i][j] = (t - sum[i][j]) - y;
        sum[i][j] = t;
      }
    __syncthreads();
  }

  // logits (+ bias) -> smem
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
      const int e = ty + 32 * j;
      if (e < E) lg[(tx + 8 * i) * (EP + 1) + e] = sum[i][j] + (p.bias ? p.bias[e] : 0.f);
    }
  for (int e = tid; e < EP; e += kThreads) picks_s[e] = 0;
  __syncthreads();

  // warp-per-token epilogue
  const int warp = tid >> 5, lane = tid & 31;
  for (int r = warp; r < kTM; r += kThreads / 32) {
    const int t = t0 + r;
    float* row = lg + r * (EP + 1);
    if (t >= N) {
      for (int c = 0; c < EJ; ++c) if (lane + 32 * c < E) row[lane + 32 * c] = 0.f;
      continue;
    }
    float v[EJ];
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < EJ; ++c) {
      const int e = lane + 32 * c;
      v[c] = (e < E) ? row[e] : -INFINITY;
      m = fmaxf(m, v[c]);
    }
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < EJ; ++c) {
      v[c] = (lane + 32 * c < E) ? expf(v[c] - m) : 0.f;
      s += v[c];
    }
    s = warp_sum(s);
#pragma unroll
    for (int c = 0; c < EJ; ++c) {
      const int e = lane + 32 * c;
      v[c] = v[c] / s;
      if (e < E) {
        row[e] = v[c];
        if (p.probs) p.probs[(size_t)t * E + e] = v[c];
      }
    }
    // top-k: k rounds of arg-max (higher p, then lower index)
    uint32_t taken = 0;
    float sel_p[8];
    int sel_e[8];
    float ksum = 0.f;
    for (int q = 0; q < k; ++q) {
      float bp = -1.f;
      int be = 0x7fffffff;
#pragma unroll
      for (int c = 0; c < EJ; ++c) {
        const int e = lane + 32 * c;
        if (e < E && !((taken >> c) & 1u) && better(v[c], e, bp, be)) { bp = v[c]; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float op = __shfl_xor_sync(0xffffffffu, bp, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (better(op, oe, bp, be)) { bp = op; be = oe; }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      sel_p[q] = bp;
      sel_e[q] = be;
      ksum += bp;
    }
    if (lane < k) {
      float mp = 0.f;
      int me = 0;
      for (int q = 0; q < k; ++q) if (q == lane) { mp = sel_p[q]; me = sel_e[q]; }
      p.topk_idx[(size_t)t * k + lane] = me;
      p.topk_w[(size_t)t * k + lane] = mp / ksum;
      atomicAdd(&picks_s[me], 1);
    }
  }
  __syncthreads();
  // per-CTA partial statistics, summed in token order (deterministic)
  for (int e = tid; e < E; e += kThreads) {
    float acc = 0.f;
    for (int r = 0; r < kTM; ++r) acc += lg[r * (EP + 1) + e];
    p.psum_part[(size_t)blockIdx.x * E + e] = acc;
    p.picks_part[(size_t)blockIdx.x * E + e] = picks_s[e];
  }
}

__global__ void __launch_bounds__(256) route_stats_kernel(RouteStatsParams p) {
  __shared__ double contrib[256];
  const int e = threadIdx.x;
  if (e < p.E) {
    double sp = 0.0;
    long long pk = 0;
    for (int b = 0; b < p.blocks; ++b) {
      sp += (double)p.psum_part[(size_t)b * p.E + e];
      pk += p.picks_part[(size_t)b * p.E + e];
    }
    const double mean = sp / (double)p.N;
    const double freq = (double)pk / ((double)p.N * (double)p.k);
    if (p.mean_prob) p.mean_prob[e] = (float)mean;
    if (p.expert_freq) p.expert_freq[e] = (float)freq;
    contrib[e] = freq * mean;
  }
  __syncthreads();
  if (threadIdx.x == 0 && p.l_bal) {
    double s = 0.0;
    for (int i = 0; i < p.E; ++i) s += contrib[i];
    p.l_bal[0] = (float)(p.E * s);
  }
}

template <typename T, int EJ>
cudaError_t launch_route_t(const RouteParams& p, cudaStream_t s) {
  const int EP = EJ * 32;
  const size_t smem = sizeof(float) * ((size_t)kTM * kXS + (size_t)EP * kXS +
                                       (size_t)kTM * (EP + 1)) + sizeof(int) * EP;
  auto kern = route_kernel<T, EJ>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const int blocks = (p.N + kTM - 1) / kTM;
  kern<<<blocks, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_route_dt(const RouteParams& p, cudaStream_t s) {
  switch ((p.E + 31) / 32) {
    case 1: return launch_route_t<T, 1>(p, s);
    case 2: return launch_route_t<T, 2>(p, s);
    case 3: return launch_route_t<T, 3>(p, s);
    case 4: return launch_route_t<T, 4>(p, s);
    case 5: return launch_route_t<T, 5>(p, s);
    case 6: return launch_route_t<T, 6>(p, s);
    case 7: return launch_route_t<T, 7>(p, s);
    default: return launch_route_t<T, 8>(p, s);
  }
}

}  // namespace

cudaError_t launch_route(const RouteParams& p, bool bf16, cudaStream_t s) {
  return bf16 ? launch_route_dt<__nv_bfloat16>(p, s) : launch_route_dt<float>(p, s);
}

cudaError_t launch_route_stats(const RouteStatsParams& p, cudaStream_t s) {
  route_stats_kernel<<<1, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
