// Router: partial logits (fp32 layers: CUDA-core contraction here; bf16 layers:
// tensor cores, route_tc.cu), their reduction over K slices, then a
// warp-per-token finish: router bias, fp32 softmax, top-k with renormalised
// gates, and the load-balance statistics (exact fixed-point sums across CTAs,
// finished by the last CTA).
//
// «为什么MoE有效？稀疏激活的数学直觉与工程实践» §2.2 (router = bias-free linear
// map, softmax, torch.topk, renormalise); «DeepSeek-V2 ...» summary §2.2
// (expert_bias added to the logits before the softmax; load_balance_loss).
//
// The K-slice partials are summed with compensation (fp32 Kahan) in slice order,
// so the logits are within ~1e-7 of the exact value and deterministic; top-k is k rounds of a
// warp-shuffle arg-max (higher probability first, ties to the lower index).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kTM = kRouteTM;   // tokens per CUDA-core logits CTA
constexpr int kKC = 64;         // K chunk staged through shared memory
constexpr int kXS = kKC + 4;    // padded smem row (floats), 16-byte aligned rows
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ void load8f(const float* src, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(src)[0];
  const float4 b = reinterpret_cast<const float4*>(src)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// fp32 partial logits on the CUDA cores (no TF32: 1e-4 accuracy is required).
// Grid (ceil(N/32), ks); EJ = ceil(E/32).  Each K chunk is summed separately and
// folded into the running sum with Kahan compensation.
template <int EJ>
__global__ void __launch_bounds__(kThreads) route_logits_simt(RouteParams p, RouteSplit sp) {
  griddep_begin();
  extern __shared__ __align__(16) float sm[];
  const int E = p.E, d = p.d, N = p.N;
  const int EP = EJ * 32;
  float* xs = sm;                                // [kTM][kXS]
  float* ws = xs + kTM * kXS;                    // [EP][kXS]
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kTM;
  const int ks = blockIdx.y;
  const int k_begin = ks * sp.k_slice, k_end = min(d, k_begin + sp.k_slice);
  const float* x = static_cast<const float*>(p.x);
  const float* wr = static_cast<const float*>(p.w_router);
  const int tx = tid & 7, ty = tid >> 3;

  float sum[4][EJ], cmp[4][EJ];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EJ; ++j) sum[i][j] = cmp[i][j] = 0.f;

  for (int k0 = k_begin; k0 < k_end; k0 += kKC) {
    for (int v = tid; v < kTM * (kKC / 8); v += kThreads) {
      const int r = v / (kKC / 8), c = (v % (kKC / 8)) * 8;
      float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (t0 + r < N && k0 + c < k_end) load8f(x + (size_t)(t0 + r) * d + k0 + c, f);
#pragma unroll
      for (int q = 0; q < 8; ++q) xs[r * kXS + c + q] = f[q];
    }
    for (int v = tid; v < EP * (kKC / 8); v += kThreads) {
      const int r = v / (kKC / 8), c = (v % (kKC / 8)) * 8;
      float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (r < E && k0 + c < k_end) load8f(wr + (size_t)r * d + k0 + c, f);
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
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + tx + 8 * i;
    if (t >= N) continue;
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
      const int e = ty + 32 * j;
      if (e < E) p.part[((size_t)ks * N + t) * E + e] = sum[i][j];
    }
  }
}

// G lanes per token (G = 8, 16 or 32, so that each lane holds EJ <= 8
// experts): logits from the partials, bias, softmax, top-k, gates.  A warp
// works on 32 / G tokens at once; the reductions over a token's experts are
// shuffles within its G-lane group.
template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int EJ, int G>
__global__ void __launch_bounds__(kThreads) route_finish_kernel(RouteParams p, RouteSplit sp) {
  griddep_begin();
  constexpr int EP = EJ * G, GW = 32 / G;
  __shared__ unsigned long long psum_w[kWarps][EP];
  __shared__ unsigned long long zh_w[kWarps][2];
  __shared__ int picks_s[EP];
  __shared__ bool last_cta;
  const int E = p.E, N = p.N, k = p.k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = lane % G, grp = lane / G, base = grp * G;   // lane in the token's group
  // bias on the logits (before the softmax) or on the selection key only
  const bool bias_logit = p.bias && !p.bias_select, bias_sel = p.bias && p.bias_select;
  for (int e = tid; e < EP; e += kThreads) picks_s[e] = 0;
  __syncthreads();
  unsigned long long psum[EJ];                  // sum of p in units of 2^-40 (exact)
#pragma unroll
  for (int c = 0; c < EJ; ++c) psum[c] = 0ull;
  unsigned long long zacc = 0ull, hacc = 0ull;  // group lane 0: lse^2 (2^-20), H (2^-40)
  float b[EJ];                                  // this lane's bias values
#pragma unroll
  for (int c = 0; c < EJ; ++c) {
    const int e = sub + G * c;
    b[c] = (p.bias && e < E) ? p.bias[e] : 0.f;
  }
  const int iters = route_finish_iters(N, GW);
  for (int i = 0; i < iters; ++i) {
    const int t_first = ((blockIdx.x * kWarps + warp) * iters + i) * GW;
    if (t_first >= N) break;                    // the whole warp leaves together
    const int t = t_first + grp;
    const bool valid = t < N;                   // groups past N compute on zeros, write nothing
    float v[EJ], raw[EJ];
    float m = -INFINITY, mr = -INFINITY;
    // logits: the K-slice partials summed in slice order (compensated fp32)
#pragma unroll
    for (int c = 0; c < EJ; ++c) {
      const int e = sub + G * c;
      if (e < E) {
        KahanF z;
        if (valid)
          for (int s0 = 0; s0 < sp.ks; ++s0) z.add(p.part[((size_t)s0 * N + t) * E + e]);
        raw[c] = z.s;
      } else {
        raw[c] = -INFINITY;
      }
      v[c] = (e < E) ? raw[c] + (bias_logit ? b[c] : 0.f) : -INFINITY;
      m = fmaxf(m, v[c]);
      mr = fmaxf(mr, raw[c]);
    }
    m = group_max<G>(m);
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < EJ; ++c) {
      v[c] = (sub + G * c < E) ? expf(v[c] - m) : 0.f;
      s += v[c];
    }
    s = group_sum<G>(s);
    if (p.z_loss) {
      // logsumexp of the bias-free logits («项目概述：为什么MoE...» §3.3)
      float lse;
      if (bias_logit) {
        mr = group_max<G>(mr);
        float sr = 0.f;
#pragma unroll
        for (int c = 0; c < EJ; ++c) sr += (sub + G * c < E) ? expf(raw[c] - mr) : 0.f;
        lse = mr + logf(group_sum<G>(sr));
      } else {
        lse = m + logf(s);
      }
      if (sub == 0 && valid) zacc += __float2ull_rn(lse * lse * 1048576.0f);
    }
    float key[EJ];   // what the top-k ranks: p, or p + b under selection-only bias
#pragma unroll
    for (int c = 0; c < EJ; ++c) {
      const int e = sub + G * c;
      v[c] = v[c] / s;
      key[c] = bias_sel ? v[c] + b[c] : v[c];
      if (e < E && valid) {
        psum[c] += __float2ull_rn(v[c] * 1099511627776.0f);
        if (p.probs) p.probs[(size_t)t * E + e] = key[c];
      }
    }
    uint32_t taken = 0;
    float ksum = 0.f, my_p = 0.f;
    int my_e = 0;
    for (int q = 0; q < k; ++q) {
      float bk = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int c = 0; c < EJ; ++c) {
        const int e = sub + G * c;
        if (e < E && !((taken >> c) & 1u) && better(key[c], e, bk, be)) { bk = key[c]; be = e; }
      }
#pragma unroll
      for (int o = G / 2; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (better(ok, oe, bk, be)) { bk = ok; be = oe; }
      }
      // the winner's probability (its key, unless the bias steered the choice)
      float pw = bk;
      if (bias_sel) {
        float mine = 0.f;
#pragma unroll
        for (int c = 0; c < EJ; ++c)
          if (c == be / G) mine = v[c];
        pw = __shfl_sync(0xffffffffu, mine, base + be % G);
      }
      if (be % G == sub) taken |= 1u << (be / G);
      if (q == sub) { my_p = pw; my_e = be; }
      ksum += pw;
    }
    const float my_w = my_p / ksum;
    if (sub < k && valid) {
      p.topk_idx[(size_t)t * k + sub] = my_e;
      p.topk_w[(size_t)t * k + sub] = my_w;
      atomicAdd(&picks_s[my_e], 1);
    }
    if (p.entropy) {
      // -sum_j w_j log2 w_j over the gates («GPT-4 Has 1.8 Trillion ...» §2.3)
      const float h = group_sum<G>((sub < k && my_w > 0.f) ? -my_w * log2f(my_w) : 0.f);
      if (sub == 0 && valid) hacc += __float2ull_rn(h * 1099511627776.0f);
    }
  }
  // the groups of a warp hold partial sums of the same experts: add them
  // (integers, so the order does not matter)
#pragma unroll
  for (int o = G; o < 32; o <<= 1) {
#pragma unroll
    for (int c = 0; c < EJ; ++c) psum[c] += __shfl_xor_sync(0xffffffffu, psum[c], o);
    zacc += __shfl_xor_sync(0xffffffffu, zacc, o);
    hacc += __shfl_xor_sync(0xffffffffu, hacc, o);
  }
  if (grp == 0) {
#pragma unroll
    for (int c = 0; c < EJ; ++c) psum_w[warp][sub + G * c] = psum[c];
  }
  if (lane == 0) { zh_w[warp][0] = zacc; zh_w[warp][1] = hacc; }
  __syncthreads();
  // integer sums are exact, so the cross-CTA atomics are order-independent
  for (int e = tid; e < E; e += kThreads) {
    unsigned long long acc = 0ull;
    for (int w = 0; w < kWarps; ++w) acc += psum_w[w][e];
    atomicAdd(&p.acc_p[e], acc);
    atomicAdd(&p.acc_pick[e], picks_s[e]);
  }
  if (tid < 2 && (tid == 0 ? p.z_loss != nullptr : p.entropy != nullptr)) {
    unsigned long long acc = 0ull;
    for (int w = 0; w < kWarps; ++w) acc += zh_w[w][tid];
    atomicAdd(&p.acc_zh[tid], acc);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last_cta = atomicAdd(p.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last_cta) return;
  // the last CTA: expert_freq, mean_prob and L_bal («DeepSeek-V2 ...» summary §2.2)
  __threadfence();
  __shared__ float contrib[kMaxExperts];
  for (int e = tid; e < E; e += kThreads) {
    const float mean = __ull2float_rn(__ldcg(&p.acc_p[e])) * (1.0f / 1099511627776.0f) / (float)N;
    const float freq = (float)__ldcg(&p.acc_pick[e]) / ((float)N * (float)k);
    if (p.mean_prob) p.mean_prob[e] = mean;
    if (p.expert_freq) p.expert_freq[e] = freq;
    contrib[e] = freq * mean;
  }
  __syncthreads();
  if (tid == 0 && p.l_bal) {
    KahanF s;
    for (int e = 0; e < E; ++e) s.add(contrib[e]);
    p.l_bal[0] = (float)E * s.s;
  }
  if (tid == 32 && p.z_loss)
    p.z_loss[0] = (float)(0.001 * (__ull2double_rn(__ldcg(&p.acc_zh[0])) / 1048576.0) / N);
  if (tid == 64 && p.entropy)
    p.entropy[0] = (float)(__ull2double_rn(__ldcg(&p.acc_zh[1])) / 1099511627776.0 / N);
}

// Auxiliary-loss-free balancing step («为什么MoE有效？...» §2.4): lower the
// bias of an expert that got more than N*k/E picks, raise it below that.
__global__ void bias_update_kernel(const int* picks, float* bias, int N, int E, int k, float gamma) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const long long load = (long long)picks[e] * E, mean = (long long)N * k;
  if (load > mean) bias[e] = bias[e] - gamma;
  else if (load < mean) bias[e] = bias[e] + gamma;
}

template <int EJ>
cudaError_t launch_simt_t(const RouteParams& p, const RouteSplit& sp, cudaStream_t s) {
  const size_t smem = sizeof(float) * ((size_t)kTM * kXS + (size_t)EJ * 32 * kXS);
  auto kern = route_logits_simt<EJ>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if ((err = launch_chained(kern, dim3((p.N + kTM - 1) / kTM, sp.ks), kThreads, smem, s, p, sp)) !=
      cudaSuccess)
    return err;
  count_launch();
  return cudaSuccess;
}

template <int EJ, int G>
cudaError_t launch_finish_t(const RouteParams& p, const RouteSplit& sp, cudaStream_t s) {
  const cudaError_t err = launch_chained(route_finish_kernel<EJ, G>, route_finish_blocks(p.N, 32 / G),
                                         kThreads, 0, s, p, sp);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

// lanes per token: the fewest of 8, 16, 32 that keep a lane at <= 8 experts
cudaError_t launch_finish(const RouteParams& p, const RouteSplit& sp, cudaStream_t s) {
  if (p.E <= 64) {
    switch ((p.E + 7) / 8) {
      case 1: return launch_finish_t<1, 8>(p, sp, s);
      case 2: return launch_finish_t<2, 8>(p, sp, s);
      case 3: return launch_finish_t<3, 8>(p, sp, s);
      case 4: return launch_finish_t<4, 8>(p, sp, s);
      case 5: return launch_finish_t<5, 8>(p, sp, s);
      case 6: return launch_finish_t<6, 8>(p, sp, s);
      case 7: return launch_finish_t<7, 8>(p, sp, s);
      default: return launch_finish_t<8, 8>(p, sp, s);
    }
  }
  if (p.E <= 128) {
    switch ((p.E + 15) / 16) {
      case 5: return launch_finish_t<5, 16>(p, sp, s);
      case 6: return launch_finish_t<6, 16>(p, sp, s);
      case 7: return launch_finish_t<7, 16>(p, sp, s);
      default: return launch_finish_t<8, 16>(p, sp, s);
    }
  }
  switch ((p.E + 31) / 32) {
    case 5: return launch_finish_t<5, 32>(p, sp, s);
    case 6: return launch_finish_t<6, 32>(p, sp, s);
    case 7: return launch_finish_t<7, 32>(p, sp, s);
    default: return launch_finish_t<8, 32>(p, sp, s);
  }
}

#define MOE_EJ_SWITCH(E, F, ...)                  \
  switch (((E) + 31) / 32) {                      \
    case 1: return F<1>(__VA_ARGS__);             \
    case 2: return F<2>(__VA_ARGS__);             \
    case 3: return F<3>(__VA_ARGS__);             \
    case 4: return F<4>(__VA_ARGS__);             \
    case 5: return F<5>(__VA_ARGS__);             \
    case 6: return F<6>(__VA_ARGS__);             \
    case 7: return F<7>(__VA_ARGS__);             \
    default: return F<8>(__VA_ARGS__);            \
  }

}  // namespace

// Iterations of a finish warp: one (its gw tokens), whatever N.  The kernel is
// a latency chain per token, so more CTAs beat more tokens per warp: with up
// to 8 tokens per warp for large batches the 64-expert route stage took
// 57.7 us, with one iteration 45.6 us (DeepSeek-V2 87.7 -> 81.0 us).
__host__ __device__ int route_finish_iters(int N, int gw) {
  (void)N;
  (void)gw;
  return 1;
}

int route_finish_blocks(int N, int gw) {
  const int per_cta = kWarps * route_finish_iters(N, gw) * gw;
  return (N + per_cta - 1) / per_cta;
}

RouteSplit route_split(int N, int d, int E, bool bf16) {
  const int tile = bf16 ? 128 : kTM;
  const int tiles = N > 0 ? (N + tile - 1) / tile : 1;
  const int kblocks = (d + 63) / 64;
  // at most one CTA per SM (the tensor-core router holds an SM's TMEM), so
  // one wave: a second, partial wave would double the time; at most 16
  // slices (each slice is one more partial per logit to read back)
  int ks = 148 / tiles;
  ks = ks < 1 ? 1 : (ks > 16 ? 16 : ks);
  // a one-tile batch with many experts: the finish kernel's share (ks partials
  // of E logits per token) outweighs the contraction's, so fewer slices
  // (DeepSeek-V2 decode, E = 160: route stage 29.0 -> 27.2 us with 8; E = 8
  // keeps 16, where 8 measured 1.4 us slower)
  if (tiles == 1 && E > 64 && ks > 8) ks = 8;
  ks = ks > kblocks ? kblocks : ks;
  const int k_slice = (kblocks + ks - 1) / ks * 64;
  RouteSplit r;
  r.k_slice = k_slice;
  r.ks = (d + k_slice - 1) / k_slice;
  return r;
}

cudaError_t launch_bias_update(const int* picks, float* bias, int N, int E, int k, float gamma,
                               cudaStream_t s) {
  bias_update_kernel<<<(E + 255) / 256, 256, 0, s>>>(picks, bias, N, E, k, gamma);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_route(const RouteParams& p, bool bf16, cudaStream_t s) {
  const RouteSplit sp = route_split(p.N, p.d, p.E, bf16);
  cudaError_t err;
  if (bf16) {
    err = launch_route_logits_tc(sp, p.x, p.w_router, p.N, p.E, p.d, p.part, p.status, s);
  } else {
    err = [&]() -> cudaError_t { MOE_EJ_SWITCH(p.E, launch_simt_t, p, sp, s) }();
  }
  if (err != cudaSuccess) return err;
  return launch_finish(p, sp, s);
}


}  // namespace moe
