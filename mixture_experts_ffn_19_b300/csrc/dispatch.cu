// Dispatch: per-expert histogram, scan, expert capacity (drop or reroute),
// segment layout, and the permutation of token rows into expert order.
//
// «大模型MoE架构揭秘：如何用2%参数实现万亿级算力调度» §3.1 (capacity
// C = floor(k N / E) x alpha; overflow forced to the next-best expert), §4.2
// code (an expert keeps its first C tokens in ascending token order).
//
// Three kernels, no atomics on anything whose order matters:
//   rank    one CTA per 256 tokens: a per-expert bitmap of the CTA's tokens
//           gives each assignment its rank among earlier tokens of the CTA
//           (popcount of the lower bits) and the CTA's per-expert count.
//   plan    one CTA: per-expert exclusive scan over the token chunks (so an
//           assignment's rank within its expert is chunk base + local rank,
//           i.e. its position in token order), capacity, the reroute rounds,
//           segment offsets, counts and drop/reroute totals.
//   scatter one CTA per token: final expert, row, perm entry, and the 16-byte
//           vector copy of x[t] into every row the token owns.
// Reroute rounds: each pending slot proposes the most probable expert (ties to
// the lower index) that was not full when the round started and that its token
// neither holds nor proposed earlier in the round, slots in slot order; each
// expert accepts proposals in ascending token order while it has room.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPendingMark = -2;

__global__ void __launch_bounds__(kRankTC) dispatch_rank_kernel(DispatchParams p) {
  extern __shared__ uint32_t bits[];             // [E][kRankTC/32]
  constexpr int W = kRankTC / 32;
  const int E = p.E, k = p.k;
  const int tid = threadIdx.x;
  const int t = blockIdx.x * kRankTC + tid;
  for (int i = tid; i < E * W; i += kRankTC) bits[i] = 0;
  __syncthreads();
  int my_e[kMaxTopk];
  if (t < p.N) {
    for (int j = 0; j < k; ++j) {
      int e = p.topk_idx[(size_t)t * k + j];
      if (e < 0 || e >= E) {          // not an expert index: record it, never index with it
        set_status(p.status, kDevBadState);
        e = -1;
      }
      my_e[j] = e;
      if (e >= 0) atomicOr(&bits[e * W + (tid >> 5)], 1u << (tid & 31));
    }
  }
  __syncthreads();
  if (t < p.N) {
    for (int j = 0; j < k; ++j) {
      const int e = my_e[j];
      if (e < 0) { p.local_rank[(size_t)t * k + j] = 0; continue; }
      int r = 0;
      for (int w = 0; w < (tid >> 5); ++w) r += __popc(bits[e * W + w]);
      r += __popc(bits[e * W + (tid >> 5)] & lanemask_lt());
      p.local_rank[(size_t)t * k + j] = r;
    }
  }
  for (int e = tid; e < E; e += kRankTC) {
    int c = 0;
    for (int w = 0; w < W; ++w) c += __popc(bits[e * W + w]);
    p.chunk_cnt[(size_t)blockIdx.x * E + e] = c;
  }
}

// Block-wide compaction of `n` candidates in order: writes the kept ones to
// out[] (which may alias the source as long as out index <= source index).
// Returns the number kept (same value in every thread).
template <typename Pred, typename Val>
__device__ int block_compact(int n, Pred keep, Val value, int32_t* out, int* warp_tot, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int base = 0;
  for (int c0 = 0; c0 < n; c0 += kPlanThreads) {
    const int i = c0 + tid;
    const bool f = (i < n) && keep(i);
    const int v = (i < n) ? value(i) : 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      for (int w = 0; w < kPlanThreads / 32; ++w) { const int c = warp_tot[w]; warp_tot[w] = run; run += c; }
      *total = run;
    }
    __syncthreads();
    if (f) out[base + warp_tot[warp] + __popc(bal & lanemask_lt())] = v;
    base += *total;
    __syncthreads();
  }
  return base;
}

__global__ void __launch_bounds__(kPlanThreads) dispatch_plan_kernel(DispatchParams p) {
  extern __shared__ uint32_t dyn[];
  const int E = p.E, k = p.k, N = p.N, S = p.S, C = p.C;
  uint32_t* bits = dyn;                                         // [E][32]
  int* pre = reinterpret_cast<int*>(dyn + E * 32);              // [E][32]
  __shared__ int fill[kMaxExperts], total[kMaxExperts];
  __shared__ int prop_cnt[kMaxExperts], chunk_tot[kMaxExperts];
  __shared__ unsigned char full_s[kMaxExperts];
  __shared__ int warp_tot[kPlanThreads / 32];
  __shared__ int s_total, s_any, s_npend;
  const int tid = threadIdx.x, lane = tid & 31;

  // 1. per-expert exclusive scan over token chunks
  for (int e = tid; e < E; e += kPlanThreads) {
    int run = 0;
    for (int c = 0; c < p.n_chunks; ++c) {
      const int v = p.chunk_cnt[(size_t)c * E + e];
      p.chunk_cnt[(size_t)c * E + e] = run;
      run += v;
    }
    total[e] = run;
    fill[e] = min(run, C);
  }
  __syncthreads();

  if (p.cap_mode == 2) {
    // 2. primary pass: keep rank < C, mark the rest pending
    for (int a = tid; a < N * k; a += kPlanThreads) {
      const int t = a / k;
      const int e = p.topk_idx[a];
      if (e < 0 || e >= E) { p.final_idx[a] = -1; p.slot[a] = -1; continue; }
      const int rank = p.chunk_cnt[(size_t)(t / kRankTC) * E + e] + p.local_rank[a];
      if (rank < C) { p.final_idx[a] = e; p.slot[a] = rank; }
      else { p.final_idx[a] = kPendingMark; p.slot[a] = -1; }
    }
    __syncthreads();
    auto has_pending = [&](int t) {
      for (int j = 0; j < k; ++j) if (p.final_idx[(size_t)t * k + j] == kPendingMark) return true;
      return false;
    };
    int npend = block_compact(N, has_pending, [](int t) { return t; }, p.pend, warp_tot, &s_total);
    // 3. reroute rounds
    int round = 0;
    while (npend > 0) {
      if (round > E + 1) {               // cannot happen: every round fills an expert or ends
        set_status(p.status, kDevBadState);
        break;
      }
      for (int e = tid; e < E; e += kPlanThreads) { full_s[e] = fill[e] >= C; prop_cnt[e] = 0; }
      if (tid == 0) s_any = 0;
      __syncthreads();
      for (int c0 = 0; c0 < npend; c0 += kPlanThreads) {
        for (int i = tid; i < E * 32; i += kPlanThreads) bits[i] = 0;
        __syncthreads();
        const int i = tid;
        const int t = (c0 + i < npend) ? p.pend[c0 + i] : -1;
        int prop[kMaxTopk];
        if (t >= 0) {
          int held[kMaxTopk];
          for (int j = 0; j < k; ++j) held[j] = p.final_idx[(size_t)t * k + j];
          for (int j = 0; j < k; ++j) {
            prop[j] = -1;
            if (held[j] != kPendingMark) continue;
            float bp = -1.f;
            int be = -1;
            const float* pr = p.probs + (size_t)t * E;
            for (int e = 0; e < E; ++e) {
              if (full_s[e]) continue;
              bool skip = false;
              for (int jj = 0; jj < k; ++jj) skip |= (held[jj] == e) | (jj < j && prop[jj] == e);
              if (skip) continue;
              const float pe = pr[e];
              if (be < 0 || better(pe, e, bp, be)) { bp = pe; be = e; }
            }
            prop[j] = be;
            if (be < 0) {
              p.final_idx[(size_t)t * k + j] = -1;          // nothing left: dropped
            } else {
              atomicOr(&bits[be * 32 + (i >> 5)], 1u << (i & 31));
              s_any = 1;
            }
          }
        }
        __syncthreads();
        for (int e = tid; e < E; e += kPlanThreads) {
          int run = 0;
          for (int w = 0; w < 32; ++w) { pre[e * 32 + w] = run; run += __popc(bits[e * 32 + w]); }
          chunk_tot[e] = run;
        }
        __syncthreads();
        if (t >= 0) {
          for (int j = 0; j < k; ++j) {
            const int e = prop[j];
            if (e < 0) continue;
            const int rank = prop_cnt[e] + pre[e * 32 + (i >> 5)] +
                             __popc(bits[e * 32 + (i >> 5)] & lanemask_lt());
            const int s = fill[e] + rank;
            if (s < C) { p.final_idx[(size_t)t * k + j] = e; p.slot[(size_t)t * k + j] = s; }
          }
        }
        __syncthreads();
        for (int e = tid; e < E; e += kPlanThreads) prop_cnt[e] += chunk_tot[e];
        __syncthreads();
      }
      for (int e = tid; e < E; e += kPlanThreads) fill[e] = min(C, fill[e] + prop_cnt[e]);
      __syncthreads();
      if (!s_any) break;
      npend = block_compact(npend, [&](int q) { return has_pending(p.pend[q]); },
                            [&](int q) { return p.pend[q]; }, p.pend, warp_tot, &s_total);
      ++round;
    }
    // anything still pending after a bad state is dropped
    for (int a = tid; a < N * k; a += kPlanThreads)
      if (p.final_idx[a] == kPendingMark) p.final_idx[a] = -1;
    __syncthreads();
  }

  // 4. totals: dropped and rerouted
  int nd = 0, nr = 0;
  if (p.cap_mode == 2) {
    for (int a = tid; a < N * k; a += kPlanThreads) {
      const int f = p.final_idx[a];
      nd += (f < 0);
      nr += (f >= 0 && f != p.topk_idx[a]);
    }
  } else {
    for (int e = tid; e < E; e += kPlanThreads) nd += total[e] - fill[e];
  }
  nd = __reduce_add_sync(0xffffffffu, nd);
  nr = __reduce_add_sync(0xffffffffu, nr);
  if (lane == 0) warp_tot[tid >> 5] = nd;
  __syncthreads();
  if (tid == 0) { int s = 0; for (int w = 0; w < kPlanThreads / 32; ++w) s += warp_tot[w]; s_total = s; }
  __syncthreads();
  const int n_dropped = s_total;
  __syncthreads();
  if (lane == 0) warp_tot[tid >> 5] = nr;
  __syncthreads();
  if (tid == 0) {
    int s = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) s += warp_tot[w];
    if (p.n_dropped) *p.n_dropped = n_dropped;
    if (p.n_rerouted) *p.n_rerouted = s;
    // 5. segment layout: routed experts, then shared experts
    int row = 0;
    for (int e = 0; e < E; ++e) {
      p.offsets[e] = row;
      row += (fill[e] + kAlign - 1) / kAlign * kAlign;
    }
    const int nseg = (N + kAlign - 1) / kAlign * kAlign;
    for (int s2 = 0; s2 < S; ++s2) { p.offsets[E + s2] = row; row += nseg; }
    p.offsets[E + S] = row;
  }
  for (int e = tid; e < E; e += kPlanThreads) if (p.counts) p.counts[e] = fill[e];
  __syncthreads();
  // 6. perm = -1 on the padding rows of routed segments (one warp per expert)
  for (int e = tid >> 5; e < E; e += kPlanThreads / 32) {
    const int r0 = p.offsets[e] + fill[e];
    const int r1 = p.offsets[e + 1];
    for (int r = r0 + lane; r < r1; r += 32) p.perm[r] = -1;
  }
}

template <typename T>
__global__ void __launch_bounds__(128) dispatch_scatter_kernel(DispatchParams p) {
  const int t = blockIdx.x;
  const int k = p.k, E = p.E;
  __shared__ int rows[kMaxTopk];
  if (threadIdx.x < k) {
    const size_t a = (size_t)t * k + threadIdx.x;
    int f, sl;
    if (p.cap_mode == 2) {
      f = p.final_idx[a];
      sl = p.slot[a];
    } else {
      const int e = p.topk_idx[a];
      if (e >= 0 && e < E) {
        sl = p.chunk_cnt[(size_t)(t / kRankTC) * E + e] + p.local_rank[a];
        f = (sl < p.C) ? e : -1;
      } else {
        sl = -1;
        f = -1;
      }
      p.final_idx[a] = f;
    }
    const int row = (f >= 0) ? p.offsets[f] + sl : -1;
    p.pos[a] = row;
    if (row >= 0) p.perm[row] = t;
    rows[threadIdx.x] = row;
  }
  __syncthreads();
  const int nvec = p.d * (int)sizeof(T) / 16;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.x) + (size_t)t * p.d);
  uint4* dst = reinterpret_cast<uint4*>(p.x_perm);
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const uint4 val = src[v];
    for (int j = 0; j < k; ++j) {
      const int row = rows[j];
      if (row >= 0) dst[(size_t)row * nvec + v] = val;
    }
  }
}

}  // namespace

cudaError_t launch_dispatch(const DispatchParams& p, bool bf16, cudaStream_t s) {
  const int W = kRankTC / 32;
  dispatch_rank_kernel<<<p.n_chunks, kRankTC, sizeof(uint32_t) * p.E * W, s>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t plan_smem = (size_t)p.E * 32 * 8;
  err = cudaFuncSetAttribute(dispatch_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)plan_smem);
  if (err != cudaSuccess) return err;
  dispatch_plan_kernel<<<1, kPlanThreads, plan_smem, s>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (bf16) dispatch_scatter_kernel<__nv_bfloat16><<<p.N, 128, 0, s>>>(p);
  else dispatch_scatter_kernel<float><<<p.N, 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
