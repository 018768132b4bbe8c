// Dispatch: per-expert histogram, scan, expert capacity (drop or reroute),
// segment layout, and the permutation of token rows into expert order.
//
// «大模型MoE架构揭秘：如何用2%参数实现万亿级算力调度» §3.1 (capacity
// C = floor(k N / E) x alpha; overflow forced to the next-best expert), §4.2
// code (an expert keeps its first C tokens in ascending token order).
//
// Kernels, no atomics on anything whose order matters:
//   rank    one CTA per 256 tokens: a per-expert bitmap of the CTA's tokens
//           gives each assignment its rank among earlier tokens of the CTA
//           (popcount of the lower bits) and the CTA's per-expert count.
//   plan    one CTA: per-expert exclusive scan over the token chunks, so an
//           assignment's rank within its expert is chunk base + local rank
//           (its position in token order); capacity; segment offsets, counts
//           and drop totals (reroute: initial fill levels only).
//   reroute (reroute only) one cooperative launch of co-resident CTAs: the
//           primary keep/pending decision per assignment, then the rounds,
//           phases separated by a bounded grid barrier:
//             A  every pending slot proposes the most probable expert (ties to
//                the lower index) that was not full when the round started and
//                that its token neither holds nor proposed earlier in the
//                round (slots in slot order); bitmap ranks per chunk of tokens
//             B  per-expert scan over the chunks; next fill levels
//             C  an expert accepts proposals in token order while it has room
//           a round with no proposal ends it; then the segment layout, as plan
//           does for the other modes.
//   scatter one CTA per token: final expert, row, perm entry, and the 16-byte
//           vector copy of x[t] into every row the token owns.
#include "common.cuh"
#include "kernels.h"

// When the row-copying dispatch kernels let their successor (the expert
// GEMMs, one large CTA per SM) launch: at their start (1) or at their end (0).
#ifndef MOE_DISPATCH_EARLY_TRIGGER
#define MOE_DISPATCH_EARLY_TRIGGER 0
#endif

namespace moe {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPendingMark = -2;
constexpr int kRrThreads = 128;     // reroute CTA = one chunk of 128 pending tokens
constexpr int kRrWords = kRrThreads / 32;
constexpr int kFusedScanInts = 16384;   // per-chunk count table summed by every reroute CTA

__device__ __forceinline__ bool valid_expert(int e, int E) { return e >= 0 && e < E; }

// In-place exclusive scan of column e of a row-major [n, E] int matrix by one
// warp (32 rows per step, shuffle scan); returns the column total.  Loads go
// through L2 so values written by other CTAs of a cooperative launch are seen.
__device__ int warp_exclusive_scan_column(int32_t* m, int n, int E, int e, int lane) {
  int carry = 0;
  for (int r0 = 0; r0 < n; r0 += 32) {
    const int r = r0 + lane;
    const int v = r < n ? __ldcg(&m[(size_t)r * E + e]) : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (r < n) m[(size_t)r * E + e] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  return carry;
}

// In-place exclusive scan of a contiguous int row by one warp; returns the
// row total.  Loads go through L2, as in the column scan.
__device__ int warp_exclusive_scan_row(int32_t* m, int n, int lane) {
  int carry = 0;
  for (int r0 = 0; r0 < n; r0 += 32) {
    const int r = r0 + lane;
    const int v = r < n ? __ldcg(&m[r]) : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (r < n) m[r] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  return carry;
}

__global__ void __launch_bounds__(kRankTC) dispatch_rank_kernel(DispatchParams p) {
  griddep_begin();
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
      if (!valid_expert(e, E)) {        // not an expert index: record it, never index with it
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

// Segment layout, counts and drop/reroute totals from the final per-expert
// fill levels; perm = -1 on the padding rows.  Executed by one whole CTA.
// The segment starts are scanned by warp 0 into shared memory and every
// later step reads them there: read back from global memory inside the
// padding loop (which also stores), each expert cost an L2 round trip.
constexpr int kLayoutInts = kMaxExperts + 8 + 1;   // routed + shared segments + end
__device__ void write_layout(const DispatchParams& p, const int* fill, int* offs_s, int n_dropped,
                             int n_rerouted) {
  const int E = p.E, S = p.S, N = p.N;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (wid == 0) {
    // exclusive scan of the 128-row-padded fills
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? (fill[e] + kAlign - 1) / kAlign * kAlign : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < E) offs_s[e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      const int nseg = (N + kAlign - 1) / kAlign * kAlign;
      for (int sh = 0; sh <= S; ++sh) offs_s[E + sh] = carry + sh * nseg;
      if (p.n_dropped) *p.n_dropped = n_dropped;
      if (p.n_rerouted) *p.n_rerouted = n_rerouted;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= E + S; i += blockDim.x) p.offsets[i] = offs_s[i];
  for (int e = threadIdx.x; e < E; e += blockDim.x) if (p.counts) p.counts[e] = fill[e];
  for (int e = wid; e < E; e += nw) {
    const int r0 = offs_s[e] + fill[e];
    const int r1 = offs_s[e + 1];
    for (int r = r0 + lane; r < r1; r += 32) p.perm[r] = -1;
  }
}

__global__ void __launch_bounds__(kPlanThreads) dispatch_plan_kernel(DispatchParams p) {
  griddep_begin();
  const int E = p.E, C = p.C;
  __shared__ int fill[kMaxExperts], total[kMaxExperts];
  __shared__ int offs_s[kLayoutInts];
  __shared__ int warp_tot[kPlanThreads / 32];
  __shared__ int s_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // per-expert exclusive scan over token chunks (a warp per expert)
  for (int e = warp; e < E; e += kPlanThreads / 32) {
    const int run = warp_exclusive_scan_column(p.chunk_cnt, p.n_chunks, E, e, lane);
    if (lane == 0) { total[e] = run; fill[e] = min(run, C); }
  }
  __syncthreads();

  if (p.cap_mode != 2) {
    int nd = 0;
    for (int e = tid; e < E; e += kPlanThreads) nd += total[e] - fill[e];
    nd = __reduce_add_sync(0xffffffffu, nd);
    if (lane == 0) warp_tot[warp] = nd;
    __syncthreads();
    if (tid == 0) { int s = 0; for (int w = 0; w < kPlanThreads / 32; ++w) s += warp_tot[w]; s_total = s; }
    __syncthreads();
    write_layout(p, fill, offs_s, s_total, 0);
    return;
  }

  // reroute: the cooperative kernel takes the assignments from here
  int kept = 0;
  for (int e = tid; e < E; e += kPlanThreads) { p.rr->fill[0][e] = fill[e]; kept += fill[e]; }
  kept = __reduce_add_sync(0xffffffffu, kept);
  if (lane == 0) warp_tot[warp] = kept;
  __syncthreads();
  if (tid == 0) {
    int s = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) s += warp_tot[w];
    p.rr->primary_kept = s;
    p.rr->bar.count = 0;
    p.rr->bar.abort = 0;
  }
  for (int r = tid; r < kMaxRounds; r += kPlanThreads) p.rr->any_prop[r] = 0;
}

__global__ void __launch_bounds__(kRrThreads) dispatch_reroute_kernel(DispatchParams p) {
  const int E = p.E, k = p.k, C = p.C, N = p.N;
  RerouteState* rr = p.rr;
  constexpr int TE = 64;                         // experts per staged probability tile
  __shared__ uint32_t bits[kMaxExperts * kRrWords];
  __shared__ float prob_s[kRrThreads][TE + 1];
  __shared__ unsigned long long full_m[kMaxExperts / 64];   // bit e: expert e was full at round start
  __shared__ int fill_s[kMaxExperts];            // fill levels at the start of the round
  __shared__ int pre_s[kMaxExperts], tot_s[kMaxExperts];
  __shared__ int offs_s[kLayoutInts];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nch = (N + kRrThreads - 1) / kRrThreads;
  // With one chunk per CTA, the chunk's staged probabilities (E <= TE) and its
  // tokens' held experts stay on chip from round to round.
  const bool own_one = nch <= (int)gridDim.x;
  // While the per-chunk count table is small, every CTA sums it itself: the
  // per-expert scan folds into the acceptance phase and a round needs one grid
  // barrier instead of two.  The table is then double-buffered by round
  // parity, so a CTA already proposing in the next round never overwrites
  // counts another CTA is still summing.
  const bool fused = (size_t)nch * E <= (size_t)kFusedScanInts;

  // primary decisions: an assignment keeps its expert if its rank in token
  // order (chunk base + rank inside the chunk) is below C, else it is pending
  for (int c = blockIdx.x; c < nch; c += gridDim.x) {
    const int t = c * kRrThreads + tid;
    if (t >= N) continue;
    for (int j = 0; j < k; ++j) {
      const size_t a = (size_t)t * k + j;
      const int e = p.topk_idx[a];
      if (!valid_expert(e, E)) { p.final_idx[a] = -1; p.slot[a] = -1; continue; }
      const int rank = p.chunk_cnt[(size_t)(t / kRankTC) * E + e] + p.local_rank[a];
      if (rank < C) { p.final_idx[a] = e; p.slot[a] = rank; }
      else { p.final_idx[a] = kPendingMark; p.slot[a] = -1; }
    }
  }
  if (fused) {
    for (int e = tid; e < E; e += kRrThreads) fill_s[e] = __ldcg(&rr->fill[0][e]);
  }

  int cur = 0;                                   // (two barriers a round) rr->fill[cur]: start levels
  int tile_chunk = -1;                           // chunk whose probabilities are in prob_s (E <= TE)
  // held / prop / prank stay in registers: every index below is a
  // compile-time constant after unrolling (slots past k are guarded); with one
  // chunk per CTA they carry from phase A to phase C and on to the next round
  int held[kMaxTopk], prop[kMaxTopk], prank[kMaxTopk];
  for (int round = 0;; ++round) {
    if (round >= kMaxRounds || round > E + 1) { set_status(p.status, kDevBadState); break; }
    int32_t* cnt = p.rr_chunk + (fused ? (size_t)(round & 1) * nch * E : 0);
    // ---- phase A: proposals, per-chunk bitmap ranks and counts
    if (!fused) {
      __syncthreads();
      for (int e = tid; e < E; e += kRrThreads) fill_s[e] = __ldcg(&rr->fill[cur][e]);
    }
    for (int w = tid; w < kMaxExperts / 64; w += kRrThreads) full_m[w] = 0ull;
    __syncthreads();
    for (int e = tid; e < E; e += kRrThreads)
      if (fill_s[e] >= C) atomicOr(&full_m[e >> 6], 1ull << (e & 63));
    __syncthreads();
    for (int c = blockIdx.x; c < nch; c += gridDim.x) {
      for (int i = tid; i < E * kRrWords; i += kRrThreads) bits[i] = 0;
      const int t = c * kRrThreads + tid;
      bool mine = false;
#pragma unroll
      for (int j = 0; j < kMaxTopk; ++j) {
        if (!own_one || round == 0) held[j] = (j < k && t < N) ? p.final_idx[(size_t)t * k + j] : -1;
        prop[j] = -1;
        mine |= held[j] == kPendingMark;
      }
      bool any = false;
      if (__syncthreads_or(mine)) {
#pragma unroll
        for (int j = 0; j < kMaxTopk; ++j) {
          if (j >= k) break;
          const bool need = held[j] == kPendingMark;
          if (!__syncthreads_or(need)) continue;
          float bp = -1.f;
          int be = -1;
          for (int e0 = 0; e0 < E; e0 += TE) {
            if (E > TE || tile_chunk != c) {
              tile_chunk = E > TE ? -1 : c;
              // stage probabilities [tokens of the chunk][e0, e0+TE): coalesced,
              // 16 independent loads in flight per thread
              __syncthreads();
              for (int i0 = 0; i0 < kRrThreads * TE; i0 += kRrThreads * 16) {
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                  const int i = i0 + u * kRrThreads + tid;
                  const int r = i / TE, col = i % TE;
                  const int tt = c * kRrThreads + r;
                  v[u] = (tt < N && e0 + col < E) ? __ldcg(&p.probs[(size_t)tt * E + e0 + col]) : -1.f;
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                  const int i = i0 + u * kRrThreads + tid;
                  prob_s[i / TE][i % TE] = v[u];
                }
              }
              __syncthreads();
            }
            if (need) {
              // experts of this tile the slot may not take: full at the start of
              // the round, held by the token, or proposed by an earlier slot
              uint64_t excl = full_m[e0 >> 6];
#pragma unroll
              for (int jj = 0; jj < kMaxTopk; ++jj) {
                const int eh = held[jj] - e0, ep = prop[jj] - e0;
                if (jj < k && eh >= 0 && eh < TE) excl |= 1ull << eh;
                if (jj < j && ep >= 0 && ep < TE) excl |= 1ull << ep;
              }
              const int ncol = min(TE, E - e0);
              // four independent arg-max chains over interleaved columns,
              // merged at the end: better() is a total order (higher p, then
              // lower index), so the winner does not depend on the grouping.
              // The test is evaluated without short-circuits and applied as a
              // select, so lanes never branch apart column by column.
              float qp[4] = {bp, -1.f, -1.f, -1.f};
              int qe[4] = {be, -1, -1, -1};
#pragma unroll
              for (int col = 0; col < TE; ++col) {
                const float pe = prob_s[tid][col];
                const int e = e0 + col, q = col & 3;
                const bool take = (col < ncol) & !((excl >> col) & 1ull) &
                                  ((qe[q] < 0) | (pe > qp[q]) | ((pe == qp[q]) & (e < qe[q])));
                qp[q] = take ? pe : qp[q];
                qe[q] = take ? e : qe[q];
              }
#pragma unroll
              for (int q = 1; q < 4; ++q)
                if (qe[q] >= 0 && (qe[0] < 0 || better(qp[q], qe[q], qp[0], qe[0]))) {
                  qp[0] = qp[q];
                  qe[0] = qe[q];
                }
              bp = qp[0];
              be = qe[0];
            }
          }
          if (need) {
            prop[j] = be;
            if (be < 0) {
              p.final_idx[(size_t)t * k + j] = -1;        // nothing left: dropped
              held[j] = -1;
            } else {
              any = true;
            }
          }
          // lanes proposing the same expert set their bits with one atomic
          {
            const unsigned act = __ballot_sync(0xffffffffu, need && be >= 0);
            if (need && be >= 0) {
              const unsigned same = __match_any_sync(act, be);
              if ((tid & 31) == __ffs(same) - 1) atomicOr(&bits[be * kRrWords + (tid >> 5)], same);
            }
          }
        }
      }
      __syncthreads();
      if (mine) {
#pragma unroll
        for (int j = 0; j < kMaxTopk; ++j) {
          if (j >= k) break;
          const int e = prop[j];
          int r = -1;
          if (e >= 0) {
            r = 0;
            for (int w = 0; w < (tid >> 5); ++w) r += __popc(bits[e * kRrWords + w]);
            r += __popc(bits[e * kRrWords + (tid >> 5)] & lanemask_lt());
          }
          prank[j] = r;
          if (!own_one) {
            p.rr_prop[(size_t)t * k + j] = e;
            p.rr_rank[(size_t)t * k + j] = r;
          }
        }
      }
      for (int e = tid; e < E; e += kRrThreads) {
        int n = 0;
        for (int w = 0; w < kRrWords; ++w) n += __popc(bits[e * kRrWords + w]);
        cnt[(size_t)e * nch + c] = n;
      }
      // every CTA that proposed stores the same 1; the grid barrier publishes it
      if (__syncthreads_or(any) && tid == 0) *(volatile int*)&rr->any_prop[round] = 1;
    }
    // a barrier that timed out (status recorded) ends the kernel for every CTA
    if (!grid_barrier(&rr->bar, p.status)) return;
    if (!__ldcg(&rr->any_prop[round])) break;    // nothing proposed: every slot is placed or dropped
    if (!fused) {
      // ---- phase B: per-expert exclusive scan over chunks (a warp per
      //      expert), next fill levels
      const int nwarps = gridDim.x * (kRrThreads / 32);
      for (int e = blockIdx.x * (kRrThreads / 32) + wid; e < E; e += nwarps) {
        const int carry = warp_exclusive_scan_row(cnt + (size_t)e * nch, nch, lane);
        if (lane == 0) rr->fill[cur ^ 1][e] = min(C, __ldcg(&rr->fill[cur][e]) + carry);
      }
      if (!grid_barrier(&rr->bar, p.status)) return;
    }
    // ---- phase C: acceptance in token order while the expert has room
    for (int c = blockIdx.x; c < nch; c += gridDim.x) {
      if (fused) {
        // this chunk's base per expert (proposals in earlier chunks) and the
        // round's totals: a warp takes 8 experts at a time, its lanes stride
        // over the chunks (the table is [expert][chunk], so loads coalesce),
        // 8 x 4 loads in flight per lane; integer sums reduced by the warp.
        constexpr int EB = 8;
        for (int e0 = wid * EB; e0 < E; e0 += EB * (kRrThreads / 32)) {
          int tot[EB], pre[EB];
#pragma unroll
          for (int b = 0; b < EB; ++b) tot[b] = pre[b] = 0;
#pragma unroll 4
          for (int c2 = lane; c2 < nch; c2 += 32) {
#pragma unroll
            for (int b = 0; b < EB; ++b) {
              const int v = e0 + b < E ? __ldcg(&cnt[(size_t)(e0 + b) * nch + c2]) : 0;
              tot[b] += v;
              pre[b] += c2 < c ? v : 0;
            }
          }
#pragma unroll
          for (int b = 0; b < EB; ++b) {
            const int tt = __reduce_add_sync(0xffffffffu, tot[b]);
            const int pp = __reduce_add_sync(0xffffffffu, pre[b]);
            if (lane == 0 && e0 + b < E) { tot_s[e0 + b] = tt; pre_s[e0 + b] = pp; }
          }
        }
        __syncthreads();
      }
      const int t = c * kRrThreads + tid;
      if (t < N) {
#pragma unroll
        for (int j = 0; j < kMaxTopk; ++j) {
          if (j >= k) break;
          const size_t a = (size_t)t * k + j;
          if (held[j] != kPendingMark && own_one) continue;
          if (!own_one && p.final_idx[a] != kPendingMark) continue;
          const int e = own_one ? prop[j] : p.rr_prop[a];
          const int base = fused ? pre_s[e] : __ldcg(&cnt[(size_t)e * nch + c]);
          const int s = fill_s[e] + base + (own_one ? prank[j] : p.rr_rank[a]);
          if (s < C) {
            p.final_idx[a] = e;
            p.slot[a] = s;
            held[j] = e;
          }
        }
      }
      __syncthreads();
    }
    if (fused) {
      for (int e = tid; e < E; e += kRrThreads) fill_s[e] = min(C, fill_s[e] + tot_s[e]);
    }
    cur ^= 1;
  }
  // ---- layout from the final fill levels (CTA 0)
  if (blockIdx.x == 0) {
    __shared__ int s_kept;
    __syncthreads();
    if (!fused)
      for (int e = tid; e < E; e += kRrThreads) fill_s[e] = __ldcg(&rr->fill[cur][e]);
    __syncthreads();
    if (tid == 0) {
      int kept = 0;
      for (int e = 0; e < E; ++e) kept += fill_s[e];
      s_kept = kept;
    }
    __syncthreads();
    write_layout(p, fill_s, offs_s, N * k - s_kept, s_kept - __ldcg(&rr->primary_kept));
  }
}

template <typename T>
__global__ void __launch_bounds__(128) dispatch_scatter_kernel(DispatchParams p) {
  griddep_wait();
  if (MOE_DISPATCH_EARLY_TRIGGER) griddep_launch_dependents();
  const int t = blockIdx.x;
  const int k = p.k, E = p.E;
  __shared__ int rows[kMaxTopk];
  if (threadIdx.x < k) {
    const size_t a = (size_t)t * k + threadIdx.x;
    int f, sl;
    if (p.cap_mode == 2) {
      f = p.final_idx[a];
      sl = p.slot[a];
      if (f < 0) { f = -1; p.final_idx[a] = -1; }
    } else {
      const int e = p.topk_idx[a];
      if (valid_expert(e, E)) {
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
  if (!MOE_DISPATCH_EARLY_TRIGGER) griddep_launch_dependents();
}

// Small batches without reroute (N k <= kSmallAssign): the whole dispatch in
// one launch, a CTA per token.  Every CTA reads all N k expert indices (a few
// KB), so it knows the per-expert totals, and counts the earlier tokens that
// hold each of its own experts: that count is the assignment's rank in token
// order, the same rank the chunked rank/plan kernels produce.  CTA 0 writes
// the segment layout; each CTA writes its own slots and copies its row.
constexpr int kSmallThreads = 128;
constexpr int kSmallAssign = 4096;

template <typename T>
__global__ void __launch_bounds__(kSmallThreads) dispatch_small_kernel(DispatchParams p) {
  griddep_wait();
  if (MOE_DISPATCH_EARLY_TRIGGER) griddep_launch_dependents();
  __shared__ int idx_s[kSmallAssign];
  __shared__ int hist[kMaxExperts], fill[kMaxExperts], offs[kLayoutInts];
  __shared__ int my_e[kMaxTopk], my_rank[kMaxTopk], rows[kMaxTopk];
  __shared__ int s_dropped;
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const int E = p.E, k = p.k, nk = p.N * p.k;
  for (int e = tid; e < E; e += kSmallThreads) hist[e] = 0;
  if (tid < kMaxTopk) my_rank[tid] = 0;
  if (tid == 0) s_dropped = 0;
  __syncthreads();
  for (int i = tid; i < nk; i += kSmallThreads) {
    int e = p.topk_idx[i];
    if (!valid_expert(e, E)) {          // not an expert index: record it, never index with it
      if (i / k == t) set_status(p.status, kDevBadState);
      e = -1;
    }
    idx_s[i] = e;
    if (e >= 0) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  if (tid < k) my_e[tid] = idx_s[t * k + tid];
  for (int e = tid; e < E; e += kSmallThreads) {
    fill[e] = min(hist[e], p.C);
    if (hist[e] > fill[e]) atomicAdd(&s_dropped, hist[e] - fill[e]);
  }
  __syncthreads();
  // rank of each own slot: earlier tokens holding the same expert (a token
  // holds an expert at most once); integer sums, so the order does not matter
  for (int j = 0; j < k; ++j) {
    const int e = my_e[j];
    if (e < 0) continue;
    int c = 0;
    for (int i = tid; i < t * k; i += kSmallThreads) c += idx_s[i] == e;
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0 && c) atomicAdd(&my_rank[j], c);
  }
  // segment starts: exclusive scan of the 128-row-padded fills (one warp)
  if (tid < 32) {
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? (fill[e] + kAlign - 1) / kAlign * kAlign : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < E) offs[e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  if (tid < k) {
    const int e = my_e[tid], r = my_rank[tid];
    const size_t a = (size_t)t * k + tid;
    int f = -1, row = -1;
    if (e >= 0 && r < p.C) { f = e; row = offs[e] + r; }
    p.final_idx[a] = f;
    p.pos[a] = row;
    if (row >= 0) p.perm[row] = t;
    rows[tid] = row;
  }
  if (blockIdx.x == 0) write_layout(p, fill, offs, s_dropped, 0);   // whole CTA
  __syncthreads();
  const int nvec = p.d * (int)sizeof(T) / 16;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.x) + (size_t)t * p.d);
  uint4* dst = reinterpret_cast<uint4*>(p.x_perm);
  for (int v = tid; v < nvec; v += kSmallThreads) {
    const uint4 val = src[v];
    for (int j = 0; j < k; ++j) {
      const int row = rows[j];
      if (row >= 0) dst[(size_t)row * nvec + v] = val;
    }
  }
  if (!MOE_DISPATCH_EARLY_TRIGGER) griddep_launch_dependents();
}

}  // namespace

size_t reroute_scratch_ints(int N, int k, int E) {
  const size_t chunks = (size_t)(N + kRrThreads - 1) / kRrThreads;
  return 2 * (size_t)N * k + 2 * chunks * E;   // rr_prop, rr_rank, two count tables
}

cudaError_t launch_dispatch(const DispatchParams& p, bool bf16, cudaStream_t s) {
  cudaError_t err;
  if (p.cap_mode != 2 && (int64_t)p.N * p.k <= kSmallAssign) {
    err = bf16 ? launch_chained(dispatch_small_kernel<__nv_bfloat16>, p.N, kSmallThreads, 0, s, p)
               : launch_chained(dispatch_small_kernel<float>, p.N, kSmallThreads, 0, s, p);
    if (err != cudaSuccess) return err;
    count_launch();
    return cudaSuccess;
  }
  const int W = kRankTC / 32;
  err = launch_chained(dispatch_rank_kernel, p.n_chunks, kRankTC, sizeof(uint32_t) * p.E * W, s, p);
  if (err != cudaSuccess) return err;
  count_launch();
  err = launch_chained(dispatch_plan_kernel, 1, kPlanThreads, 0, s, p);
  if (err != cudaSuccess) return err;
  count_launch();
  if (p.cap_mode == 2) {
    int dev = 0, sms = 0, per_sm = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return err;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_reroute_kernel,
                                                             kRrThreads, 0)) != cudaSuccess)
      return err;
    const int max_chunks = (p.N + kRrThreads - 1) / kRrThreads;
    int grid = sms * (per_sm < 2 ? per_sm : 2);
    if (grid > max_chunks) grid = max_chunks;
    if (grid < 1) grid = 1;
    DispatchParams q = p;
    void* args[] = {&q};
    err = cudaLaunchCooperativeKernel((const void*)dispatch_reroute_kernel, dim3(grid),
                                      dim3(kRrThreads), args, 0, s);
    if (err != cudaSuccess) return err;
    count_launch();
  }
  err = bf16 ? launch_chained(dispatch_scatter_kernel<__nv_bfloat16>, p.N, 128, 0, s, p)
             : launch_chained(dispatch_scatter_kernel<float>, p.N, 128, 0, s, p);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

}  // namespace moe
