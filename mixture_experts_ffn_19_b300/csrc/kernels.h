// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "grid_barrier.h"

namespace moe {

// Launch `kernel` on `s` with programmatic stream serialisation (the kernel
// calls griddep_wait() before touching its predecessor's data), so its launch
// and set-up overlap the predecessor's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

constexpr int kAlign = 128;        // rows per expert segment granule (= GEMM tile M)
constexpr int kRouteTM = 32;       // tokens per router CTA
constexpr int kRankTC = 256;       // tokens per dispatch-rank CTA
constexpr int kMaxTopk = 8;        // = MOE_MAX_TOPK
constexpr int kMaxExperts = 256;   // = MOE_MAX_EXPERTS

struct RouteParams {
  const void* x;             // [N, d]
  const void* w_router;      // [E, d]
  const float* bias;         // [E] or null
  int bias_select;           // 1: the bias only steers the top-k (p + b)
  int N, d, E, k;
  int32_t* topk_idx;         // [N, k]
  float* topk_w;             // [N, k]
  float* probs;              // [N, E] or null
  float* part;               // [ks, N, E] partial logits (one per K slice)
  // load-balance statistics: exact fixed-point sums of p (2^-40 units) and pick
  // counts, accumulated across CTAs (zeroed before the router runs); the last
  // CTA to finish turns them into the outputs below (each nullable)
  unsigned long long* acc_p; // [E]
  int* acc_pick;             // [E]
  unsigned* ticket;          // [1]
  // z-loss and entropy: sums of lse^2 (2^-24 units) and of H (2^-40 units)
  unsigned long long* acc_zh; // [2]
  float* expert_freq;        // [E]
  float* mean_prob;          // [E]
  float* l_bal;              // [1]
  float* z_loss;             // [1]
  float* entropy;            // [1]
  int* status;
};

cudaError_t launch_quantize_fp8(const void* w, int n_mat, int64_t per_mat, uint8_t* q, float* scales,
                                int num_sms, cudaStream_t s);

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_barrier_selftest(int* status, GridBarrier* bar, uint64_t limit_ns,
                                    int n_barriers, cudaStream_t s);

cudaError_t launch_bias_update(const int* picks, float* bias, int N, int E, int k, float gamma,
                               cudaStream_t s);

// Split of the router contraction over K: ks slices of k_slice (a multiple of 64).
struct RouteSplit {
  int ks, k_slice;
};
RouteSplit route_split(int N, int d, int E, bool bf16);
int route_finish_blocks(int N, int gw);
__host__ __device__ int route_finish_iters(int N, int gw);
cudaError_t launch_route_logits_tc(const RouteSplit& s, const void* x, const void* w_router,
                                   int N, int E, int d, float* part, int* status,
                                   cudaStream_t stream);


constexpr int kMaxRounds = 260;   // reroute rounds never exceed E + 1 <= 257

// Device state shared by the CTAs of the cooperative reroute launch.
struct RerouteState {
  int fill[2][kMaxExperts];      // per-expert fill levels, double-buffered by round
  int any_prop[kMaxRounds];      // round r made at least one proposal
  int primary_kept;
  GridBarrier bar;               // grid barrier of the cooperative kernel
};
size_t reroute_scratch_ints(int N, int k, int E);

struct DispatchParams {
  int N, E, k, S, d, cap_mode, C;
  int n_chunks;
  const int32_t* topk_idx;
  const float* probs;
  const void* x;
  int32_t* chunk_cnt;        // [n_chunks, E]; counts, then exclusive bases
  int32_t* local_rank;       // [N, k]
  int32_t* final_idx;        // [N, k]
  int32_t* slot;             // [N, k]
  int32_t* pos;              // [N, k]
  int32_t* offsets;          // [E+S+1]
  int32_t* perm;             // [max_rows]
  void* x_perm;              // [max_rows, d]
  RerouteState* rr;          // reroute state (workspace)
  int32_t* rr_prop;          // [N, k] proposal of each pending slot in the round
  int32_t* rr_rank;          // [N, k] rank of each proposal inside its 128-token chunk
  int32_t* rr_chunk;         // 2 x [E, ceil(N/128)] proposal counts per chunk (then bases)
  int32_t* counts;           // [E] nullable
  int32_t* n_dropped;        // nullable
  int32_t* n_rerouted;       // nullable
  int* status;
};

struct FfnParams {
  int N, d, F, E, S, k, act;
  const int32_t* offsets;    // [E+S+1]
  const int32_t* counts;     // [E] valid rows of the routed segments, or null
  const void* x;             // [N, d]
  const void* x_perm;        // [max_rows, d]
  const void* w_gate;        // [E+S, F, d]
  const void* w_up;          // [E+S, F, d] or null
  const void* w_down;        // [E+S, d, F]
  const void* b1;            // [E+S, F] or null
  const void* b2;            // [E+S, d] or null
  void* h;                   // [max_total_rows, F]
  void* y_perm;              // [max_total_rows, d]
  int64_t max_rows, max_total_rows;
  int* status;
  int* tile_ctr;             // [2] zeroed ints: GEMM-1's tile-claim and done counters
  int num_sms;
  // E4M3 weights: w_gate / w_up / w_down hold codes and w_scales [3][E+S] the
  // gate, up and down scale of each expert; null for bf16 weights
  const float* w_scales;
  // E4M3 weights: f16 copies of the token rows the gate/up GEMM reads, at
  // x_perm's row indices ([max_rows, d]; may be x_perm itself) and of x for
  // the shared experts ([N, d]); H is then f16 as well
  void* tok16;
  void* x16;
};

struct CombineParams {
  int N, d, E, k, S;
  const void* y_perm;
  const int32_t* offsets;
  const int32_t* final_idx;
  const int32_t* pos;
  const float* topk_w;
  void* y;
};

// Kernels this library has launched in this process (host-side count).
void count_launch();

cudaError_t launch_route(const RouteParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_dispatch(const DispatchParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_ffn_simt(const FfnParams& p, cudaStream_t s, cudaEvent_t mid);
cudaError_t launch_ffn_tc(const FfnParams& p, cudaStream_t s, cudaEvent_t mid);
cudaError_t launch_combine(const CombineParams& p, bool bf16, cudaStream_t s);

}  // namespace moe
