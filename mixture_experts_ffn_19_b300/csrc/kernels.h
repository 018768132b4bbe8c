// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kAlign = 128;        // rows per expert segment granule (= GEMM tile M)
constexpr int kRouteTM = 32;       // tokens per router CTA
constexpr int kRankTC = 256;       // tokens per dispatch-rank CTA
constexpr int kMaxTopk = 8;        // = MOE_MAX_TOPK
constexpr int kMaxExperts = 256;   // = MOE_MAX_EXPERTS

struct RouteParams {
  const void* x;             // [N, d]
  const void* w_router;      // [E, d]
  const float* bias;         // [E] or null
  int N, d, E, k;
  int32_t* topk_idx;         // [N, k]
  float* topk_w;             // [N, k]
  float* probs;              // [N, E] or null
  float* psum_part;          // [blocks, E]
  int32_t* picks_part;       // [blocks, E]
};

struct RouteStatsParams {
  const float* psum_part;
  const int32_t* picks_part;
  int blocks, N, E, k;
  float* expert_freq;        // nullable
  float* mean_prob;          // nullable
  float* l_bal;              // nullable
};

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
  int32_t* pend;             // [N] scratch (pending token list)
  int32_t* counts;           // [E] nullable
  int32_t* n_dropped;        // nullable
  int32_t* n_rerouted;       // nullable
  int* status;
};

struct FfnParams {
  int N, d, F, E, S, act;
  const int32_t* offsets;    // [E+S+1]
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
  int num_sms;
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

cudaError_t launch_route(const RouteParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_route_stats(const RouteStatsParams& p, cudaStream_t s);
cudaError_t launch_dispatch(const DispatchParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_ffn_simt(const FfnParams& p, cudaStream_t s, cudaEvent_t mid);
cudaError_t launch_ffn_tc(const FfnParams& p, cudaStream_t s, cudaEvent_t mid);
cudaError_t launch_combine(const CombineParams& p, bool bf16, cudaStream_t s);

}  // namespace moe
