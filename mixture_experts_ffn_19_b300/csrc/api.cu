// C ABI of libmoe (declared in include/moe.h): argument checks, workspace
// layout, and the launch sequence of the layer on one stream.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "moe.h"

namespace moe {
namespace {

constexpr size_t kWsAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int64_t align_rows(int64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Layout {
  size_t status, acc_p, acc_pick, ticket, acc_zh, tile_ctr, zero_end;  // [status .. zero_end) is cleared per call
  size_t topk_idx, topk_w, probs, final_idx, slot, pos, offsets, counts, perm;
  size_t part, chunk_cnt, local_rank, rr_state, rr_scratch;
  size_t x_perm, h, y_perm, total;
};

int64_t max_rows_of(const moe_config* c) {
  return (int64_t)c->n_tokens * c->top_k + (int64_t)c->n_experts * (kAlign - 1);
}
int64_t max_total_rows_of(const moe_config* c) {
  return max_rows_of(c) + (int64_t)c->n_shared * align_rows(c->n_tokens);
}

Layout layout_of(const moe_config* c) {
  Layout L;
  const size_t N = (size_t)c->n_tokens, k = (size_t)c->top_k, E = (size_t)c->n_experts;
  const size_t es = c->dtype == MOE_BF16 ? 2 : 4;
  const RouteSplit rs = route_split(c->n_tokens, c->d_model, c->n_experts, c->dtype == MOE_BF16);
  const size_t chunks = (N + kRankTC - 1) / kRankTC;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = align_up(off + bytes, kWsAlign); return o; };
  L.status = take(sizeof(int32_t));
  L.acc_p = take(E * 8);
  L.acc_pick = take(E * 4);
  L.ticket = take(4);
  L.acc_zh = take(2 * 8);
  L.tile_ctr = take(2 * 4);
  L.zero_end = off;
  L.topk_idx = take(N * k * 4);
  L.topk_w = take(N * k * 4);
  L.probs = take(N * E * 4);
  L.final_idx = take(N * k * 4);
  L.slot = take(N * k * 4);
  L.pos = take(N * k * 4);
  L.offsets = take((E + c->n_shared + 1) * 4);
  L.counts = take(E * 4);
  L.perm = take((size_t)max_rows_of(c) * 4);
  L.part = take((size_t)rs.ks * N * E * 4);
  L.chunk_cnt = take(chunks * E * 4);
  L.local_rank = take(N * k * 4);
  L.rr_state = take(sizeof(RerouteState));
  L.rr_scratch = take(reroute_scratch_ints(c->n_tokens, c->top_k, c->n_experts) * 4);
  L.x_perm = take((size_t)max_rows_of(c) * c->d_model * es);
  L.h = take((size_t)max_total_rows_of(c) * c->d_ff * es);
  L.y_perm = take((size_t)max_total_rows_of(c) * c->d_model * es);
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

int capacity_of(const moe_config* c) {
  if (c->cap_mode == MOE_CAP_NONE) return INT32_MAX;
  const double base = (double)(((int64_t)c->top_k * c->n_tokens) / c->n_experts);
  const double cap = floor(base * c->alpha);
  return cap >= (double)INT32_MAX ? INT32_MAX : (int)cap;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

int check_ws(const moe_config* c, const void* ws, size_t bytes) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (bytes < layout_of(c).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

void record(const moe_timing* t, int i, cudaStream_t s) {
  if (t && t->events[i]) cudaEventRecord(static_cast<cudaEvent_t>(t->events[i]), s);
}

int route_impl(const moe_config* c, const void* x, const void* w_router, const float* bias,
               int32_t* topk_idx, float* topk_w, float* probs, const moe_stats* stats, void* ws,
               cudaStream_t s) {
  const Layout L = layout_of(c);
  RouteParams rp{};
  rp.x = x; rp.w_router = w_router; rp.bias = c->has_router_bias ? bias : nullptr;
  rp.bias_select = c->bias_mode == MOE_BIAS_SELECT;
  rp.N = c->n_tokens; rp.d = c->d_model; rp.E = c->n_experts; rp.k = c->top_k;
  rp.topk_idx = topk_idx; rp.topk_w = topk_w; rp.probs = probs;
  rp.part = at<float>(ws, L.part);
  rp.acc_p = at<unsigned long long>(ws, L.acc_p);
  rp.acc_pick = at<int>(ws, L.acc_pick);
  rp.ticket = at<unsigned>(ws, L.ticket);
  rp.acc_zh = at<unsigned long long>(ws, L.acc_zh);
  if (stats) {
    rp.expert_freq = stats->expert_freq; rp.mean_prob = stats->mean_prob; rp.l_bal = stats->l_bal;
    rp.z_loss = stats->z_loss; rp.entropy = stats->router_entropy;
  }
  rp.status = at<int>(ws, L.status);
  return launch_route(rp, c->dtype == MOE_BF16, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int dispatch_impl(const moe_config* c, const int32_t* topk_idx, const float* probs, const void* x,
                  int32_t* final_idx, int32_t* pos, int32_t* offsets, int32_t* perm, void* x_perm,
                  const moe_stats* stats, void* ws, cudaStream_t s) {
  const Layout L = layout_of(c);
  DispatchParams dp{};
  dp.N = c->n_tokens; dp.E = c->n_experts; dp.k = c->top_k; dp.S = c->n_shared;
  dp.d = c->d_model; dp.cap_mode = c->cap_mode; dp.C = capacity_of(c);
  dp.n_chunks = (c->n_tokens + kRankTC - 1) / kRankTC;
  dp.topk_idx = topk_idx; dp.probs = probs; dp.x = x;
  dp.chunk_cnt = at<int32_t>(ws, L.chunk_cnt);
  dp.local_rank = at<int32_t>(ws, L.local_rank);
  dp.final_idx = final_idx; dp.slot = at<int32_t>(ws, L.slot); dp.pos = pos;
  dp.offsets = offsets; dp.perm = perm; dp.x_perm = x_perm;
  dp.rr = at<RerouteState>(ws, L.rr_state);
  dp.rr_prop = at<int32_t>(ws, L.rr_scratch);
  dp.rr_rank = dp.rr_prop + (size_t)c->n_tokens * c->top_k;
  dp.rr_chunk = dp.rr_rank + (size_t)c->n_tokens * c->top_k;
  dp.counts = stats ? stats->counts : nullptr;
  dp.n_dropped = stats ? stats->n_dropped : nullptr;
  dp.n_rerouted = stats ? stats->n_rerouted : nullptr;
  dp.status = at<int>(ws, L.status);
  return launch_dispatch(dp, c->dtype == MOE_BF16, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int ffn_impl(const moe_config* c, const void* x, const void* x_perm, const int32_t* offsets,
             const int32_t* counts, const void* w_gate, const void* w_up, const void* w_down,
             const void* b1, const void* b2, const float* w_scales, void* y_perm, void* ws,
             cudaStream_t s, cudaEvent_t mid) {
  const Layout L = layout_of(c);
  FfnParams fp{};
  fp.N = c->n_tokens; fp.d = c->d_model; fp.F = c->d_ff; fp.E = c->n_experts;
  fp.S = c->n_shared; fp.k = c->top_k; fp.act = c->act; fp.offsets = offsets; fp.counts = counts;
  fp.x = x; fp.x_perm = x_perm;
  fp.w_gate = w_gate; fp.w_up = w_up; fp.w_down = w_down;
  fp.b1 = c->has_ffn_bias ? b1 : nullptr; fp.b2 = c->has_ffn_bias ? b2 : nullptr;
  fp.h = at<void>(ws, L.h); fp.y_perm = y_perm;
  fp.max_rows = max_rows_of(c); fp.max_total_rows = max_total_rows_of(c);
  fp.status = at<int>(ws, L.status);
  fp.tile_ctr = at<int>(ws, L.tile_ctr);
  fp.num_sms = num_sms();
  fp.w_scales = w_scales;
  if (w_scales) {
    // f16 token copies for the E4M3 GEMMs: the routed rows in the workspace's
    // x_perm (in place when the caller's x_perm is that buffer, as in
    // moe_forward_fp8), the shared experts' copy of x past the routed rows of
    // the workspace's y_perm, which the down GEMM only writes afterwards
    fp.tok16 = at<void>(ws, L.x_perm);
    fp.x16 = c->n_shared > 0 ? static_cast<void*>(at<char>(ws, L.y_perm) +
                                                  (size_t)max_rows_of(c) * c->d_model * 2)
                             : at<void>(ws, L.x_perm);
  }
  const cudaError_t err = c->dtype == MOE_BF16 ? launch_ffn_tc(fp, s, mid) : launch_ffn_simt(fp, s, mid);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int combine_impl(const moe_config* c, const void* y_perm, const int32_t* offsets,
                 const int32_t* final_idx, const int32_t* pos, const float* topk_w, void* y,
                 cudaStream_t s) {
  CombineParams cp{c->n_tokens, c->d_model, c->n_experts, c->top_k, c->n_shared,
                   y_perm, offsets, final_idx, pos, topk_w, y};
  return launch_combine(cp, c->dtype == MOE_BF16, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// The layer, after the caller-specific weight checks: the bf16/fp32 weights
// (w_scales null) or E4M3 codes with their scales.
int forward_impl(const moe_config* c, const void* x, const void* w_router, const float* bias,
                 const void* w_gate, const void* w_up, const void* w_down, const void* b1,
                 const void* b2, const float* w_scales, void* y, const moe_stats* stats, void* ws,
                 size_t ws_bytes, void* stream, const moe_timing* timing) {
  int st = check_ws(c, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (!x || !w_router || !w_gate || !w_down || !y) return MOE_ERR_INVALID_ARG;
  if (c->has_router_bias && !bias) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w_gate) || !aligned16(w_down) ||
      !aligned16(y) || (w_up && !aligned16(w_up)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = layout_of(c);
  if (cudaMemsetAsync(ws, 0, L.zero_end, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (c->n_tokens == 0) return MOE_OK;
  float* probs = c->cap_mode == MOE_CAP_REROUTE ? at<float>(ws, L.probs) : nullptr;
  record(timing, 0, s);
  st = route_impl(c, x, w_router, bias, at<int32_t>(ws, L.topk_idx), at<float>(ws, L.topk_w),
                  probs, stats, ws, s);
  if (st != MOE_OK) return st;
  record(timing, 1, s);
  // the expert GEMMs read the per-expert counts: the caller's array when given
  moe_stats st_fwd{};
  if (stats) st_fwd = *stats;
  if (!st_fwd.counts) st_fwd.counts = at<int32_t>(ws, L.counts);
  st = dispatch_impl(c, at<int32_t>(ws, L.topk_idx), probs, x, at<int32_t>(ws, L.final_idx),
                     at<int32_t>(ws, L.pos), at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.perm),
                     at<void>(ws, L.x_perm), &st_fwd, ws, s);
  if (st != MOE_OK) return st;
  record(timing, 2, s);
  st = ffn_impl(c, x, at<void>(ws, L.x_perm), at<int32_t>(ws, L.offsets), st_fwd.counts, w_gate,
                w_up, w_down, b1, b2, w_scales, at<void>(ws, L.y_perm), ws, s,
                timing ? static_cast<cudaEvent_t>(timing->events[3]) : nullptr);
  if (st != MOE_OK) return st;
  record(timing, 4, s);
  st = combine_impl(c, at<void>(ws, L.y_perm), at<int32_t>(ws, L.offsets),
                    at<int32_t>(ws, L.final_idx), at<int32_t>(ws, L.pos), at<float>(ws, L.topk_w),
                    y, s);
  if (st != MOE_OK) return st;
  record(timing, 5, s);
  return MOE_OK;
}

// E4M3 weights: SwiGLU bf16 layer, rows of 16 bytes for the E4M3 maps.
int validate_fp8(const moe_config* c, const void* w_gate, const void* w_up, const void* w_down,
                 const float* scales) {
  int st = moe_validate_config(c);
  if (st != MOE_OK) return st;
  if (c->dtype != MOE_BF16 || c->act != MOE_ACT_SWIGLU || c->has_ffn_bias) return MOE_ERR_UNSUPPORTED;
  if (c->d_model % 16 != 0 || c->d_ff % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (!w_gate || !w_up || !w_down || !scales || !aligned16(w_up) || !aligned16(scales))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

namespace moe {
namespace {
std::atomic<long long> g_launches{0};
}  // namespace
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace moe

using namespace moe;

extern "C" {

int64_t moe_kernel_launches(void) { return (int64_t)g_launches.load(std::memory_order_relaxed); }

const char* moe_status_string(int st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE: return "device-side check failed";
    default: return "unknown status";
  }
}

int moe_validate_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->n_tokens < 0 || c->n_tokens > MOE_MAX_TOKENS) return MOE_ERR_INVALID_ARG;
  if (c->d_model < 8 || c->d_model > MOE_MAX_DIM || c->d_model % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (c->d_ff < 8 || c->d_ff > MOE_MAX_DIM || c->d_ff % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (c->n_experts < 1 || c->n_experts > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  if (c->top_k < 1 || c->top_k > std::min(c->n_experts, MOE_MAX_TOPK)) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || c->n_shared > MOE_MAX_SHARED) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_GELU && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->cap_mode < MOE_CAP_NONE || c->cap_mode > MOE_CAP_REROUTE) return MOE_ERR_INVALID_ARG;
  if (c->cap_mode != MOE_CAP_NONE && !(c->alpha > 0.0 && isfinite(c->alpha)))
    return MOE_ERR_INVALID_ARG;
  if (c->bias_mode != MOE_BIAS_LOGIT && c->bias_mode != MOE_BIAS_SELECT) return MOE_ERR_INVALID_ARG;
  if (c->has_ffn_bias && c->act != MOE_ACT_GELU) return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_BF16 && (c->act == MOE_ACT_GELU || c->has_ffn_bias)) return MOE_ERR_UNSUPPORTED;
  if (max_total_rows_of(c) >= INT32_MAX) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int32_t moe_capacity(const moe_config* c) {
  if (moe_validate_config(c) != MOE_OK || c->cap_mode == MOE_CAP_NONE) return -1;
  return capacity_of(c);
}

int64_t moe_max_rows(const moe_config* c) {
  return moe_validate_config(c) == MOE_OK ? max_rows_of(c) : -1;
}

int64_t moe_max_total_rows(const moe_config* c) {
  return moe_validate_config(c) == MOE_OK ? max_total_rows_of(c) : -1;
}

size_t moe_workspace_size(const moe_config* c) {
  return moe_validate_config(c) == MOE_OK ? layout_of(c).total : 0;
}

int moe_workspace_views(const moe_config* c, void* ws, size_t bytes, moe_views* out) {
  int st = moe_validate_config(c);
  if (st != MOE_OK) return st;
  if (!out) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(c, ws, bytes)) != MOE_OK) return st;
  const Layout L = layout_of(c);
  out->topk_idx = at<int32_t>(ws, L.topk_idx);
  out->topk_w = at<float>(ws, L.topk_w);
  out->probs = at<float>(ws, L.probs);
  out->final_idx = at<int32_t>(ws, L.final_idx);
  out->pos = at<int32_t>(ws, L.pos);
  out->offsets = at<int32_t>(ws, L.offsets);
  out->perm = at<int32_t>(ws, L.perm);
  out->x_perm = at<void>(ws, L.x_perm);
  out->h = at<void>(ws, L.h);
  out->y_perm = at<void>(ws, L.y_perm);
  return MOE_OK;
}

int moe_route(const moe_config* c, const void* x, const void* w_router, const float* bias,
              int32_t* topk_idx, float* topk_w, float* probs, const moe_stats* stats, void* ws,
              size_t ws_bytes, void* stream) {
  int st = moe_validate_config(c);
  if (st != MOE_OK) return st;
  if ((st = check_ws(c, ws, ws_bytes)) != MOE_OK) return st;
  if (!x || !w_router || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (c->has_router_bias && !bias) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, layout_of(c).zero_end, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (c->n_tokens == 0) return MOE_OK;
  return route_impl(c, x, w_router, bias, topk_idx, topk_w, probs, stats, ws, s);
}

int moe_router_bias_update(const moe_config* c, const void* ws, size_t ws_bytes, float* bias,
                           float gamma, void* stream) {
  int st = moe_validate_config(c);
  if (st != MOE_OK) return st;
  if ((st = check_ws(c, ws, ws_bytes)) != MOE_OK) return st;
  if (!bias || !aligned16(bias) || !isfinite(gamma)) return MOE_ERR_INVALID_ARG;
  if (c->n_tokens == 0) return MOE_OK;
  const Layout L = layout_of(c);
  return launch_bias_update(at<const int>(const_cast<void*>(ws), L.acc_pick), bias, c->n_tokens,
                            c->n_experts, c->top_k, gamma, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

int moe_dispatch(const moe_config* c, const int32_t* topk_idx, const float* probs, const void* x,
                 int32_t* final_idx, int32_t* pos, int32_t* offsets, int32_t* perm, void* x_perm,
                 const moe_stats* stats, void* ws, size_t ws_bytes, void* stream) {
  int st = moe_validate_config(c);
  if (st != MOE_OK) return st;
  if ((st = check_ws(c, ws, ws_bytes)) != MOE_OK) return st;
  if (!topk_idx || !x || !final_idx || !pos || !offsets || !perm || !x_perm)
    return MOE_ERR_INVALID_ARG;
  if (c->cap_mode == MOE_CAP_REROUTE && !probs) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  if (c->n_tokens == 0) return MOE_OK;
  return dispatch_impl(c, topk_idx, probs, x, final_idx, pos, offsets, perm, x_perm, stats, ws,
                       static_cast<cudaStream_t>(stream));
}

int moe_expert_ffn(const moe_config* c, const void* x, const void* x_perm, const int32_t* offsets,
                   const int32_t* counts, const void* w_gate, const void* w_up,
                   const void* w_down, const void* b1, const void* b2, void* y_perm, void* ws,
                   size_t ws_bytes, void* stream) {
  int st = moe_validate_config(c);
  if (st != MOE_OK) return st;
  if ((st = check_ws(c, ws, ws_bytes)) != MOE_OK) return st;
  if (!x || !x_perm || !offsets || !w_gate || !w_down || !y_perm) return MOE_ERR_INVALID_ARG;
  if (c->act == MOE_ACT_SWIGLU && !w_up) return MOE_ERR_INVALID_ARG;
  if (c->has_ffn_bias && (!b1 || !b2)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_down) ||
      !aligned16(y_perm) || (w_up && !aligned16(w_up)))
    return MOE_ERR_INVALID_ARG;
  if (c->n_tokens == 0) return MOE_OK;
  return ffn_impl(c, x, x_perm, offsets, counts, w_gate, w_up, w_down, b1, b2, nullptr, y_perm, ws,
                  static_cast<cudaStream_t>(stream), nullptr);
}

int moe_combine(const moe_config* c, const void* y_perm, const int32_t* offsets,
                const int32_t* final_idx, const int32_t* pos, const float* topk_w, void* y,
                void* stream) {
  int st = moe_validate_config(c);
  if (st != MOE_OK) return st;
  if (!y_perm || !offsets || !final_idx || !pos || !topk_w || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  if (c->n_tokens == 0) return MOE_OK;
  return combine_impl(c, y_perm, offsets, final_idx, pos, topk_w, y,
                      static_cast<cudaStream_t>(stream));
}

int moe_forward(const moe_config* c, const void* x, const void* w_router, const float* bias,
                const void* w_gate, const void* w_up, const void* w_down, const void* b1,
                const void* b2, void* y, const moe_stats* stats, void* ws, size_t ws_bytes,
                void* stream, const moe_timing* timing) {
  int st = moe_validate_config(c);
  if (st != MOE_OK) return st;
  if (c->act == MOE_ACT_SWIGLU && !w_up) return MOE_ERR_INVALID_ARG;
  if (c->has_ffn_bias && (!b1 || !b2)) return MOE_ERR_INVALID_ARG;
  return forward_impl(c, x, w_router, bias, w_gate, w_up, w_down, b1, b2, nullptr, y, stats, ws,
                      ws_bytes, stream, timing);
}

int moe_quantize_fp8(const void* w, int32_t n_mat, int64_t rows, int64_t cols, uint8_t* q,
                     float* scales, void* stream) {
  if (!w || !q || !scales || !aligned16(w) || !aligned16(q) || !aligned16(scales))
    return MOE_ERR_INVALID_ARG;
  if (n_mat < 1 || n_mat > 65535 || rows < 1 || cols < 1 || (rows * cols) % 16 != 0)
    return MOE_ERR_INVALID_ARG;
  return launch_quantize_fp8(w, n_mat, rows * cols, q, scales, num_sms(),
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

int moe_expert_ffn_fp8(const moe_config* c, const void* x, const void* x_perm,
                       const int32_t* offsets, const int32_t* counts, const uint8_t* w_gate,
                       const uint8_t* w_up, const uint8_t* w_down, const float* scales,
                       void* y_perm, void* ws, size_t ws_bytes, void* stream) {
  int st = validate_fp8(c, w_gate, w_up, w_down, scales);
  if (st != MOE_OK) return st;
  if ((st = check_ws(c, ws, ws_bytes)) != MOE_OK) return st;
  if (!x || !x_perm || !offsets || !counts || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
  // the call writes f16 copies of the token rows into the workspace's x_perm
  const Layout L = layout_of(c);
  if (x_perm == at<void>(ws, L.x_perm)) return MOE_ERR_INVALID_ARG;
  if (c->n_tokens == 0) return MOE_OK;
  return ffn_impl(c, x, x_perm, offsets, counts, w_gate, w_up, w_down, nullptr, nullptr, scales,
                  y_perm, ws, static_cast<cudaStream_t>(stream), nullptr);
}

int moe_forward_fp8(const moe_config* c, const void* x, const void* w_router, const float* bias,
                    const uint8_t* w_gate, const uint8_t* w_up, const uint8_t* w_down,
                    const float* scales, void* y, const moe_stats* stats, void* ws,
                    size_t ws_bytes, void* stream, const moe_timing* timing) {
  const int st = validate_fp8(c, w_gate, w_up, w_down, scales);
  if (st != MOE_OK) return st;
  return forward_impl(c, x, w_router, bias, w_gate, w_up, w_down, nullptr, nullptr, scales, y,
                      stats, ws, ws_bytes, stream, timing);
}

int moe_selftest_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream) {
  if (!ws || !aligned16(ws) || ws_bytes < sizeof(int32_t)) return MOE_ERR_INVALID_ARG;
  if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  return launch_wait_selftest(static_cast<int*>(ws), (uint64_t)limit_us * 1000ull,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

int moe_selftest_barrier_timeout(void* ws, size_t ws_bytes, uint32_t limit_us,
                                 uint32_t n_barriers, void* stream) {
  if (!ws || !aligned16(ws) || ws_bytes < 16 + sizeof(GridBarrier)) return MOE_ERR_INVALID_ARG;
  if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  if (n_barriers < 1 || n_barriers > 4096) return MOE_ERR_INVALID_ARG;
  // the status word is the workspace's first 4 bytes; the barrier state sits at byte 16
  GridBarrier* bar = reinterpret_cast<GridBarrier*>(static_cast<char*>(ws) + 16);
  return launch_barrier_selftest(static_cast<int*>(ws), bar, (uint64_t)limit_us * 1000ull,
                                 (int)n_barriers, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

int moe_device_status(void* ws, void* stream, int32_t* status_out) {
  if (!ws || !status_out) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  *status_out = v == kDevOk ? MOE_OK : (v == kDevTimeout ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE);
  return MOE_OK;
}

}  // extern "C"
