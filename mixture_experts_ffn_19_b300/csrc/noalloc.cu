// moe_dispatch_noalloc: the dispatch step (histogram, scan, capacity with drop
// or reroute, segment layout, row permutation) for callers that cannot hand
// the library a workspace.
//
// Some programs cannot call cudaMalloc when they run the layer: a serving
// process that reserved all of its device memory up front and hands out
// nothing afterwards, or a host loop that must not pay the implicit device
// synchronisation an allocation or a free may cause.  This entry point needs
// no workspace: its scratch (per-chunk counts, in-chunk ranks, reroute state
// and the device status word) lives in one file-scope device array of
// kScratchBytes, part of the library's device image.  Every GPU that loads the
// library holds that array until the process exits.
//
// Rules of use:
//  * Sizes whose scratch exceeds kScratchBytes are rejected with
//    MOE_ERR_WORKSPACE before any launch (roughly 60k tokens at E=256, k=8;
//    the 64-expert top-2 layer at 16k tokens needs under 1 MiB).
//  * The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (once per device, cached); make that first call
//    before any stream capture begins.
//  * Every call shares the one array and it keeps the previous call's
//    contents: each call clears the status word before its kernels run, and
//    every other scratch byte is written before it is read.  Two calls whose
//    kernels overlap on the GPU (different streams, or different host
//    threads without ordering) race on the array and give wrong results.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "moe.h"

namespace moe {
namespace {

constexpr size_t kScratchBytes = 8u << 20;   // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_scratch);
    if (err != cudaSuccess) return err;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

struct ScratchLayout {
  size_t chunk_cnt, local_rank, slot, rr_state, rr_scratch, total;
};

ScratchLayout scratch_layout(const moe_config* c) {
  ScratchLayout L;
  const size_t N = (size_t)c->n_tokens, k = (size_t)c->top_k, E = (size_t)c->n_experts;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = up256(off + bytes); return o; };
  L.chunk_cnt = take((N + kRankTC - 1) / kRankTC * E * 4);
  L.local_rank = take(N * k * 4);
  L.slot = take(N * k * 4);
  L.rr_state = take(sizeof(RerouteState));
  L.rr_scratch = take(reroute_scratch_ints(c->n_tokens, c->top_k, c->n_experts) * 4);
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_dispatch_noalloc(const moe_config* cfg, const int32_t* topk_idx,
                                    const float* probs, const void* x, int32_t* final_idx,
                                    int32_t* pos, int32_t* offsets, int32_t* perm, void* x_perm,
                                    const moe_stats* stats, int32_t* device_status,
                                    void* stream) {
  using namespace moe;
  int st = moe_validate_config(cfg);
  if (st != MOE_OK) return st;
  // device_status is required: the scratch array is not readable through any
  // entry point, so a failure recorded there would go unreported
  if (!topk_idx || !x || !final_idx || !pos || !offsets || !perm || !x_perm || !device_status)
    return MOE_ERR_INVALID_ARG;
  if (cfg->cap_mode == MOE_CAP_REROUTE && !probs) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  const ScratchLayout L = scratch_layout(cfg);
  if (L.total > kScratchBytes) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = nullptr;
  if (scratch_address(reinterpret_cast<void**>(&base)) != cudaSuccess) return MOE_ERR_CUDA;
  int* status = device_status;
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cfg->n_tokens == 0) return MOE_OK;

  DispatchParams dp{};
  dp.N = cfg->n_tokens; dp.E = cfg->n_experts; dp.k = cfg->top_k; dp.S = cfg->n_shared;
  dp.d = cfg->d_model; dp.cap_mode = cfg->cap_mode;
  dp.C = cfg->cap_mode == MOE_CAP_NONE ? INT32_MAX : moe_capacity(cfg);
  dp.n_chunks = (cfg->n_tokens + kRankTC - 1) / kRankTC;
  dp.topk_idx = topk_idx; dp.probs = probs; dp.x = x;
  dp.chunk_cnt = reinterpret_cast<int32_t*>(base + L.chunk_cnt);
  dp.local_rank = reinterpret_cast<int32_t*>(base + L.local_rank);
  dp.final_idx = final_idx;
  dp.slot = reinterpret_cast<int32_t*>(base + L.slot);
  dp.pos = pos; dp.offsets = offsets; dp.perm = perm; dp.x_perm = x_perm;
  dp.rr = reinterpret_cast<RerouteState*>(base + L.rr_state);
  dp.rr_prop = reinterpret_cast<int32_t*>(base + L.rr_scratch);
  dp.rr_rank = dp.rr_prop + (size_t)cfg->n_tokens * cfg->top_k;
  dp.rr_chunk = dp.rr_rank + (size_t)cfg->n_tokens * cfg->top_k;
  dp.counts = stats ? stats->counts : nullptr;
  dp.n_dropped = stats ? stats->n_dropped : nullptr;
  dp.n_rerouted = stats ? stats->n_rerouted : nullptr;
  dp.status = status;
  return launch_dispatch(dp, cfg->dtype == MOE_BF16, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
