/*
 * moe.h -- C ABI of libmoe: the forward pass of one Mixture-of-Experts FFN
 * layer on one NVIDIA B300 (sm_103a).
 *
 * The layer (pages cited by title and section):
 *   router      z = x W_r^T (+ b)          «为什么MoE有效？稀疏激活的数学直觉与工程实践» §2.2;
 *                                           «DeepSeek-V2 ...» summary §2.2 (expert_bias)
 *   softmax     p = softmax(z) in fp32      same sections
 *   top-k       k largest p, gates renormalised to sum 1 (ties -> lower expert index)
 *   capacity    C = floor(floor(k N / E) * alpha); overflow dropped in token order
 *               or rerouted to the next-best expert with room
 *                                           «大模型MoE架构揭秘：如何用2%参数实现万亿级算力调度» §3.1, §4.2
 *   experts     SwiGLU  y = (silu(x Wg^T) * (x Wu^T)) Wd^T   (same page, §3.2)
 *               GELU    y = GELU(x W1^T + b1) W2^T + b2       («为什么MoE有效？» §3 code)
 *               plus S shared experts applied to every token  («DeepSeek-V2 ...» summary §2.3)
 *   combine     y_t = sum_s shared_s(x_t) + sum_j g_tj * expert_{e_tj}(x_t)
 *                                           («为什么MoE有效？» §2.1)
 *   statistics  expert_freq, mean_prob, L_bal = E * sum_e freq_e * P_e
 *                                           («DeepSeek-V2 ...» summary §2.2 load_balance_loss)
 *
 * Conventions for every call:
 *   - Every tensor pointer is a DEVICE pointer, allocated and owned by the
 *     caller.  The library allocates and frees nothing.
 *   - `stream` is a cudaStream_t (passed as void*).  Calls enqueue work on it
 *     and return without synchronising, except moe_device_status().
 *   - A call returns MOE_OK after enqueueing, or a negative moe_status from the
 *     host-side checks done before any launch; then nothing was written.
 *     A failed launch returns MOE_ERR_CUDA.
 *   - Device-side failures (a bounded wait that ran out, an expert index out
 *     of range) are recorded in a status word inside the workspace; read it
 *     with moe_device_status().  moe_route and moe_forward clear it (and the
 *     statistics accumulators next to it) when they start; moe_dispatch and
 *     moe_expert_ffn only add to it, so a fresh workspace used first by one of
 *     those must be zero-filled once (or moe_device_status called once).
 *   - Layouts are row-major.  Weight matrices are nn.Linear style [out, in].
 *     Shared experts are experts E .. E+S-1 of the expert weight arrays.
 *   - dtype MOE_BF16: x, w_router, expert weights, x_perm, y_perm and y are
 *     bf16; router_bias, probabilities and gates are fp32.  MOE_F32: all fp32.
 *   - Alignment: every pointer 16-byte aligned; for bf16, d_model and d_ff are
 *     multiples of 8 (16-byte rows for the tensor-memory-access engine).
 *   - Integer outputs are bit-exact and deterministic; float outputs are
 *     deterministic run to run (no floating-point atomics anywhere).
 *
 * Expert-row space.  Dispatch sorts assignments into one segment per routed
 * expert e (rows offsets[e] .. offsets[e]+counts[e]-1, padded up to a multiple
 * of MOE_SEGMENT_ALIGN rows), followed by one segment of n_tokens rows per
 * shared expert (row offsets[E+s] + t holds token t).  x_perm holds the routed
 * rows; y_perm holds routed and shared rows.  Padding rows hold unspecified
 * values and are never read by the combine.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad size or field     */
  MOE_ERR_UNSUPPORTED = -2,   /* valid but not implemented (e.g. bf16 + GELU)    */
  MOE_ERR_WORKSPACE = -3,     /* workspace smaller than moe_workspace_size()     */
  MOE_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed            */
  MOE_ERR_TIMEOUT = -5,       /* a device-side bounded wait ran out              */
  MOE_ERR_DEVICE = -6         /* another device-side check failed                */
} moe_status;

typedef enum { MOE_ACT_GELU = 0, MOE_ACT_SWIGLU = 1 } moe_act;
typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum { MOE_CAP_NONE = 0, MOE_CAP_DROP = 1, MOE_CAP_REROUTE = 2 } moe_cap_mode;
/* How router_bias enters the routing.  LOGIT: added to the logits before the
 * softmax («DeepSeek-V2 ...» summary §2.2 TopKRouter).  SELECT: the softmax is
 * of the bias-free logits and the bias only steers the choice, top-k of
 * p + b with gates renormalised from p («为什么MoE有效？...» §2.4, the
 * DeepSeek-V3 auxiliary-loss-free scheme). */
typedef enum { MOE_BIAS_LOGIT = 0, MOE_BIAS_SELECT = 1 } moe_bias_mode;

#define MOE_MAX_EXPERTS 256      /* routed experts E                      */
#define MOE_MAX_TOPK 8           /* k <= min(E, 8)                        */
#define MOE_MAX_SHARED 8         /* shared experts S                      */
#define MOE_MAX_TOKENS (1 << 22) /* N                                     */
#define MOE_MAX_DIM 65536        /* d and F: keeps the stacked weights'    *
                                  * row coordinates, (E+S)*F and (E+S)*d,  *
                                  * inside the int32 range of a TMA copy   */
#define MOE_SEGMENT_ALIGN 128    /* rows; segment starts are multiples    */

/* Layer shape and options (plain values, read on the host only). */
typedef struct moe_config {
  int32_t n_tokens;        /* N >= 0 (N = 0 is a no-op)                    */
  int32_t d_model;         /* d, 8 .. MOE_MAX_DIM, a multiple of 8        */
  int32_t n_experts;       /* E routed experts, 1 .. MOE_MAX_EXPERTS       */
  int32_t top_k;           /* k, 1 .. min(E, MOE_MAX_TOPK)                 */
  int32_t d_ff;            /* F, expert hidden width, like d               */
  int32_t n_shared;        /* S, 0 .. MOE_MAX_SHARED                       */
  int32_t act;             /* moe_act                                      */
  int32_t dtype;           /* moe_dtype                                    */
  int32_t cap_mode;        /* moe_cap_mode                                 */
  double alpha;            /* capacity factor (> 0 unless MOE_CAP_NONE), in
                            * double: floor(floor(kN/E) * alpha) must see
                            * the factor as written (0.7 as a float is
                            * 0.69999999, which turns 1250 * 0.7 = 875
                            * into 874)                                   */
  int32_t has_ffn_bias;    /* GELU experts: b1 [E+S, F], b2 [E+S, d]       */
  int32_t has_router_bias; /* router_bias [E] fp32 is given                */
  int32_t bias_mode;       /* moe_bias_mode (with has_router_bias)         */
} moe_config;

/* Statistics outputs (device pointers; each may be NULL = not written). */
typedef struct moe_stats {
  float* expert_freq;  /* [E]  pre-capacity top-k picks of e / (N k)          */
  float* mean_prob;    /* [E]  (1/N) sum_t p[t,e]                              */
  float* l_bal;        /* [1]  E * sum_e expert_freq[e] * mean_prob[e]         */
  int32_t* counts;     /* [E]  assignments kept per routed expert (post-cap)  */
  int32_t* n_dropped;  /* [1]  assignments dropped by capacity                */
  int32_t* n_rerouted; /* [1]  assignments moved to another expert            */
  float* z_loss;       /* [1]  0.001 * mean_t logsumexp(z_t)^2 on the bias-free
                                logits («项目概述：为什么MoE...» §3.3)           */
  float* router_entropy; /* [1] mean_t -sum_j w_tj log2 w_tj over the gates, bits
                                («GPT-4 Has 1.8 Trillion Parameters...» §2.3)  */
} moe_stats;

/* Optional stage timing for moe_forward: cudaEvent_t handles (as void*),
 * recorded on `stream` before the router [0], after the router [1], after
 * dispatch [2], after the first expert GEMM [3], after the second expert GEMM
 * [4] and after the combine [5].  NULL entries are skipped. */
typedef struct moe_timing {
  void* events[6];
} moe_timing;

/* Device pointers into a moe_forward workspace (for inspection and tests). */
typedef struct moe_views {
  int32_t* topk_idx;  /* [N, k]   */
  float* topk_w;      /* [N, k]   */
  float* probs;       /* [N, E]   (written only when cap_mode == REROUTE) */
  int32_t* final_idx; /* [N, k]   */
  int32_t* pos;       /* [N, k]   */
  int32_t* offsets;   /* [E+S+1]  */
  int32_t* perm;      /* [max_rows] */
  void* x_perm;       /* [max_rows, d]        */
  void* h;            /* [max_total_rows, F]  */
  void* y_perm;       /* [max_total_rows, d]  */
} moe_views;

/* ---- host-only queries (no device work, no CUDA context needed) ---------- */

/* Text for a moe_status value. */
const char* moe_status_string(int status);

/* MOE_OK if the configuration is valid and implemented, else the status. */
int moe_validate_config(const moe_config* cfg);

/* Expert capacity C = floor(floor(k*N/E) * alpha) for DROP/REROUTE, -1 for
 * MOE_CAP_NONE or an invalid config («大模型MoE架构揭秘» §3.1). */
int32_t moe_capacity(const moe_config* cfg);

/* Routed rows of x_perm/perm including segment padding (upper bound). */
int64_t moe_max_rows(const moe_config* cfg);

/* Rows of y_perm (routed + shared segments, with padding). */
int64_t moe_max_total_rows(const moe_config* cfg);

/* Bytes of device workspace that every call below needs (0 on error).  The
 * same size serves every call; 256-byte aligned. */
size_t moe_workspace_size(const moe_config* cfg);

/* Pointers into a workspace laid out by moe_forward. */
int moe_workspace_views(const moe_config* cfg, void* workspace, size_t workspace_bytes,
                        moe_views* out);

/* Number of CUDA kernels this library has launched in this process so far
 * (host-side count, every entry point included). */
int64_t moe_kernel_launches(void);

/* ---- device calls ---------------------------------------------------------- */

/* Router: logits, fp32 softmax, top-k with renormalised gates, and the
 * pre-capacity statistics (expert_freq, mean_prob, l_bal, z_loss,
 * router_entropy).
 *   x        [N, d]      w_router [E, d]      router_bias [E] fp32 (NULL unless
 *   has_router_bias)
 *   topk_idx [N, k] int32 out, slot 0 = highest selection score
 *   topk_w   [N, k] fp32  out, renormalised gates (sum 1 per token)
 *   probs    [N, E] fp32  out, nullable: the selection scores the top-k ranks
 *            (the probabilities; p + b under MOE_BIAS_SELECT), which is what
 *            moe_dispatch's reroute ranks by
 *   stats    nullable; expert_freq, mean_prob, l_bal, z_loss, router_entropy
 *            are written where non-NULL (mean_prob averages the probabilities,
 *            never p + b). */
int moe_route(const moe_config* cfg, const void* x, const void* w_router,
              const float* router_bias, int32_t* topk_idx, float* topk_w, float* probs,
              const moe_stats* stats, void* workspace, size_t workspace_bytes, void* stream);

/* Dispatch: per-expert histogram, scan, capacity (drop or reroute), segment
 * layout and the permutation of token rows into x_perm.
 *   topk_idx  [N, k] int32 in (as written by moe_route)
 *   probs     [N, E] fp32 in, required when cap_mode == REROUTE: the
 *             selection scores moe_route wrote (candidate order), else may be NULL
 *   x         [N, d] in
 *   final_idx [N, k] int32 out: expert of the slot after capacity, -1 dropped
 *   pos       [N, k] int32 out: row of the slot in the expert-row space, -1 dropped
 *   offsets   [E+S+1] int32 out: segment start rows; offsets[E+S] = total rows
 *   perm      [moe_max_rows] int32 out: token of each routed row, -1 on padding
 *   x_perm    [moe_max_rows, d] out: x_perm[pos[t,j]] = x[t]
 *   stats     nullable; counts, n_dropped, n_rerouted are written if non-NULL.
 * Within a routed expert, rows are its kept assignments in ascending token
 * order, then rerouted ones in (round, token, slot) order. */
int moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const float* probs,
                 const void* x, int32_t* final_idx, int32_t* pos, int32_t* offsets,
                 int32_t* perm, void* x_perm, const moe_stats* stats, void* workspace,
                 size_t workspace_bytes, void* stream);

/* Expert FFNs of every segment as one grouped computation.
 *   x       [N, d]   in (rows of the shared-expert segments)
 *   x_perm  [moe_max_rows, d] in (rows of the routed segments)
 *   offsets [E+S+1]  in (segment layout from moe_dispatch)
 *   counts  [E]      in, nullable: kept rows per routed expert (stats->counts
 *           of moe_dispatch).  With counts, batches with few tokens per expert
 *           run a variant with the weights as the wide MMA operand; without,
 *           every padded row of every segment is computed (the same sums up to
 *           fp32 summation order)
 *   w_gate  [E+S, F, d]  SwiGLU gate weight | GELU W1
 *   w_up    [E+S, F, d]  SwiGLU up weight   | GELU: NULL
 *   w_down  [E+S, d, F]  down weight (W2)
 *   b1 [E+S, F], b2 [E+S, d]  GELU biases (NULL unless has_ffn_bias)
 *   y_perm  [moe_max_total_rows, d] out
 * bf16 runs on the tensor cores (fp32 accumulation, the SwiGLU product is
 * rounded to bf16 between the two GEMMs); fp32 runs in fp32 on the CUDA cores. */
int moe_expert_ffn(const moe_config* cfg, const void* x, const void* x_perm,
                   const int32_t* offsets, const int32_t* counts, const void* w_gate,
                   const void* w_up, const void* w_down, const void* b1, const void* b2,
                   void* y_perm, void* workspace, size_t workspace_bytes, void* stream);

/* Combine: y[t] = sum_s y_perm[offsets[E+s] + t] + sum_j topk_w[t,j] *
 * y_perm[pos[t,j]] over kept slots, summed in fp32 in that fixed order.
 *   y [N, d] out (dtype). */
int moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* offsets,
                const int32_t* final_idx, const int32_t* pos, const float* topk_w, void* y,
                void* stream);

/* The whole layer: route -> dispatch -> expert FFNs -> combine, all on
 * `stream`, intermediates in `workspace` (see moe_workspace_views).
 *   y [N, d] out; stats nullable; timing nullable. */
int moe_forward(const moe_config* cfg, const void* x, const void* w_router,
                const float* router_bias, const void* w_gate, const void* w_up,
                const void* w_down, const void* b1, const void* b2, void* y,
                const moe_stats* stats, void* workspace, size_t workspace_bytes,
                void* stream, const moe_timing* timing);

/* Auxiliary-loss-free balancing step («为什么MoE有效？...» §2.4): for each
 * expert e, router_bias[e] -= gamma if e got more than N*k/E pre-capacity
 * picks in the last moe_route / moe_forward run on `workspace`, += gamma if
 * fewer, unchanged if equal (fp32 arithmetic).  router_bias [E] fp32 device,
 * updated in place on `stream`, ordered after that run.  The pages give no
 * gamma. */
int moe_router_bias_update(const moe_config* cfg, const void* workspace, size_t workspace_bytes,
                           float* router_bias, float gamma, void* stream);

/* ---- FP8 (E4M3) expert weights --------------------------------------------
 * «大模型MoE架构揭秘：如何用2%参数实现万亿级算力调度» §5.4 and «GPT-4 Has 1.8
 * Trillion Parameters...» §4.4: expert weights in low precision with
 * per-expert scales, router kept in high precision.  Format: OCP FP8 E4M3
 * (bias 7, 3 mantissa bits, subnormals, largest finite 448, no infinities).
 * Weights only: the dequantised weight is scale * value(code); accumulation
 * is fp32.  The tensor cores take the codes widened to f16 (exact) times f16
 * copies of the bf16 token rows (exact from 2^-14 to 65504; smaller values
 * round to f16 subnormals, an absolute error below 2^-25), and H is stored in
 * f16 (finer than the bf16 layer's H).  A finite token value past +-65504,
 * or an H value past it (infinities included), has no f16 form: the call then
 * records MOE_ERR_DEVICE in the device status and its results are not valid. */

/* Quantise n_mat bf16 matrices of rows x cols each (contiguous, row-major):
 * per matrix scale = amax / 448 in fp32 (1 if the matrix is all zero), code =
 * round-to-nearest-even of the fp32 quotient w / scale, saturated to +-448.
 *   w      [n_mat, rows, cols] bf16 in     q [n_mat, rows, cols] uint8 out
 *   scales [n_mat] fp32 out
 * rows * cols must be a multiple of 16; 1 <= n_mat <= 65535. */
int moe_quantize_fp8(const void* w, int32_t n_mat, int64_t rows, int64_t cols, uint8_t* q,
                     float* scales, void* stream);

/* moe_expert_ffn with E4M3 weights (dtype MOE_BF16, MOE_ACT_SWIGLU, no FFN
 * bias; d_model and d_ff multiples of 16).
 *   w_gate, w_up [E+S, F, d] and w_down [E+S, d, F] E4M3 codes
 *   scales [3, E+S] fp32: gate, up and down scale of each expert
 *   counts [E] required (kept rows per routed expert)
 * The f16 token copies go into the workspace (its x_perm and y_perm regions),
 * so x_perm may not be the workspace's own x_perm (moe_workspace_views):
 * MOE_ERR_INVALID_ARG.  Other arguments as moe_expert_ffn. */
int moe_expert_ffn_fp8(const moe_config* cfg, const void* x, const void* x_perm,
                       const int32_t* offsets, const int32_t* counts, const uint8_t* w_gate,
                       const uint8_t* w_up, const uint8_t* w_down, const float* scales,
                       void* y_perm, void* workspace, size_t workspace_bytes, void* stream);

/* moe_forward with E4M3 expert weights (same conditions as
 * moe_expert_ffn_fp8); the router runs on the bf16 w_router as in moe_forward.
 * Afterwards the workspace's x_perm (moe_workspace_views) holds the f16 copies
 * of the kept token rows, and its H is f16. */
int moe_forward_fp8(const moe_config* cfg, const void* x, const void* w_router,
                    const float* router_bias, const uint8_t* w_gate, const uint8_t* w_up,
                    const uint8_t* w_down, const float* scales, void* y, const moe_stats* stats,
                    void* workspace, size_t workspace_bytes, void* stream,
                    const moe_timing* timing);

/* Dispatch without a workspace.  No page has a counterpart: it exists for
 * callers that cannot allocate device memory when they run the layer (a
 * serving process that reserved all its memory up front, or a loop that must
 * not pay the device synchronisation cudaMalloc/cudaFree may cause).  Same
 * arguments and results as moe_dispatch, with the scratch kept in a fixed
 * 8 MiB device array inside the library, which every GPU that loads the
 * library holds until exit; nothing is allocated.
 *   device_status  [1] int32 device pointer, required (MOE_ERR_INVALID_ARG if
 *                  null): cleared by the call, then set to a nonzero code by
 *                  a device-side failure (1 = a wait timed out, 2 = a bad
 *                  expert index or internal check).  It is the only place
 *                  such a failure is reported.
 * Returns MOE_ERR_WORKSPACE when the scratch for these sizes exceeds 8 MiB
 * (about 60k tokens at E=256, k=8).  The first call on a device looks up the
 * array's address (cudaGetSymbolAddress, once per device): make it before any
 * stream capture.  All calls share the array and it keeps the previous call's
 * contents (each call clears what must start at zero); calls whose kernels
 * overlap on the GPU race and give wrong results. */
int moe_dispatch_noalloc(const moe_config* cfg, const int32_t* topk_idx, const float* probs,
                         const void* x, int32_t* final_idx, int32_t* pos, int32_t* offsets,
                         int32_t* perm, void* x_perm, const moe_stats* stats,
                         int32_t* device_status, void* stream);

/* Failure-path self-test (no page has a counterpart: it exercises this
 * library's error handling).  Launches one kernel on `stream` whose bounded
 * wait on an mbarrier that nothing arrives on runs out after limit_us
 * microseconds (1 .. 1,000,000); like a stalled pipeline it records
 * MOE_ERR_TIMEOUT in the workspace status word (read it with
 * moe_device_status) and returns, leaving the context usable.  No fault,
 * trap or unbounded wait is involved.  The status word is the first 4 bytes
 * of any workspace, so any workspace of at least 4 bytes serves. */
int moe_selftest_timeout(void* workspace, size_t workspace_bytes, uint32_t limit_us, void* stream);

/* Grid-barrier failure-path self-test (no page has a counterpart: it exercises
 * this library's error handling).  Launches one cooperative kernel of four
 * CTAs on `stream`: CTA 0 never reaches the grid barrier -- the bounded
 * barrier the cooperative reroute kernel uses -- while the other three run a
 * chain of n_barriers (1 .. 4096) barriers.  Their first wait runs out after
 * limit_us microseconds (1 .. 1,000,000): the first CTA to give up records
 * MOE_ERR_TIMEOUT in the workspace status word and raises the barrier's abort
 * flag, and every CTA then leaves at once, so the kernel ends after about one
 * limit whatever n_barriers is.  The barrier state occupies workspace bytes
 * 16..27 (zeroed by the call, stream-ordered), so the workspace must hold at
 * least 28 bytes; it is overwritten.  No fault, trap or unbounded wait is
 * involved; the context stays usable. */
int moe_selftest_barrier_timeout(void* workspace, size_t workspace_bytes, uint32_t limit_us,
                                 uint32_t n_barriers, void* stream);

/* Synchronises `stream`, then copies the workspace's device status word to
 * *status_out (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE) and clears it. */
int moe_device_status(void* workspace, void* stream, int32_t* status_out);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
