/* CPU oracle of the MoE-FFN forward layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain C++17 loops, one file per stage, every sum accumulated in double in the
 * order its definition writes it.  Only the tests, the smoke check and the CPU
 * baseline of the benchmark load this library; the CUDA library never does,
 * and the two share no code, header or table.
 *
 * Pages cited (by title; section numbers as printed on each page):
 *   [P1] «大模型MoE架构揭秘：如何用2%参数实现万亿级算力调度» (mhpn.cn)
 *   [P2] «项目概述：为什么MoE成了大模型突围的“秘密武器”» (mooersco.com)
 *   [P3] «DeepSeek-V2: A Strong, Economical, and Efficient Mixture-of-Experts
 *        Language Model» -- paper summary page (wzjinhao.cn)
 *   [P4] «GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per Token.» --
 *        rebuttal page (l189.com)
 *   [P5] «为什么MoE有效？稀疏激活的数学直觉与工程实践» (ai.learningdata.cn)
 *
 * Files: numbers.cpp (widening, FP8 E4M3 codec and quantiser), router.cpp
 * (logits, softmax, top-k, gates, statistics, z-loss, entropy, selection
 * bias), capacity.cpp (capacity, drop, reroute, segment membership),
 * experts.cpp (GELU / SwiGLU expert FFN), combine.cpp (gate-weighted sum),
 * layer.cpp (the whole layer over a subset of output tokens).
 *
 * Conventions: arrays are row-major and caller-owned; nothing is allocated
 * that outlives a call.  Tensor element types are given by ORC_* codes.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2, ORC_E4M3 = 3 };

/* One matrix (or vector) operand: element (r, c) is widen(data[r*cols + c]),
 * times `scale` when dtype is ORC_E4M3 (per-matrix scale, reading R16). */
typedef struct {
    const void* data;   /* NULL: absent (a bias that is not there) */
    int32_t dtype;
    float scale;
} orc_mat;

/* ---- threads (OpenMP) ---------------------------------------------------- */
int orc_set_threads(int n);                 /* returns the thread count now in use */
int orc_threads(void);
int orc_hardware_concurrency(void);         /* std::thread::hardware_concurrency() */

/* ---- numbers.cpp ---------------------------------------------------------- */
void orc_widen(const void* src, int32_t dtype, int64_t n, double* dst);
void orc_e4m3_encode(const float* v, int64_t n, uint8_t* codes);
void orc_e4m3_decode(const uint8_t* codes, int64_t n, double* v);
/* one expert matrix of n elements (bf16 / f32) -> codes and per-matrix scale */
void orc_quantize_fp8(const void* w, int32_t dtype, int64_t n, uint8_t* codes, float* scale);
/* scale * value(code), exact in double */
void orc_dequantize_fp8(const uint8_t* codes, int64_t n, float scale, double* v);

/* ---- router.cpp ([P5] §2.2, [P3] §2.2, [P2] §3.3, [P4] §2.3, [P5] §2.4) ---- */
void orc_router_logits(int32_t N, int32_t d, int32_t E, const void* x, int32_t x_dtype,
                       const void* w_router, int32_t w_dtype, const float* bias, double* z);
void orc_softmax_fp32(int32_t N, int32_t E, const double* z, float* p);
void orc_topk(int32_t N, int32_t E, int32_t k, const float* key, int32_t* idx);
void orc_topk_margin(int32_t N, int32_t E, int32_t k, const float* key, double* margin);
void orc_renormalise(int32_t N, int32_t E, int32_t k, const float* p, const int32_t* idx,
                     float* w);
void orc_balance_stats(int32_t N, int32_t E, int32_t k, const float* p, const int32_t* idx,
                       double* freq, double* mean_prob, double* l_bal, int64_t* picks);
double orc_z_loss(int32_t N, int32_t E, const double* z);
double orc_router_entropy(int32_t N, int32_t k, const float* w);
void orc_selection_keys(int32_t N, int32_t E, const float* p, const float* bias, float* key);
void orc_router_bias_update(int32_t E, const float* bias, const int64_t* picks, int64_t n_tokens,
                            int32_t k, float gamma, float* out);

typedef struct {
    double* logits;      /* [N,E] router logits without the expert bias */
    float* p;            /* [N,E] probabilities (float32) */
    float* key;          /* [N,E] what top-k and reroute rank by */
    int32_t* idx;        /* [N,k] */
    float* w;            /* [N,k] renormalised gates */
    double* margin;      /* [N] */
    double* freq;        /* [E] */
    double* mean_prob;   /* [E] */
    int64_t* picks;      /* [E] */
    double l_bal, z_loss, router_entropy;
} orc_route_out;

/* The router stage.  bias_mode 0: bias added to the logits ([P3] §2.2);
 * 1: bias steers the selection only (reading R15).  idx_given (nullable)
 * replaces the top-k selection (one of several equally valid selections of a
 * near-tied token); gates and statistics are then taken for that selection. */
void orc_route(int32_t N, int32_t d, int32_t E, int32_t k, const void* x, int32_t x_dtype,
               const void* w_router, int32_t w_dtype, const float* bias, int32_t bias_mode,
               const int32_t* idx_given, orc_route_out* out);

/* ---- capacity.cpp ([P1] §3.1, §4.2, §5.3) ------------------------------- */
double orc_alpha_for_batch(int64_t n_tokens);
int64_t orc_capacity(int64_t n_tokens, int32_t E, int32_t k, double alpha);

typedef struct {
    int32_t* final_idx;      /* [N,k], -1 = dropped */
    int32_t* members;        /* [N*k] tokens of expert 0, then 1, ... in row order */
    int32_t* member_start;   /* [E+1] */
    int64_t n_dropped, n_rerouted, rounds;
} orc_dispatch_out;

/* cap_mode 0: no limit, 1: drop, 2: reroute.  key [N,E] ranks the reroute
 * candidates (nullable unless cap_mode is 2). */
int orc_dispatch(int32_t N, int32_t E, int32_t k, int32_t cap_mode, int64_t cap,
                 const int32_t* idx, const float* key, orc_dispatch_out* out);

/* ---- experts.cpp ([P1] §3.2, [P5] §3, [P3] §2.3) ------------------------- */
double orc_gelu(double a);
double orc_silu(double a);
void orc_gelu_n(const double* a, int64_t n, double* out);
void orc_silu_n(const double* a, int64_t n, double* out);
/* y[r,:] = FFN(x[r,:]) for R rows.  act 0: GELU(x W1^T + b1) W2^T + b2 with
 * W1 = w_gate [F,d], W2 = w_down [d,F]; act 1: (silu(x Wg^T) * (x Wu^T)) Wd^T. */
void orc_expert_ffn(int32_t act, int32_t d, int32_t F, int64_t R, const double* x,
                    orc_mat w_gate, orc_mat w_up, orc_mat w_down, orc_mat b1, orc_mat b2,
                    double* y);

/* ---- combine.cpp ([P5] §2.1, [P3] §2.3) ---------------------------------- */
/* y = sum_s shared[s] + sum_j gates[j] * routed[j], in that order. */
void orc_combine_token(int32_t d, int32_t S, const double* const* shared, int32_t n_routed,
                       const double* const* routed, const float* gates, double* y);

/* ---- layer.cpp ------------------------------------------------------------ */
/* Experts and combine for the output rows of tokens[0..n_out): routed expert e
 * of token t runs when final_idx[t,j] == e >= 0, shared experts E..E+S-1 run
 * for every token.  experts[(E+S)*5]: w_gate, w_up, w_down, b1, b2 of each
 * expert (an expert that no listed token uses may have NULL data). */
int orc_layer_rows(int32_t N, int32_t d, int32_t E, int32_t k, int32_t F, int32_t S,
                   int32_t act, const void* x, int32_t x_dtype, const int32_t* final_idx,
                   const float* gates, const int64_t* tokens, int64_t n_out,
                   const orc_mat* experts, double* y);

#ifdef __cplusplus
}
#endif
#endif
