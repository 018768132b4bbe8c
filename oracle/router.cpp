// Router stage of the MoE-FFN layer -- test infrastructure only.
//
// Steps and sources:
//   logits   z[t,e] = sum_j x[t,j] Wr[e,j]          [P5] §2.2 (bias-free Linear d -> E)
//   bias     z + b[e] before the softmax              [P3] §2.2 (TopKRouter expert_bias)
//   softmax  p = exp(z - max z) / sum, then float32   [P5] §2.2, [P2] §2.2
//   top-k    k largest, ties to the lower index       [P5] §2.2, reading R1 ([P1] §5.5 "stable")
//   gates    w = p[idx] / sum_j p[idx_j]              [P5] §2.2, [P3] §2.2
//   stats    freq, mean prob, L_bal = E sum f P       [P3] §2.2 (reading R5)
//   z-loss   0.001 mean_t (logsumexp_e z)^2           [P2] §3.3 (reading R13)
//   entropy  mean_t -sum_j w_j log2 w_j               [P4] §2.3, §3.1 (reading R14)
//   selection-only bias and its update rule          [P5] §2.4 (reading R15)
// Every decision (top-k, margins) is taken on the float32 probabilities, as the
// layer's fp32 softmax produces them.
#include <algorithm>
#include <cmath>
#include <functional>
#include <vector>

#include "internal.hpp"

extern "C" {

void orc_router_logits(int32_t N, int32_t d, int32_t E, const void* x, int32_t x_dtype,
                       const void* w_router, int32_t w_dtype, const float* bias, double* z) {
    std::vector<double> wr(static_cast<size_t>(E) * d);
    for (int64_t i = 0; i < static_cast<int64_t>(E) * d; ++i)
        wr[i] = orc_element_raw(w_router, w_dtype, i);
#pragma omp parallel for schedule(dynamic, 16)
    for (int32_t t = 0; t < N; ++t) {
        std::vector<double> xt(d);
        for (int32_t j = 0; j < d; ++j)
            xt[j] = orc_element_raw(x, x_dtype, static_cast<int64_t>(t) * d + j);
        for (int32_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int32_t j = 0; j < d; ++j) acc += xt[j] * wr[static_cast<size_t>(e) * d + j];
            if (bias) acc += static_cast<double>(bias[e]);
            z[static_cast<int64_t>(t) * E + e] = acc;
        }
    }
}

void orc_softmax_fp32(int32_t N, int32_t E, const double* z, float* p) {
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < N; ++t) {
        const double* zt = z + static_cast<int64_t>(t) * E;
        double m = zt[0];
        for (int32_t e = 1; e < E; ++e) m = std::max(m, zt[e]);
        double s = 0.0;
        for (int32_t e = 0; e < E; ++e) s += std::exp(zt[e] - m);
        for (int32_t e = 0; e < E; ++e)
            p[static_cast<int64_t>(t) * E + e] = static_cast<float>(std::exp(zt[e] - m) / s);
    }
}

// Slot j holds the j-th largest key; among equal keys the lower expert index
// comes first (a strict comparison keeps the earlier index).
void orc_topk(int32_t N, int32_t E, int32_t k, const float* key, int32_t* idx) {
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < N; ++t) {
        const float* kt = key + static_cast<int64_t>(t) * E;
        std::vector<char> taken(E, 0);
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || kt[e] > kt[best])) best = e;
            taken[best] = 1;
            idx[static_cast<int64_t>(t) * k + j] = best;
        }
    }
}

// Smallest gap between consecutive keys among the k+1 largest (all E when
// k = E): below 1e-6 a device that rounds the keys differently may choose a
// different set or order its slots differently (reading R17).
void orc_topk_margin(int32_t N, int32_t E, int32_t k, const float* key, double* margin) {
    const int32_t n = std::min(k + 1, E);
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < N; ++t) {
        std::vector<double> s(E);
        for (int32_t e = 0; e < E; ++e) s[e] = static_cast<double>(key[static_cast<int64_t>(t) * E + e]);
        std::sort(s.begin(), s.end(), std::greater<double>());
        double m = INFINITY;
        for (int32_t i = 0; i + 1 < n; ++i) m = std::min(m, s[i] - s[i + 1]);
        margin[t] = m;
    }
}

void orc_renormalise(int32_t N, int32_t E, int32_t k, const float* p, const int32_t* idx, float* w) {
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < N; ++t) {
        double s = 0.0;
        for (int32_t j = 0; j < k; ++j)
            s += static_cast<double>(p[static_cast<int64_t>(t) * E + idx[static_cast<int64_t>(t) * k + j]]);
        for (int32_t j = 0; j < k; ++j) {
            const double pj = p[static_cast<int64_t>(t) * E + idx[static_cast<int64_t>(t) * k + j]];
            w[static_cast<int64_t>(t) * k + j] = static_cast<float>(pj / s);
        }
    }
}

// [P3] §2.2: freq_e = picks_e / (N k) over the pre-capacity top-k picks,
// P_e = (1/N) sum_t p[t,e], L_bal = E sum_e freq_e P_e.
void orc_balance_stats(int32_t N, int32_t E, int32_t k, const float* p, const int32_t* idx,
                       double* freq, double* mean_prob, double* l_bal, int64_t* picks) {
    for (int32_t e = 0; e < E; ++e) picks[e] = 0;
    for (int64_t i = 0; i < static_cast<int64_t>(N) * k; ++i) picks[idx[i]] += 1;
    double l = 0.0;
    for (int32_t e = 0; e < E; ++e) {
        double s = 0.0;
        for (int32_t t = 0; t < N; ++t) s += static_cast<double>(p[static_cast<int64_t>(t) * E + e]);
        freq[e] = N > 0 ? static_cast<double>(picks[e]) / (static_cast<double>(N) * k) : 0.0;
        mean_prob[e] = N > 0 ? s / N : 0.0;
        l += freq[e] * mean_prob[e];
    }
    *l_bal = E * l;
}

double orc_z_loss(int32_t N, int32_t E, const double* z) {
    if (N == 0) return 0.0;
    double s = 0.0;
    for (int32_t t = 0; t < N; ++t) {
        const double* zt = z + static_cast<int64_t>(t) * E;
        double m = zt[0];
        for (int32_t e = 1; e < E; ++e) m = std::max(m, zt[e]);
        double se = 0.0;
        for (int32_t e = 0; e < E; ++e) se += std::exp(zt[e] - m);
        const double lse = m + std::log(se);
        s += lse * lse;
    }
    return 0.001 * (s / N);
}

double orc_router_entropy(int32_t N, int32_t k, const float* w) {
    if (N == 0) return 0.0;
    double s = 0.0;
    for (int32_t t = 0; t < N; ++t) {
        double h = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            const double v = w[static_cast<int64_t>(t) * k + j];
            if (v > 0.0) h += -v * std::log2(v);      // 0 log 0 = 0
        }
        s += h;
    }
    return s / N;
}

// key[t,e] = p[t,e] + b[e] in float32 arithmetic.
void orc_selection_keys(int32_t N, int32_t E, const float* p, const float* bias, float* key) {
    for (int64_t t = 0; t < N; ++t)
        for (int32_t e = 0; e < E; ++e) {
            const float v = p[t * E + e] + bias[e];
            key[t * E + e] = v;
        }
}

// b_e - gamma when picks_e > N k / E, b_e + gamma when below, unchanged when
// equal; picks_e * E is compared with N * k so that no division rounds.
void orc_router_bias_update(int32_t E, const float* bias, const int64_t* picks, int64_t n_tokens,
                            int32_t k, float gamma, float* out) {
    for (int32_t e = 0; e < E; ++e) {
        const int64_t load = picks[e] * E;
        const int64_t mean = n_tokens * k;
        float b = bias[e];
        if (load > mean) b = b - gamma;
        else if (load < mean) b = b + gamma;
        out[e] = b;
    }
}

void orc_route(int32_t N, int32_t d, int32_t E, int32_t k, const void* x, int32_t x_dtype,
               const void* w_router, int32_t w_dtype, const float* bias, int32_t bias_mode,
               const int32_t* idx_given, orc_route_out* o) {
    orc_router_logits(N, d, E, x, x_dtype, w_router, w_dtype, nullptr, o->logits);
    const int64_t NE = static_cast<int64_t>(N) * E;
    if (bias && bias_mode == 1) {
        orc_softmax_fp32(N, E, o->logits, o->p);
        orc_selection_keys(N, E, o->p, bias, o->key);
    } else {
        std::vector<double> zb(o->logits, o->logits + NE);
        if (bias)
            for (int64_t t = 0; t < N; ++t)
                for (int32_t e = 0; e < E; ++e) zb[t * E + e] += static_cast<double>(bias[e]);
        orc_softmax_fp32(N, E, zb.data(), o->p);
        for (int64_t i = 0; i < NE; ++i) o->key[i] = o->p[i];
    }
    if (idx_given)
        for (int64_t i = 0; i < static_cast<int64_t>(N) * k; ++i) o->idx[i] = idx_given[i];
    else
        orc_topk(N, E, k, o->key, o->idx);
    orc_renormalise(N, E, k, o->p, o->idx, o->w);
    orc_topk_margin(N, E, k, o->key, o->margin);
    orc_balance_stats(N, E, k, o->p, o->idx, o->freq, o->mean_prob, &o->l_bal, o->picks);
    o->z_loss = orc_z_loss(N, E, o->logits);
    o->router_entropy = orc_router_entropy(N, k, o->w);
}

}  // extern "C"
