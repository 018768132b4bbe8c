// The MoE-FFN layer's expert and combine stages over a subset of output rows
// -- test infrastructure only.
//
// Routing and capacity couple every token of a batch, so they always run over
// the whole batch (router.cpp, capacity.cpp).  Once each token's kept experts
// and gates are known, an output row depends on its own token only ([P5] §2.1:
// y = sum_i g_i(x) Expert_i(x)), so the rows of any subset of tokens can be
// computed alone: each routed expert runs on the listed tokens that kept it,
// each shared expert on every listed token ([P3] §2.3), then the combine sums
// them per token in a fixed order (shared experts, then slots in order).
#include <vector>

#include "internal.hpp"

extern "C" {

int orc_layer_rows(int32_t N, int32_t d, int32_t E, int32_t k, int32_t F, int32_t S,
                   int32_t act, const void* x, int32_t x_dtype, const int32_t* final_idx,
                   const float* gates, const int64_t* tokens, int64_t n_out,
                   const orc_mat* experts, double* y) {
    for (int64_t i = 0; i < n_out; ++i)
        if (tokens[i] < 0 || tokens[i] >= N) return -1;
    auto x_row = [&](int64_t t, double* dst) {
        for (int32_t j = 0; j < d; ++j) dst[j] = orc_element_raw(x, x_dtype, t * d + j);
    };
    auto run_expert = [&](int32_t e, const std::vector<int64_t>& toks, double* out) {
        std::vector<double> xs(toks.size() * static_cast<size_t>(d));
        for (size_t r = 0; r < toks.size(); ++r) x_row(toks[r], xs.data() + r * d);
        const orc_mat* m = experts + static_cast<int64_t>(e) * 5;
        orc_expert_ffn(act, d, F, static_cast<int64_t>(toks.size()), xs.data(), m[0], m[1], m[2],
                       m[3], m[4], out);
    };

    // routed experts: out_routed[(i k + j) d ...] for kept slot j of listed token i
    std::vector<double> out_routed(static_cast<size_t>(n_out) * k * d, 0.0);
    for (int32_t e = 0; e < E; ++e) {
        std::vector<int64_t> toks, where;
        for (int64_t i = 0; i < n_out; ++i)
            for (int32_t j = 0; j < k; ++j)
                if (final_idx[tokens[i] * k + j] == e) {
                    toks.push_back(tokens[i]);
                    where.push_back(i * k + j);
                }
        if (toks.empty()) continue;
        const orc_mat* m = experts + static_cast<int64_t>(e) * 5;
        if (!m[0].data || !m[2].data || (act == 1 && !m[1].data)) return -2;
        std::vector<double> ye(toks.size() * static_cast<size_t>(d));
        run_expert(e, toks, ye.data());
        for (size_t r = 0; r < toks.size(); ++r)
            for (int32_t c = 0; c < d; ++c) out_routed[where[r] * d + c] = ye[r * d + c];
    }

    // shared experts: every listed token
    std::vector<std::vector<double>> out_shared(S);
    std::vector<int64_t> all(tokens, tokens + n_out);
    for (int32_t s = 0; s < S; ++s) {
        const orc_mat* m = experts + static_cast<int64_t>(E + s) * 5;
        if (!m[0].data || !m[2].data || (act == 1 && !m[1].data)) return -2;
        out_shared[s].assign(static_cast<size_t>(n_out) * d, 0.0);
        if (n_out > 0) run_expert(E + s, all, out_shared[s].data());
    }

    for (int64_t i = 0; i < n_out; ++i) {
        std::vector<const double*> sh(S), rt;
        std::vector<float> g;
        for (int32_t s = 0; s < S; ++s) sh[s] = out_shared[s].data() + i * d;
        for (int32_t j = 0; j < k; ++j)
            if (final_idx[tokens[i] * k + j] >= 0) {
                rt.push_back(out_routed.data() + (i * k + j) * d);
                g.push_back(gates[tokens[i] * k + j]);
            }
        orc_combine_token(d, S, sh.data(), static_cast<int32_t>(rt.size()), rt.data(), g.data(),
                          y + i * d);
    }
    return 0;
}

}  // extern "C"
