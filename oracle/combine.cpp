// Combine stage of the MoE-FFN layer -- test infrastructure only.
//
//   y_t = sum_s Shared_s(x_t) + sum_j g_j Expert_{e_j}(x_t)
// [P5] §2.1 writes the layer as y = sum_i g_i(x) Expert_i(x); [P3] §2.3 adds the
// always-on shared experts' outputs.  Dropped slots are not passed in: they
// contribute nothing and their gate is not given to the other slots (reading R3).
#include "internal.hpp"

extern "C" {

void orc_combine_token(int32_t d, int32_t S, const double* const* shared, int32_t n_routed,
                       const double* const* routed, const float* gates, double* y) {
    for (int32_t i = 0; i < d; ++i) {
        double v = 0.0;
        for (int32_t s = 0; s < S; ++s) v += shared[s][i];
        for (int32_t j = 0; j < n_routed; ++j) v += static_cast<double>(gates[j]) * routed[j][i];
        y[i] = v;
    }
}

}  // extern "C"
