// Expert FFNs of the MoE-FFN layer -- test infrastructure only.
//
//   SwiGLU expert   y = (silu(x Wg^T) * (x Wu^T)) Wd^T       [P1] §3.2 names SwiGLU experts
//                   silu(a) = a / (1 + e^-a)                 (reading R6: gate on the silu branch)
//   GELU expert     y = GELU(x W1^T + b1) W2^T + b2          [P5] §3 code: Linear -> GELU -> Linear
//                   GELU(a) = a Phi(a) = 0.5 a (1 + erf(a / sqrt 2))   (reading R7: erf form)
//   shared experts  the same FFN, applied to every token     [P3] §2.3
// Everything is accumulated in double; the intermediate h stays in double
// (the definition; reading R10).  Weights are widened where they are read.
#include <cmath>
#include <vector>

#include "internal.hpp"

extern "C" {

double orc_gelu(double a) { return 0.5 * a * (1.0 + std::erf(a / std::sqrt(2.0))); }

double orc_silu(double a) { return a / (1.0 + std::exp(-a)); }

void orc_gelu_n(const double* a, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_gelu(a[i]);
}

void orc_silu_n(const double* a, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_silu(a[i]);
}

void orc_expert_ffn(int32_t act, int32_t d, int32_t F, int64_t R, const double* x,
                    orc_mat w_gate, orc_mat w_up, orc_mat w_down, orc_mat b1, orc_mat b2,
                    double* y) {
    const std::vector<double> bb1 = (act == 0 && b1.data) ? orc_widened(b1, F) : std::vector<double>();
    const std::vector<double> bb2 = (act == 0 && b2.data) ? orc_widened(b2, d) : std::vector<double>();

    // rows one after another; the output features of a row are independent,
    // so each parallel loop shares them out over the threads
    std::vector<double> h(F);
    for (int64_t r = 0; r < R; ++r) {
        const double* xr = x + r * d;
#pragma omp parallel for schedule(static)
        for (int32_t f = 0; f < F; ++f) {
            const int64_t row = static_cast<int64_t>(f) * d;
            double a = orc_dot_row(xr, w_gate, row, d);           // (x W^T)[f]
            if (act == 0) {
                if (!bb1.empty()) a += bb1[f];
                h[f] = orc_gelu(a);
            } else {
                const double u = orc_dot_row(xr, w_up, row, d);
                h[f] = orc_silu(a) * u;
            }
        }
#pragma omp parallel for schedule(static)
        for (int32_t i = 0; i < d; ++i) {
            double v = orc_dot_row(h.data(), w_down, static_cast<int64_t>(i) * F, F);
            if (!bb2.empty()) v += bb2[i];
            y[r * d + i] = v;
        }
    }
}

}  // extern "C"
