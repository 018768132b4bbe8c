// Helpers shared by the oracle's own files (test infrastructure only).
#pragma once

#include <cstdint>
#include <vector>

#include "moe_oracle.h"

// Exact value of element i of an operand (E4M3 codes times their scale).
double orc_element(const orc_mat& m, int64_t i);
// Exact value of element i of a bf16 / f32 / f64 array.
double orc_element_raw(const void* src, int32_t dtype, int64_t i);

// sum_{j < n} x[j] * m[offset + j], j ascending, in double: one row of a
// row-major operand against a vector, each element widened where it is read.
double orc_dot_row(const double* x, const orc_mat& m, int64_t offset, int32_t n);

// n consecutive elements of an operand, widened to double (short vectors).
inline std::vector<double> orc_widened(const orc_mat& m, int64_t n) {
    std::vector<double> out(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) out[static_cast<size_t>(i)] = orc_element(m, i);
    return out;
}
