// Number formats of the layer's inputs -- test infrastructure only.
//
// Widening: bf16 is the top half of a binary32 pattern, so a bf16 value is the
// binary32 with sixteen zero low bits; binary32 and binary64 values widen to
// double exactly.
//
// FP8 E4M3 (reading R16; [P1] §5.4 and [P4] §4.4 ask for low-precision expert
// weights with per-expert scales and leave the format open): the OCP 8-bit
// format with 1 sign bit, 4 exponent bits of bias 7 and 3 mantissa bits.  A
// code with exponent field e = 1..15 and mantissa m is (1 + m/8) * 2^(e-7);
// e = 0 is the subnormal m * 2^-9; S.1111.111 is NaN and there is no infinity,
// so the largest finite value is 1.75 * 2^8 = 448.  Encoding rounds to the
// nearest code, ties to the even code, and saturates at 448.
#include "internal.hpp"

#include <cfenv>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include <omp.h>

namespace {

double widen_one(const void* src, int32_t dtype, int64_t i) {
    switch (dtype) {
    case ORC_F32: return static_cast<double>(static_cast<const float*>(src)[i]);
    case ORC_F64: return static_cast<const double*>(src)[i];
    case ORC_BF16: {
        uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(src)[i]) << 16;
        float f;
        std::memcpy(&f, &bits, 4);
        return static_cast<double>(f);
    }
    default: return NAN;
    }
}

double e4m3_value(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double mag;
    if ((c & 0x7F) == 0x7F) return NAN;
    if (e == 0) mag = m * std::ldexp(1.0, -9);
    else mag = (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);
    return s ? -mag : mag;
}

uint8_t e4m3_code(float v) {
    // round-half-even of a real quotient: nearbyint under the default rounding mode
    const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
    const double a = std::fabs(static_cast<double>(v));
    int code;
    if (a >= 448.0) {
        code = 0x7E;                                   // saturate
    } else if (a < std::ldexp(1.0, -6)) {
        // subnormal range: multiples of 2^-9; a result of 8 is the smallest normal
        code = static_cast<int>(std::nearbyint(a / std::ldexp(1.0, -9)));
    } else {
        int ex;
        std::frexp(a, &ex);                            // a = f * 2^ex, f in [0.5, 1)
        int e = ex - 1;                                // a in [2^e, 2^(e+1))
        int m = static_cast<int>(std::nearbyint(a / std::ldexp(1.0, e - 3)));   // 8..16
        if (m == 16) { ++e; m = 8; }
        code = ((e + 7) << 3) | (m - 8);
    }
    return static_cast<uint8_t>(code) | sign;
}

}  // namespace

extern "C" {

int orc_set_threads(int n) {
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
}

int orc_threads(void) { return omp_get_max_threads(); }

int orc_hardware_concurrency(void) {
    return static_cast<int>(std::thread::hardware_concurrency());
}

void orc_widen(const void* src, int32_t dtype, int64_t n, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = widen_one(src, dtype, i);
}

void orc_e4m3_encode(const float* v, int64_t n, uint8_t* codes) {
    std::fesetround(FE_TONEAREST);
    for (int64_t i = 0; i < n; ++i) codes[i] = e4m3_code(v[i]);
}

void orc_e4m3_decode(const uint8_t* codes, int64_t n, double* v) {
    for (int64_t i = 0; i < n; ++i) v[i] = e4m3_value(codes[i]);
}

// scale = amax / 448 in float32 (1 for an all-zero matrix); code = E4M3 of the
// float32 quotient w / scale.
void orc_quantize_fp8(const void* w, int32_t dtype, int64_t n, uint8_t* codes, float* scale) {
    std::fesetround(FE_TONEAREST);
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = std::fabs(static_cast<float>(widen_one(w, dtype, i)));
        if (a > amax) amax = a;
    }
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float q = static_cast<float>(widen_one(w, dtype, i)) / s;
        codes[i] = e4m3_code(q);
    }
    *scale = s;
}

void orc_dequantize_fp8(const uint8_t* codes, int64_t n, float scale, double* v) {
    for (int64_t i = 0; i < n; ++i) v[i] = e4m3_value(codes[i]) * static_cast<double>(scale);
}

}  // extern "C"

// Widening used by the other oracle files (declared where used).
double orc_element(const orc_mat& m, int64_t i) {
    if (m.dtype == ORC_E4M3)
        return e4m3_value(static_cast<const uint8_t*>(m.data)[i]) * static_cast<double>(m.scale);
    return widen_one(m.data, m.dtype, i);
}

double orc_element_raw(const void* src, int32_t dtype, int64_t i) { return widen_one(src, dtype, i); }

namespace {

template <typename Load>
double dot_loop(const double* x, int32_t n, Load load) {
    double a = 0.0;
    for (int32_t j = 0; j < n; ++j) a += x[j] * load(j);
    return a;
}

}  // namespace

double orc_dot_row(const double* x, const orc_mat& m, int64_t offset, int32_t n) {
    switch (m.dtype) {
    case ORC_F32: {
        const float* p = static_cast<const float*>(m.data) + offset;
        return dot_loop(x, n, [p](int32_t j) { return static_cast<double>(p[j]); });
    }
    case ORC_F64: {
        const double* p = static_cast<const double*>(m.data) + offset;
        return dot_loop(x, n, [p](int32_t j) { return p[j]; });
    }
    case ORC_BF16: {
        const uint16_t* p = static_cast<const uint16_t*>(m.data) + offset;
        return dot_loop(x, n, [p](int32_t j) {
            const uint32_t bits = static_cast<uint32_t>(p[j]) << 16;
            float f;
            std::memcpy(&f, &bits, 4);
            return static_cast<double>(f);
        });
    }
    case ORC_E4M3: {
        static const std::vector<double> value = [] {
            std::vector<double> v(256);
            for (int c = 0; c < 256; ++c) v[c] = e4m3_value(static_cast<uint8_t>(c));
            return v;
        }();
        const uint8_t* p = static_cast<const uint8_t*>(m.data) + offset;
        const double s = static_cast<double>(m.scale);
        return dot_loop(x, n, [p, s](int32_t j) { return value[p[j]] * s; });
    }
    default: return NAN;
    }
}
