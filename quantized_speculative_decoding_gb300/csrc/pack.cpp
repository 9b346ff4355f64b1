// Host-side weight packers of libsd.so: sd_w4_pack, sd_wb_pack and sd_w8_pack.
//
// Weight formats of the pages: the INT4 (AWQ / GPTQ-style) group-quantised
// target and draft ("The Free Half of Speculative Decoding", para. 3; "When Do
// Quantized Drafts Help Speculative Decoding?", pilot setup), and the GPTQ
// INT8 draft (same page).  The exact rounding rules are stated in sd.h.
//
// fp16 conversions here work on the IEEE-754 bit patterns with integer
// arithmetic (round to nearest even).
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/sd.h"

namespace {

uint16_t half_bits_from_double(double d) {
    uint64_t b;
    std::memcpy(&b, &d, sizeof b);
    const uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    const int dexp = (int)((b >> 52) & 0x7ff);
    const uint64_t frac = b & ((1ull << 52) - 1);
    if (dexp == 0x7ff) return (uint16_t)(sign | 0x7c00u | (frac ? 0x200u : 0u));
    if (dexp == 0) return sign;  // zero or a double subnormal: far below fp16's range
    const int e = dexp - 1023;   // value = sig * 2^(e - 52), sig has 53 bits
    const uint64_t sig = frac | (1ull << 52);
    int shift;                   // low bits of sig dropped by the rounding
    int hexp;                    // biased fp16 exponent (0 = subnormal)
    if (e >= -14) {
        shift = 42;
        hexp = e + 15;
    } else {
        shift = 42 + (-14 - e);
        hexp = 0;
    }
    if (shift > 63) return sign;
    uint64_t q = sig >> shift;
    const uint64_t rem = sig & ((1ull << shift) - 1);
    const uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1))) ++q;
    if (hexp == 0) return (uint16_t)(sign | (uint16_t)q);  // q == 1024 is the least normal
    if (q == 2048) {
        q = 1024;
        ++hexp;
    }
    if (hexp >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(hexp << 10) | (uint16_t)(q - 1024));
}

double double_from_half_bits(uint16_t h) {
    const int hexp = (h >> 10) & 31;
    const int frac = h & 1023;
    const double sgn = (h & 0x8000u) ? -1.0 : 1.0;
    if (hexp == 31) return frac ? NAN : sgn * INFINITY;
    if (hexp == 0) return sgn * std::ldexp((double)frac, -24);
    return sgn * std::ldexp((double)(frac | 1024), hexp - 25);
}

// Smallest fp16 scale s with limit * s >= span, starting from the rounded
// quotient span / limit; 0 if it overflows.
bool scale_for_span(double span, double limit, uint16_t* s_bits) {
    if (span == 0.0) {
        *s_bits = 0x3c00u;  // 1.0
        return true;
    }
    uint16_t s = half_bits_from_double(span / limit);
    if (limit * double_from_half_bits(s) < span) s = (uint16_t)(s + 1u);
    if ((s & 0x7c00u) == 0x7c00u) return false;
    *s_bits = s;
    return true;
}

double clampd(double v, double lo, double hi) { return v < lo ? lo : (v > hi ? hi : v); }

}  // namespace

extern "C" sd_status sd_w4_pack_impl(const float* w, int N, int K, int group, uint32_t* qweight,
                                     uint16_t* scales, uint16_t* zeros) {
    if (!w || !qweight || !scales || !zeros) return SD_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || group <= 0 || K % 8 != 0 || K % group != 0) return SD_ERR_INVALID_ARG;
    const int G = K / group;
    const int words = K / 8;
    for (int n = 0; n < N; ++n) {
        const float* row = w + (size_t)n * K;
        uint32_t* qrow = qweight + (size_t)n * words;
        for (int c = 0; c < words; ++c) qrow[c] = 0u;
        for (int g = 0; g < G; ++g) {
            double lo = 0.0, hi = 0.0;
            for (int t = 0; t < group; ++t) {
                const double v = row[g * group + t];
                if (!std::isfinite(v)) return SD_ERR_INVALID_ARG;
                lo = v < lo ? v : lo;
                hi = v > hi ? v : hi;
            }
            uint16_t s_bits;
            if (!scale_for_span(hi - lo, 15.0, &s_bits)) return SD_ERR_INVALID_ARG;
            const double s = double_from_half_bits(s_bits);
            const double z = clampd(std::nearbyint(-lo / s), 0.0, 15.0);
            scales[(size_t)n * G + g] = s_bits;
            zeros[(size_t)n * G + g] = half_bits_from_double(z);
            for (int t = 0; t < group; ++t) {
                const int k = g * group + t;
                const double qv = clampd(std::nearbyint(row[k] / s) + z, 0.0, 15.0);
                qrow[k >> 3] |= (uint32_t)qv << (4 * (k & 7));
            }
        }
    }
    return SD_OK;
}

// b-bit weights (INT4 / INT3 / INT2 targets of "Speculative Decoding in
// Quantized Regimes", sec. 4.1-4.2): the sd_w4_pack rules with 2^b - 1
// levels, each row's codes one little-endian bit stream along K.
extern "C" sd_status sd_wb_pack_impl(const float* w, int N, int K, int group, int bits, uint32_t* packed,
                                     uint16_t* scales, uint16_t* zeros) {
    if (!w || !packed || !scales || !zeros) return SD_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || group <= 0 || K % group != 0) return SD_ERR_INVALID_ARG;
    if (bits < 2 || bits > 4) return SD_ERR_UNSUPPORTED;
    if (((long long)K * bits) % 32 != 0) return SD_ERR_INVALID_ARG;
    const double levels = (double)((1 << bits) - 1);
    const int G = K / group;
    const long long words = (long long)K * bits / 32;
    for (int n = 0; n < N; ++n) {
        const float* row = w + (size_t)n * K;
        uint32_t* prow = packed + (size_t)n * words;
        for (long long c = 0; c < words; ++c) prow[c] = 0u;
        for (int g = 0; g < G; ++g) {
            double lo = 0.0, hi = 0.0;
            for (int t = 0; t < group; ++t) {
                const double v = row[g * group + t];
                if (!std::isfinite(v)) return SD_ERR_INVALID_ARG;
                lo = v < lo ? v : lo;
                hi = v > hi ? v : hi;
            }
            uint16_t s_bits;
            if (!scale_for_span(hi - lo, levels, &s_bits)) return SD_ERR_INVALID_ARG;
            const double s = double_from_half_bits(s_bits);
            const double z = clampd(std::nearbyint(-lo / s), 0.0, levels);
            scales[(size_t)n * G + g] = s_bits;
            zeros[(size_t)n * G + g] = half_bits_from_double(z);
            for (int t = 0; t < group; ++t) {
                const long long k = (long long)g * group + t;
                const uint64_t code = (uint64_t)clampd(std::nearbyint(row[k] / s) + z, 0.0, levels);
                // bits b k .. b k + b - 1 of the stream, possibly across two words
                const long long bit = k * bits;
                const uint64_t shifted = code << (bit & 31);
                prow[bit >> 5] |= (uint32_t)shifted;
                if ((shifted >> 32) != 0) prow[(bit >> 5) + 1] |= (uint32_t)(shifted >> 32);
            }
        }
    }
    return SD_OK;
}

extern "C" sd_status sd_w8_pack_impl(const float* w, int N, int K, int8_t* qweight,
                                     uint16_t* scales) {
    if (!w || !qweight || !scales) return SD_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0) return SD_ERR_INVALID_ARG;
    for (int n = 0; n < N; ++n) {
        const float* row = w + (size_t)n * K;
        double amax = 0.0;
        for (int k = 0; k < K; ++k) {
            const double v = row[k];
            if (!std::isfinite(v)) return SD_ERR_INVALID_ARG;
            amax = std::fabs(v) > amax ? std::fabs(v) : amax;
        }
        uint16_t s_bits;
        if (!scale_for_span(amax, 127.0, &s_bits)) return SD_ERR_INVALID_ARG;
        const double s = double_from_half_bits(s_bits);
        scales[n] = s_bits;
        for (int k = 0; k < K; ++k)
            qweight[(size_t)n * K + k] = (int8_t)clampd(std::nearbyint(row[k] / s), -127.0, 127.0);
    }
    return SD_OK;
}
