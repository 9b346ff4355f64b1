/*
 * Plain CPU oracle for the quantized speculative-decoding hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * restatement of what the GPU library computes.  It shares no code, header,
 * table or constant generator with the CUDA path (quantized_speculative_
 * decoding_gb300/csrc).  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference arm may load it.
 *
 * Floating point is fp64 throughout (the pages fix no precision for the
 * math).  Loops are sequential and unblocked, in the order of the
 * definitions, so that each function can be checked against its source by
 * eye.
 *
 * Sources (pages):
 *   [FreeHalf]      "The Free Half of Speculative Decoding" (devlinliles.com)
 *                   para. 3: INT4 (AWQ) target, quantized draft;
 *                   para. 4: draft proposes a run, target verifies each token.
 *   [QuantDrafts]   "When Do Quantized Drafts Help Speculative Decoding?"
 *                   "Current pilot setup": gamma=4, batch 1, BF16 / GPTQ INT8 /
 *                   GPTQ INT4 draft; References [2] Leviathan et al. 2023,
 *                   [3] Chen et al. 2023 (the speculative-sampling rule),
 *                   [4] AWQ (group-wise INT4 weights).
 *   [QuantRegimes]  "Speculative Decoding in Quantized Regimes", sec. 2.1
 *                   (its alpha = 1 - KL formula is NOT used; the closed form
 *                   of refs [2],[3], alpha = sum_v min(p_v, q_v), is);
 *                   sec. 4.1-4.2: INT4, INT3 and INT2 targets.
 *   [QSPEC]         [QuantDrafts] "What is open" and Reference [1] (QSPEC):
 *                   a W4A4 draft that shares the target's W4 weights.
 *   Philox4x32-10:  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *                   Easy as 1, 2, 3", SC'11 (the counter-based generator the
 *                   uniforms are drawn from).
 *
 * Readings where the pages are silent:
 *   R1 quantiser range includes 0; s = RN_fp16((hi-lo)/15), stepped up one
 *      fp16 ulp if 15*s < hi-lo; s = 1 for an all-zero group; integer zero
 *      point z = clamp(RNE(-lo/s), 0, 15); q = clamp(RNE(w/s) + z, 0, 15);
 *      w' = (q - z) * s.
 *   R2 packed layout: qweight[n][c] uint32, nibble j (bits 4j..4j+3) holds
 *      q[n][8c+j]; scales/zeros fp16 [N][K/group].
 *   R3 INT8 per-channel: s = RN_fp16(max|w|/127) stepped up if 127*s < max|w|,
 *      s = 1 for an all-zero row; q8 = clamp(RNE(w/s), -127, 127).
 *   R4 one temperature T for draft and target; T = 0 is greedy.
 *   R5 accept iff u*q(x) < p(x), u in [0,1) (strict <; q(x)=0 accepts iff
 *      p(x) > 0).  Every u_i is drawn.
 *   R6 Philox mapping: key = (seed lo32, seed hi32);
 *      accept uniform of position i, batch b: counter (i, b, 0, 0), word 0,
 *      u = (word >> 8) * 2^-24;
 *      race variate of slot j, vocab v, batch b: counter (v>>2, b, 1+j, 0),
 *      word v&3, t = (word + 1/2) * 2^-32, E = -ln(1 - t).
 *   R7 residual / bonus sampling by the exponential race:
 *      x = argmax_{v: r_v > 0} r_v / E_v, lowest v on equal keys; an exact
 *      sampler of r / sum(r) (Gumbel-max / exponential clocks).  If the
 *      residual max(0, p - q) is all zero, sample from p instead.
 *   R8 greedy: accept iff x_i == argmax_v target_i (lowest index on ties);
 *      the emitted token is argmax of the first rejected (or bonus) row.
 *   R11 b-bit weights (b = 2, 3, 4): R1 with L = 2^b - 1 levels in place of
 *      15; each row's codes form one little-endian bit stream along K (code
 *      k in bits b k .. b k + b - 1), stored as uint32 words (word c holds
 *      bits 32 c .. 32 c + 31); K b must be a multiple of 32.  b = 4 is R1/R2.
 *   R12 W4A4 activations: per row m and 128-input group g, symmetric int4
 *      with an fp32 scale s = fl32(max|x| / 7) (s = 1 for an all-zero
 *      group) and codes q = clamp(RNE(fl32(x / s)), -8, 7), both decided in
 *      fp32; y = sum_g s_x s_w sum_{k in g} q_x (q_w - z).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* R12 decides codes by fp32 divisions: float arithmetic must be evaluated in
 * fp32 (true of x86-64 SSE and aarch64). */
#if FLT_EVAL_METHOD != 0
#error "float expressions must be evaluated in binary32"
#endif

/* ------------------------------------------------------------------------
 * Philox4x32-10 (Salmon et al., SC'11).  One round maps the counter
 * (c0,c1,c2,c3) with key (k0,k1) to
 *     (hi(B*c2) ^ c1 ^ k0,  lo(B*c2),  hi(A*c0) ^ c3 ^ k1,  lo(A*c0))
 * with the paper's multipliers A = 0xD2511F53, B = 0xCD9E8D57; between rounds
 * the key advances by the Weyl constants (0x9E3779B9, 0xBB67AE85).
 * ---------------------------------------------------------------------- */
void oracle_philox4x32(const uint32_t ctr[4], const uint32_t key[2], int rounds,
                       uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < rounds; ++r) {
        uint64_t pa = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t pb = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(pb >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)pb;
        uint32_t n2 = (uint32_t)(pa >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)pa;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static uint32_t philox_word(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2,
                            uint32_t c3, int word) {
    uint32_t ctr[4] = {c0, c1, c2, c3};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32(ctr, key, 10, out);
    return out[word];
}

/* R6: accept uniform of draft position i for batch element b. */
double oracle_accept_uniform(uint64_t seed, uint32_t b, uint32_t i) {
    uint32_t w = philox_word(seed, i, b, 0u, 0u, 0);
    return (double)(w >> 8) * 0x1p-24;
}

/* R6: exponential race variate E for (batch b, slot j, vocab index v) on
 * stream `stream` (0 = verification; 1 = the test-only draft sampler). */
double oracle_race_exponential(uint64_t seed, uint32_t b, uint32_t slot, uint32_t v,
                               uint32_t stream) {
    uint32_t w = philox_word(seed, v >> 2, b, 1u + slot, stream, (int)(v & 3u));
    double t = ((double)w + 0.5) * 0x1p-32;           /* exact in fp64 */
    double one_minus_t = ((double)(~w) + 0.5) * 0x1p-32; /* exact: 1 - t */
    /* -ln(1 - t), evaluated where each form is accurate */
    return (t < 0.5) ? -log1p(-t) : -log(one_minus_t);
}

/* ------------------------------------------------------------------------
 * IEEE binary16 / bfloat16 rounding from fp64, round to nearest even,
 * written from the formats' definitions (sign, biased exponent, fraction).
 * ---------------------------------------------------------------------- */
static uint16_t round_to_small_float(double x, int mant_bits, int exp_bias, int exp_max) {
    /* exp_max: largest unbiased exponent of a finite value */
    uint16_t sign = signbit(x) ? (uint16_t)(1u << 15) : 0;
    uint16_t inf_bits = (uint16_t)(((1u << (15 - mant_bits)) - 1u) << mant_bits);
    if (isnan(x)) return (uint16_t)(sign | inf_bits | (1u << (mant_bits - 1)));
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | inf_bits);
    if (a == 0.0) return sign;
    int emin = 1 - exp_bias; /* smallest normal exponent */
    int e;
    frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1) */
    int E = e - 1;           /* a = 1.f * 2^E */
    if (E < emin) {
        /* subnormal range: integer multiples of 2^(emin - mant_bits) */
        double units = ldexp(a, mant_bits - emin);
        double r = nearbyint(units);
        /* r == 2^mant_bits rolls into the smallest normal: same bit pattern */
        return (uint16_t)(sign | (uint16_t)r);
    }
    double units = ldexp(a, mant_bits - E); /* in [2^m, 2^(m+1)) */
    double r = nearbyint(units);
    if (r == ldexp(1.0, mant_bits + 1)) { r = ldexp(1.0, mant_bits); E += 1; }
    if (E > exp_max) return (uint16_t)(sign | inf_bits);
    uint32_t frac = (uint32_t)r - (1u << mant_bits);
    return (uint16_t)(sign | (uint16_t)((uint32_t)(E + exp_bias) << mant_bits) | frac);
}

static double small_float_value(uint16_t h, int mant_bits, int exp_bias) {
    int exp_field_bits = 15 - mant_bits;
    uint32_t expo = (h >> mant_bits) & ((1u << exp_field_bits) - 1u);
    uint32_t frac = h & ((1u << mant_bits) - 1u);
    double s = (h >> 15) ? -1.0 : 1.0;
    if (expo == (1u << exp_field_bits) - 1u) return frac ? NAN : s * INFINITY;
    if (expo == 0) return s * ldexp((double)frac, 1 - exp_bias - mant_bits);
    return s * ldexp((double)(frac + (1u << mant_bits)), (int)expo - exp_bias - mant_bits);
}

uint16_t oracle_f64_to_f16(double x) { return round_to_small_float(x, 10, 15, 15); }
double oracle_f16_to_f64(uint16_t h) { return small_float_value(h, 10, 15); }
uint16_t oracle_f64_to_bf16(double x) { return round_to_small_float(x, 7, 127, 127); }
double oracle_bf16_to_f64(uint16_t h) { return small_float_value(h, 7, 127); }

/* next fp16 value above a positive finite fp16 (the encoding is monotone) */
static uint16_t f16_next_up(uint16_t h) { return (uint16_t)(h + 1u); }

/* ------------------------------------------------------------------------
 * R1: asymmetric uint4 round-to-nearest group quantiser ([FreeHalf] para. 3,
 * "INT4 using AWQ"; [QuantDrafts] pilot setup, "GPTQ INT4"; group along K).
 * q: uint8 [N][K] in 0..15;  scales, zeros: fp16 bits [N][K/group].
 * Returns 0, or -1 on bad sizes / non-finite input / scale overflow.
 * ---------------------------------------------------------------------- */
int oracle_quantize_w4(const float* w, int N, int K, int group, uint8_t* q,
                       uint16_t* scales, uint16_t* zeros) {
    if (N <= 0 || K <= 0 || group <= 0 || K % group != 0) return -1;
    int G = K / group;
    for (int n = 0; n < N; ++n) {
        for (int g = 0; g < G; ++g) {
            const float* wg = w + (size_t)n * K + (size_t)g * group;
            double lo = 0.0, hi = 0.0;
            for (int t = 0; t < group; ++t) {
                double v = (double)wg[t];
                if (!isfinite(v)) return -1;
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            uint16_t s16;
            if (hi == lo) {
                s16 = oracle_f64_to_f16(1.0);
            } else {
                double range = hi - lo; /* exact: both are fp32 values */
                s16 = oracle_f64_to_f16(range / 15.0);
                if (15.0 * oracle_f16_to_f64(s16) < range) s16 = f16_next_up(s16);
                if (!isfinite(oracle_f16_to_f64(s16))) return -1;
            }
            double s = oracle_f16_to_f64(s16);
            double z = nearbyint(-lo / s);
            if (z < 0.0) z = 0.0;
            if (z > 15.0) z = 15.0;
            for (int t = 0; t < group; ++t) {
                double qv = nearbyint((double)wg[t] / s) + z;
                if (qv < 0.0) qv = 0.0;
                if (qv > 15.0) qv = 15.0;
                q[(size_t)n * K + (size_t)g * group + t] = (uint8_t)qv;
            }
            scales[(size_t)n * G + g] = s16;
            zeros[(size_t)n * G + g] = oracle_f64_to_f16(z);
        }
    }
    return 0;
}

/* R2: unpack the K-packed uint32 nibble layout into q[N][K]. */
void oracle_unpack_w4(const uint32_t* qweight, int N, int K, uint8_t* q) {
    int C = K / 8;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            uint32_t word = qweight[(size_t)n * C + k / 8];
            q[(size_t)n * K + k] = (uint8_t)((word >> (4 * (k % 8))) & 0xFu);
        }
}

/* w'[n][k] = (q - z) * s in fp64 (exact: small integer times an fp16). */
void oracle_dequant_w4(const uint8_t* q, const uint16_t* scales, const uint16_t* zeros,
                       int N, int K, int group, double* wdq) {
    int G = K / group;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            double s = oracle_f16_to_f64(scales[(size_t)n * G + k / group]);
            double z = oracle_f16_to_f64(zeros[(size_t)n * G + k / group]);
            wdq[(size_t)n * K + k] = ((double)q[(size_t)n * K + k] - z) * s;
        }
}

/* y[m][n] = sum_k x[m][k] * w'[n][k]: the W4A16 linear on the packed layout,
 * sequential fp64 accumulation.  x is bf16 bits [M][K]. */
void oracle_w4a16_linear(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                         const uint16_t* zeros, int group, int M, int N, int K, double* y) {
    int C = K / 8, G = K / group;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) {
                uint32_t word = qweight[(size_t)n * C + k / 8];
                double qv = (double)((word >> (4 * (k % 8))) & 0xFu);
                double s = oracle_f16_to_f64(scales[(size_t)n * G + k / group]);
                double z = oracle_f16_to_f64(zeros[(size_t)n * G + k / group]);
                acc += oracle_bf16_to_f64(x[(size_t)m * K + k]) * ((qv - z) * s);
            }
            y[(size_t)m * N + n] = acc;
        }
}

/* ------------------------------------------------------------------------
 * R11: b-bit asymmetric group quantiser ([QuantRegimes] sec. 4.1-4.2, INT4 /
 * INT3 / INT2 targets): R1 with L = 2^b - 1 levels.  q: uint8 [N][K] in
 * 0..L; scales, zeros: fp16 bits [N][K/group].  Returns 0, or -1 on bad
 * sizes, bits outside {2, 3, 4}, non-finite input or scale overflow.
 * ---------------------------------------------------------------------- */
int oracle_quantize_wb(const float* w, int N, int K, int group, int bits, uint8_t* q,
                       uint16_t* scales, uint16_t* zeros) {
    if (N <= 0 || K <= 0 || group <= 0 || K % group != 0 || bits < 2 || bits > 4) return -1;
    const double L = (double)((1 << bits) - 1);
    int G = K / group;
    for (int n = 0; n < N; ++n) {
        for (int g = 0; g < G; ++g) {
            const float* wg = w + (size_t)n * K + (size_t)g * group;
            double lo = 0.0, hi = 0.0;
            for (int t = 0; t < group; ++t) {
                double v = (double)wg[t];
                if (!isfinite(v)) return -1;
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            uint16_t s16;
            if (hi == lo) {
                s16 = oracle_f64_to_f16(1.0);
            } else {
                double range = hi - lo;
                s16 = oracle_f64_to_f16(range / L);
                if (L * oracle_f16_to_f64(s16) < range) s16 = f16_next_up(s16);
                if (!isfinite(oracle_f16_to_f64(s16))) return -1;
            }
            double s = oracle_f16_to_f64(s16);
            double z = nearbyint(-lo / s);
            if (z < 0.0) z = 0.0;
            if (z > L) z = L;
            for (int t = 0; t < group; ++t) {
                double qv = nearbyint((double)wg[t] / s) + z;
                if (qv < 0.0) qv = 0.0;
                if (qv > L) qv = L;
                q[(size_t)n * K + (size_t)g * group + t] = (uint8_t)qv;
            }
            scales[(size_t)n * G + g] = s16;
            zeros[(size_t)n * G + g] = oracle_f64_to_f16(z);
        }
    }
    return 0;
}

/* R11 layout: code k of row n in bits b k .. b k + b - 1 of the row's stream
 * of K b / 32 uint32 words.  Returns 0, or -1 if K b is not a multiple of 32. */
int oracle_pack_wb(const uint8_t* q, int N, int K, int bits, uint32_t* packed) {
    if (N <= 0 || K <= 0 || bits < 2 || bits > 4 || ((long)K * bits) % 32 != 0) return -1;
    long W = (long)K * bits / 32;
    for (int n = 0; n < N; ++n) {
        for (long c = 0; c < W; ++c) packed[(size_t)n * W + c] = 0u;
        for (int k = 0; k < K; ++k)
            for (int t = 0; t < bits; ++t) {
                long bit = (long)k * bits + t;
                uint32_t v = (uint32_t)((q[(size_t)n * K + k] >> t) & 1u);
                packed[(size_t)n * W + bit / 32] |= v << (bit % 32);
            }
    }
    return 0;
}

void oracle_unpack_wb(const uint32_t* packed, int N, int K, int bits, uint8_t* q) {
    long W = (long)K * bits / 32;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            uint32_t v = 0;
            for (int t = 0; t < bits; ++t) {
                long bit = (long)k * bits + t;
                v |= ((packed[(size_t)n * W + bit / 32] >> (bit % 32)) & 1u) << t;
            }
            q[(size_t)n * K + k] = (uint8_t)v;
        }
}

/* y = x . w'^T on the R11 layout, w' = (q - z) s; fp64, sequential.  x bf16
 * bits [M][K]. */
void oracle_wb_linear(const uint16_t* x, const uint32_t* packed, const uint16_t* scales,
                      const uint16_t* zeros, int group, int bits, int M, int N, int K, double* y) {
    uint8_t* q = (uint8_t*)malloc((size_t)N * K);
    if (!q) return;
    oracle_unpack_wb(packed, N, K, bits, q);
    int G = K / group;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) {
                double s = oracle_f16_to_f64(scales[(size_t)n * G + k / group]);
                double z = oracle_f16_to_f64(zeros[(size_t)n * G + k / group]);
                acc += oracle_bf16_to_f64(x[(size_t)m * K + k]) * (((double)q[(size_t)n * K + k] - z) * s);
            }
            y[(size_t)m * N + n] = acc;
        }
    free(q);
}

/* ------------------------------------------------------------------------
 * R12: the W4A4 draft's activations ([QSPEC]): per row and 128-input group,
 * s = fl32(max|x| / 7) (1 for an all-zero group), q = clamp(RNE(fl32(x / s)),
 * -8, 7).  The two divisions are IEEE fp32 (float operands, round to
 * nearest), the precision the codes are decided in.  x bf16 bits [M][K];
 * qx int8 [M][K]; sx fp32 [M][K/128].  Returns 0, or -1 on bad sizes or
 * non-finite input.
 * ---------------------------------------------------------------------- */
int oracle_quantize_a4(const uint16_t* x, int M, int K, int8_t* qx, float* sx) {
    if (M <= 0 || K <= 0 || K % 128 != 0) return -1;
    int G = K / 128;
    for (int m = 0; m < M; ++m)
        for (int g = 0; g < G; ++g) {
            const uint16_t* xg = x + (size_t)m * K + (size_t)g * 128;
            float amax = 0.0f;
            for (int t = 0; t < 128; ++t) {
                float v = (float)oracle_bf16_to_f64(xg[t]); /* exact */
                if (!isfinite(v)) return -1;
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            float s = amax > 0.0f ? amax / 7.0f : 1.0f;
            for (int t = 0; t < 128; ++t) {
                float r = (float)oracle_bf16_to_f64(xg[t]) / s;
                double qv = nearbyint((double)r);
                if (qv < -8.0) qv = -8.0;
                if (qv > 7.0) qv = 7.0;
                qx[(size_t)m * K + (size_t)g * 128 + t] = (int8_t)qv;
            }
            sx[(size_t)m * G + g] = s;
        }
    return 0;
}

/* The W4A4 linear ([QSPEC]): the R12 activation codes against the shared W4
 * weights (R1/R2), y = sum_g s_x s_w sum_{k in g} q_x (q_w - z); the inner
 * sums are exact integers; fp64. */
int oracle_w4a4_linear(const uint16_t* x, const uint32_t* qweight, const uint16_t* scales,
                       const uint16_t* zeros, int M, int N, int K, double* y) {
    int G = K / 128, C = K / 8;
    int8_t* qx = (int8_t*)malloc((size_t)M * K);
    float* sx = (float*)malloc(sizeof(float) * (size_t)M * G);
    if (!qx || !sx || oracle_quantize_a4(x, M, K, qx, sx) != 0) {
        free(qx);
        free(sx);
        return -1;
    }
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int g = 0; g < G; ++g) {
                double z = oracle_f16_to_f64(zeros[(size_t)n * G + g]);
                double dot = 0.0;
                for (int k = g * 128; k < (g + 1) * 128; ++k) {
                    uint32_t word = qweight[(size_t)n * C + k / 8];
                    double qw = (double)((word >> (4 * (k % 8))) & 0xFu);
                    dot += (double)qx[(size_t)m * K + k] * (qw - z);
                }
                acc += (double)sx[(size_t)m * G + g] * oracle_f16_to_f64(scales[(size_t)n * G + g]) * dot;
            }
            y[(size_t)m * N + n] = acc;
        }
    free(qx);
    free(sx);
    return 0;
}

/* R3: symmetric INT8 per-output-channel quantiser ([QuantDrafts] pilot setup,
 * "GPTQ INT8" draft).  q8: int8 [N][K]; scales: fp16 bits [N]. */
int oracle_quantize_w8(const float* w, int N, int K, int8_t* q8, uint16_t* scales) {
    if (N <= 0 || K <= 0) return -1;
    for (int n = 0; n < N; ++n) {
        const float* wr = w + (size_t)n * K;
        double amax = 0.0;
        for (int k = 0; k < K; ++k) {
            double v = (double)wr[k];
            if (!isfinite(v)) return -1;
            if (fabs(v) > amax) amax = fabs(v);
        }
        uint16_t s16;
        if (amax == 0.0) {
            s16 = oracle_f64_to_f16(1.0);
        } else {
            s16 = oracle_f64_to_f16(amax / 127.0);
            if (127.0 * oracle_f16_to_f64(s16) < amax) s16 = f16_next_up(s16);
            if (!isfinite(oracle_f16_to_f64(s16))) return -1;
        }
        double s = oracle_f16_to_f64(s16);
        for (int k = 0; k < K; ++k) {
            double v = nearbyint((double)wr[k] / s);
            if (v < -127.0) v = -127.0;
            if (v > 127.0) v = 127.0;
            q8[(size_t)n * K + k] = (int8_t)v;
        }
        scales[n] = s16;
    }
    return 0;
}

/* y = x . (q8 * s)^T, fp64. */
void oracle_w8a16_linear(const uint16_t* x, const int8_t* q8, const uint16_t* scales,
                         int M, int N, int K, double* y) {
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double s = oracle_f16_to_f64(scales[n]);
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += oracle_bf16_to_f64(x[(size_t)m * K + k]) * ((double)q8[(size_t)n * K + k] * s);
            y[(size_t)m * N + n] = acc;
        }
}

/* y = x . W^T with bf16 W [N][K] (the BF16 draft of [QuantDrafts]), fp64. */
void oracle_bf16_linear(const uint16_t* x, const uint16_t* w, int M, int N, int K, double* y) {
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += oracle_bf16_to_f64(x[(size_t)m * K + k]) * oracle_bf16_to_f64(w[(size_t)n * K + k]);
            y[(size_t)m * N + n] = acc;
        }
}

/* Round fp64 values to bf16 bits (for the bit-exact one-hot probes). */
void oracle_round_bf16(const double* y, size_t n, uint16_t* out) {
    for (size_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(y[i]);
}

/* ------------------------------------------------------------------------
 * Softmax at temperature T > 0 (R4): p_v = exp(l_v/T - m) / Z,
 * m = max_v l_v/T, Z = sum_v exp(l_v/T - m).  fp64.
 * ---------------------------------------------------------------------- */
void oracle_softmax(const float* logits, int V, double T, double* p) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double a = (double)logits[v] / T;
        if (a > m) m = a;
    }
    double Z = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp((double)logits[v] / T - m);
        Z += p[v];
    }
    for (int v = 0; v < V; ++v) p[v] /= Z;
}

/* argmax with the lowest index winning ties (R8). */
static int argmax_f32(const float* row, int V) {
    int best = 0;
    for (int v = 1; v < V; ++v)
        if (row[v] > row[best]) best = v;
    return best;
}

/* ------------------------------------------------------------------------
 * The statistics a softmax row is normalised by (R4), in raw logit units:
 * m = max_v l_v and Z = sum_v exp((l_v - m) / T), so that
 * p_v = exp((l_v - m) / T) / Z.  Z is returned only for T > 0.  *arg is the
 * argmax with the lowest index winning ties (R8), for any T.  Given a slice of
 * a row, these are that slice's partial statistics: the row's are
 * m = max_i m_i and Z = sum_i Z_i exp((m_i - m) / T).  fp64.  Returns 0, or
 * -1 on bad arguments.
 * ---------------------------------------------------------------------- */
int oracle_softmax_stats(const float* logits, int V, double T, double* m_out, double* z_out,
                         int32_t* arg_out) {
    if (V < 1 || !(T >= 0.0)) return -1;
    int arg = argmax_f32(logits, V);
    double m = (double)logits[arg];
    double Z = 0.0;
    if (T > 0.0)
        for (int v = 0; v < V; ++v) Z += exp(((double)logits[v] - m) / T);
    *m_out = m;
    *z_out = Z;
    *arg_out = arg;
    return 0;
}

/* Near-tie windows.  The accept window is the +-1e-6 band around
 * min(1, p/q).  A race is flagged when the best key is within the sum of the
 * two keys' relative error windows of the runner-up, each window being
 * 4e-6 scaled by (p_v + q_v) / r_v, which is how much fp32 rounding of p and
 * q is amplified by the cancellation in p - q (q = 0 for rows of p alone). */
#define ACCEPT_TIE_WINDOW 1e-6
#define RACE_REL_WINDOW 4e-6
#define FLAG_RACE (1 << 30)

typedef struct {
    int winner;
    int flagged;
} race_result;

/* R7: exponential race over weights r (r_v > 0 competes), ties to lowest v. */
static race_result race_sample(const double* r, const double* pq_sum, int V, uint64_t seed,
                               uint32_t b, uint32_t slot, uint32_t stream) {
    int best = -1, second = -1;
    double kbest = 0.0, ksecond = 0.0;
    for (int v = 0; v < V; ++v) {
        if (!(r[v] > 0.0)) continue;
        double E = oracle_race_exponential(seed, b, slot, (uint32_t)v, stream);
        double key = r[v] / E; /* E > 0 always (t < 1) */
        if (best < 0 || key > kbest) {
            second = best; ksecond = kbest;
            best = v; kbest = key;
        } else if (second < 0 || key > ksecond) {
            second = v; ksecond = key;
        }
    }
    race_result res = {best, 0};
    if (best >= 0 && second >= 0) {
        double wb = RACE_REL_WINDOW * (pq_sum ? pq_sum[best] / r[best] : 1.0);
        double ws = RACE_REL_WINDOW * (pq_sum ? pq_sum[second] / r[second] : 1.0);
        if (ksecond * (1.0 + wb + ws) >= kbest) res.flagged = 1;
    }
    return res;
}

/* ------------------------------------------------------------------------
 * Speculative-sampling verification ([FreeHalf] para. 4; [QuantDrafts]
 * refs [2],[3]).  For each batch element b:
 *   q_i = softmax(draft_i / T), p_i = softmax(target_i / T), i < gamma;
 *   p_gamma = softmax(target_gamma / T);
 *   accept position i iff u_i * q_i(x_i) < p_i(x_i)   (R5, R6);
 *   accept_len = first rejected i, or gamma;
 *   new token: rejected at j < gamma -> race over max(0, p_j - q_j)
 *              (all zero -> over p_j); all accepted -> race over p_gamma (R7).
 * T == 0: greedy (R8).
 * out_tokens [B][gamma+1]: accepted drafts, the new token, then -1.
 * flags [B]: bit i = accept decision i was within the near-tie window,
 *            bit 30 = the race was a near tie.  Only decisions that reach the
 *            output are flagged (positions <= accept_len, and the race).
 * Returns 0, or -1 on bad arguments.
 * ---------------------------------------------------------------------- */
int oracle_verify(const float* draft_logits, const float* target_logits,
                  const int32_t* draft_tokens, int gamma, int B, int V, double T,
                  uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len,
                  int32_t* flags) {
    if (gamma < 1 || B < 0 || V < 1 || !(T >= 0.0)) return -1;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    double* pq = (double*)malloc(sizeof(double) * (size_t)V);
    if (!p || !q || !r || !pq) { free(p); free(q); free(r); free(pq); return -1; }
    for (int b = 0; b < B; ++b) {
        const float* dl = draft_logits + (size_t)b * gamma * V;
        const float* tl = target_logits + (size_t)b * (gamma + 1) * V;
        const int32_t* xt = draft_tokens + (size_t)b * gamma;
        int32_t* out = out_tokens + (size_t)b * (gamma + 1);
        int32_t flag = 0;
        for (int i = 0; i < gamma; ++i)
            if (xt[i] < 0 || xt[i] >= V) { free(p); free(q); free(r); free(pq); return -1; }
        int j = gamma;
        int new_token;
        if (T == 0.0) {
            for (int i = 0; i < gamma; ++i) {
                if (xt[i] != argmax_f32(tl + (size_t)i * V, V)) { j = i; break; }
            }
            new_token = argmax_f32(tl + (size_t)j * V, V);
        } else {
            for (int i = 0; i < gamma; ++i) {
                oracle_softmax(dl + (size_t)i * V, V, T, q);
                oracle_softmax(tl + (size_t)i * V, V, T, p);
                int x = xt[i];
                double u = oracle_accept_uniform(seed, (uint32_t)b, (uint32_t)i);
                int accept = u * q[x] < p[x];
                double ratio = (q[x] > 0.0) ? fmin(1.0, p[x] / q[x]) : (p[x] > 0.0 ? 1.0 : 0.0);
                if (fabs(u - ratio) < ACCEPT_TIE_WINDOW) flag |= (1 << i);
                if (!accept) { j = i; break; }
            }
            race_result rr;
            if (j < gamma) {
                /* p and q of row j are still in p[], q[] */
                double mass = 0.0;
                for (int v = 0; v < V; ++v) {
                    double d = p[v] - q[v];
                    r[v] = d > 0.0 ? d : 0.0;
                    pq[v] = p[v] + q[v];
                    mass += r[v];
                }
                if (mass > 0.0) {
                    rr = race_sample(r, pq, V, seed, (uint32_t)b, (uint32_t)j, 0u);
                    if (mass < 1e-5) rr.flagged = 1;
                } else {
                    rr = race_sample(p, NULL, V, seed, (uint32_t)b, (uint32_t)j, 0u);
                    rr.flagged = 1;
                }
            } else {
                oracle_softmax(tl + (size_t)gamma * V, V, T, p);
                rr = race_sample(p, NULL, V, seed, (uint32_t)b, (uint32_t)gamma, 0u);
            }
            new_token = rr.winner;
            if (rr.flagged) flag |= FLAG_RACE;
        }
        for (int i = 0; i < j; ++i) out[i] = xt[i];
        out[j] = new_token;
        for (int i = j + 1; i <= gamma; ++i) out[i] = -1;
        out_accept_len[b] = j;
        if (flags) flags[b] = flag;
    }
    free(p); free(q); free(r); free(pq);
    return 0;
}

/* Draft-side sampler (the draft step before the verification: "When Do
 * Quantized Drafts Help Speculative Decoding?", pilot setup; References [2],
 * [3]): x ~ softmax(logits / T) by the exponential race of R7 on Philox
 * stream 1 (counter word 3 = 1), slot = draft position, batch index b.
 * T == 0 returns the argmax (lowest index on ties).  *flagged (if not NULL)
 * is set when the race's top two keys are within the near-tie window. */
int oracle_sample_flag(const float* logits, int V, double T, uint64_t seed, uint32_t b,
                       uint32_t slot, int32_t* flagged) {
    if (flagged) *flagged = 0;
    if (V < 1 || !(T >= 0.0)) return -1;
    if (T == 0.0) return argmax_f32(logits, V);
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    if (!p) return -1;
    oracle_softmax(logits, V, T, p);
    race_result rr = race_sample(p, NULL, V, seed, b, slot, 1u);
    free(p);
    if (flagged) *flagged = rr.flagged;
    return rr.winner;
}

int oracle_sample(const float* logits, int V, double T, uint64_t seed, uint32_t b,
                  uint32_t slot) {
    return oracle_sample_flag(logits, V, T, seed, b, slot, NULL);
}

/* Repeated trials on one fixed set of logits (statistical pins).  Trial t
 * uses seed seed0 + t, batch index 0: draft tokens x_i ~ q_i from stream 1,
 * then oracle_verify.  Accumulates:
 *   hist_len[gamma+1]        accept_len counts
 *   hist_tok[(gamma+1)*V]    counts of the token emitted at each position
 *                            (only positions that are emitted, i <= accept_len)
 *   hist_new[(gamma+1)*V]    counts of the new (resampled / bonus) token,
 *                            by accept_len
 *   accepted[gamma], reached[gamma]: per-position accept / reach counts.
 * Returns the number of flagged trials, or -1. */
long oracle_verify_trials(const float* draft_logits, const float* target_logits, int gamma,
                          int V, double T, uint64_t seed0, long ntrials, int64_t* hist_len,
                          int64_t* hist_tok, int64_t* hist_new, int64_t* accepted,
                          int64_t* reached) {
    int32_t* xt = (int32_t*)malloc(sizeof(int32_t) * (size_t)gamma);
    int32_t* out = (int32_t*)malloc(sizeof(int32_t) * (size_t)(gamma + 1));
    if (!xt || !out) { free(xt); free(out); return -1; }
    long nflag = 0;
    for (long t = 0; t < ntrials; ++t) {
        uint64_t seed = seed0 + (uint64_t)t;
        for (int i = 0; i < gamma; ++i)
            xt[i] = oracle_sample(draft_logits + (size_t)i * V, V, T, seed, 0u, (uint32_t)i);
        int32_t len, flag;
        if (oracle_verify(draft_logits, target_logits, xt, gamma, 1, V, T, seed, out, &len, &flag)) {
            free(xt); free(out); return -1;
        }
        if (flag) nflag++;
        hist_len[len]++;
        for (int i = 0; i <= len; ++i) hist_tok[(size_t)i * V + out[i]]++;
        hist_new[(size_t)len * V + out[len]]++;
        for (int i = 0; i < gamma && i <= len; ++i) {
            reached[i]++;
            if (i < len) accepted[i]++;
        }
    }
    free(xt); free(out);
    return nflag;
}
