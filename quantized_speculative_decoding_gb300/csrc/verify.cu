// Fused speculative-sampling verification (sd_verify).
//
// The rule of the works cited by "When Do Quantized Drafts Help Speculative
// Decoding?" (References [2] Leviathan et al., [3] Chen et al.), as the target
// model's check of the drafted run ("The Free Half of Speculative Decoding",
// para. 4): position i is accepted with probability min(1, p_i(x_i)/q_i(x_i));
// the first rejected position j is resampled from norm(max(0, p_j - q_j)); if
// all gamma are accepted a bonus token is drawn from p_gamma.  Greedy (T = 0)
// accepts the prefix where the draft token is the target argmax.
//
// Kernels (no spin-waits):
//   stats: grid (chunks, rows).  Each CTA streams one vocabulary chunk of one
//     logit row (float4 loads) and reduces it to (running max, sum of
//     exp((l - max)/T)) -- or (max, argmax) when T = 0 -- written to the
//     workspace.  The last CTA to finish for a batch element (atomicInc
//     counter that wraps back to zero) merges the chunks of its rows in fp64,
//     evaluates the gamma accept decisions with fp64 p(x)/q(x) against the
//     Philox uniforms, and writes accept_len, the accepted tokens and the -1
//     padding (for T = 0 also the new token).
//     For sd_verify_parts each CTA merges a chunk of the softmax partials
//     that the lm_head (logits mode) wrote beside its logits instead of a
//     chunk of the row: the logits are read only at the draft tokens and in
//     the race.
//   race (T > 0 only): grid (chunks, batch).  Each CTA evaluates, over its
//     chunk of the selected row, r_v = max(0, p_v - q_v) (or p_v for the
//     bonus) and the race key r_v / E_v with E_v from Philox, keeps the best
//     (key, index) -- and the best over p_v alone for the all-zero-residual
//     case -- and the last CTA per batch element picks the winner.
#include <float.h>
#include <math.h>

#include <atomic>

#include "../../include/sd.h"
#include "device_common.cuh"
#include "launch.cuh"
#include "sd_internal.h"

namespace sd {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxRowsPerBatch = 2 * 16 + 1;

struct Decision {
    int j;          // accept_len
    float m_p;      // max logit of the p row (raw logit units)
    float inv_z_p;  // 1 / sum exp((l - m_p)/T)
    float m_q;
    float inv_z_q;
    int pad[3];
};

struct Layout {
    int nrows, rows_per_b, nchunk, chunk, nchunk2, chunk2;
    size_t off_stats, off_dec, off_race, total;
};

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// lm_head partials per statistics CTA (sd_verify_parts).
constexpr int kPartChunk = 1024;

// parts > 0: the statistics kernel merges lm_head partials (at most `parts`
// per row) in chunks of kPartChunk instead of reading the logits.
Layout make_layout(int gamma, int batch, int vocab, float T, int sms, int parts = 0) {
    Layout L;
    L.rows_per_b = T > 0.f ? 2 * gamma + 1 : gamma + 1;
    L.nrows = batch * L.rows_per_b;
    const int max_chunks = (vocab + 2047) / 2048;
    if (parts > 0) {
        L.chunk = kPartChunk;
        L.nchunk = (parts + kPartChunk - 1) / kPartChunk;
    } else {
        int want = (4 * sms + L.nrows - 1) / (L.nrows > 0 ? L.nrows : 1);
        want = want < 1 ? 1 : (want > max_chunks ? max_chunks : want);
        L.chunk = (((vocab + want - 1) / want) + 3) & ~3;
        L.nchunk = (vocab + L.chunk - 1) / L.chunk;
    }
    int want2 = (2 * sms + batch - 1) / (batch > 0 ? batch : 1);
    want2 = want2 < 1 ? 1 : (want2 > max_chunks ? max_chunks : want2);
    L.chunk2 = (((vocab + want2 - 1) / want2) + 3) & ~3;
    L.nchunk2 = (vocab + L.chunk2 - 1) / L.chunk2;
    L.off_stats = 0;
    L.off_dec = L.off_stats + align256((size_t)L.nrows * L.nchunk * sizeof(float2));
    L.off_race = L.off_dec + align256((size_t)batch * sizeof(Decision));
    L.total = L.off_race + align256((size_t)batch * L.nchunk2 * sizeof(float4));
    return L;
}

struct Params {
    const float* draft;
    const float* target;
    const int32_t* tokens;
    int gamma, batch, vocab;
    float T, invT, c;  // c = log2(e) / T
    uint32_t k0, k1;
    int32_t* out_tokens;
    int32_t* out_len;
    unsigned* cnt_stats;
    unsigned* cnt_race;
    float2* stats;
    Decision* dec;
    float4* race;
    int rows_per_b, nchunk, chunk, nchunk2, chunk2;
    int* err;
    // sd_verify_parts: the lm_head's softmax partials (logits mode), which the
    // statistics kernel merges instead of reading the logits; target
    // [batch][gamma + 1][tparts], draft [batch][gamma][dparts].  tstats ==
    // nullptr (sd_verify): the statistics kernel reads the logit rows.
    const float2* tstats;
    const float2* dstats;
    int tparts, dparts;
};

__device__ __forceinline__ const float* row_ptr(const Params& P, int b, int lr) {
    // lr in [0, gamma]: target row lr; lr > gamma: draft row lr - gamma - 1
    if (lr <= P.gamma) return P.target + ((size_t)b * (P.gamma + 1) + lr) * P.vocab;
    return P.draft + ((size_t)b * P.gamma + (lr - P.gamma - 1)) * P.vocab;
}

// ---- (max, sum exp) online pairs -------------------------------------
struct MS {
    float m, s;
};

// exp((l - m) / T) as exp2(l c - m c) with c = log2(e) / T: one FMA and one
// exp2 per logit.
__device__ __forceinline__ float exp_scaled(float l, float c, float mc) { return exp2f(fmaf(l, c, -mc)); }

__device__ __forceinline__ MS ms_merge(MS a, MS b, float c) {
    if (a.m == -INFINITY) return b;
    if (b.m == -INFINITY) return a;
    const float m = fmaxf(a.m, b.m);
    return MS{m, a.s * exp_scaled(a.m, c, m * c) + b.s * exp_scaled(b.m, c, m * c)};
}

__device__ __forceinline__ void ms_add4(MS& a, float4 v, float c) {
    const float lm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (lm == -INFINITY) return;
    if (lm > a.m) {
        a.s = (a.m == -INFINITY) ? 0.f : a.s * exp_scaled(a.m, c, lm * c);
        a.m = lm;
    }
    const float mc = a.m * c;
    a.s += exp_scaled(v.x, c, mc) + exp_scaled(v.y, c, mc) + exp_scaled(v.z, c, mc) + exp_scaled(v.w, c, mc);
}

// ---- (value, index) argmax pairs, lowest index wins ties -----------------
struct VI {
    float v;
    int i;
};

__device__ __forceinline__ VI vi_better(VI a, VI b) {
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

template <typename T, typename F>
__device__ __forceinline__ T block_reduce(T v, F merge, T* smem) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        T other;
        static_assert(sizeof(T) == 8 || sizeof(T) == 16, "pair types only");
        if constexpr (sizeof(T) == 8) {
            unsigned long long bits = *reinterpret_cast<unsigned long long*>(&v);
            bits = __shfl_xor_sync(0xffffffffu, bits, o);
            other = *reinterpret_cast<T*>(&bits);
        } else {
            float4 f = *reinterpret_cast<float4*>(&v);
            f.x = __shfl_xor_sync(0xffffffffu, f.x, o);
            f.y = __shfl_xor_sync(0xffffffffu, f.y, o);
            f.z = __shfl_xor_sync(0xffffffffu, f.z, o);
            f.w = __shfl_xor_sync(0xffffffffu, f.w, o);
            other = *reinterpret_cast<T*>(&f);
        }
        v = merge(v, other);
    }
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = smem[lane < kThreads / 32 ? lane : 0];
        for (int w = 1; w < kThreads / 32; ++w)
            if (lane == 0) v = merge(v, smem[w]);
    }
    return v;  // valid in thread 0
}

// Last-arrival test: every CTA of a group calls this once (all threads); it
// returns true in exactly one CTA, the last to arrive, after a fence that
// makes the other CTAs' workspace writes visible.
__device__ __forceinline__ bool last_arrival(unsigned* counter, unsigned total) {
    __shared__ int is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicInc(counter, total - 1);
        is_last = (prev == total - 1);
    }
    __syncthreads();
    if (is_last) __threadfence();
    return is_last;
}

// ---- decisions for batch element b (one CTA, all threads) ----
// Merges each row's chunk statistics, evaluates the gamma accept decisions with fp64
// p(x)/q(x) against the Philox uniforms, and writes accept_len, the accepted
// tokens, the -1 padding (for T = 0 also the new token) and, for T > 0, the
// race's Decision.
__device__ __forceinline__ void decide(const Params& P, int b) {
    __shared__ float row_m[kMaxRowsPerBatch];
    __shared__ double row_z[kMaxRowsPerBatch];
    __shared__ int row_arg[kMaxRowsPerBatch];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int rr = warp; rr < P.rows_per_b; rr += kThreads / 32) {
        const float2* s = P.stats + ((size_t)b * P.rows_per_b + rr) * P.nchunk;
        const int ns = P.nchunk;
        if (P.T > 0.f) {
            float m = -INFINITY;
            for (int i = lane; i < ns; i += 32) m = fmaxf(m, __ldcg(&s[i].x));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            // chunk sums rescaled to the row max in fp32 (factors <= 1), added in fp64
            double z = 0.0;
            for (int i = lane; i < ns; i += 32) {
                const float2 e = __ldcg(&s[i]);
                if (e.x != -INFINITY) z += (double)e.y * (double)exp_scaled(e.x, P.c, m * P.c);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            if (lane == 0) {
                row_m[rr] = m;
                row_z[rr] = z;
            }
        } else {
            VI best{-INFINITY, 0x7fffffff};
            for (int i = lane; i < ns; i += 32) {
                const float2 e = __ldcg(&s[i]);
                best = vi_better(best, VI{e.x, __float_as_int(e.y)});
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                VI other{__shfl_xor_sync(0xffffffffu, best.v, o), __shfl_xor_sync(0xffffffffu, best.i, o)};
                best = vi_better(best, other);
            }
            if (lane == 0) row_arg[rr] = best.i;
        }
    }
    __syncthreads();

    if (warp == 0) {
        // lane i < gamma evaluates the accept decision of position i
        bool accept = true;
        int x = 0;
        if (lane < P.gamma) {
            x = P.tokens[(size_t)b * P.gamma + lane];
            if (x < 0 || x >= P.vocab) {
                record_error(P.err, kDevErrInvalidArg);
                accept = false;
            } else if (P.T > 0.f) {
                const double T = (double)P.T;
                const double lt = (double)P.target[((size_t)b * (P.gamma + 1) + lane) * P.vocab + x];
                const double ld = (double)P.draft[((size_t)b * P.gamma + lane) * P.vocab + x];
                const double p = exp((lt - (double)row_m[lane]) / T) / row_z[lane];
                const int dq = P.gamma + 1 + lane;
                const double q = exp((ld - (double)row_m[dq]) / T) / row_z[dq];
                const uint4 u4 = philox4x32_10(make_uint4((uint32_t)lane, (uint32_t)b, 0u, 0u), P.k0, P.k1);
                const double u = (double)(u4.x >> 8) * 0x1p-24;
                accept = u * q < p;
            } else {
                accept = (x == row_arg[lane]);
            }
        }
        const unsigned rej = __ballot_sync(0xffffffffu, !accept) & ((1u << P.gamma) - 1u);
        const int j = rej ? __ffs(rej) - 1 : P.gamma;
        int32_t* out = P.out_tokens + (size_t)b * (P.gamma + 1);
        if (lane < P.gamma + 1) {
            if (lane < j) out[lane] = x;
            else if (lane > j) out[lane] = -1;
            else if (P.T == 0.f) out[lane] = row_arg[j];
        }
        if (lane == 0) {
            P.out_len[b] = j;
            if (P.T > 0.f) {
                Decision d;
                d.j = j;
                d.m_p = row_m[j];
                d.inv_z_p = (float)(1.0 / row_z[j]);
                if (j < P.gamma) {
                    d.m_q = row_m[P.gamma + 1 + j];
                    d.inv_z_q = (float)(1.0 / row_z[P.gamma + 1 + j]);
                } else {
                    d.m_q = 0.f;
                    d.inv_z_q = 0.f;
                }
                P.dec[b] = d;
            }
        }
    }
}

// =========================== kernel 1: row statistics + decisions
__global__ void __launch_bounds__(kThreads) verify_stats_kernel(Params P) {
    griddep_launch_dependents();
    griddep_wait();  // logits and the workspace may come from the previous kernel
    const int r = blockIdx.x / P.nchunk;
    const int c = blockIdx.x - r * P.nchunk;
    const int b = r / P.rows_per_b, lr = r - b * P.rows_per_b;
    const float* row = row_ptr(P, b, lr);
    const int v0 = c * P.chunk;
    const int v1 = min(P.vocab, v0 + P.chunk);
    const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15) == 0);

    if (P.tstats != nullptr) {
        // chunk c of the row's lm_head partials (sd_verify_parts); a draft row
        // may have fewer partials than the chunks cover
        const float2* src;
        int n;
        if (lr <= P.gamma) {
            src = P.tstats + ((size_t)b * (P.gamma + 1) + lr) * P.tparts;
            n = P.tparts;
        } else {
            src = P.dstats + ((size_t)b * P.gamma + (lr - P.gamma - 1)) * P.dparts;
            n = P.dparts;
        }
        const int i1 = min(n, v0 + P.chunk);  // partials can outnumber a tiny vocabulary
        if (P.T > 0.f) {
            MS acc{-INFINITY, 0.f};
            const float cc = P.c;
#pragma unroll 4
            for (int i = v0 + threadIdx.x; i < i1; i += kThreads) {
                const float2 e = __ldg(src + i);
                acc = ms_merge(acc, MS{e.x, e.y}, cc);
            }
            __shared__ MS redp[kThreads / 32];
            acc = block_reduce(acc, [cc](MS a, MS bb) { return ms_merge(a, bb, cc); }, redp);
            if (threadIdx.x == 0) P.stats[(size_t)r * P.nchunk + c] = make_float2(acc.m, acc.s);
        } else {
            VI acc{-INFINITY, 0x7fffffff};
#pragma unroll 4
            for (int i = v0 + threadIdx.x; i < i1; i += kThreads) {
                const float2 e = __ldg(src + i);
                acc = vi_better(acc, VI{e.x, __float_as_int(e.y)});
            }
            __shared__ VI redv[kThreads / 32];
            acc = block_reduce(acc, [](VI a, VI bb) { return vi_better(a, bb); }, redv);
            if (threadIdx.x == 0)
                P.stats[(size_t)r * P.nchunk + c] = make_float2(acc.v, __int_as_float(acc.i));
        }
    } else if (P.T > 0.f) {
        MS acc{-INFINITY, 0.f};
        const float cc = P.c;
        if (vec) {
            const float4* p4 = reinterpret_cast<const float4*>(row + v0);
            const int n4 = (v1 - v0) >> 2;
            const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            // four independent loads in flight before any arithmetic
            for (int i = threadIdx.x; i < n4; i += 4 * kThreads) {
                float4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = i + u * kThreads < n4 ? __ldg(p4 + i + u * kThreads) : ninf;
#pragma unroll
                for (int u = 0; u < 4; ++u) ms_add4(acc, v[u], cc);
            }
            for (int v = v0 + 4 * n4 + threadIdx.x; v < v1; v += kThreads)
                ms_add4(acc, make_float4(row[v], -INFINITY, -INFINITY, -INFINITY), cc);
        } else {
            for (int v = v0 + threadIdx.x; v < v1; v += kThreads)
                ms_add4(acc, make_float4(row[v], -INFINITY, -INFINITY, -INFINITY), cc);
        }
        __shared__ MS red[kThreads / 32];
        acc = block_reduce(acc, [cc](MS a, MS bb) { return ms_merge(a, bb, cc); }, red);
        if (threadIdx.x == 0) P.stats[(size_t)r * P.nchunk + c] = make_float2(acc.m, acc.s);
    } else {
        VI acc{-INFINITY, 0x7fffffff};
        for (int v = v0 + threadIdx.x; v < v1; v += kThreads) acc = vi_better(acc, VI{row[v], v});
        __shared__ VI red[kThreads / 32];
        acc = block_reduce(acc, [](VI a, VI bb) { return vi_better(a, bb); }, red);
        if (threadIdx.x == 0)
            P.stats[(size_t)r * P.nchunk + c] = make_float2(acc.v, __int_as_float(acc.i));
    }

    if (!last_arrival(&P.cnt_stats[b], (unsigned)(P.nchunk * P.rows_per_b))) return;
    decide(P, b);
}

// =========================== kernel 2: residual / bonus race
// (key, index) of the best race entry so far; key -1 means none.  A larger
// key wins, the lower index on equal keys.
__device__ __forceinline__ VI race_better(VI a, VI b) {
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

// The race of row j of batch element b over [v0, v1): keys r_v / E_v for
// r_v > 0, with r_v = p_v - q_v (residual, has_q) or p_v (bonus, or the
// fallback when the whole residual is zero).  E_v is drawn only where r_v > 0;
// four consecutive v share one Philox call (counter v >> 2).
__device__ __forceinline__ VI race_range(const Params& P, const Decision& d, int b, int j, bool has_q,
                                         int v0, int v1, int step) {
    const float* prow = P.target + ((size_t)b * (P.gamma + 1) + j) * P.vocab;
    const float* qrow = has_q ? P.draft + ((size_t)b * P.gamma + j) * P.vocab : nullptr;
    const float c = P.c, mpc = d.m_p * c, mqc = d.m_q * c;
    const bool vec = ((reinterpret_cast<uintptr_t>(prow) | reinterpret_cast<uintptr_t>(qrow)) & 15) == 0;
    VI acc{-1.f, 0x7fffffff};
    for (int g = (v0 >> 2) + (int)threadIdx.x; 4 * g < v1; g += step) {
        float r[4];
        bool any = false;
        if (vec && 4 * g >= v0 && 4 * g + 3 < v1) {
            const float4 pl = __ldg(reinterpret_cast<const float4*>(prow) + g);
            const float4 ql = has_q ? __ldg(reinterpret_cast<const float4*>(qrow) + g) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float pa[4] = {pl.x, pl.y, pl.z, pl.w}, qa[4] = {ql.x, ql.y, ql.z, ql.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float pv = exp_scaled(pa[t], c, mpc) * d.inv_z_p;
                const float qv = has_q ? exp_scaled(qa[t], c, mqc) * d.inv_z_q : 0.f;
                r[t] = pv - qv;
                any |= r[t] > 0.f;
            }
        } else {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int v = 4 * g + t;
                r[t] = 0.f;
                if (v >= v0 && v < v1) {
                    const float pv = exp_scaled(__ldg(prow + v), c, mpc) * d.inv_z_p;
                    const float qv = has_q ? exp_scaled(__ldg(qrow + v), c, mqc) * d.inv_z_q : 0.f;
                    r[t] = pv - qv;
                    any |= r[t] > 0.f;
                }
            }
        }
        if (!any) continue;
        const uint4 ph = philox4x32_10(make_uint4((uint32_t)g, (uint32_t)b, 1u + (uint32_t)j, 0u), P.k0, P.k1);
        const uint32_t words[4] = {ph.x, ph.y, ph.z, ph.w};
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (r[t] > 0.f) {
                const float key = r[t] / race_exponential(words[t]);
                if (key > acc.v) acc = VI{key, 4 * g + t};
            }
    }
    return acc;
}

__global__ void __launch_bounds__(kThreads) verify_race_kernel(Params P) {
    griddep_launch_dependents();
    griddep_wait();  // the decisions come from the statistics kernel
    const int b = blockIdx.x / P.nchunk2;
    const int c = blockIdx.x - b * P.nchunk2;
    const Decision d = P.dec[b];
    const int j = min(max(d.j, 0), P.gamma);  // always in range, whatever the workspace holds
    const int v0 = c * P.chunk2;
    const int v1 = min(P.vocab, v0 + P.chunk2);
    VI acc = race_range(P, d, b, j, j < P.gamma, v0, v1, kThreads);
    __shared__ VI red[kThreads / 32];
    acc = block_reduce(acc, [](VI a, VI bb) { return race_better(a, bb); }, red);
    if (threadIdx.x == 0) P.race[(size_t)b * P.nchunk2 + c] = make_float4(acc.v, __int_as_float(acc.i), 0.f, 0.f);

    if (!last_arrival(&P.cnt_race[b], (unsigned)P.nchunk2)) return;
    __shared__ VI best_s;
    if (threadIdx.x < 32) {
        VI best{-1.f, 0x7fffffff};
        for (int i = threadIdx.x; i < P.nchunk2; i += 32) {
            const float4 f = __ldcg(&P.race[(size_t)b * P.nchunk2 + i]);
            best = race_better(best, VI{f.x, __float_as_int(f.y)});
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            VI other{__shfl_xor_sync(0xffffffffu, best.v, o), __shfl_xor_sync(0xffffffffu, best.i, o)};
            best = race_better(best, other);
        }
        if (threadIdx.x == 0) best_s = best;
    }
    __syncthreads();
    VI best = best_s;
    if (best.v <= 0.f) {
        // the residual is zero everywhere (only fp rounding gets here): the
        // race over p_j itself, the whole row in this CTA
        VI f = race_range(P, d, b, j, false, 0, P.vocab, kThreads);
        f = block_reduce(f, [](VI a, VI bb) { return race_better(a, bb); }, red);
        if (threadIdx.x == 0) best = f;
    }
    if (threadIdx.x == 0) P.out_tokens[(size_t)b * (P.gamma + 1) + j] = best.i;
}

// =========================== draft-side sampler (sd_sample)
// x_b ~ softmax(l_b / T) by the exponential race on Philox stream 1: the key
// of v is p_v / E_v with E_v from counter (v >> 2, b, 1 + slot, 1), word v & 3;
// the largest key wins, the lowest v on equal keys.  Each CTA takes one chunk
// of one row: a first pass finds the chunk max m_c, a second forms the keys
// exp((l_v - m_c) / T) / E_v; the last CTA of the row rescales the chunk
// winners by exp((m_c - m) / T) to the row max m and picks the winner.
// T = 0: the argmax, lowest index on ties.
struct SampleParams {
    const float* logits;  // [B][V]
    int batch, vocab, chunk, nchunk;
    float T, c;           // c = log2(e) / T
    uint32_t k0, k1, slot;
    int32_t* out;         // [B]
    float4* part;         // [B][nchunk]: (chunk max, best key or logit, index)
    unsigned* cnt;        // [B], zero on entry and on exit
};

__global__ void __launch_bounds__(kThreads) sample_kernel(SampleParams P) {
    griddep_launch_dependents();
    griddep_wait();  // the logits may come from the previous kernel
    const int b = blockIdx.x / P.nchunk;
    const int ch = blockIdx.x - b * P.nchunk;
    const float* row = P.logits + (size_t)b * P.vocab;
    const int v0 = ch * P.chunk;
    const int v1 = min(P.vocab, v0 + P.chunk);
    __shared__ VI red[kThreads / 32];
    __shared__ float m_s;
    float4 res;
    if (P.T > 0.f) {
        float m = -INFINITY;
        for (int v = v0 + (int)threadIdx.x; v < v1; v += kThreads) m = fmaxf(m, __ldg(row + v));
        VI mv = block_reduce(VI{m, 0}, [](VI a, VI bb) { return a.v >= bb.v ? a : bb; }, red);
        if (threadIdx.x == 0) m_s = mv.v;
        __syncthreads();
        const float mc = m_s, c = P.c, mcc = mc * c;
        VI acc{-1.f, 0x7fffffff};
        for (int g = (v0 >> 2) + (int)threadIdx.x; 4 * g < v1; g += kThreads) {
            const uint4 ph = philox4x32_10(make_uint4((uint32_t)g, (uint32_t)b, 1u + P.slot, 1u), P.k0, P.k1);
            const uint32_t words[4] = {ph.x, ph.y, ph.z, ph.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int v = 4 * g + t;
                if (v < v0 || v >= v1) continue;
                const float pv = exp_scaled(__ldg(row + v), c, mcc);
                if (pv > 0.f) {
                    const float key = pv / race_exponential(words[t]);
                    if (key > acc.v) acc = VI{key, v};
                }
            }
        }
        __syncthreads();  // red is reused
        acc = block_reduce(acc, [](VI a, VI bb) { return race_better(a, bb); }, red);
        res = make_float4(mc, acc.v, __int_as_float(acc.i), 0.f);
    } else {
        VI acc{-INFINITY, 0x7fffffff};
        for (int v = v0 + (int)threadIdx.x; v < v1; v += kThreads) acc = vi_better(acc, VI{__ldg(row + v), v});
        acc = block_reduce(acc, [](VI a, VI bb) { return vi_better(a, bb); }, red);
        res = make_float4(0.f, acc.v, __int_as_float(acc.i), 0.f);
    }
    if (threadIdx.x == 0) P.part[(size_t)b * P.nchunk + ch] = res;

    if (!last_arrival(&P.cnt[b], (unsigned)P.nchunk)) return;
    if (threadIdx.x < 32) {
        const float4* pr = P.part + (size_t)b * P.nchunk;
        VI best;
        if (P.T > 0.f) {
            float m = -INFINITY;
            for (int i = threadIdx.x; i < P.nchunk; i += 32) m = fmaxf(m, __ldcg(&pr[i].x));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            best = VI{-1.f, 0x7fffffff};
            for (int i = threadIdx.x; i < P.nchunk; i += 32) {
                const float4 e = __ldcg(&pr[i]);
                if (e.y > 0.f) best = race_better(best, VI{e.y * exp_scaled(e.x, P.c, m * P.c), __float_as_int(e.z)});
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                best = race_better(best, VI{__shfl_xor_sync(0xffffffffu, best.v, o), __shfl_xor_sync(0xffffffffu, best.i, o)});
        } else {
            best = VI{-INFINITY, 0x7fffffff};
            for (int i = threadIdx.x; i < P.nchunk; i += 32) {
                const float4 e = __ldcg(&pr[i]);
                best = vi_better(best, VI{e.y, __float_as_int(e.z)});
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                best = vi_better(best, VI{__shfl_xor_sync(0xffffffffu, best.v, o), __shfl_xor_sync(0xffffffffu, best.i, o)});
        }
        if (threadIdx.x == 0) P.out[b] = best.i;
    }
}


}  // namespace

size_t verify_workspace_bytes(int gamma, int batch, int vocab, float temperature, int sms, int parts) {
    return make_layout(gamma, batch, vocab, temperature, sms, parts).total;
}

size_t verify_counter_count(int batch) { return (size_t)2 * batch; }

namespace {

// The kernels' parameters for problem a over workspace ws (layout L).
Params make_params(const VerifyArgs& a, const Layout& L, void* ws, unsigned* counters, int* err) {
    char* base = static_cast<char*>(ws);
    Params P;
    P.draft = a.draft;
    P.target = a.target;
    P.tokens = a.tokens;
    P.gamma = a.gamma;
    P.batch = a.batch;
    P.vocab = a.vocab;
    P.T = a.temperature;
    P.invT = a.temperature > 0.f ? 1.f / a.temperature : 0.f;
    P.c = a.temperature > 0.f ? (float)(1.4426950408889634 / (double)a.temperature) : 0.f;
    P.k0 = (uint32_t)(a.seed & 0xffffffffu);
    P.k1 = (uint32_t)(a.seed >> 32);
    P.out_tokens = a.out_tokens;
    P.out_len = a.out_len;
    P.cnt_stats = counters;
    P.cnt_race = counters + a.batch;
    P.stats = reinterpret_cast<float2*>(base + L.off_stats);
    P.dec = reinterpret_cast<Decision*>(base + L.off_dec);
    P.race = reinterpret_cast<float4*>(base + L.off_race);
    P.rows_per_b = L.rows_per_b;
    P.nchunk = L.nchunk;
    P.chunk = L.chunk;
    P.nchunk2 = L.nchunk2;
    P.chunk2 = L.chunk2;
    P.err = err;
    P.tstats = nullptr;
    P.dstats = nullptr;
    P.tparts = 0;
    P.dparts = 0;
    return P;
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, void* ws, size_t ws_bytes, unsigned* counters,
                          int sms, int* err, cudaStream_t s) {
    const Layout L = make_layout(a.gamma, a.batch, a.vocab, a.temperature, sms);
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    const Params P = make_params(a, L, ws, counters, err);
    cudaError_t e = launch_pdl(verify_stats_kernel, dim3(L.nchunk * L.nrows), dim3(kThreads), 0, s, P);
    if (e != cudaSuccess || a.temperature == 0.f) return e;
    return launch_pdl(verify_race_kernel, dim3(L.nchunk2 * a.batch), dim3(kThreads), 0, s, P);
}

cudaError_t launch_verify_parts(const VerifyArgs& a, const void* draft_stats, int draft_parts,
                                const void* target_stats, int target_parts, void* ws, size_t ws_bytes,
                                unsigned* counters, int sms, int* err, cudaStream_t s) {
    if (target_parts < 1 || (a.temperature > 0.f && draft_parts < 1)) return cudaErrorInvalidValue;
    const int parts = a.temperature > 0.f && draft_parts > target_parts ? draft_parts : target_parts;
    const Layout L = make_layout(a.gamma, a.batch, a.vocab, a.temperature, sms, parts);
    if (ws_bytes < L.total) return cudaErrorInvalidValue;
    Params P = make_params(a, L, ws, counters, err);
    P.tstats = static_cast<const float2*>(target_stats);
    P.dstats = static_cast<const float2*>(draft_stats);
    P.tparts = target_parts;
    P.dparts = draft_parts;
    cudaError_t e = launch_pdl(verify_stats_kernel, dim3(L.nchunk * L.nrows), dim3(kThreads), 0, s, P);
    if (e != cudaSuccess || a.temperature == 0.f) return e;
    return launch_pdl(verify_race_kernel, dim3(L.nchunk2 * a.batch), dim3(kThreads), 0, s, P);
}

// Chunks per row for the sampler: about four CTAs per SM over all rows,
// chunks of at least 2048 logits, a multiple of 4 (Philox groups).
static void sample_layout(int batch, int vocab, int sms, int* chunk, int* nchunk) {
    const int max_chunks = (vocab + 2047) / 2048;
    int want = (4 * sms + batch - 1) / batch;
    want = want < 1 ? 1 : (want > max_chunks ? max_chunks : want);
    *chunk = (((vocab + want - 1) / want) + 3) & ~3;
    *nchunk = (vocab + *chunk - 1) / *chunk;
}

size_t sample_workspace_bytes(int batch, int vocab, int sms) {
    int chunk, nchunk;
    sample_layout(batch, vocab, sms, &chunk, &nchunk);
    return (size_t)batch * nchunk * sizeof(float4);
}

cudaError_t launch_sample(const float* logits, int batch, int vocab, float temperature, uint64_t seed, int slot,
                          int32_t* out, void* ws, size_t ws_bytes, unsigned* counters, int sms, cudaStream_t s) {
    SampleParams P;
    sample_layout(batch, vocab, sms, &P.chunk, &P.nchunk);
    if (ws_bytes < (size_t)batch * P.nchunk * sizeof(float4)) return cudaErrorInvalidValue;
    P.logits = logits;
    P.batch = batch;
    P.vocab = vocab;
    P.T = temperature;
    P.c = temperature > 0.f ? (float)(1.4426950408889634 / (double)temperature) : 0.f;
    P.k0 = (uint32_t)(seed & 0xffffffffu);
    P.k1 = (uint32_t)(seed >> 32);
    P.slot = (uint32_t)slot;
    P.out = out;
    P.part = static_cast<float4*>(ws);
    P.cnt = counters;
    return launch_pdl(sample_kernel, dim3(P.nchunk * batch), dim3(kThreads), 0, s, P);
}

// ------------------------------------------------------------------------
// Allocation-free variant (sd_verify_noalloc): the same two kernels, with
// their scratch in a fixed array of device memory that the library declares
// at file scope, so that no call ever allocates.  Every GPU that loads the
// library holds the array until the process exits.  In host code the array's
// name is only a host-side stand-in, so its device address is looked up once
// per device with cudaGetSymbolAddress (the first call on a device, with that
// device current) and passed to the kernels.  All calls on a device share the
// array: calls that may overlap on the GPU race with one another.
constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB per device
constexpr int kMaxStaticDevices = 64;

static __device__ __align__(256) unsigned char g_verify_scratch[kStaticScratchBytes];
static __device__ int g_verify_scratch_err;

namespace {

std::atomic<void*> g_scratch_addr[kMaxStaticDevices];
std::atomic<int*> g_scratch_err_addr[kMaxStaticDevices];

// Device addresses of the scratch array and its error word on `dev` (the
// current device); false if the lookup fails.
bool static_scratch(int dev, void** base, int** err) {
    if (dev < 0 || dev >= kMaxStaticDevices) return false;
    void* b = g_scratch_addr[dev].load(std::memory_order_acquire);
    int* e = g_scratch_err_addr[dev].load(std::memory_order_acquire);
    if (!b || !e) {
        if (cudaGetSymbolAddress(&b, g_verify_scratch) != cudaSuccess) return false;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&e), g_verify_scratch_err) != cudaSuccess)
            return false;
        g_scratch_addr[dev].store(b, std::memory_order_release);
        g_scratch_err_addr[dev].store(e, std::memory_order_release);
    }
    *base = b;
    *err = e;
    return true;
}

}  // namespace


int* verify_static_error_word(int dev) {
    void* b = nullptr;
    int* e = nullptr;
    return static_scratch(dev, &b, &e) ? e : nullptr;
}

int launch_verify_static(const VerifyArgs& a, int dev, int sms, cudaStream_t s) {
    void* base = nullptr;
    int* err = nullptr;
    if (!static_scratch(dev, &base, &err)) return SD_ERR_CUDA;
    const size_t counter_bytes = align256(verify_counter_count(a.batch) * sizeof(unsigned));
    const size_t ws_bytes = verify_workspace_bytes(a.gamma, a.batch, a.vocab, a.temperature, sms);
    if (counter_bytes + ws_bytes > kStaticScratchBytes) return SD_ERR_INVALID_ARG;
    // the counters must start at zero; the array keeps whatever the last call left
    if (cudaMemsetAsync(base, 0, counter_bytes, s) != cudaSuccess) return SD_ERR_CUDA;
    const cudaError_t e = launch_verify(a, static_cast<char*>(base) + counter_bytes, ws_bytes,
                                        static_cast<unsigned*>(base), sms, err, s);
    return e == cudaSuccess ? SD_OK : SD_ERR_CUDA;
}

}  // namespace sd
