// Tensor-core W4A16 GEMM for small M (1 <= M <= 32) on sm_103a: TMA weight
// stream, dequantisation into tensor memory, group scaling after the MMA.
//
// The verify-time linear of "When Do Quantized Drafts Help Speculative
// Decoding?" (pilot setup: target at M = batch * (gamma + 1) = 5; draft at
// M = 1) is HBM-bound, and on GB300 the CUDA cores cannot afford the M fp32
// FMAs plus an exact dequantisation per weight at HBM speed.  Here the
// dequantisation shrinks to one LOP3 per two weights and the multiply-adds go
// to the tensor core:
//
//   y[m][n] = sum_g s_g[n] * ( D_g[n][m] - (128 + z_g[n]) * X_g[m] ),
//   D_g[n][m] = sum_{k in g} (128 + q[n][k]) * x[m][k],   X_g[m] = sum_{k in g} x[m][k]
//
// which is exactly sum_k (q - z) s x.  128 + q is exact in bf16 and one
// LOP3 builds two of them, (w >> 4i) & 0x000F000F | 0x43004300, pairing
// nibbles i and i + 4 of a 32-bit word; x is staged in the same k order so
// that the K permutation cancels in the contraction.
//
// CTA = 15 warps, one 128-row tile of W and one K-slice, one 128-wide stage
// per quantisation group, every role decoupled by mbarriers:
//   warp 12 (lane 0)  weight producer: 128 rows x 64 bytes of packed int4 per
//                     stage (one 2D TMA box) into a 16-deep shared ring;
//   warp 13 (lane 0)  x producer: the M rows x 128 bf16 of x of each stage
//                     (2D TMA) into an 8-deep ring;
//   warps 0-7         dequantisation: warp w serves TMEM lanes 32(w%4)..+31
//                     (rows) and half w/4 of the stage; each thread builds 32
//                     bf16x2 words of (128 + q) from its 32 bytes and stores
//                     them into its TMEM lane (A operand, 4 buffers);
//   warp 14 (lane 0)  issues 8 tcgen05.mma (K = 16, A from TMEM, B from shared
//                     memory) per stage into one of 8 TMEM accumulators;
//   warps 8-11        permute the x of each stage (shared to shared) into a
//                     128B-swizzled tile (B operand, 8 buffers) with its group
//                     sums X_g, and, four stages behind the MMAs, load D_g from
//                     TMEM and accumulate s (D - (128 + z) X) in fp32.
// One CTA per SM; the grid is sized to one wave where the shape allows.
// Launched with programmatic dependent launch: the weights, scales and zeros
// stream in before the kernel waits for the previous kernel of the stream;
// x, the workspace and the output are touched only after that wait.
// Split-K slices meet through fp32 partials and a last-arrival counter,
// summed in fixed order.
//
// All waits are bounded (about 2^31 SM cycles) and watch a CTA-wide abort
// flag; on expiry the kernel records SD_ERR_TIMEOUT, frees its TMEM and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>

#include "device_common.cuh"
#include "launch.cuh"
#include "sd_internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace sd {
namespace {

using namespace tc;

constexpr int kDqWarps = 8;                     // warps 0-7
constexpr int kEpWarp0 = 8;                     // warps 8-11
constexpr int kWProdWarp = 12, kXProdWarp = 13, kMmaWarp = 14;
constexpr int kThreads = 15 * 32;
constexpr int kGK = 128;                        // K per stage = one group
constexpr int kWStage = 128 * kGK / 2;          // 8 KB packed int4 per stage
constexpr int kNX = 8;                          // x ring depth
constexpr int kNA = 4, kNB = 8, kND = 8;        // A (TMEM), B (smem), D (TMEM) buffers
constexpr int kLag = 4;                         // epilogue runs kLag stages behind
constexpr int kXS = 8;                          // group-sum ring depth (> kLag + 1)
constexpr uint32_t kTmemCols = 512;             // A: 4 x 64 cols, D: 8 x MP cols (MP <= 32)
constexpr uint32_t kColA0 = 0, kColD0 = 256;

// Bounded wait on phase `parity`.  Gives up (false) after about 2^31 SM
// cycles (about 1 s) or when another thread of the CTA has set *abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort = 1;
            return false;
        }
    }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

struct Tc2Params {
    const __nv_bfloat16* x;
    const __half* scales;     // [N][K/128]
    const __half* zeros;
    __nv_bfloat16* out;
    float* partial;      // [splits][M][N] (splits > 1)
    unsigned* counters;  // [tiles] (splits > 1)
    int* err;
    int M, N, K, splits;
};

template <int MP>
struct Tc2Cfg {
    static constexpr int kBStage = MP * kGK * 2;            // two 64-wide SW128 atoms
    static constexpr int kXStage = MP * kGK * 2;            // x rows of a stage, natural order
    static constexpr int kNS = MP <= 16 ? 16 : 8;           // weight ring depth (227 KB limit)
    static constexpr int kSmem = kNS * kWStage + kNX * kXStage + kNB * kBStage + 1024;
};

template <int MP>
__global__ void __launch_bounds__(kThreads, 1)
w4a16_tc2_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                 Tc2Params P) {
    using C = Tc2Cfg<MP>;
    constexpr int NS = C::kNS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_wfull[NS], bar_wempty[NS];
    __shared__ __align__(8) uint64_t bar_xfull[kNX], bar_xempty[kNX];
    __shared__ __align__(8) uint64_t bar_aready[kNA], bar_afree[kNA];
    __shared__ __align__(8) uint64_t bar_bready[kNB], bar_bfree[kNB];
    __shared__ __align__(8) uint64_t bar_dfull[kND], bar_dfree[kND];
    __shared__ float xsum[kXS][MP];
    // per-row scale and zero of 16 groups, double-buffered; each epilogue
    // thread reads and writes only its own row's entries
    __shared__ __half2 sz_s[2][16][128];
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    __shared__ int is_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x / P.splits;
    const int split = blockIdx.x - tile * P.splits;
    const int n0 = tile * 128;
    const int M = P.M, N = P.N, K = P.K;
    const int ngr = K / kGK;
    const int g0 = (int)((long long)split * ngr / P.splits);
    const int g1 = (int)((long long)(split + 1) * ngr / P.splits);
    const int nit = g1 - g0;
    // Stage `it` handles group grp(it): each tile starts its slice at a
    // different group so that the CTAs of a launch do not all read the same
    // rows of x from the same L2 lines at the same time.
    const int rot = tile % (nit > 0 ? nit : 1);
    auto grp = [&](int it) -> int {
        const int r = it + rot;
        return g0 + (r >= nit ? r - nit : r);
    };

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t wring = smem_u32(smem);                  // NS x 8 KB weights
    const uint32_t xring = wring + NS * kWStage;           // kNX x kXStage x rows
    const uint32_t btile = xring + kNX * C::kXStage;       // kNB x kBStage

    griddep_launch_dependents();
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_wfull[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bar_wempty[i])),
                         "r"(kDqWarps * 32));
        }
        for (int i = 0; i < kNX; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_xfull[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;" ::"r"(smem_u32(&bar_xempty[i])));
        }
        for (int i = 0; i < kNA; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bar_aready[i])),
                         "r"(kDqWarps * 32));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_afree[i])));
        }
        for (int i = 0; i < kNB; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;" ::"r"(smem_u32(&bar_bready[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_bfree[i])));
        }
        for (int i = 0; i < kND; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_dfull[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 128;" ::"r"(smem_u32(&bar_dfree[i])));
        }
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_s)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    // TMEM lanes this warp may touch (a warp reaches lanes 32 * (warp % 4) ..)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    // Waits are taken by every lane and then voted over the warp, so that
    // warp-wide tcgen05 instructions always run converged.  A warp that gives
    // up keeps iterating in `skip` mode and still takes every named barrier.
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
        const bool ok = mbar_wait(smem_u32(bar), parity, &abort_s);
        return __all_sync(0xffffffffu, ok);
    };

    float acc[MP];
#pragma unroll
    for (int m = 0; m < MP; ++m) acc[m] = 0.f;

    if (warp == kWProdWarp) {
        // ---------------- weight producer (constant data: no wait for the previous kernel)
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
            for (int it = 0; it < nit; ++it) {
                const int slot = it % NS;
                if (it >= NS &&
                    !mbar_wait(smem_u32(&bar_wempty[slot]), ((it / NS) - 1) & 1, &abort_s))
                    break;
                mbar_expect_tx(smem_u32(&bar_wfull[slot]), kWStage);
                tma_load_2d(wring + slot * kWStage, &wmap, grp(it) * (kGK / 2), n0,
                            smem_u32(&bar_wfull[slot]));
            }
        }
    } else if (warp == kXProdWarp) {
        // ---------------- x producer (x may come from the previous kernel)
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
            griddep_wait();
            for (int it = 0; it < nit; ++it) {
                const int slot = it % kNX;
                if (it >= kNX &&
                    !mbar_wait(smem_u32(&bar_xempty[slot]), ((it / kNX) - 1) & 1, &abort_s))
                    break;
                mbar_expect_tx(smem_u32(&bar_xfull[slot]), M * kGK * 2);
                tma_load_2d(xring + slot * C::kXStage, &xmap, grp(it) * kGK, 0,
                            smem_u32(&bar_xfull[slot]));
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, MP);
            for (int it = 0; it < nit; ++it) {
                const int a = it % kNA, bb = it % kNB, d = it % kND;
                if (!mbar_wait(smem_u32(&bar_aready[a]), (it / kNA) & 1, &abort_s)) break;
                if (!mbar_wait(smem_u32(&bar_bready[bb]), (it / kNB) & 1, &abort_s)) break;
                if (it >= kND && !mbar_wait(smem_u32(&bar_dfree[d]), ((it / kND) - 1) & 1, &abort_s))
                    break;
                tc_fence_after();
                const uint32_t a_col = tmem + kColA0 + 64 * a;
                const uint32_t d_col = tmem + kColD0 + MP * d;
                const uint32_t bt = btile + bb * C::kBStage;
#pragma unroll
                for (int kk = 0; kk < kGK / 16; ++kk)
                    mma_bf16_ta(d_col, a_col + 8 * kk,
                               desc_sw128(bt + (kk >> 2) * (MP * 128) + (kk & 3) * 32), idesc,
                               kk > 0 ? 1u : 0u);
                mma_commit(smem_u32(&bar_afree[a]));
                mma_commit(smem_u32(&bar_bfree[bb]));
                mma_commit(smem_u32(&bar_dfull[d]));
            }
        }
    } else if (warp < kDqWarps) {
        // ---------------- dequantisation: row 32 * (warp % 4) + lane, half warp / 4
        const int r = (warp & 3) * 32 + lane;
        const int h = warp >> 2;
        for (int it = 0; it < nit; ++it) {
            const int slot = it % NS, a = it % kNA;
            if (!wait_warp(&bar_wfull[slot], (it / NS) & 1)) break;
            // the stage's 64 bytes of row r, 16-byte chunk c at c ^ ((r >> 1) & 3)
            const uint32_t rbase = wring + slot * kWStage + r * 64;
            const uint4 w0 = lds128(rbase + (((2 * h) ^ ((r >> 1) & 3)) << 4));
            const uint4 w1 = lds128(rbase + (((2 * h + 1) ^ ((r >> 1) & 3)) << 4));
            mbar_arrive(smem_u32(&bar_wempty[slot]));
            if (it >= kNA && !wait_warp(&bar_afree[a], ((it / kNA) - 1) & 1)) break;
            const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            uint32_t av[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t w = words[j];
                av[4 * j + 0] = (w & 0x000f000fu) | 0x43004300u;
                av[4 * j + 1] = ((w >> 4) & 0x000f000fu) | 0x43004300u;
                av[4 * j + 2] = ((w >> 8) & 0x000f000fu) | 0x43004300u;
                av[4 * j + 3] = ((w >> 12) & 0x000f000fu) | 0x43004300u;
            }
            tmem_st32(tmem + lane_base + kColA0 + 64 * a + 32 * h, av);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_aready[a]));
        }
    } else {
        // ---------------- x stager + epilogue, row 32 * (warp % 4) + lane
        const int e = warp - kEpWarp0;  // 0..3, equal to warp % 4
        const int et = e * 32 + lane;   // 0..127
        const int row = min(n0 + et, N - 1);
        const __half* srow = P.scales + (size_t)row * ngr;  // + group
        const __half* zrow = P.zeros + (size_t)row * ngr;
        // Scales and zeros are staged 16 stages at a time: window w (stages
        // 16w .. 16w + 15) lives in sz_s[w & 1].  Window w + 1 is loaded into
        // registers at stage 16w + 8 and stored at stage 16w + 12, so no stage
        // waits on their global loads.
        __half2 pend[16];
        auto load_window = [&](int w) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int it = 16 * w + j;
                pend[j] = it < nit ? __halves2half2(__ldg(srow + grp(it)),
                                                    __ldg(zrow + grp(it)))
                                   : __halves2half2(__float2half(0.f), __float2half(0.f));
            }
        };
        auto store_window = [&](int w) {
#pragma unroll
            for (int j = 0; j < 16; ++j) sz_s[w & 1][j][et] = pend[j];
        };
        load_window(0);
        store_window(0);
        bool skip = false;  // warp-uniform
        for (int it = 0; it < nit + kLag; ++it) {
            // (a) x of stage it -> B tile it % kNB (k order of the A pairs), sums -> xsum ring
            if (it < nit && !skip) {
                const int bb = it % kNB;
                const int slot = it % kNX;
                if (!wait_warp(&bar_xfull[slot], (it / kNX) & 1)) skip = true;
                if (!skip && it >= kNB && !wait_warp(&bar_bfree[bb], ((it / kNB) - 1) & 1)) skip = true;
                if (!skip) {
                    const uint32_t bt = btile + bb * C::kBStage;
                    const uint32_t xs = xring + slot * C::kXStage;  // M rows x 256 bytes
#pragma unroll
                    for (int i0 = 0; i0 < MP * 16; i0 += 128) {
                        const int i = i0 + et;  // MP * 16 is a multiple of 128
                        const int m = i >> 4, c = i & 15;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (m < M) v = lds128(xs + m * 256 + c * 16);
                        uint4 pv;
                        pv.x = __byte_perm(v.x, v.z, 0x5410);
                        pv.y = __byte_perm(v.x, v.z, 0x7632);
                        pv.z = __byte_perm(v.y, v.w, 0x5410);
                        pv.w = __byte_perm(v.y, v.w, 0x7632);
                        sts128(bt + (c >> 3) * (MP * 128) + m * 128 + (((c & 7) ^ (m & 7)) << 4), pv);
                        float sum = bf16lo_to_float(v.x) + bf16hi_to_float(v.x) + bf16lo_to_float(v.y) +
                                    bf16hi_to_float(v.y) + bf16lo_to_float(v.z) + bf16hi_to_float(v.z) +
                                    bf16lo_to_float(v.w) + bf16hi_to_float(v.w);
                        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
                        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                        if (c == 0) xsum[it % kXS][m] = sum;
                    }
                    mbar_arrive(smem_u32(&bar_xempty[slot]));
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive(smem_u32(&bar_bready[bb]));
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");  // xsum of stage it visible
            // (b) epilogue of group g = it - kLag
            const int g = it - kLag;
            if (g >= 0 && !skip) {
                const int d = g % kND;
                if ((g & 15) == 8 && 16 * ((g >> 4) + 1) < nit) load_window((g >> 4) + 1);
                if ((g & 15) == 12 && 16 * ((g >> 4) + 1) < nit) store_window((g >> 4) + 1);
                const __half2 sz = sz_s[(g >> 4) & 1][g & 15][et];
                const float s = __low2float(sz);
                const float corr = 128.f + __high2float(sz);
                if (!wait_warp(&bar_dfull[d], (g / kND) & 1)) {
                    skip = true;
                } else {
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < MP; c0 += 16) {
                        uint32_t rv[16];
                        tmem_ld16(tmem + lane_base + kColD0 + MP * d + c0, rv);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            acc[c0 + j] = fmaf(s, fmaf(-corr, xsum[g % kXS][c0 + j], __uint_as_float(rv[j])),
                                               acc[c0 + j]);
                    }
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bar_dfree[d]));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool aborted = abort_s != 0;
    const bool epi = warp >= kEpWarp0 && warp < kEpWarp0 + 4;
    const int n = n0 + (warp - kEpWarp0) * 32 + lane;
    if (epi || tid == 0) griddep_wait();  // before any global write
    if (aborted && tid == 0) record_error(P.err, kDevErrTimeout);
    if (epi && !aborted && n < N) {
#pragma unroll
        for (int m = 0; m < MP; ++m) {
            if (m < M) {
                if (P.splits == 1) P.out[(size_t)m * N + n] = __float2bfloat16_rn(acc[m]);
                else P.partial[((size_t)split * M + m) * N + n] = acc[m];
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
    if (P.splits == 1) return;

    // split-K: the last slice of the tile sums the partials in order (an
    // aborted slice still arrives so that the counter returns to zero)
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        is_last = atomicInc(&P.counters[tile], (unsigned)(P.splits - 1)) == (unsigned)(P.splits - 1);
    }
    __syncthreads();
    if (!is_last || aborted || !epi) return;
    __threadfence();
    if (n < N) {
        for (int m = 0; m < M; ++m) {
            float v = 0.f;
            for (int sp = 0; sp < P.splits; ++sp) v += __ldcg(P.partial + ((size_t)sp * M + m) * N + n);
            P.out[(size_t)m * N + n] = __float2bfloat16_rn(v);
        }
    }
}

template <int MP>
cudaError_t launch_mp(const CUtensorMap& map, const CUtensorMap& xmap, const Tc2Params& P, int tiles,
                      cudaStream_t s) {
    using C = Tc2Cfg<MP>;
    static std::atomic<unsigned long long> attr_set{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(w4a16_tc2_kernel<MP>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit, std::memory_order_release);
    }
    return launch_pdl(w4a16_tc2_kernel<MP>, dim3(tiles * P.splits), dim3(kThreads),
                      (size_t)C::kSmem, s, map, xmap, P);
}

cudaError_t launch_impl(const void* x, const void* qweight, const void* scales,
                        const void* zeros, int M, int N, int K, void* out, void* ws, size_t ws_bytes,
                        unsigned* counters, int sms, int* err, cudaStream_t s) {
    if (M < 1 || M > 32 || K % kGK != 0) return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const cuuint32_t estride[2] = {1, 1};
    CUtensorMap map;
    std::memset(&map, 0, sizeof map);
    const cuuint64_t gdim[2] = {(cuuint64_t)K / 2, (cuuint64_t)N};  // bytes along K, rows
    const cuuint64_t gstride[1] = {(cuuint64_t)K / 2};
    const cuuint32_t box[2] = {kGK / 2, 128};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(qweight), gdim, gstride, box,
               estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // x [M][K] bf16: one box = all M rows x 128 elements (256 bytes), no swizzle
    CUtensorMap xmap;
    const cuuint64_t xdim[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t xstride[1] = {(cuuint64_t)K * 2};
    const cuuint32_t xbox[2] = {kGK, (cuuint32_t)M};
    if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), xdim, xstride, xbox,
               estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    Tc2Params P;
    P.x = static_cast<const __nv_bfloat16*>(x);
    P.scales = static_cast<const __half*>(scales);
    P.zeros = static_cast<const __half*>(zeros);
    P.out = static_cast<__nv_bfloat16*>(out);
    P.err = err;
    P.M = M;
    P.N = N;
    P.K = K;
    P.splits = w4a16_tc2_splits(M, N, K, sms);
    const int tiles = (N + 127) / 128;
    if (P.splits > 1) {
        if (ws_bytes < w4a16_tc2_workspace_bytes(M, N, K, sms) || !counters)
            return cudaErrorInvalidValue;
        P.partial = static_cast<float*>(ws);
        P.counters = counters;
    } else {
        P.partial = nullptr;
        P.counters = nullptr;
    }
    return M <= 16 ? launch_mp<16>(map, xmap, P, tiles, s) : launch_mp<32>(map, xmap, P, tiles, s);
}

}  // namespace

int w4a16_tc2_splits(int M, int N, int K, int sms) {
    // one CTA per SM: split K so that tiles * splits fills (but does not
    // exceed) one wave, keeping at least one stage per slice
    const int tiles = (N + 127) / 128;
    const int ngr = K / kGK;
    int splits = sms / tiles;
    if (splits > ngr) splits = ngr;
    if (splits < 1) splits = 1;
    (void)M;
    return splits;
}

size_t w4a16_tc2_workspace_bytes(int M, int N, int K, int sms) {
    const int splits = w4a16_tc2_splits(M, N, K, sms);
    return splits == 1 ? 0 : (size_t)splits * M * N * sizeof(float);
}

cudaError_t launch_w4a16_tc2(const void* x, const uint32_t* qweight, const void* scales,
                             const void* zeros, int M, int N, int K, void* out, void* ws,
                             size_t ws_bytes, unsigned* counters, int sms, int* err,
                             cudaStream_t s) {
    return launch_impl(x, qweight, scales, zeros, M, N, K, out, ws, ws_bytes, counters, sms, err, s);
}

}  // namespace sd
