// Tensor-memory-operand W4A16 GEMM for small M (1 <= M <= 8) on the
// fragment-ordered layout of sd_w4_tile (tcgen05, sm_103a).
//
// The verify-time linears of "When Do Quantized Drafts Help Speculative
// Decoding?" (pilot setup: M = batch x (gamma + 1) = 5) read every weight once
// and do 2M flops per weight: an HBM stream whose cost is the instructions
// spent per weight byte.  The register-operand kernel (w4a16_mma.cu) spends
// them on per-warp work that does not scale with the weights: x fragment
// loads, an all-ones MMA per 16 inputs for the zero-point sums, accumulator
// bookkeeping and the mma.sync issue itself.  Here the tensor core gets its A
// operand from tensor memory instead:
//
//   - A CTA owns 128 weight rows (8 tiles of 16) = the 128 TMEM lanes = the
//     MMA's M.  Thread (warp w, lane l) owns row 32 (w % 4) + l and the K half
//     w / 4 of every quantisation group (64 inputs).
//   - Per group, every thread reads its row's 64 bytes of the tiled layout
//     (the lane units of rows g and g + 8 share them), keeps its own row's
//     nibble pairs, turns each pair into the exact bf16 pair (128 + q,
//     128 + q') with one LOP3 (the same magic-number encoding as the register
//     kernel) and writes the 32 resulting columns to its TMEM lane with one
//     tcgen05.st.  Consecutive inputs share a column, so TMEM holds A in the
//     natural K order.
//   - One thread issues 8 tcgen05.mma (K = 16 each, N = 16: the x rows padded)
//     with A from TMEM and the group's x rows from a 128B-swizzled shared
//     tile: D_g = sum (128 + q) x.  Eight more with a constant all-ones A in
//     TMEM give X_g = sum x.  Both land in a TMEM slot of 32 columns.
//   - The epilogue of group g - 1 runs while the MMAs of group g execute: each
//     thread reads D and X of its row for its 4 x rows (tcgen05.ld) and adds
//     s (D - (128 + z) X) in fp32: y = sum_g s_g sum_k (q - z) x, exactly the
//     register kernel's arithmetic.
//
// Pipelines: packed weights and scale/zero entries of a group arrive by 1D
// bulk copies (16 per group, one thread) into an 8-stage ring counted on
// per-stage mbarriers, issued before the wait on the previous kernel
// (constant data); x rows arrive by cp.async two groups ahead into a 4-slot
// ring; two TMEM slots for A and two for D/X.  Every mbarrier wait is
// bounded: on expiry the kernel records SD_ERR_TIMEOUT, lets its copies and
// MMAs drain (bounded), frees its TMEM and returns.
//
// Work split: CTA = (128-row block p, K split rank).  The S splits of a row
// block form one thread-block cluster and add their fp32 partials through
// distributed shared memory in rank order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "device_common.cuh"
#include "launch.cuh"
#include "sd_internal.h"
#include "tcgen05.cuh"

namespace sd {
namespace {

using namespace tc;

constexpr int kTmThreads = 256;  // 8 warps: TMEM lane quarter w % 4, K half w / 4
constexpr int kTmRows = 128;     // weight rows per CTA = TMEM lanes = MMA M
constexpr int kTmTiles = 8;      // 16-row tiles of the tiled layout per CTA
constexpr int kTmN = 16;         // MMA N: x rows, padded
constexpr int kTmMaxM = 8;
constexpr int kWBytes = kTmTiles * 1024;  // one group: 8 tiles x 2 chunks x 512 bytes
constexpr int kSzBytes = kTmTiles * 64;   // one group: 8 tiles x 8 entries x 8 bytes
constexpr int kWSlot = kWBytes + kSzBytes;
constexpr int kNW = 8;                    // packed-weight ring stages
constexpr int kBTile = kTmN * 256;        // x of one group: two 64-input SW128 atoms of 16 rows
constexpr int kBSlots = 4;
constexpr int kTmSmem = kBSlots * kBTile + kNW * kWSlot + 1024;  // + alignment slack: 2 CTAs / SM
constexpr int kTmMaxSplits = 16;
// TMEM columns: A slots (64 each), D/X slots (16 + 16 each), the all-ones A
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColA = 0;
constexpr uint32_t kColD = 128;
constexpr uint32_t kColOnes = 192;
constexpr uint32_t kIdesc = idesc_bf16(kTmRows, kTmN);

struct TmParams {
    const __nv_bfloat16* x;  // [M][K]
    const uint8_t* wq;       // [T][K/64][32] 16-byte lane units
    const uint8_t* wsz;      // [T][K/128][8] 8-byte entries
    __nv_bfloat16* out;      // [M][N]
    int* err;
    int M, N, K, T, G, S;
};

// pair t (0..3) of a word: nibbles t and t + 4 -> bf16 pair (128 + q_t, 128 + q_{t+4})
__device__ __forceinline__ uint32_t pair_bf16(uint32_t w) {
    uint32_t d;
    asm("lop3.b32 %0, %1, 0x000f000f, 0x43004300, 0xEA;" : "=r"(d) : "r"(w));
    return d;
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(taddr), "r"(v)
                 : "memory");
}

__global__ void __launch_bounds__(kTmThreads, 2) w4a16_tm_kernel(TmParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t wfull[kNW];
    __shared__ __align__(8) uint64_t mdone[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    griddep_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, kh = warp >> 2;
    const int S = P.S, G = P.G, K = P.K, M = P.M;
    const int p = blockIdx.x / S, rank = blockIdx.x - p * S;
    const int g0 = rank * G / S, nit = (rank + 1) * G / S - g0;  // nit >= 1 (S <= G)
    const int KC = K / 64;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bring = sbase;                     // [kBSlots][kBTile], 1024-aligned atoms
    const int woff = kBSlots * kBTile;                // [kNW][kWSlot]
    const uint32_t wring = sbase + woff;

    // this thread's row r of the block: tile r / 16, row g = r % 8 of it, the
    // lower (hi = 0) or upper (hi = 1) half of the tile's rows
    const int r = 32 * qd + lane;
    const int tt = r >> 4, gq = r & 7, hi = (r >> 3) & 1;

    if (tid == 0) {
        for (int i = 0; i < kNW; ++i) mbar_init(&wfull[i], 1);
        mbar_init(&mdone[0], 1);
        mbar_init(&mdone[1], 1);
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint32_t lane_q = (uint32_t)(32 * qd) << 16;  // TMEM lane quarter of this warp

    // group it of the split: 8 tiles x 1 KB of weights, 8 x 64 bytes of entries
    auto issue_w = [&](int it) {
        if (it >= nit) return;
        uint64_t* bar = &wfull[it % kNW];
        const uint32_t dst = wring + (it % kNW) * kWSlot;
        const int g = g0 + it;
        mbar_expect_tx(bar, kWSlot);
        for (int t = 0; t < kTmTiles; ++t) {
            const int tile = min(p * kTmTiles + t, P.T - 1);  // rows past N: any data, never stored
            bulk_load(dst + t * 1024, P.wq + ((size_t)tile * KC + 2 * g) * 512, 1024, bar);
            bulk_load(dst + kWBytes + t * 64, P.wsz + ((size_t)tile * G + g) * 64, 64, bar);
        }
    };
    // x rows of group it -> B slot it % kBSlots (rows >= M are never written:
    // they only feed D columns that are not read)
    auto issue_x = [&](int it) {
        if (it >= nit) return;
        const uint32_t b = bring + (it % kBSlots) * kBTile;
        const __nv_bfloat16* src = P.x + (size_t)(g0 + it) * 128;
        for (int i = tid; i < M * 16; i += kTmThreads) {
            const int m = i >> 4, c = i & 15;
            cp_async16(b + (c >> 3) * 2048 + sw128_off(m, c & 7), src + (size_t)m * K + 8 * c);
        }
    };

    if (tid == 0)
        for (int it = 0; it < kNW - 1; ++it) issue_w(it);
    if (kh == 0) {
        tmem_st8(tmem + lane_q + kColOnes, 0x3f803f80u);  // bf16 (1, 1)
        tmem_st_wait();
    }
    griddep_wait();  // x and the output may belong to the previous kernel of the stream
    issue_x(0);
    cp_async_commit();
    issue_x(1);
    cp_async_commit();
    int w_issued = kNW - 1 < nit ? kNW - 1 : nit;
    int mma_issued = 0;  // groups whose MMAs thread 0 has committed

    float acc[4] = {0.f, 0.f, 0.f, 0.f};  // x rows 4 kh .. 4 kh + 3 of row r
    float s_prev = 0.f, t_prev = 0.f;     // scale and s (128 + z) of group it - 1
    bool aborted = false;
    auto epilogue = [&](int j) {  // group j's D and X (its MMAs have completed)
        uint32_t d[4], xv[4];
        const uint32_t col = tmem + lane_q + kColD + 32 * (j & 1) + 4 * kh;
        tmem_ld4_nowait(col, d);
        tmem_ld4_nowait(col + 16, xv);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(s_prev, __uint_as_float(d[i]), fmaf(-t_prev, __uint_as_float(xv[i]), acc[i]));
    };

    for (int it = 0; it < nit; ++it) {
        if (tid == 0) {
            // weights of group it have landed; the MMAs of group it - 2 (the
            // last readers of A slot it % 2, D slot it % 2 and B slot
            // (it + 2) % 4) are done
            bool ok = mbar_wait_bounded(&wfull[it % kNW], (it / kNW) & 1);
            if (ok && it >= 2) ok = mbar_wait_bounded(&mdone[it & 1], ((it - 2) >> 1) & 1);
            if (!ok) {
                record_error(P.err, kDevErrTimeout);
                abort_s = 1;
            }
        }
        __syncthreads();
        tc_fence_after();
        if (abort_s) {
            aborted = true;
            break;
        }
        issue_x(it + 2);
        cp_async_commit();
        if (tid == 0 && it + kNW - 1 < nit) {
            issue_w(it + kNW - 1);  // into the stage of group it - 1, read by every thread
            ++w_issued;
        }

        // this row's K half of group it -> 32 TMEM columns of A slot it % 2
        const uint8_t* ws = smem + woff + (it % kNW) * kWSlot;
        const uint4* u = reinterpret_cast<const uint4*>(ws + tt * 1024 + kh * 512 + gq * 64);
        uint32_t a[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 q = u[c];
            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                // word s of unit c: inputs 16 c + 4 s .. + 3 of rows g (even
                // nibble pairs) and g + 8 (odd pairs)
                const uint32_t w = wv[s] >> (4 * hi);
                a[8 * c + 2 * s] = pair_bf16(w);           // inputs k0, k0 + 1
                a[8 * c + 2 * s + 1] = pair_bf16(w >> 8);  // inputs k0 + 2, k0 + 3
            }
        }
        tmem_st32(tmem + lane_q + kColA + 64 * (it & 1) + 32 * kh, a);
        const uint32_t e = *reinterpret_cast<const uint32_t*>(ws + kWBytes + tt * 64 + gq * 8 + hi * 4);
        const float s_cur = __half2float(__ushort_as_half((unsigned short)(e & 0xffffu)));
        const float t_cur = s_cur * __uint_as_float(e & 0xffff0000u);
        tmem_st_wait();

        if (it >= 1) {
            // warp-uniform outcome: the TMEM loads below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&mdone[(it - 1) & 1], ((it - 1) >> 1) & 1))) {
                record_error(P.err, kDevErrTimeout);
                abort_s = 1;
            } else {
                tc_fence_after();
                epilogue(it - 1);
            }
        }
        s_prev = s_cur;
        t_prev = t_cur;

        cp_async_wait<2>();  // this thread's x copies of group it have landed
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        if (abort_s) {
            aborted = true;
            break;
        }
        if (tid == 0) {
            tc_fence_after();
            const uint32_t b = bring + (it % kBSlots) * kBTile;
            const uint32_t dcol = tmem + kColD + 32 * (it & 1);
            const uint32_t acol = tmem + kColA + 64 * (it & 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ta(dcol, acol + 8 * kk, desc_sw128(b + (kk >> 2) * 2048 + 32 * (kk & 3)), kIdesc, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ta(dcol + 16, tmem + kColOnes, desc_sw128(b + (kk >> 2) * 2048 + 32 * (kk & 3)), kIdesc,
                            kk > 0);
            mma_commit(&mdone[it & 1]);
            ++mma_issued;
        }
    }
    // the last group's epilogue; then nothing of this CTA is in flight
    if (!aborted) {
        const int j = nit - 1;
        if (__all_sync(0xffffffffu, mbar_wait_bounded(&mdone[j & 1], (j >> 1) & 1))) {
            tc_fence_after();
            epilogue(j);
        } else {
            record_error(P.err, kDevErrTimeout);
            aborted = true;
        }
    }
    cp_async_wait<0>();
    if (tid == 0 && aborted) {
        // weight stages and MMAs still in flight complete (bounded) before the
        // memory is reused or freed
        for (int it = w_issued - kNW > 0 ? w_issued - kNW : 0; it < w_issued; ++it)
            mbar_wait_bounded(&wfull[it % kNW], (it / kNW) & 1);
        for (int j = mma_issued - 2 > 0 ? mma_issued - 2 : 0; j < mma_issued; ++j)
            mbar_wait_bounded(&mdone[j & 1], (j >> 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    aborted = aborted || abort_s;
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }

    const int n = p * kTmRows + r;
    if (S == 1) {
        if (!aborted && n < P.N)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (4 * kh + i < M) P.out[(size_t)(4 * kh + i) * P.N + n] = __float2bfloat16_rn(acc[i]);
        return;
    }
    // split-K in the cluster: partials [m][128 rows] fp32 in the x ring
    // (every copy into it has landed, every MMA reading it is done); CTA rank
    // adds the entries i = rank, rank + S, ... in rank order
    float* red = reinterpret_cast<float*>(smem);
#pragma unroll
    for (int i = 0; i < 4; ++i) red[(4 * kh + i) * kTmRows + r] = acc[i];
    cluster_sync();
    if (!aborted) {
        for (int i = rank + S * tid; i < M * kTmRows; i += S * kTmThreads) {
            const int m = i / kTmRows, rr = i - m * kTmRows;
            const int nn = p * kTmRows + rr;
            float sum = 0.f;
            for (int q0 = 0; q0 < S; q0 += 8) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q0 + q < S) v[q] = ld_cluster_f32(sbase + (uint32_t)i * 4u, (uint32_t)(q0 + q));
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q0 + q < S) sum += v[q];
            }
            if (nn < P.N) P.out[(size_t)m * P.N + nn] = __float2bfloat16_rn(sum);
        }
    }
    cluster_sync();  // no CTA leaves while its shared memory may still be read
}

// Opt-in to the dynamic shared memory and the non-portable cluster sizes
// (once per device); false if refused.
bool tm_prepare(int dev) {
    static std::atomic<int> done[64];
    if (done[dev & 63].load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(w4a16_tm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTmSmem) != cudaSuccess)
        return false;
    if (cudaFuncSetAttribute(w4a16_tm_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return false;
    done[dev & 63].store(1, std::memory_order_release);
    return true;
}

// Clusters of S CTAs the GPU holds at once (cached per device and size; 0 if
// that size cannot be launched).
int tm_max_clusters(int dev, int S) {
    static std::atomic<int> cache[64][kTmMaxSplits + 1];
    int v = cache[dev & 63][S].load(std::memory_order_acquire);
    if (v != 0) return v < 0 ? 0 : v;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S);
    cfg.blockDim = dim3(kTmThreads);
    cfg.dynamicSmemBytes = kTmSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, w4a16_tm_kernel, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = 0;
    }
    cache[dev & 63][S].store(n > 0 ? n : -1, std::memory_order_release);
    return n;
}

}  // namespace

// K splits for a shape: the S (<= 16, <= G; above 8 only while every split
// keeps 8 groups) that minimises (waves of co-resident clusters) x (groups per
// CTA + 3, the CTA's fixed cost in groups); 0 if none can be launched.
int w4a16_tm_splits(int N, int K) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !tm_prepare(dev)) return 0;
    const int P = (N + kTmRows - 1) / kTmRows, G = K / 128;
    int best = 0;
    long long best_cost = -1;
    for (int S = 1; S <= kTmMaxSplits && S <= G; ++S) {
        if (S > 8 && G < 8 * S) break;
        const long long clusters = tm_max_clusters(dev, S);
        if (clusters < 1) continue;
        const long long cost = ((P + clusters - 1) / clusters) * ((G + S - 1) / S + 3);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

cudaError_t launch_w4a16_tm(const void* x, const void* wq, const void* wsz, int M, int N, int K, void* out,
                            int* err, cudaStream_t s) {
    if (M < 1 || M > kTmMaxM || N < 1 || K < 128 || K % 128 != 0) return cudaErrorInvalidValue;
    const int S = w4a16_tm_splits(N, K);
    if (S < 1) return cudaErrorInvalidConfiguration;
    TmParams P;
    P.x = static_cast<const __nv_bfloat16*>(x);
    P.wq = static_cast<const uint8_t*>(wq);
    P.wsz = static_cast<const uint8_t*>(wsz);
    P.out = static_cast<__nv_bfloat16*>(out);
    P.err = err;
    P.M = M;
    P.N = N;
    P.K = K;
    P.T = (N + 15) / 16;
    P.G = K / 128;
    P.S = S;
    const int blocks = (N + kTmRows - 1) / kTmRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks * S);
    cfg.blockDim = dim3(kTmThreads);
    cfg.dynamicSmemBytes = kTmSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, w4a16_tm_kernel, P);
}

}  // namespace sd
