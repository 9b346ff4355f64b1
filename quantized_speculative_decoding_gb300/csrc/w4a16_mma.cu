// Register-operand tensor-core W4A16 GEMM for small M (1 <= M <= 32) on the
// fragment-ordered layout of sd_w4_tile.
//
// The verify-time linears of "When Do Quantized Drafts Help Speculative
// Decoding?" (pilot setup: M = batch x (gamma + 1) = 5 rows of x per target
// layer) read every weight once and do 2M flops per weight, far below any
// tensor-core roofline: the kernel is an HBM stream, and its design follows
// from keeping enough bytes in flight at a low instruction cost per byte.
//
//   - The fragment-ordered layout stores, for every 16 output rows and 64
//     inputs, the 32 lanes' mma.sync A operands back to back: one 16-byte
//     shared load per lane, 512 contiguous bytes per warp, no redundant bytes.
//   - Inside a 64-input chunk the input order is permuted so that lane c of a
//     quad needs inputs [16c, 16c + 16) of x: two 16-byte loads give its B
//     operands for the chunk's four k16 steps.  Weights are stored in the same
//     permuted order, so the dot product is unchanged.
//   - Each 32-bit weight word holds one lane's four A registers of one k16
//     step as nibble pairs (i, i + 4); one shift and one LOP3 turn a pair into
//     the bf16 pair (128 + q, 128 + q'), exact.
//   - Per quantisation group g (128 inputs) mma.sync m16n8k16 (bf16 operands,
//     fp32 accumulation) forms D_g = sum (128 + q) x for every row, and one more
//     MMA with an all-ones A forms X_g = sum x for every x row; the result is
//         y = sum_g s_g (D_g - (128 + z_g) X_g) = sum_k s (q - z) x,
//     accumulated in fp32.
//
// Work split: a CTA is one row block (4 warps x RT tiles of 16 rows) x one
// K split; it streams the split's quantisation groups through an NS-stage
// cp.async ring in shared memory that holds, per group, the block's weights,
// scale/zero entries and the group's x rows, one barrier per stage; warp w
// computes tiles RT w .. RT w + RT - 1 of the block.  The S K splits of a row
// block form one thread-block cluster and add their partials through
// distributed shared memory between two cluster barriers, in rank order, so
// results do not depend on scheduling and no workspace, fence or atomic is
// needed.
//
// Weights, scales and zero points are constant inputs and are requested
// before the kernel waits on the previous kernel of the stream (programmatic
// dependent launch); x and the output are touched only after the wait.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "device_common.cuh"
#include "launch.cuh"
#include "sd_internal.h"

namespace sd {
namespace {

constexpr int kChunkK = 64;  // inputs per 16-byte lane load

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_16816_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// (w >> 4t) & 0x000f000f | bf16 pair (128, 128): nibbles t and t + 4 as
// (128 + q_t, 128 + q_{t+4}), exact in bf16.  Written as one shift and one
// three-input logic op per pair (the compiler's own lowering of the C++ form
// spent about twice the instructions).
template <int T>
__device__ __forceinline__ uint32_t nib_pair(uint32_t w) {
    uint32_t d;
    if (T == 0)
        asm("lop3.b32 %0, %1, 0x000f000f, 0x43004300, 0xEA;" : "=r"(d) : "r"(w));
    else
        asm("{\n\t.reg .b32 t;\n\tshr.b32 t, %1, %2;\n\tlop3.b32 %0, t, 0x000f000f, 0x43004300, 0xEA;\n\t}"
            : "=r"(d)
            : "r"(w), "n"(4 * T));
    return d;
}

// INT2 / INT3 A operands of k16 step (h, s) from a lane's group units.  Word
// 2h + s/2 of the 16-byte 2-bit unit holds the step's four pairs at bits
// (2t, 2t + 16), t = 4 (s & 1) + i; for INT3 the third bits of pair i sit at
// bits (4s + i, 4s + i + 16) of word h of the 8-byte unit and are moved to
// bits (2, 18).  Each pair becomes the bf16 pair (128 + q, 128 + q'), exact.
template <int T>
__device__ __forceinline__ uint32_t crumb_pair(uint32_t w) {
    uint32_t d;
    if (T == 0)
        asm("lop3.b32 %0, %1, 0x00030003, 0x43004300, 0xEA;" : "=r"(d) : "r"(w));
    else
        asm("{\n\t.reg .b32 t;\n\tshr.b32 t, %1, %2;\n\tlop3.b32 %0, t, 0x00030003, 0x43004300, 0xEA;\n\t}"
            : "=r"(d)
            : "r"(w), "n"(2 * T));
    return d;
}
template <int P>
__device__ __forceinline__ uint32_t third_bit(uint32_t hi, uint32_t pair) {
    const uint32_t t = P >= 2 ? hi >> (P >= 2 ? P - 2 : 0) : hi << (P < 2 ? 2 - P : 0);
    uint32_t d;
    asm("lop3.b32 %0, %1, 0x00040004, %2, 0xEA;" : "=r"(d) : "r"(t), "r"(pair));
    return d;
}
template <int BITS, int H, int S>
__device__ __forceinline__ void lowbit_pairs_hs(const uint4& wl, const uint2& wh, uint32_t& a0, uint32_t& a1,
                                                uint32_t& a2, uint32_t& a3) {
    const uint32_t w = H == 0 ? (S < 2 ? wl.x : wl.y) : (S < 2 ? wl.z : wl.w);
    constexpr int T0 = 4 * (S & 1);
    a0 = crumb_pair<T0 + 0>(w);
    a1 = crumb_pair<T0 + 1>(w);
    a2 = crumb_pair<T0 + 2>(w);
    a3 = crumb_pair<T0 + 3>(w);
    if constexpr (BITS == 3) {
        const uint32_t hw = H == 0 ? wh.x : wh.y;
        a0 = third_bit<4 * S + 0>(hw, a0);
        a1 = third_bit<4 * S + 1>(hw, a1);
        a2 = third_bit<4 * S + 2>(hw, a2);
        a3 = third_bit<4 * S + 3>(hw, a3);
    }
}
template <int BITS>
__device__ __forceinline__ void lowbit_pairs(const uint4& wl, const uint2& wh, int h, int s, uint32_t& a0,
                                             uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    // h and s are compile-time constants at every call (unrolled loops)
    if (h == 0) {
        if (s == 0) lowbit_pairs_hs<BITS, 0, 0>(wl, wh, a0, a1, a2, a3);
        else if (s == 1) lowbit_pairs_hs<BITS, 0, 1>(wl, wh, a0, a1, a2, a3);
        else if (s == 2) lowbit_pairs_hs<BITS, 0, 2>(wl, wh, a0, a1, a2, a3);
        else lowbit_pairs_hs<BITS, 0, 3>(wl, wh, a0, a1, a2, a3);
    } else {
        if (s == 0) lowbit_pairs_hs<BITS, 1, 0>(wl, wh, a0, a1, a2, a3);
        else if (s == 1) lowbit_pairs_hs<BITS, 1, 1>(wl, wh, a0, a1, a2, a3);
        else if (s == 2) lowbit_pairs_hs<BITS, 1, 2>(wl, wh, a0, a1, a2, a3);
        else lowbit_pairs_hs<BITS, 1, 3>(wl, wh, a0, a1, a2, a3);
    }
}

// Whether half h of a quantisation group starts a fresh accumulator chain.
__device__ __forceinline__ constexpr bool s_first(int h, int hc) { return h == 0 || hc == 2; }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kXRow = 272;      // bytes per staged x row: 128 bf16 + 16 bytes of padding
constexpr int kMaxSplits = 16;  // CTAs of one cluster sharing a row block (non-portable cluster size, opted in)

// One ring stage: the row block's packed weights (BITS x 256 bytes per tile:
// 16 rows x 128 inputs), its scale/zero entries (64 bytes per tile) and the
// group's x rows (8 MT rows; in the W4A4 mode each row's activation scale sits
// in the row's padding).
template <int RT, int MT, int BITS, bool RM = false>
struct Stage {
    static constexpr int kTiles = kWarps * RT;
    static constexpr int kWTile = BITS * 256;
    static constexpr int kW = kTiles * kWTile;
    static constexpr int kSZ = kTiles * (RM ? 128 : 64);  // row-major: s pairs, then z pairs, per tile
    static constexpr int kX = 8 * MT * kXRow;
    static constexpr int kBytes = kW + kSZ + kX;
    static constexpr int kItems = kWarps * RT * MT * 32;  // float4 partials per CTA
    static constexpr int kPieces = kW / 16;               // 16-byte weight copies per stage
    static constexpr int kPiecesPerThread = (kPieces + kThreads - 1) / kThreads;
};

struct MmaParams {
    const __nv_bfloat16* x;  // [M][K], 16-byte aligned (W4A4: the activation codes)
    const float* sx;         // W4A4 only: activation scales [M][K/128]
    const uint4* wq;         // [T][K/128][BITS x 16] 16-byte units (INT4: [T][K/64][32] lane units);
                             // row-major mode: the sd_w4_pack qweight [N][K/8]
    const __half* scales;    // row-major mode: fp16 [N][K/128]
    const __half* zeros;     // row-major mode: fp16 [N][K/128]
    const uint2* wsz;        // [T][K/128][8]: {(s, 128 + z) of row g, of row g + 8}
    __nv_bfloat16* out;      // [M][N]
    int M, N, K;
    int T;                   // 16-row tiles
    int G;                   // quantisation groups (128 inputs) per row
    int S;                   // K splits = cluster size (1 .. kMaxSplits)
    // logits mode (the lm_head) only
    float* logits;           // [M] rows of stride ld_logits, fp32 (instead of out)
    float2* stats;           // [M] rows of stride ld_stats: one softmax partial per CTA
    long long ld_logits, ld_stats;
    float c;                 // log2(e) / T; 0 selects (max, argmax) partials (T = 0)
};

// One logit v (vocabulary index n) into a softmax partial (a, b): for c > 0
// (max, sum of exp2(l c - max c)), the row statistics at temperature
// T = log2(e) / c in raw logit units; for c = 0 (max, lowest index holding it).
__device__ __forceinline__ void lm_push(float& a, float& b, float v, int n, float c) {
    if (c > 0.f) {
        if (v > a) {
            b = (a == -INFINITY ? 0.f : b * exp2f(fmaf(a, c, -v * c))) + 1.f;
            a = v;
        } else {
            b += exp2f(fmaf(v, c, -a * c));
        }
    } else if (v > a || (v == a && n < __float_as_int(b))) {
        a = v;
        b = __int_as_float(n);
    }
}

// (a, b) := the merge of partials (a, b) and (a2, b2).
__device__ __forceinline__ void lm_merge(float& a, float& b, float a2, float b2, float c) {
    if (c > 0.f) {
        if (a2 == -INFINITY) return;
        if (a == -INFINITY) {
            a = a2;
            b = b2;
            return;
        }
        const float m = fmaxf(a, a2);
        b = b * exp2f(fmaf(a, c, -m * c)) + b2 * exp2f(fmaf(a2, c, -m * c));
        a = m;
    } else if (a2 > a || (a2 == a && __float_as_int(b2) < __float_as_int(b))) {
        a = a2;
        b = b2;
    }
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Exit barrier: only keeps every CTA's shared memory alive until the cluster's
// remote reads of it are done (their values are consumed before the arrive),
// so it needs no memory ordering and does not wait for the output stores.
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

// CTA (row block p, K split `rank`): the row block is kWarps x RT tiles of 16
// rows, the split is groups [rank G / S, (rank + 1) G / S).  The S CTAs of a
// row block form one cluster and add their partials through distributed
// shared memory, in rank order.
// kLM (logits mode, the lm_head): the outputs go out as fp32 logits, and each
// CTA also writes, per x row, the softmax partial of the logits it stored.
// BITS (4, 3 or 2): the weight code width of the tiled layout.
// kA4 (W4A4): x holds integer activation codes and P.sx their scales; each
// group's integer dot product is formed exactly and scaled by s_x s_w.
// kRM (row-major mode): the weights are read in the sd_w4_pack layout (row
// n's 16 words of a group are its 128 inputs in order) and the scales and
// zero points from their fp16 [N][K/128] arrays; lane c of a quad takes words
// 4c .. 4c+3 of rows g and g + 8, and k16 step (w, p) pairs nibbles (p, p+4)
// and (p+1, p+5) of word w with the same inputs of x, so that the K order
// inside the lane's 32 inputs cancels in the contraction.
template <int RT, int MT, int NS, bool kLM, int BITS, bool kA4, bool kRM>
__global__ void __launch_bounds__(kThreads, RT * MT <= 2 ? 5 : 3)
w4a16_mma_kernel(MmaParams P) {
    using S_ = Stage<RT, MT, BITS, kRM>;
    static_assert(BITS == 4 || BITS == 3 || BITS == 2, "weight code width");
    static_assert(!(kLM && (kA4 || BITS != 4)), "logits mode reads W4A16 only");
    static_assert(!(kRM && (kA4 || BITS != 4 || kLM)), "row-major mode reads W4A16 only");
    griddep_launch_dependents();
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int M = P.M, N = P.N, G = P.G, T = P.T, S = P.S;
    const int p = blockIdx.x / S, rank = blockIdx.x - (blockIdx.x / S) * S;
    const int g0 = rank * G / S, nu = (rank + 1) * G / S - g0;  // nu >= 1 (S <= G)
    const uint32_t base = smem_u32(smem);

    // x rows M .. 8 MT - 1 of a stage are never written: they only feed D
    // columns of x rows >= M, which are neither stored nor mixed into others

    // per-thread copy sources; every unit (group) advances them by a constant
    constexpr int kPT = S_::kWTile / 16;  // 16-byte pieces per tile and group
    const uint4* wsrc[S_::kPiecesPerThread];
#pragma unroll
    for (int i = 0; i < S_::kPiecesPerThread; ++i) {
        const int q = tid + kThreads * i;  // 16-byte piece of a stage's weights
        if constexpr (kRM) {
            // piece (tile, row, 16-byte chunk) of the group's 64 bytes per row
            const int n = min((p * S_::kTiles + q / kPT) * 16 + ((q % kPT) >> 2), N - 1);
            wsrc[i] = P.wq + (size_t)n * (P.K / 32) + (size_t)g0 * 4 + (q & 3);
        } else {
            const int tile = min(p * S_::kTiles + q / kPT, T - 1);
            wsrc[i] = P.wq + ((size_t)tile * G + g0) * kPT + (q % kPT);
        }
    }
    // scale/zero entries: tiled, 16 words per tile; row-major, per tile and row
    // the 4-byte pair of fp16 scales (then of zero points) of groups 2j, 2j + 1
    // holding the stage's group (G is even in this mode)
    const bool has_sz = tid < (kRM ? 32 : 16) * S_::kTiles;
    const uint32_t* szsrc;
    if constexpr (kRM) {
        const int n = min((p * S_::kTiles + (tid >> 5)) * 16 + (tid & 15), N - 1);
        szsrc = reinterpret_cast<const uint32_t*>((tid & 16 ? P.zeros : P.scales) + (size_t)n * G);
    } else {
        szsrc = reinterpret_cast<const uint32_t*>(
                    P.wsz + ((size_t)min(p * S_::kTiles + (tid >> 4), T - 1) * G + g0) * 8) + (tid & 15);
    }
    int gsz = g0;  // row-major mode: the group whose entries the next issue_w copies
    const __nv_bfloat16* xsrc[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) {
        const int q = tid + kThreads * j;  // x piece: row q / 16, 16 bytes q % 16
        xsrc[j] = P.x + (size_t)min(q >> 4, M - 1) * P.K + g0 * 128 + (q & 15) * 8;
    }
    const float* sxsrc = kA4 ? P.sx + (size_t)min(tid, M - 1) * G + g0 : nullptr;
    auto issue_w = [&](int slot) {
        const uint32_t dst = base + slot * S_::kBytes;
#pragma unroll
        for (int i = 0; i < S_::kPiecesPerThread; ++i) {
            if (S_::kPieces % kThreads == 0 || tid + kThreads * i < S_::kPieces)
                cp_async16(dst + (tid + kThreads * i) * 16, wsrc[i]);
            wsrc[i] += kPT;
        }
        if constexpr (kRM) {
            if (has_sz) cp_async4(dst + S_::kW + tid * 4, szsrc + (gsz >> 1));
            ++gsz;
        } else {
            if (has_sz) cp_async4(dst + S_::kW + tid * 4, szsrc);
            szsrc += 16;
        }
    };
    auto issue_x = [&](int slot) {
        const uint32_t dst = base + slot * S_::kBytes + S_::kW + S_::kSZ;
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            const int q = tid + kThreads * j;
            // row-major mode: chunk q of a row goes to slot (q & 12) | ((q + ((q >> 3) << 1)) & 3),
            // so that the four loads of each quad's lanes hit distinct banks
            const int slot = kRM ? ((q & 12) | ((q + (((q & 15) >> 3) << 1)) & 3)) : q;
            if (q < M * 16) cp_async16(dst + (q >> 4) * kXRow + (slot & 15) * 16, xsrc[j]);
            xsrc[j] += 128;
        }
        if constexpr (kA4) {
            if (tid < M) cp_async4(dst + tid * kXRow + 256, sxsrc);  // in the row's padding
            sxsrc += 1;
        }
    };

#pragma unroll
    for (int s = 0; s < NS - 1; ++s) {
        if (s < nu) issue_w(s);
        cp_async_commit();
    }
    griddep_wait();
    for (int s = 0; s < NS - 1 && s < nu; ++s) issue_x(s);
    cp_async_commit();

    float acc[RT][MT][4];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[r][mt][i] = 0.f;

    constexpr uint32_t kOnes = 0x3f803f80u;  // bf16 pair (1, 1)
    int slot = 0, islot = NS - 1;
    for (int u = 0; u < nu; ++u) {
        if (u == 0)
            cp_async_wait<0>();
        else
            cp_async_wait<NS - 2>();
        __syncthreads();  // stage u is complete for all threads; stage u - 1 is free
        if (u + NS - 1 < nu) {
            issue_w(islot);
            issue_x(islot);
        }
        cp_async_commit();
        islot = islot + 1 == NS ? 0 : islot + 1;

        // plain shared loads (not asm) so that the compiler may schedule them
        const uint8_t* sb = smem + slot * S_::kBytes;
        const uint8_t* wb = sb + warp * RT * S_::kWTile;
        const uint8_t* xb = sb + S_::kW + S_::kSZ;
        // INT2 / INT3: the lane's codes of the whole group in one 16-byte
        // unit (2-bit plane) and, for INT3, an 8-byte unit (third bits)
        uint4 wl[RT];
        uint2 wh[RT], wh2[RT];
        if constexpr (kRM) {
            // rows g and g + 8 of each tile: words 4c .. 4c + 3 of the group
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                wl[r] = *reinterpret_cast<const uint4*>(wb + r * 1024 + g * 64 + c * 16);
                const uint4 v = *reinterpret_cast<const uint4*>(wb + r * 1024 + (g + 8) * 64 + c * 16);
                wh[r] = make_uint2(v.x, v.y);
                wh2[r] = make_uint2(v.z, v.w);
            }
        } else if constexpr (BITS != 4) {
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                wl[r] = *reinterpret_cast<const uint4*>(wb + r * S_::kWTile + lane * 16);
                if constexpr (BITS == 3) wh[r] = *reinterpret_cast<const uint2*>(wb + r * S_::kWTile + 512 + lane * 8);
            }
        }
        // D = sum (128 + q) x per tile, and X = sum x (all-ones A) per x column.
        // With one tile and one x tile per warp the two 64-input halves
        // accumulate in separate registers (HC = 2), so that two MMA chains are
        // in flight instead of one.
        constexpr int HC = RT == 1 && MT == 1 ? 2 : 1;
        float part[HC][RT][MT][4], xs[HC][MT][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int hc = HC == 2 ? h : 0;
            const bool first = s_first(h, HC);
            uint4 xa[MT], xc[MT], wq[RT];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                if constexpr (kRM) {
                    // chunks 2h and 2h + 1 of the lane's 64 bytes (placed rotated by c & 2)
                    const uint8_t* xr = xb + (8 * mt + g) * kXRow + c * 64;
                    xa[mt] = *reinterpret_cast<const uint4*>(xr + ((2 * h + (c & 2)) & 3) * 16);
                    xc[mt] = *reinterpret_cast<const uint4*>(xr + ((2 * h + 1 + (c & 2)) & 3) * 16);
                } else {
                    const uint4* xrow = reinterpret_cast<const uint4*>(xb + (8 * mt + g) * kXRow + h * 128 + c * 32);
                    xa[mt] = xrow[0];
                    xc[mt] = xrow[1];
                }
            }
            if constexpr (BITS == 4 && !kRM) {
#pragma unroll
                for (int r = 0; r < RT; ++r)
                    wq[r] = *reinterpret_cast<const uint4*>(wb + r * 1024 + h * 512 + lane * 16);
            }
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                uint32_t b0[MT], b1[MT];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    if constexpr (kRM) {
                        // step s of half h: word w = 2h + s/2, nibble pairs p = 2 (s & 1) and p + 1:
                        // inputs (8w + p, 8w + p + 4) and (8w + p + 1, 8w + p + 5) of the lane's 32
                        const uint4& xw = s < 2 ? xa[mt] : xc[mt];
                        const uint32_t lo = (s & 1) ? xw.y : xw.x, hi = (s & 1) ? xw.w : xw.z;
                        b0[mt] = __byte_perm(lo, hi, 0x5410);
                        b1[mt] = __byte_perm(lo, hi, 0x7632);
                    } else {
                        b0[mt] = s == 0 ? xa[mt].x : s == 1 ? xa[mt].z : s == 2 ? xc[mt].x : xc[mt].z;
                        b1[mt] = s == 0 ? xa[mt].y : s == 1 ? xa[mt].w : s == 2 ? xc[mt].y : xc[mt].w;
                    }
                    if (first && s == 0)
                        mma_bf16_16816_zc(xs[hc][mt], kOnes, kOnes, kOnes, kOnes, b0[mt], b1[mt]);
                    else
                        mma_bf16_16816(xs[hc][mt], kOnes, kOnes, kOnes, kOnes, b0[mt], b1[mt]);
                }
#pragma unroll
                for (int r = 0; r < RT; ++r) {
                    uint32_t a0, a1, a2, a3;
                    if constexpr (kRM) {
                        const int w = 2 * h + (s >> 1);
                        const uint32_t vg = w == 0 ? wl[r].x : w == 1 ? wl[r].y : w == 2 ? wl[r].z : wl[r].w;
                        const uint32_t vh = w == 0 ? wh[r].x : w == 1 ? wh[r].y : w == 2 ? wh2[r].x : wh2[r].y;
                        if (s & 1) {
                            a0 = nib_pair<2>(vg);
                            a1 = nib_pair<2>(vh);
                            a2 = nib_pair<3>(vg);
                            a3 = nib_pair<3>(vh);
                        } else {
                            a0 = nib_pair<0>(vg);
                            a1 = nib_pair<0>(vh);
                            a2 = nib_pair<1>(vg);
                            a3 = nib_pair<1>(vh);
                        }
                    } else if constexpr (BITS == 4) {
                        const uint32_t wv = s == 0 ? wq[r].x : s == 1 ? wq[r].y : s == 2 ? wq[r].z : wq[r].w;
                        a0 = nib_pair<0>(wv);  // row g
                        a1 = nib_pair<1>(wv);  // row g + 8
                        a2 = nib_pair<2>(wv);  // row g, upper k
                        a3 = nib_pair<3>(wv);  // row g + 8, upper k
                    } else {
                        lowbit_pairs<BITS>(wl[r], wh[r], h, s, a0, a1, a2, a3);
                    }
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        if (first && s == 0)
                            mma_bf16_16816_zc(part[hc][r][mt], a0, a1, a2, a3, b0[mt], b1[mt]);
                        else
                            mma_bf16_16816(part[hc][r][mt], a0, a1, a2, a3, b0[mt], b1[mt]);
                    }
                }
            }
        }
        if (HC == 2) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xs[0][mt][i] += xs[HC - 1][mt][i];
#pragma unroll
                    for (int r = 0; r < RT; ++r) part[0][r][mt][i] += part[HC - 1][r][mt][i];
                }
        }
        // y += s (D - (128 + z) X): an entry word holds the fp16 scale in its
        // low half and 128 + z as bf16 (= the top half of its fp32) in its high half
#pragma unroll
        for (int r = 0; r < RT; ++r) {
            float s_g, s_h, zw_g, zw_h;
            if constexpr (kRM) {
                // fp16 scale and zero point of rows g, g + 8 for group g0 + u: half (g0 + u) & 1
                const uint8_t* e = sb + S_::kW + (warp * RT + r) * 128;
                const int sh = ((g0 + u) & 1) * 16;
                const auto f16 = [&](int off) {
                    return __half2float(__ushort_as_half((unsigned short)(*reinterpret_cast<const uint32_t*>(e + off) >> sh)));
                };
                s_g = f16(g * 4);
                s_h = f16((g + 8) * 4);
                zw_g = 128.f + f16(64 + g * 4);
                zw_h = 128.f + f16(64 + (g + 8) * 4);
            } else {
                const uint2 sz = *reinterpret_cast<const uint2*>(sb + S_::kW + (warp * RT + r) * 64 + g * 8);
                s_g = __low2float(*reinterpret_cast<const __half2*>(&sz.x));
                s_h = __low2float(*reinterpret_cast<const __half2*>(&sz.y));
                zw_g = __uint_as_float(sz.x & 0xffff0000u);
                zw_h = __uint_as_float(sz.y & 0xffff0000u);
            }
            if constexpr (kA4) {
                // integer codes: D - (128 + z) X is the exact integer
                // sum q_x (q_w - z) (every term below 2^24), then s_x s_w
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const float sx0 = *reinterpret_cast<const float*>(xb + (8 * mt + 2 * c) * kXRow + 256);
                    const float sx1 = *reinterpret_cast<const float*>(xb + (8 * mt + 2 * c + 1) * kXRow + 256);
                    acc[r][mt][0] = fmaf(s_g * sx0, fmaf(-zw_g, xs[0][mt][0], part[0][r][mt][0]), acc[r][mt][0]);
                    acc[r][mt][1] = fmaf(s_g * sx1, fmaf(-zw_g, xs[0][mt][1], part[0][r][mt][1]), acc[r][mt][1]);
                    acc[r][mt][2] = fmaf(s_h * sx0, fmaf(-zw_h, xs[0][mt][2], part[0][r][mt][2]), acc[r][mt][2]);
                    acc[r][mt][3] = fmaf(s_h * sx1, fmaf(-zw_h, xs[0][mt][3], part[0][r][mt][3]), acc[r][mt][3]);
                }
            } else {
                const float t_g = s_g * zw_g;
                const float t_h = s_h * zw_h;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    acc[r][mt][0] = fmaf(-t_g, xs[0][mt][0], fmaf(s_g, part[0][r][mt][0], acc[r][mt][0]));
                    acc[r][mt][1] = fmaf(-t_g, xs[0][mt][1], fmaf(s_g, part[0][r][mt][1], acc[r][mt][1]));
                    acc[r][mt][2] = fmaf(-t_h, xs[0][mt][2], fmaf(s_h, part[0][r][mt][2], acc[r][mt][2]));
                    acc[r][mt][3] = fmaf(-t_h, xs[0][mt][3], fmaf(s_h, part[0][r][mt][3], acc[r][mt][3]));
                }
            }
        }
        slot = slot + 1 == NS ? 0 : slot + 1;
    }

    // D element i of lane l: row 16 tile + l / 4 (+8 for i >= 2), x row 8 mt + 2 (l % 4) + (i & 1).
    // Logits mode: the softmax partials of this thread's two x rows in each x
    // tile (every item a thread stores has the same l).
    float lm_a[MT][2], lm_b[MT][2];
    if constexpr (kLM) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                lm_a[t][h] = -INFINITY;
                lm_b[t][h] = P.c > 0.f ? 0.f : __int_as_float(0x7fffffff);
            }
    }
    auto store4 = [&](int w, int r, int mt, int l, const float4& v) {
        const int tile = p * S_::kTiles + w * RT + r;
        if (tile >= T) return;
        const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = tile * 16 + (l >> 2) + (i >= 2 ? 8 : 0);
            const int m = 8 * mt + 2 * (l & 3) + (i & 1);
            if constexpr (kLM) {
                if (n < N && m < M) {
                    P.logits[(size_t)m * P.ld_logits + n] = e[i];
#pragma unroll
                    for (int t = 0; t < MT; ++t)
                        if (t == mt) lm_push(lm_a[t][i & 1], lm_b[t][i & 1], e[i], n, P.c);
                }
            } else {
                if (n < N && m < M) P.out[(size_t)m * N + n] = __float2bfloat16_rn(e[i]);
            }
        }
    };
    if (S == 1) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                store4(warp, r, mt, lane, make_float4(acc[r][mt][0], acc[r][mt][1], acc[r][mt][2], acc[r][mt][3]));
        if constexpr (!kLM) return;
    } else {
        // the cluster's partials: item (w, r, mt, l) of every CTA at the same
        // offset of its ring memory, added in rank order by CTA item % S
        cp_async_wait<0>();
        __syncthreads();  // every warp is done with the ring
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                float4* dst = reinterpret_cast<float4*>(smem) + ((warp * RT + r) * MT + mt) * 32 + lane;
                *dst = make_float4(acc[r][mt][0], acc[r][mt][1], acc[r][mt][2], acc[r][mt][3]);
            }
        cluster_sync();
        for (int it = rank + S * tid; it < S_::kItems; it += S * kThreads) {
            const int l = it & 31, rm = it >> 5;
            const int mt = rm % MT, wr = rm / MT;
            if (8 * mt + 2 * (l & 3) >= M) continue;  // all four x columns past M
            // remote loads eight at a time in flight, added in rank order
            float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int q0 = 0; q0 < S; q0 += 8) {
                float4 v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q0 + q < S) v[q] = ld_cluster_f4(base + it * 16, (uint32_t)(q0 + q));
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q0 + q < S) {
                        sum.x += v[q].x;
                        sum.y += v[q].y;
                        sum.z += v[q].z;
                        sum.w += v[q].w;
                    }
            }
            store4(wr / RT, wr % RT, mt, l, sum);
        }
        cluster_sync_relaxed();  // no CTA leaves while its shared memory may still be read
    }

    if constexpr (kLM) {
        // Lanes with equal lane % 4 hold the same x rows: l % 4 is
        // (rank + S lane) % 4 (rank 0, S 1 without a cluster).  Merge them by
        // shuffles, then each x row's classes across the warps.
        __shared__ float2 lm_s[kWarps][4][MT][2];
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int o = 4; o < 32; o <<= 1)
                    lm_merge(lm_a[t][h], lm_b[t][h], __shfl_xor_sync(0xffffffffu, lm_a[t][h], o),
                             __shfl_xor_sync(0xffffffffu, lm_b[t][h], o), P.c);
                if (lane < 4) lm_s[warp][lane][t][h] = make_float2(lm_a[t][h], lm_b[t][h]);
            }
        __syncthreads();
        if (tid < 8 * MT) {
            const int m = tid, t = m >> 3, h = m & 1, pair = (m & 7) >> 1;
            float a = -INFINITY, b = P.c > 0.f ? 0.f : __int_as_float(0x7fffffff);
            for (int w = 0; w < kWarps; ++w)
                for (int cl = 0; cl < 4; ++cl)
                    if (((rank + S * cl) & 3) == pair) {
                        const float2 e = lm_s[w][cl][t][h];
                        lm_merge(a, b, e.x, e.y, P.c);
                    }
            if (m < M) P.stats[(size_t)m * P.ld_stats + blockIdx.x] = make_float2(a, b);
        }
    }
}

// sd_w4_pack layout -> fragment-ordered layout, one thread per 16-byte lane
// unit (tile t, chunk j, lane l = 4 g + c).  Word s of the unit is the lane's
// k16 step s; with k0 = 64 j + 16 c + 4 s its nibbles (low to high) are
//   (g, k0) (g+8, k0) (g, k0+2) (g+8, k0+2) (g, k0+1) (g+8, k0+1) (g, k0+3) (g+8, k0+3)
// (rows relative to 16 t).  Rows past N are zero, scale and zero point 0.
// Scale/zero entry (t, group, g) holds, for row 16 t + g and then row
// 16 t + g + 8, the fp16 scale in the low half and 128 + z as bf16 in the high
// half.  Records SD_ERR_INVALID_ARG when a zero point is not an integer in
// [0, 15].
__global__ void w4_tile_kernel(const uint32_t* __restrict__ qw, const __half* __restrict__ scales,
                               const __half* __restrict__ zeros, int N, int K, uint4* __restrict__ wq,
                               uint2* __restrict__ wsz, int* err) {
    const int KC = K / kChunkK, G = K / 128, T = (N + 15) / 16;
    const size_t units = (size_t)T * KC * 32;
    const int wpr = K / 8;  // packed words per row
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < units;
         i += (size_t)gridDim.x * blockDim.x) {
        const int l = (int)(i & 31);
        const size_t tj = i >> 5;
        const int j = (int)(tj % KC);
        const int t = (int)(tj / KC);
        const int g = l >> 2, c = l & 3;
        const int ng = t * 16 + g, nh = ng + 8;
        // inputs 64 j + 16 c + [0, 16) of rows ng and nh: packed words 8 j + 2 c, + 1
        const size_t wi = (size_t)8 * j + 2 * c;
        const uint64_t rg = ng < N ? ((uint64_t)qw[(size_t)ng * wpr + wi + 1] << 32) | qw[(size_t)ng * wpr + wi] : 0;
        const uint64_t rh = nh < N ? ((uint64_t)qw[(size_t)nh * wpr + wi + 1] << 32) | qw[(size_t)nh * wpr + wi] : 0;
        uint32_t w[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint32_t a = (uint32_t)(rg >> (16 * s)) & 0xffffu;  // row g, k0 .. k0+3
            const uint32_t b = (uint32_t)(rh >> (16 * s)) & 0xffffu;  // row g+8
            w[s] = (a & 0xf) | (b & 0xf) << 4 | ((a >> 8) & 0xf) << 8 | ((b >> 8) & 0xf) << 12 |
                   ((a >> 4) & 0xf) << 16 | ((b >> 4) & 0xf) << 20 | ((a >> 12) & 0xf) << 24 |
                   ((b >> 12) & 0xf) << 28;
        }
        wq[i] = make_uint4(w[0], w[1], w[2], w[3]);
        if ((j & 1) == 0 && c == 0) {
            // entry (t, gr, g): {fp16 s, bf16 128 + z} of row ng, then of row nh
            const int gr = j >> 1;
            uint32_t e[2] = {0x43000000u, 0x43000000u};  // rows past N: s = 0, z = 0
            const int rows[2] = {ng, nh};
            for (int h = 0; h < 2; ++h) {
                if (rows[h] >= N) continue;
                const __half sc = scales[(size_t)rows[h] * G + gr];
                const float z = __half2float(zeros[(size_t)rows[h] * G + gr]);
                if (!(z >= 0.f && z <= 15.f && z == rintf(z))) record_error(err, kDevErrInvalidArg);
                const uint32_t zi = z >= 0.f && z <= 15.f ? (uint32_t)z : 0u;
                e[h] = (uint32_t)__half_as_ushort(sc) | (0x4300u + zi) << 16;
            }
            uint2 v;
            v.x = e[0];
            v.y = e[1];
            wsz[((size_t)t * G + gr) * 8 + g] = v;
        }
    }
}

template <int RT, int MT, int NS, bool kLM = false, int BITS = 4, bool kA4 = false, bool kRM = false>
struct Config {
    using St = Stage<RT, MT, BITS, kRM>;
    static constexpr int kTiles = St::kTiles;
    static constexpr size_t kSmem = (size_t)NS * St::kBytes;
    static_assert(St::kItems * 16 <= (int)kSmem && kTiles == kWarps * RT, "partials fit in the ring");
    static void (*kernel())(MmaParams) { return w4a16_mma_kernel<RT, MT, NS, kLM, BITS, kA4, kRM>; }
    using Logits = Config<RT, MT, NS, true, BITS, kA4, kRM>;  // the same shape in logits mode
};
// x rows in tiles of 8 (MT); row blocks of 8 tiles (RT = 2) for tall
// matrices, 4 tiles (RT = 1) when more row blocks are needed to fill the GPU.
// One family per weight format (code width BITS, W4A4 activations A4).
template <int BITS, bool A4, bool RM = false>
struct Family {
    using Cfg1w = Config<2, 1, 8, false, BITS, A4, RM>;
    using Cfg1n = Config<1, 1, 8, false, BITS, A4, RM>;
    using Cfg2 = Config<1, 2, 5, false, BITS, A4, RM>;
    using Cfg3 = Config<1, 3, 4, false, BITS, A4, RM>;
    using Cfg4 = Config<1, 4, 4, false, BITS, A4, RM>;
    static constexpr int kMaxM = BITS == 4 && !A4 ? 32 : 8;  // the other formats serve M <= 8
};
using W4 = Family<4, false>;
using W4RowMajor = Family<4, false, true>;

struct Shape {
    int cfg;  // 0 = Cfg1w, 1 = Cfg1n, 2..4 = Cfg2..Cfg4
    int T, G, P, S;
};

// Opts the configuration into its dynamic shared memory and returns its
// resident CTAs per SM (once per device; later calls read the cache), or -1.
template <class C>
int resident_ctas(int dev) {
    static std::atomic<int> cache[64];
    int v = cache[dev & 63].load(std::memory_order_acquire);
    if (v > 0) return v;
    int n = 0;
    if (cudaFuncSetAttribute(C::kernel(), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
        return -1;
    if (cudaFuncSetAttribute(C::kernel(), cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return -1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, C::kernel(), kThreads, C::kSmem) != cudaSuccess || n < 1)
        return -1;
    cache[dev & 63].store(n, std::memory_order_release);
    return n;
}

// Clusters of S CTAs the GPU holds at once (queried once per device and
// cluster size; 0 if that size cannot be launched).
template <class C>
int max_clusters(int dev, int S) {
    static std::atomic<int> cache[64][kMaxSplits + 1];
    int v = cache[dev & 63][S].load(std::memory_order_acquire);
    if (v != 0) return v < 0 ? 0 : v;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, C::kernel(), &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();  // leave no sticky error behind a refused size
        n = 0;
    }
    cache[dev & 63][S].store(n > 0 ? n : -1, std::memory_order_release);
    return n;
}

// Row blocks P = ceil(T / tiles per block); K splits S per row block (= the
// cluster size, at most kMaxSplits and G; above 8 only while every split keeps
// 8 groups), the S that minimises (waves of co-resident clusters) x (groups
// per CTA + 2, the CTA's fixed cost).  S = 0 when the configuration cannot be
// launched.
template <class C>
void fill(Shape& sh, int cfg, int N, int K, int sms) {
    (void)sms;
    sh.cfg = cfg;
    sh.T = (N + 15) / 16;
    sh.G = K / 128;
    sh.P = (sh.T + C::kTiles - 1) / C::kTiles;
    sh.S = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    if (resident_ctas<C>(dev) < 1) return;
    long long best_cost = -1;
    for (int S = 1; S <= kMaxSplits && S <= sh.G; ++S) {
        if (S > 8 && sh.G < 8 * S) break;  // clusters past 8 only for long K
        const long long clusters = max_clusters<C>(dev, S);
        if (clusters < 1) continue;
        const long long cost = ((sh.P + clusters - 1) / clusters) * ((sh.G + S - 1) / S + 2);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            sh.S = S;
        }
    }
}

template <class F>
Shape shape_for(int M, int N, int K, int sms) {
    Shape sh;
    switch ((M + 7) / 8) {
        case 1: {
            // tall row blocks while they alone give most of a wave's CTAs
            fill<typename F::Cfg1w>(sh, 0, N, K, sms);
            int dev = 0;
            cudaGetDevice(&dev);
            const long long wave = (long long)sms * resident_ctas<typename F::Cfg1w>(dev);
            if (sh.S > 0 && (long long)sh.P * sh.S * 4 < wave * 3) fill<typename F::Cfg1n>(sh, 1, N, K, sms);
            return sh;
        }
        default:
            if constexpr (F::kMaxM > 8) {
                if (M <= 16) fill<typename F::Cfg2>(sh, 2, N, K, sms);
                else if (M <= 24) fill<typename F::Cfg3>(sh, 3, N, K, sms);
                else fill<typename F::Cfg4>(sh, 4, N, K, sms);
            } else {
                sh.S = 0;  // the format serves M <= 8 only
            }
            return sh;
    }
}

template <class C>
cudaError_t launch_cfg(const MmaParams& P, int blocks, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks * P.S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = P.S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, C::kernel(), P);
}

}  // namespace

void w4_tiled_sizes(int N, int K, size_t* q_bytes, size_t* sz_bytes) {
    const size_t T = (N + 15) / 16;
    *q_bytes = T * (K / kChunkK) * 32 * 16;
    *sz_bytes = T * (K / 128) * 8 * 8;
}

cudaError_t launch_w4_tile(const uint32_t* qweight, const void* scales, const void* zeros, int N,
                           int K, void* wq, void* wsz, int* err, int sms, cudaStream_t s) {
    const size_t units = (size_t)((N + 15) / 16) * (K / kChunkK) * 32;
    size_t blocks = (units + 255) / 256;
    if (blocks > (size_t)sms * 16) blocks = (size_t)sms * 16;
    if (blocks < 1) blocks = 1;
    w4_tile_kernel<<<(unsigned)blocks, 256, 0, s>>>(qweight, static_cast<const __half*>(scales),
                                                    static_cast<const __half*>(zeros), N, K,
                                                    static_cast<uint4*>(wq), static_cast<uint2*>(wsz), err);
    return cudaGetLastError();
}

namespace {
// One linear of weight format F: plan, then launch the planned configuration.
template <class F>
cudaError_t launch_family(MmaParams P, int sms, cudaStream_t s) {
    const int M = P.M, N = P.N, K = P.K;
    if (M < 1 || M > F::kMaxM || N < 1 || K < 128 || K % 128 != 0) return cudaErrorInvalidValue;
    if ((long long)((N + 15) / 16) * (K / 128) * 64 >= (1LL << 31)) return cudaErrorInvalidValue;
    const Shape sh = shape_for<F>(M, N, K, sms);
    if (sh.S < 1) return cudaErrorInvalidConfiguration;
    P.T = sh.T;
    P.G = sh.G;
    P.S = sh.S;
    switch (sh.cfg) {
        case 0: return launch_cfg<typename F::Cfg1w>(P, sh.P, s);
        case 1: return launch_cfg<typename F::Cfg1n>(P, sh.P, s);
        default:
            if constexpr (F::kMaxM > 8) {
                switch (sh.cfg) {
                    case 2: return launch_cfg<typename F::Cfg2>(P, sh.P, s);
                    case 3: return launch_cfg<typename F::Cfg3>(P, sh.P, s);
                    default: return launch_cfg<typename F::Cfg4>(P, sh.P, s);
                }
            }
            return cudaErrorInvalidValue;
    }
}

MmaParams linear_params(const void* x, const void* wq, const void* wsz, int M, int N, int K, void* out) {
    MmaParams P = {};
    P.x = static_cast<const __nv_bfloat16*>(x);
    P.wq = static_cast<const uint4*>(wq);
    P.wsz = static_cast<const uint2*>(wsz);
    P.out = static_cast<__nv_bfloat16*>(out);
    P.M = M;
    P.N = N;
    P.K = K;
    return P;
}

// R11 bit stream -> the b-bit fragment-ordered layout, one thread per
// (tile t, group gr, lane l = 4 g + c) unit.  Step (h, s) of the lane covers
// inputs k0 .. k0 + 3, k0 = 128 gr + 64 h + 16 c + 4 s, of rows g and g + 8
// (relative to 16 t), as four pairs i: (g, k0 | k0+1), (g+8, k0 | k0+1),
// (g, k0+2 | k0+3), (g+8, k0+2 | k0+3) -- the INT4 layout's k order.  The low
// two bits of pair i go to word 2h + s/2 of the 16-byte unit at bits
// (2t, 2t + 16), t = 4 (s & 1) + i; for b = 3 the third bits go to word h of
// the 8-byte unit at bits (4s + i, 4s + i + 16).  Rows past N are zero with
// scale and zero point 0; the scale/zero entries are those of the INT4
// layout.  Records SD_ERR_INVALID_ARG when a zero point is not an integer in
// [0, 2^b - 1].
__device__ __forceinline__ uint32_t stream_code(const uint32_t* row, long words, int bits, int k) {
    const long bit = (long)bits * k;
    const long w = bit >> 5;
    const uint64_t lo = row[w];
    const uint64_t hi = w + 1 < words ? row[w + 1] : 0u;
    return (uint32_t)(((hi << 32 | lo) >> (bit & 31)) & ((1u << bits) - 1u));
}

__global__ void wb_tile_kernel(const uint32_t* __restrict__ packed, const __half* __restrict__ scales,
                               const __half* __restrict__ zeros, int bits, int N, int K, uint8_t* __restrict__ wq,
                               uint2* __restrict__ wsz, int* err) {
    const int G = K / 128, T = (N + 15) / 16;
    const long words = (long)K * bits / 32;
    const size_t units = (size_t)T * G * 32;
    const int zmax = (1 << bits) - 1;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < units; i += (size_t)gridDim.x * blockDim.x) {
        const int l = (int)(i & 31);
        const size_t tg = i >> 5;
        const int gr = (int)(tg % G);
        const int t = (int)(tg / G);
        const int g = l >> 2, c = l & 3;
        const int rows[2] = {t * 16 + g, t * 16 + g + 8};
        uint32_t lo[4] = {0u, 0u, 0u, 0u}, hi[2] = {0u, 0u};
        for (int h = 0; h < 2; ++h)
            for (int st = 0; st < 4; ++st) {
                const int k0 = 128 * gr + 64 * h + 16 * c + 4 * st;
                for (int pi = 0; pi < 4; ++pi) {
                    const int row = rows[pi & 1];
                    const int k = k0 + (pi >> 1) * 2;  // pair (k, k + 1)
                    uint32_t q0 = 0u, q1 = 0u;
                    if (row < N) {
                        const uint32_t* r = packed + (size_t)row * words;
                        q0 = stream_code(r, words, bits, k);
                        q1 = stream_code(r, words, bits, k + 1);
                    }
                    const int tt = 4 * (st & 1) + pi;
                    lo[2 * h + (st >> 1)] |= (q0 & 3u) << (2 * tt) | (q1 & 3u) << (2 * tt + 16);
                    if (bits == 3) hi[h] |= (q0 >> 2) << (4 * st + pi) | (q1 >> 2) << (4 * st + pi + 16);
                }
            }
        uint8_t* unit = wq + tg * (size_t)(bits * 256);
        reinterpret_cast<uint4*>(unit)[l] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if (bits == 3) reinterpret_cast<uint2*>(unit + 512)[l] = make_uint2(hi[0], hi[1]);
        if (c == 0) {
            uint32_t e[2] = {0x43000000u, 0x43000000u};  // rows past N: s = 0, z = 0
            for (int hh = 0; hh < 2; ++hh) {
                if (rows[hh] >= N) continue;
                const __half sc = scales[(size_t)rows[hh] * G + gr];
                const float z = __half2float(zeros[(size_t)rows[hh] * G + gr]);
                const bool ok = z >= 0.f && z <= (float)zmax && z == rintf(z);
                if (!ok) record_error(err, kDevErrInvalidArg);
                e[hh] = (uint32_t)__half_as_ushort(sc) | (0x4300u + (ok ? (uint32_t)z : 0u)) << 16;
            }
            wsz[tg * 8 + g] = make_uint2(e[0], e[1]);
        }
    }
}

// W4A4 activation codes: one warp per (row m, group g); amax in fp32 (exact
// from bf16), s = amax / 7 and each code RNE(x / s) clamped to [-8, 7], both
// divisions IEEE fp32 round-to-nearest; s = 1 for an all-zero group.  Codes
// go out as bf16 integers.  Records SD_ERR_INVALID_ARG for a non-finite input.
__global__ void a4_quantize_kernel(const __nv_bfloat16* __restrict__ x, int M, int K,
                                   __nv_bfloat16* __restrict__ qx, float* __restrict__ sx, int* err) {
    griddep_launch_dependents();
    griddep_wait();
    const int G = K / 128;
    const long long warps = (long long)M * G;
    const int lane = threadIdx.x & 31;
    for (long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; w < warps;
         w += ((long long)gridDim.x * blockDim.x) >> 5) {
        const int m = (int)(w / G), g = (int)(w % G);
        const size_t off = (size_t)m * K + (size_t)g * 128 + lane * 4;
        const uint2 raw = *reinterpret_cast<const uint2*>(x + off);
        float v[4];
        v[0] = __uint_as_float(raw.x << 16);
        v[1] = __uint_as_float(raw.x & 0xffff0000u);
        v[2] = __uint_as_float(raw.y << 16);
        v[3] = __uint_as_float(raw.y & 0xffff0000u);
        bool finite = true;
        uint32_t amax = 0u;  // |v| bit patterns order like the values
        for (int i = 0; i < 4; ++i) {
            finite = finite && isfinite(v[i]);
            amax = max(amax, __float_as_uint(fabsf(v[i])));
        }
        amax = __reduce_max_sync(0xffffffffu, amax);
        const bool all_finite = __all_sync(0xffffffffu, finite);
        if (!all_finite && lane == 0) record_error(err, kDevErrInvalidArg);
        const float a = __uint_as_float(amax);
        const float sc = a > 0.f ? __fdiv_rn(a, 7.0f) : 1.0f;
        uint32_t out[2];
        for (int i = 0; i < 2; ++i) {
            float q0 = rintf(__fdiv_rn(v[2 * i], sc)), q1 = rintf(__fdiv_rn(v[2 * i + 1], sc));
            q0 = fminf(fmaxf(q0, -8.f), 7.f);
            q1 = fminf(fmaxf(q1, -8.f), 7.f);
            // small integers: the top half of the fp32 is their exact bf16
            out[i] = (__float_as_uint(q0) >> 16) | (__float_as_uint(q1) & 0xffff0000u);
        }
        *reinterpret_cast<uint2*>(qx + off) = make_uint2(out[0], out[1]);
        if (lane == 0) sx[(size_t)m * G + g] = sc;
    }
}
}  // namespace

cudaError_t launch_w4a16_mma(const void* x, const void* wq, const void* wsz, int M, int N, int K,
                             void* out, int sms, cudaStream_t s) {
    return launch_family<W4>(linear_params(x, wq, wsz, M, N, K, out), sms, s);
}

bool w4a16_mma_rowmajor_ok(const void* qweight, const void* scales, const void* zeros, int M, int K) {
    const auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
    return M >= 1 && M <= 32 && K >= 256 && K % 256 == 0 && al(qweight, 16) && al(scales, 4) && al(zeros, 4);
}

cudaError_t launch_w4a16_mma_rowmajor(const void* x, const uint32_t* qweight, const void* scales, const void* zeros,
                                      int M, int N, int K, void* out, int sms, cudaStream_t s) {
    if (!w4a16_mma_rowmajor_ok(qweight, scales, zeros, M, K)) return cudaErrorInvalidValue;
    MmaParams P = linear_params(x, qweight, nullptr, M, N, K, out);
    P.scales = static_cast<const __half*>(scales);
    P.zeros = static_cast<const __half*>(zeros);
    return launch_family<W4RowMajor>(P, sms, s);
}

void wb_tiled_sizes(int N, int K, int bits, size_t* q_bytes, size_t* sz_bytes) {
    const size_t T = (N + 15) / 16;
    *q_bytes = T * (K / 128) * (size_t)bits * 256;
    *sz_bytes = T * (K / 128) * 8 * 8;
}

cudaError_t launch_wb_tile(const uint32_t* packed, const void* scales, const void* zeros, int bits, int N,
                           int K, void* wq, void* wsz, int* err, int sms, cudaStream_t s) {
    if (bits != 2 && bits != 3) return cudaErrorInvalidValue;
    const size_t units = (size_t)((N + 15) / 16) * (K / 128) * 32;
    size_t blocks = (units + 255) / 256;
    if (blocks > (size_t)sms * 16) blocks = (size_t)sms * 16;
    if (blocks < 1) blocks = 1;
    wb_tile_kernel<<<(unsigned)blocks, 256, 0, s>>>(packed, static_cast<const __half*>(scales),
                                                    static_cast<const __half*>(zeros), bits, N, K,
                                                    static_cast<uint8_t*>(wq), static_cast<uint2*>(wsz), err);
    return cudaGetLastError();
}

cudaError_t launch_wb_mma(const void* x, const void* wq, const void* wsz, int bits, int M, int N, int K, void* out,
                          int sms, cudaStream_t s) {
    const MmaParams P = linear_params(x, wq, wsz, M, N, K, out);
    switch (bits) {
        case 2: return launch_family<Family<2, false>>(P, sms, s);
        case 3: return launch_family<Family<3, false>>(P, sms, s);
        case 4: return launch_family<W4>(P, sms, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_a4_quantize(const void* x, int M, int K, void* qx, float* sx, int* err, int sms,
                               cudaStream_t s) {
    if (M < 1 || K < 128 || K % 128 != 0) return cudaErrorInvalidValue;
    const long long warps = (long long)M * (K / 128);
    long long blocks = (warps + 7) / 8;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, a4_quantize_kernel, static_cast<const __nv_bfloat16*>(x), M, K,
                              static_cast<__nv_bfloat16*>(qx), sx, err);
}

cudaError_t launch_w4a4_mma(const void* qx, const float* sx, const void* wq, const void* wsz, int M, int N, int K,
                            void* out, int sms, cudaStream_t s) {
    MmaParams P = linear_params(qx, wq, wsz, M, N, K, out);
    P.sx = sx;
    return launch_family<Family<4, true>>(P, sms, s);
}

int w4a16_lm_head_parts(int M, int N, int K, int sms) {
    if (M < 1 || M > 32 || N < 1 || K < 128 || K % 128 != 0) return -1;
    const Shape sh = shape_for<W4>(M, N, K, sms);
    return sh.S < 1 ? -1 : sh.P * sh.S;
}

namespace {
// The logits-mode launch of configuration C for shape sh: its own opt-ins
// (shared memory, cluster size) and a check that its clusters fit.
template <class C>
cudaError_t launch_logits_cfg(const MmaParams& P, int blocks, cudaStream_t s) {
    using L = typename C::Logits;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (resident_ctas<L>(dev) < 1 || max_clusters<L>(dev, P.S) < 1) return cudaErrorInvalidConfiguration;
    return launch_cfg<L>(P, blocks, s);
}
}  // namespace

cudaError_t launch_w4a16_lm_head(const void* x, const void* wq, const void* wsz, int M, int N, int K,
                                 float temperature, float* logits, long long ld_logits, void* stats,
                                 long long ld_stats, int sms, cudaStream_t s) {
    if (M < 1 || M > 32 || N < 1 || K < 128 || K % 128 != 0 || ld_logits < N) return cudaErrorInvalidValue;
    if ((long long)((N + 15) / 16) * (K / kChunkK) >= (1LL << 31)) return cudaErrorInvalidValue;
    const Shape sh = shape_for<W4>(M, N, K, sms);
    if (sh.S < 1) return cudaErrorInvalidConfiguration;
    if (ld_stats < (long long)sh.P * sh.S) return cudaErrorInvalidValue;
    MmaParams P = {};
    P.x = static_cast<const __nv_bfloat16*>(x);
    P.wq = static_cast<const uint4*>(wq);
    P.wsz = static_cast<const uint2*>(wsz);
    P.out = nullptr;
    P.M = M;
    P.N = N;
    P.K = K;
    P.T = sh.T;
    P.G = sh.G;
    P.S = sh.S;
    P.logits = logits;
    P.stats = static_cast<float2*>(stats);
    P.ld_logits = ld_logits;
    P.ld_stats = ld_stats;
    P.c = temperature > 0.f ? (float)(1.4426950408889634 / (double)temperature) : 0.f;
    switch (sh.cfg) {
        case 0: return launch_logits_cfg<W4::Cfg1w>(P, sh.P, s);
        case 1: return launch_logits_cfg<W4::Cfg1n>(P, sh.P, s);
        case 2: return launch_logits_cfg<W4::Cfg2>(P, sh.P, s);
        case 3: return launch_logits_cfg<W4::Cfg3>(P, sh.P, s);
        default: return launch_logits_cfg<W4::Cfg4>(P, sh.P, s);
    }
}

}  // namespace sd
