// Tensor-core W4A16 GEMM for sm_103a (tcgen05 + TMEM): y = x . W'^T.
//
// The batched verification regime of "When Do Quantized Drafts Help
// Speculative Decoding?" (What is open: batch 8 / 16 / 32 with gamma = 4, so
// M = batch * (gamma + 1) = 40 / 80 / 160), where the W4A16 linear is a real
// dense contraction.
//
// Swap-AB: the MMA's M side is 128 weight rows (output features n), its N
// side is the M_PAD = roundup16(M) rows of x, so that D[n][m] = sum_k W'[n][k]
// x[m][k] sits in TMEM as 128 lanes x M_PAD fp32 columns.
//
// One CTA = 4 warps = one 128-row tile of W and one K-slice.  Per 64-wide K
// stage, thread t loads the 32 bytes of packed int4 of row n0 + t (prefetched
// one stage ahead in registers), dequantises them exactly in fp32 ((q - z) s
// with f = 1 + q/16 built by a mantissa insert, f * 16s - (16 + z)s in one
// FMA), rounds to bf16 and stores them into a 128B-swizzled K-major shared
// tile; the x stage goes into a second swizzled tile.  After a proxy fence
// and a CTA barrier one thread issues four tcgen05.mma (K = 16 each) and
// commits them to the stage's mbarrier; the tile is overwritten only after
// that mbarrier completes (two stages in flight).  The epilogue reads the
// accumulator with tcgen05.ld.  With split-K, each slice writes its fp32
// partial tile to a workspace and the last CTA of the tile (atomicInc
// counter, wraps back to zero) sums the slices in order and writes bf16.
//
// Every wait on an mbarrier is bounded (about 2^31 SM cycles); on
// expiry the kernel records SD_ERR_TIMEOUT in the device error word, waits
// once more (bounded) for its in-flight MMAs, frees its TMEM and returns.
#include "device_common.cuh"
#include "launch.cuh"
#include "sd_internal.h"

namespace sd {
namespace {

constexpr int kThreads = 128;
constexpr int kStageK = 64;                  // K elements per pipeline stage
constexpr int kATileBytes = 128 * kStageK * 2;  // 16 KB
constexpr long long kWaitCycles = 1ll << 31;  // bounded waits: about 1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the completion of phase `parity` (about 2^31 SM cycles,
// about 1 s); false on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_test(bar, parity)) return true;
        if (clock64() - t0 > kWaitCycles) return false;
    }
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand with 128-byte swizzle:
// start address >> 4 in bits 0-13, stride byte offset (1024 B between 8-row
// groups) >> 4 in bits 32-45, descriptor version 1 in bits 46-47, layout
// type 2 (SWIZZLE_128B) in bits 61-63.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9 = 1, 10-12 = 1), both K-major, N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int J>
__device__ __forceinline__ float nib16(uint32_t w) {
    uint32_t b;
    if constexpr (J <= 4) b = (w << (19 - 4 * J)) & 0x00780000u;
    else b = (w >> (4 * J - 19)) & 0x00780000u;
    return __uint_as_float(b | 0x3f800000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 8 nibbles of one word -> 8 exact (q - z) s values rounded to bf16.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, float s16, float c0) {
    uint4 o;
    o.x = pack_bf16x2(fmaf(nib16<0>(w), s16, c0), fmaf(nib16<1>(w), s16, c0));
    o.y = pack_bf16x2(fmaf(nib16<2>(w), s16, c0), fmaf(nib16<3>(w), s16, c0));
    o.z = pack_bf16x2(fmaf(nib16<4>(w), s16, c0), fmaf(nib16<5>(w), s16, c0));
    o.w = pack_bf16x2(fmaf(nib16<6>(w), s16, c0), fmaf(nib16<7>(w), s16, c0));
    return o;
}

// byte offset of 16-byte chunk c (0..7) of row r in a 128B-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

template <int MP>
struct TcCfg {
    static constexpr int kBTileBytes = MP * 128;
    static constexpr int kStageBytes = kATileBytes + kBTileBytes;
    static constexpr int kSmemBytes = 2 * kStageBytes + 1024;
    static constexpr uint32_t kTmemCols = MP <= 32 ? 32 : MP <= 64 ? 64 : MP <= 128 ? 128 : 256;
};

struct TcParams {
    const __nv_bfloat16* x;
    const uint32_t* qweight;
    const __half* scales;
    const __half* zeros;
    __nv_bfloat16* out;
    float* partial;      // [splits][M][N] fp32 (splits > 1)
    unsigned* counters;  // [tiles] (splits > 1)
    int* err;
    int M, N, K, splits;
};

template <int MP>
__global__ void __launch_bounds__(kThreads, 1) w4a16_tc_kernel(TcParams P) {
    using C = TcCfg<MP>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t mbar[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    griddep_launch_dependents();
    griddep_wait();  // x, the workspace and the output may be in use by the previous kernel
    const int tid = threadIdx.x, warp = tid >> 5;
    const int tile = blockIdx.x / P.splits;
    const int split = blockIdx.x - tile * P.splits;
    const int n0 = tile * 128;
    const int K = P.K, N = P.N, M = P.M;
    const int nst = K / kStageK;
    const int st0 = (int)((long long)split * nst / P.splits);
    const int st1 = (int)((long long)(split + 1) * nst / P.splits);

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);

    if (tid == 0) {
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_s)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = tmem_base_s;

    // this thread's weight row (rows past N read row N-1; results discarded)
    const int row = min(n0 + tid, N - 1);
    const uint4* wrow = reinterpret_cast<const uint4*>(P.qweight + (size_t)row * (K / 8));
    const int G = K / 128;
    const __half* srow = P.scales + (size_t)row * G;
    const __half* zrow = P.zeros + (size_t)row * G;
    constexpr uint32_t idesc = idesc_bf16(128, MP);

    uint4 wcur0 = make_uint4(0, 0, 0, 0), wcur1 = wcur0;
    if (st0 < st1) {
        wcur0 = ld_stream_u4(wrow + 2 * st0);
        wcur1 = ld_stream_u4(wrow + 2 * st0 + 1);
    }
    bool aborted = false;
    for (int st = st0; st < st1; ++st) {
        const int it = st - st0;
        const int b = it & 1;
        if (it >= 2) {
            if (tid == 0 && !mbar_wait_bounded(&mbar[b], ((it - 2) >> 1) & 1)) {
                record_error(P.err, kDevErrTimeout);
                abort_s = 1;
            }
            __syncthreads();
            if (abort_s) {
                aborted = true;
                break;
            }
        }
        // prefetch next stage's weights
        uint4 wn0 = wcur0, wn1 = wcur1;
        if (st + 1 < st1) {
            wn0 = ld_stream_u4(wrow + 2 * (st + 1));
            wn1 = ld_stream_u4(wrow + 2 * (st + 1) + 1);
        }
        const int k0 = st * kStageK;
        const float s = __half2float(__ldg(srow + (k0 >> 7)));
        const float z = __half2float(__ldg(zrow + (k0 >> 7)));
        const float s16 = 16.f * s, c0 = -(16.f + z) * s;
        const uint32_t a_tile = sbase + b * C::kStageBytes;
        const uint32_t b_tile = a_tile + kATileBytes;
        const uint32_t wv[8] = {wcur0.x, wcur0.y, wcur0.z, wcur0.w, wcur1.x, wcur1.y, wcur1.z, wcur1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) st_shared_u4(a_tile + sw128_off(tid, c), dequant_word(wv[c], s16, c0));
        // x stage: MP rows x 8 chunks of 16 bytes, rows >= M are zero
        for (int i = tid; i < MP * 8; i += kThreads) {
            const int m = i >> 3, c = i & 7;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (m < M) v = __ldg(reinterpret_cast<const uint4*>(P.x + (size_t)m * K + k0 + 8 * c));
            st_shared_u4(b_tile + sw128_off(m, c), v);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kStageK / 16; ++kk)
                mma_bf16(tmem_d, desc_sw128(a_tile + 32 * kk), desc_sw128(b_tile + 32 * kk), idesc,
                         (it > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&mbar[b]);
        }
        wcur0 = wn0;
        wcur1 = wn1;
    }

    // wait for the last commit (it covers every MMA this thread issued)
    const int nit = st1 - st0;
    if (nit > 0) {
        const int last = nit - 1;
        if (tid == 0 && !mbar_wait_bounded(&mbar[last & 1], (last >> 1) & 1)) {
            record_error(P.err, kDevErrTimeout);
            abort_s = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    aborted = aborted || abort_s;

    if (!aborted) {
        const int n = n0 + tid;
        const uint32_t lane_addr = tmem_d + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
        for (int c0 = 0; c0 < MP; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(lane_addr + c0, r);
            if (n < N) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int m = c0 + j;
                    if (m < M) {
                        const float v = nit > 0 ? __uint_as_float(r[j]) : 0.f;
                        if (P.splits == 1) P.out[(size_t)m * N + n] = __float2bfloat16_rn(v);
                        else P.partial[((size_t)split * M + m) * N + n] = v;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_d),
                     "r"(C::kTmemCols)
                     : "memory");
    }
    if (P.splits == 1) return;

    // split-K: the last slice to finish for this tile sums the partials in
    // order.  An aborted slice still arrives, so that the counter returns to
    // zero; the (then incomplete) tile has its error recorded.
    __shared__ int is_last;
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        is_last = atomicInc(&P.counters[tile], (unsigned)(P.splits - 1)) == (unsigned)(P.splits - 1);
    }
    __syncthreads();
    if (!is_last || aborted) return;
    __threadfence();
    const int n = n0 + tid;
    if (n < N) {
        for (int m = 0; m < M; ++m) {
            float v = 0.f;
            for (int sp = 0; sp < P.splits; ++sp) v += __ldcg(P.partial + ((size_t)sp * M + m) * N + n);
            P.out[(size_t)m * N + n] = __float2bfloat16_rn(v);
        }
    }
}

template <int MP>
cudaError_t launch_mp(const TcParams& P0, int tiles, cudaStream_t s) {
    using C = TcCfg<MP>;
    static unsigned long long attr_set = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&attr_set, __ATOMIC_ACQUIRE) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(w4a16_tc_kernel<MP>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&attr_set, bit, __ATOMIC_RELEASE);
    }
    return launch_pdl(w4a16_tc_kernel<MP>, dim3(tiles * P0.splits), dim3(kThreads),
                      (size_t)C::kSmemBytes, s, P0);
}

}  // namespace

int w4a16_tc_splits(int M, int N, int K, int sms) {
    const int tiles = (N + 127) / 128;
    const int nst = K / kStageK;
    int splits = (2 * sms + tiles - 1) / tiles;
    if (splits > nst / 2) splits = nst / 2;
    if (splits < 1) splits = 1;
    (void)M;
    return splits;
}

size_t w4a16_tc_workspace_bytes(int M, int N, int K, int sms) {
    const int splits = w4a16_tc_splits(M, N, K, sms);
    if (splits == 1) return 0;
    return (size_t)splits * M * N * sizeof(float);
}

cudaError_t launch_w4a16_tc(const void* x, const uint32_t* qweight, const void* scales,
                            const void* zeros, int M, int N, int K, void* out, void* ws,
                            size_t ws_bytes, unsigned* counters, int sms, int* err,
                            cudaStream_t s) {
    TcParams P;
    P.x = static_cast<const __nv_bfloat16*>(x);
    P.qweight = qweight;
    P.scales = static_cast<const __half*>(scales);
    P.zeros = static_cast<const __half*>(zeros);
    P.out = static_cast<__nv_bfloat16*>(out);
    P.err = err;
    P.M = M;
    P.N = N;
    P.K = K;
    P.splits = w4a16_tc_splits(M, N, K, sms);
    const int tiles = (N + 127) / 128;
    if (P.splits > 1) {
        if (ws_bytes < w4a16_tc_workspace_bytes(M, N, K, sms) || !counters)
            return cudaErrorInvalidValue;
        P.counters = counters;
        P.partial = static_cast<float*>(ws);
    } else {
        P.counters = nullptr;
        P.partial = nullptr;
    }
    const int mp = (M + 15) & ~15;
    switch (mp) {
        case 16: return launch_mp<16>(P, tiles, s);
        case 32: return launch_mp<32>(P, tiles, s);
        case 48: return launch_mp<48>(P, tiles, s);
        case 64: return launch_mp<64>(P, tiles, s);
        case 80: return launch_mp<80>(P, tiles, s);
        case 96: return launch_mp<96>(P, tiles, s);
        case 112: return launch_mp<112>(P, tiles, s);
        case 128: return launch_mp<128>(P, tiles, s);
        case 144: return launch_mp<144>(P, tiles, s);
        case 160: return launch_mp<160>(P, tiles, s);
        case 176: return launch_mp<176>(P, tiles, s);
        case 192: return launch_mp<192>(P, tiles, s);
        case 208: return launch_mp<208>(P, tiles, s);
        case 224: return launch_mp<224>(P, tiles, s);
        case 240: return launch_mp<240>(P, tiles, s);
        case 256: return launch_mp<256>(P, tiles, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sd
