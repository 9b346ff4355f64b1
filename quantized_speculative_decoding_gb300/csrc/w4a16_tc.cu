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
// One CTA = 8 warps = one 128-row tile of W and one K-slice, with a 4-slot
// ring of (A, B) tiles and a 12-stage ring of packed weights.  Per 64-wide K
// stage, two threads per row dequantise its 32 bytes of packed int4 (one 2D
// TMA box of 128 rows x 32 bytes per stage, issued 11 stages ahead with its own
// mbarrier) exactly in fp32 ((q - z) s with f = 1 + q/16 built by a mantissa
// insert, f * 16s - (16 + z)s in one FMA), rounds to bf16 and stores them into
// the stage's 128B-swizzled K-major A tile; the stage's x rows reach the B
// tile by cp.async, issued two stages ahead.  After a proxy fence and a CTA
// barrier one thread issues four tcgen05.mma (K = 16 each) and commits them
// to the slot's mbarrier; a slot is refilled only after the MMAs that read it
// have completed.  The epilogue reads the accumulator with tcgen05.ld.  The
// S <= 8 K splits of a tile form one thread-block cluster: each CTA stages its
// fp32 partial tile in its own shared memory, and CTA r adds the S partials of
// its share of the x rows through distributed shared memory, in rank order.
//
// Every wait on an mbarrier is bounded (about 2^31 SM cycles); on
// expiry the kernel records SD_ERR_TIMEOUT in the device error word, waits
// once more (bounded) for its in-flight MMAs, frees its TMEM and returns.
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

constexpr int kThreads = 256;  // 8 warps: two threads per weight row (one per 32-wide half of a stage)
constexpr int kStageK = 64;                  // K elements per pipeline stage
constexpr int kATileBytes = 128 * kStageK * 2;  // 16 KB
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

constexpr int kSlots = 4;     // (A, B) ring slots: A(it) goes to it % 4, x(it + 2) to (it + 2) % 4
constexpr int kWStagesMax = 12;  // packed-weight ring: 128 rows x 32 bytes per stage
constexpr int kWStageBytes = 128 * 32;

template <int MP>
struct TcCfg {
    static constexpr int kBTileBytes = MP * 128;
    static constexpr int kStageBytes = kATileBytes + kBTileBytes;  // a multiple of 1024
    static constexpr int kRingBytes = kSlots * kStageBytes;
    // a shorter weight ring for small M keeps two CTAs per SM
    static constexpr int kWS = MP <= 64 ? 6 : kWStagesMax;
    static constexpr int kSmemBytes = kRingBytes + kWS * kWStageBytes + 1024;
    static constexpr uint32_t kTmemCols = MP <= 32 ? 32 : MP <= 64 ? 64 : MP <= 128 ? 128 : 256;
};

struct TcParams {
    const __nv_bfloat16* x;
    const uint32_t* qweight;
    const __half* scales;
    const __half* zeros;
    __nv_bfloat16* out;
    int* err;
    int M, N, K, splits;  // splits = cluster size
};

constexpr int kMaxSplits = 8;  // portable cluster size

template <int MP>
__global__ void __launch_bounds__(kThreads) w4a16_tc_kernel(const __grid_constant__ CUtensorMap wmap, TcParams P) {
    using C = TcCfg<MP>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t mbar[kSlots];
    __shared__ __align__(8) uint64_t wfull[kWStagesMax];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    griddep_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5;
    const int r = tid & 127, half = tid >> 7;  // weight row within the tile, half of the stage's 64 k
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
        for (int i = 0; i < kSlots; ++i) mbar_init(&mbar[i], 1);
        for (int i = 0; i < C::kWS; ++i) mbar_init(&wfull[i], 1);
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
    const int row = min(n0 + r, N - 1);
    const int G = K / 128;
    const __half* srow = P.scales + (size_t)row * G;
    const __half* zrow = P.zeros + (size_t)row * G;
    constexpr uint32_t idesc = idesc_bf16(128, MP);

    const int nit = st1 - st0;
    const uint32_t wring = sbase + C::kRingBytes;  // [kWS stages][128 rows][32 bytes]
    // x rows of stage it -> B tile of slot it % kSlots; rows >= M are never
    // written: they only feed D columns that are not stored
    auto issue_x = [&](int it) {
        if (it >= nit) return;
        const uint32_t b_tile = sbase + (it % kSlots) * C::kStageBytes + kATileBytes;
        const int k0 = (st0 + it) * kStageK;
        for (int i = tid; i < M * 8; i += kThreads) {
            const int m = i >> 3, c = i & 7;
            cp_async16(b_tile + sw128_off(m, c), P.x + (size_t)m * K + k0 + 8 * c);
        }
    };
    // packed weights of stage it: one TMA box (128 rows x 32 bytes) into weight
    // ring slot it % kWS, issued by thread 0 (constant data: may start
    // before the dependency wait)
    auto issue_w = [&](int it) {
        if (it >= nit) return;
        uint64_t* bar = &wfull[it % C::kWS];
        mbar_expect_tx(bar, kWStageBytes);
        tma_load_2d(wring + (it % C::kWS) * kWStageBytes, &wmap, (st0 + it) * (kStageK / 2), n0, bar);
    };
    if (tid == 0)
        for (int it = 0; it < C::kWS - 1; ++it) issue_w(it);
    griddep_wait();  // x and the output may belong to the previous kernel of the stream
    issue_x(0);
    cp_async_commit();
    issue_x(1);
    cp_async_commit();
    int w_issued = C::kWS - 1 < nit ? C::kWS - 1 : nit;

    bool aborted = false;
    for (int it = 0; it < nit; ++it) {
        const int slot = it % kSlots;
        if (tid == 0) {
            // the MMAs of stage it - 2 (and so of it - 4) are done: slots
            // (it + 2) % 4 and it % 4 may be refilled; the weights of stage it
            // have landed
            const int pj = it - 2;
            if ((it >= 2 && !mbar_wait_bounded(&mbar[pj % kSlots], (pj / kSlots) & 1)) ||
                !mbar_wait_bounded(&wfull[it % C::kWS], (it / C::kWS) & 1)) {
                record_error(P.err, kDevErrTimeout);
                abort_s = 1;
            }
        }
        __syncthreads();
        if (abort_s) {
            aborted = true;
            break;
        }
        // x(it + 2) by cp.async; the weights of stage it + kWS - 1 into
        // the ring slot of stage it - 1, which every thread is done with
        issue_x(it + 2);
        cp_async_commit();
        if (tid == 0 && it + C::kWS - 1 < nit) {
            issue_w(it + C::kWS - 1);
            ++w_issued;
        }
        cp_async_wait<2>();  // this thread's x copies of stage it have landed

        const int k0 = (st0 + it) * kStageK;
        const float s = __half2float(__ldg(srow + (k0 >> 7)));
        const float z = __half2float(__ldg(zrow + (k0 >> 7)));
        const float s16 = 16.f * s, c0 = -(16.f + z) * s;
        const uint32_t a_tile = sbase + slot * C::kStageBytes;
        const uint32_t b_tile = a_tile + kATileBytes;
        const uint4 w = *reinterpret_cast<const uint4*>(smem + C::kRingBytes + (it % C::kWS) * kWStageBytes + r * 32 +
                                                      half * 16);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) st_shared_u4(a_tile + sw128_off(r, 4 * half + c), dequant_word(wv[c], s16, c0));
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kStageK / 16; ++kk)
                mma_bf16(tmem_d, desc_sw128(a_tile + 32 * kk), desc_sw128(b_tile + 32 * kk), idesc,
                         (it > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&mbar[slot]);
        }
    }
    cp_async_wait<0>();  // no copy into the ring is left in flight
    if (aborted && tid == 0) {
        // weight stages still in flight land (bounded) before the memory is reused
        for (int it = w_issued - C::kWS > 0 ? w_issued - C::kWS : 0; it < w_issued; ++it)
            mbar_wait_bounded(&wfull[it % C::kWS], (it / C::kWS) & 1);
    }

    // wait for the last commit (it covers every MMA this thread issued)
    if (nit > 0) {
        const int last = nit - 1;
        if (tid == 0 && !mbar_wait_bounded(&mbar[last % kSlots], (last / kSlots) & 1)) {
            record_error(P.err, kDevErrTimeout);
            abort_s = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    aborted = aborted || abort_s;

    // the accumulator: TMEM lane = row, column = x row m.  Warp w reads lanes
    // 32 (w % 4) .. + 31; warps 0-3 take the even 16-column chunks, 4-7 the odd
    const int erow = 32 * (warp & 3) + (tid & 31);
    const int n = n0 + erow;
    const uint32_t lane_addr = tmem_d + ((uint32_t)(32 * (warp & 3)) << 16);
    float* red = reinterpret_cast<float*>(smem);  // [MP][128] fp32, split-K only
#pragma unroll 1
    for (int c0 = 16 * (warp >> 2); c0 < MP; c0 += 32) {
        uint32_t r[16];
        tmem_ld16(lane_addr + c0, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int m = c0 + j;
            const float v = nit > 0 ? __uint_as_float(r[j]) : 0.f;
            if (P.splits == 1) {
                if (!aborted && n < N && m < M) P.out[(size_t)m * N + n] = __float2bfloat16_rn(v);
            } else {
                red[m * 128 + erow] = v;
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

    // split-K within the cluster: CTA `split` adds the partials of x rows
    // [split MP / S, (split + 1) MP / S) in rank order.  Every CTA takes part in
    // both cluster barriers, aborted or not.
    cluster_sync();
    if (!abort_s && n0 + r < N) {
        // thread (r, half): row n0 + r, every other x row of this CTA's share
        const int S = P.splits;
        const int m0 = split * MP / S, m1 = min((split + 1) * MP / S, M);
        for (int m = m0 + half; m < m1; m += 2) {
            float v = 0.f;
            for (int q = 0; q < S; ++q) v += ld_cluster_f32(sbase + (uint32_t)(m * 128 + r) * 4u, (uint32_t)q);
            P.out[(size_t)m * N + n0 + r] = __float2bfloat16_rn(v);
        }
    }
    cluster_sync();  // no CTA leaves while its shared memory may still be read
}

// One-time (per device) opt-in to the configuration's dynamic shared memory.
template <int MP>
cudaError_t prepare(int dev) {
    static std::atomic<unsigned long long> attr_set{0};  // one bit per device
    const unsigned long long bit = 1ull << (dev & 63);
    if (attr_set.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(w4a16_tc_kernel<MP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               TcCfg<MP>::kSmemBytes);
    if (e == cudaSuccess) attr_set.fetch_or(bit, std::memory_order_release);
    return e;
}

// Clusters of `sp` CTAs that the GPU holds at once (queried once per device
// and cluster size): the cluster-packing of the SMs, not just their count.
template <int MP>
int max_clusters(int dev, int sp) {
    static std::atomic<int> cache[64][kMaxSplits + 1];
    int v = cache[dev & 63][sp].load(std::memory_order_acquire);
    if (v > 0) return v;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sp);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)TcCfg<MP>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sp;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, w4a16_tc_kernel<MP>, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();  // leave no sticky error behind a failed query
        n = 1;
    }
    cache[dev & 63][sp].store(n, std::memory_order_release);
    return n;
}

// K splits per 128-row tile (= cluster size): the count that minimises
// (waves of clusters) x (stages per CTA), with at least 8 stages per split.
template <int MP>
int choose_splits(int dev, int tiles, int nst) {
    int best = 1;
    long long best_cost = -1;
    for (int sp = 1; sp <= kMaxSplits && sp <= nst / 8; ++sp) {
        const long long clusters = max_clusters<MP>(dev, sp);
        const long long cost = ((tiles + clusters - 1) / clusters) * ((nst + sp - 1) / sp);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = sp;
        }
    }
    return best;
}

template <int MP>
cudaError_t launch_mp(const CUtensorMap& wmap, TcParams P, int tiles, cudaStream_t s) {
    using C = TcCfg<MP>;
    static_assert(MP * 128 * 4 <= C::kRingBytes, "partial tile fits in the ring");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const cudaError_t e = prepare<MP>(dev);
    if (e != cudaSuccess) return e;
    P.splits = choose_splits<MP>(dev, tiles, P.K / kStageK);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * P.splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)C::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = P.splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<MP>, wmap, P);
}

}  // namespace

size_t w4a16_tc_workspace_bytes(int M, int N, int K, int sms) {
    (void)M;
    (void)N;
    (void)K;
    (void)sms;
    return 0;  // K splits meet in distributed shared memory
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
    P.splits = 1;  // chosen per configuration at launch
    (void)sms;
    const int tiles = (N + 127) / 128;
    (void)ws;
    (void)ws_bytes;
    (void)counters;
    // packed weights as a 2D uint8 tensor: K/2 bytes per row, N rows; one box =
    // 32 bytes (64 k) x 128 rows, no swizzle; rows past N read as zero
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap wmap;
    std::memset(&wmap, 0, sizeof wmap);
    const cuuint64_t gdim[2] = {(cuuint64_t)K / 2, (cuuint64_t)N};
    const cuuint64_t gstride[1] = {(cuuint64_t)K / 2};
    const cuuint32_t box[2] = {kStageK / 2, 128};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(qweight), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int mp = (M + 15) & ~15;  // at most 160 rows of x per launch
    switch (mp) {
        case 16: return launch_mp<16>(wmap, P, tiles, s);
        case 32: return launch_mp<32>(wmap, P, tiles, s);
        case 48: return launch_mp<48>(wmap, P, tiles, s);
        case 64: return launch_mp<64>(wmap, P, tiles, s);
        case 80: return launch_mp<80>(wmap, P, tiles, s);
        case 96: return launch_mp<96>(wmap, P, tiles, s);
        case 112: return launch_mp<112>(wmap, P, tiles, s);
        case 128: return launch_mp<128>(wmap, P, tiles, s);
        case 144: return launch_mp<144>(wmap, P, tiles, s);
        case 160: return launch_mp<160>(wmap, P, tiles, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sd
