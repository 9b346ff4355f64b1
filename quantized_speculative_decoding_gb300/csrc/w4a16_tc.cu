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
// One CTA = one 128-row tile of W and one K-slice, 18 warps in three roles
// that meet only on mbarriers (no CTA barrier inside the K loop):
//   - warp 16 (one thread) is the TMA producer.  Per 64-wide K stage it loads
//     the packed weights (one 2D box of 128 rows x 32 bytes) into a 6-stage
//     ring, issued before the wait on the previous kernel (constant data),
//     and the stage's x rows (one 2D box of 64 inputs x MP rows, 128-byte
//     swizzle: the MMA's K-major B layout, rows past M zero) into the B ring.
//     x and weights run ahead independently, each gated by its own empty
//     barriers.
//   - warps 0-15 dequantise, in two groups of 8 warps that take alternate
//     stages: two threads per weight row read its 32 bytes of the stage,
//     release the weight stage, and write the exact fp32 (q - z) s
//     (f = 1 + q/16 by a mantissa insert, f * 16s - (16 + z)s in one FMA),
//     rounded to bf16, into an A slot's 128B-swizzled K-major tile; then a
//     proxy fence and an arrive on the slot's full barrier.  Scales and zero
//     points are prefetched two groups ahead.
//   - warp 17 (one thread) owns TMEM and issues four
//     tcgen05.mma.cta_group::1.kind::f16 per stage once its A and B slots are
//     full; its commits free both slots.  A final commit marks the
//     accumulator complete.
// The epilogue reads the accumulator with tcgen05.ld.  The S <= 4 K splits
// of a tile form one thread-block cluster: each CTA stages its fp32 partial
// tile in its own shared memory, and CTA r adds the S partials of its share
// of the x rows through distributed shared memory, in rank order.
//
// Every wait on an mbarrier is bounded (about 2^31 SM cycles).  On expiry
// the kernel records SD_ERR_TIMEOUT in the device error word, every role
// leaves its loop, the copies and MMAs in flight complete (bounded waits),
// TMEM is freed and the kernel returns without writing its output.
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

constexpr int kThreads = 576;  // 18 warps: 2 x 8 dequantise, 1 TMA producer, 1 MMA issuer
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

constexpr int kWStages = 6;            // packed-weight ring: 128 rows x 32 bytes per stage
constexpr int kWStageBytes = 128 * 32;
constexpr int kDequantThreads = 256;   // one dequantisation group: two threads per weight row
constexpr int kDequantGroups = 2;      // warps 0-7 take the even stages, warps 8-15 the odd ones
constexpr int kProducerWarp = 16;      // TMA for weights and x
constexpr int kMmaWarp = 17;           // TMEM owner, MMA issue

// Rings: A (dequantised weights, 16 KB a stage) and B (x rows, MP x 128
// bytes a stage) are separate, so that each is as deep as the shared memory
// allows: a slot returns only after its MMAs complete, about 1.5 us after it
// was filled.  One CTA per SM (576 threads), about 216 KB of rings, 6 A slots
// up to MP = 96.  (At MP = 48 one smaller combination, 3 A and 6 B slots in
// 108 KB, gave wrong split-K sums, cause not found; 3 A with 8 B slots and
// 6 A with 6 B slots checked exact, as does this configuration.)
template <int MP>
struct TcCfg {
    static constexpr int kBTileBytes = MP * 128;                   // MP rows x 64 bf16, 128B swizzle
    static constexpr int kASlots = MP <= 96 ? 6 : 3;
    static constexpr int kBudget = 216 * 1024 - kWStages * kWStageBytes - kASlots * kATileBytes;
    static constexpr int kBSlots = kBudget / kBTileBytes < 8 ? kBudget / kBTileBytes : 8;
    static constexpr int kABytes = kASlots * kATileBytes;          // a multiple of 1024
    static constexpr int kRingBytes = kABytes + kBSlots * kBTileBytes;
    static constexpr int kSmemBytes = kRingBytes + kWStages * kWStageBytes + 1024;
    static constexpr uint32_t kTmemCols = MP <= 32 ? 32 : MP <= 64 ? 64 : MP <= 128 ? 128 : 256;
    static_assert(kBSlots >= 3, "x ring depth");
    static_assert(kBTileBytes % 1024 == 0, "B tiles stay 1024-aligned (128B swizzle)");
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

// K splits (cluster size) at most 4, the counts the parity tests cover.
constexpr int kMaxSplits = 4;

// Bounded wait that also gives up once another role has recorded an abort.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_test(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) return false;
    }
}

template <int MP>
__global__ void __launch_bounds__(kThreads) w4a16_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                                                            const __grid_constant__ CUtensorMap xmap, TcParams P) {
    using C = TcCfg<MP>;
    constexpr int NA = C::kASlots, NB = C::kBSlots;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t wfull[kWStages], wempty[kWStages];
    __shared__ __align__(8) uint64_t afull[NA], aempty[NA], bfull[NB], bempty[NB];
    __shared__ __align__(8) uint64_t dfull;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    griddep_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x / P.splits;
    const int split = blockIdx.x - tile * P.splits;
    const int n0 = tile * 128;
    const int K = P.K, N = P.N, M = P.M;
    const int nst = K / kStageK;
    const int st0 = (int)((long long)split * nst / P.splits);
    const int nit = (int)((long long)(split + 1) * nst / P.splits) - st0;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t wring = sbase + C::kRingBytes;  // [kWStages][128 rows][32 bytes]

    if (tid == 0) {
        for (int i = 0; i < kWStages; ++i) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wempty[i], kDequantThreads);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(&afull[i], kDequantThreads);
            mbar_init(&aempty[i], 1);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(&bfull[i], 1);
            mbar_init(&bempty[i], 1);
        }
        mbar_init(&dfull, 1);
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
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
    volatile int* abort_flag = &abort_s;
    auto fail = [&]() {
        record_error(P.err, kDevErrTimeout);
        abort_s = 1;
    };

    if (warp == kProducerWarp) {
        // ---- producer: packed weights (constant: before the dependency wait),
        // then x.  x runs up to NB stages ahead (its slot is free once the
        // MMAs of stage it - NB are done), weights up to kWStages ahead (their
        // stage is free once every dequantising thread has read it); neither
        // waits for the other.
        if (lane == 0) {
            int wi = 0, xi = 0;
            for (; wi < kWStages && wi < nit; ++wi) {
                mbar_expect_tx(&wfull[wi], kWStageBytes);
                tma_load_2d(wring + wi * kWStageBytes, &wmap, (st0 + wi) * (kStageK / 2), n0, &wfull[wi]);
            }
            griddep_wait();  // x may belong to the previous kernel of the stream
            long long t0 = clock64();
            while ((xi < nit || wi < nit) && !abort_s) {
                bool progress = false;
                if (xi < nit && (xi < NB || mbar_test(&bempty[xi % NB], ((xi / NB) - 1) & 1))) {
                    const int j = xi % NB;
                    mbar_expect_tx(&bfull[j], C::kBTileBytes);
                    tma_load_2d(sbase + C::kABytes + j * C::kBTileBytes, &xmap, (st0 + xi) * kStageK, 0, &bfull[j]);
                    ++xi;
                    progress = true;
                }
                if (wi < nit && mbar_test(&wempty[wi % kWStages], ((wi / kWStages) - 1) & 1)) {
                    const int ws = wi % kWStages;
                    mbar_expect_tx(&wfull[ws], kWStageBytes);
                    tma_load_2d(wring + ws * kWStageBytes, &wmap, (st0 + wi) * (kStageK / 2), n0, &wfull[ws]);
                    ++wi;
                    progress = true;
                }
                if (progress) {
                    t0 = clock64();
                } else if (clock64() - t0 > kWaitCycles) {
                    fail();
                    break;
                }
            }
            // copies still in flight land (bounded) before the CTA may leave
            for (int it = wi - kWStages > 0 ? wi - kWStages : 0; it < wi; ++it)
                mbar_wait_bounded(&wfull[it % kWStages], (it / kWStages) & 1);
            for (int it = xi - NB > 0 ? xi - NB : 0; it < xi; ++it)
                mbar_wait_bounded(&bfull[it % NB], (it / NB) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ---- MMA issue: one thread; each stage's commits free its A and B slots
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, MP);
            int issued = 0;
            for (int it = 0; it < nit; ++it) {
                const int ja = it % NA, jb = it % NB;
                if (!wait_or_abort(&afull[ja], (it / NA) & 1, abort_flag) ||
                    !wait_or_abort(&bfull[jb], (it / NB) & 1, abort_flag)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t a_tile = sbase + ja * kATileBytes;
                const uint32_t b_tile = sbase + C::kABytes + jb * C::kBTileBytes;
#pragma unroll
                for (int kk = 0; kk < kStageK / 16; ++kk)
                    mma_bf16(tmem_d, desc_sw128(a_tile + 32 * kk), desc_sw128(b_tile + 32 * kk), idesc,
                             (it > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&aempty[ja]);
                mma_commit(&bempty[jb]);
                ++issued;
            }
            mma_commit(&dfull);  // covers every MMA issued above
            if (!mbar_wait_bounded(&dfull, 0)) fail();
            (void)issued;
        }
    } else {
        // ---- dequantisation: group grp takes the stages it = grp (mod 2), so
        // that two stages are in flight; thread (r, half) of the group writes
        // row r's 32 inputs of each of them
        const int grp = tid / kDequantThreads, t = tid % kDequantThreads;
        const int r = t & 127, half = t >> 7;
        const int row = min(n0 + r, N - 1);  // rows past N read row N - 1; results discarded
        const int G = K / 128;
        const __half* srow = P.scales + (size_t)row * G;
        const __half* zrow = P.zeros + (size_t)row * G;
        // the row's scale and zero point for the current group and the next
        // two, loaded two groups ahead so that no L2 round trip sits between a
        // stage's arrival and its dequantisation
        int gcur = (st0 * kStageK) >> 7;
        __half s_c = __ldg(srow + gcur), z_c = __ldg(zrow + gcur);
        __half s_n = __ldg(srow + min(gcur + 1, G - 1)), z_n = __ldg(zrow + min(gcur + 1, G - 1));
        __half s_f = __ldg(srow + min(gcur + 2, G - 1)), z_f = __ldg(zrow + min(gcur + 2, G - 1));
        for (int it = grp; it < nit; it += kDequantGroups) {
            const int ws = it % kWStages, j = it % NA;
            if (!wait_or_abort(&wfull[ws], (it / kWStages) & 1, abort_flag) ||
                (it >= NA && !wait_or_abort(&aempty[j], ((it / NA) - 1) & 1, abort_flag))) {
                fail();
                break;
            }
            const uint4 w = *reinterpret_cast<const uint4*>(smem + C::kRingBytes + ws * kWStageBytes + r * 32 + half * 16);
            mbar_arrive(&wempty[ws]);  // the stage's bytes are in registers
            const int g = ((st0 + it) * kStageK) >> 7;
            if (g != gcur) {  // next group: rotate, fetch the one two ahead
                gcur = g;
                s_c = s_n;
                z_c = z_n;
                s_n = s_f;
                z_n = z_f;
                s_f = __ldg(srow + min(g + 2, G - 1));
                z_f = __ldg(zrow + min(g + 2, G - 1));
            }
            const float s = __half2float(s_c);
            const float z = __half2float(z_c);
            const float s16 = 16.f * s, c0 = -(16.f + z) * s;
            const uint32_t a_tile = sbase + j * kATileBytes;
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) st_shared_u4(a_tile + sw128_off(r, 4 * half + c), dequant_word(wv[c], s16, c0));
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
            mbar_arrive(&afull[j]);
        }
    }

    griddep_wait();  // (returns at once by now) before any global write
    // every role is done issuing; the accumulator is complete once dfull has fired
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool aborted = abort_s != 0;

    // the accumulator: TMEM lane = row, column = x row m.  Warp w < 8 reads lanes
    // 32 (w % 4) .. + 31; warps 0-3 take the even 16-column chunks, 4-7 the odd
    float* red = reinterpret_cast<float*>(smem);  // [MP][128] fp32, split-K only
    if (warp < 8) {
        const int erow = 32 * (warp & 3) + lane;
        const int n = n0 + erow;
        const uint32_t lane_addr = tmem_d + ((uint32_t)(32 * (warp & 3)) << 16);
#pragma unroll 1
        for (int c0 = 16 * (warp >> 2); c0 < MP; c0 += 32) {
            uint32_t rr[16];
            tmem_ld16(lane_addr + c0, rr);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int m = c0 + jj;
                const float v = nit > 0 ? __uint_as_float(rr[jj]) : 0.f;
                if (P.splits == 1) {
                    if (!aborted && n < N && m < M) P.out[(size_t)m * N + n] = __float2bfloat16_rn(v);
                } else {
                    red[m * 128 + erow] = v;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
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
    if (!aborted) {
        const int S = P.splits;
        const int m0 = split * MP / S, m1 = min((split + 1) * MP / S, M);
        for (int i = tid; i < (m1 - m0) * 128; i += kThreads) {
            const int m = m0 + i / 128, rr = i % 128;
            if (n0 + rr >= N) continue;
            float v = 0.f;
            for (int q = 0; q < S; ++q) v += ld_cluster_f32(sbase + (uint32_t)(m * 128 + rr) * 4u, (uint32_t)q);
            P.out[(size_t)m * N + n0 + rr] = __float2bfloat16_rn(v);
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

// K splits per 128-row tile (= cluster size): the largest count (at most
// kMaxSplits, at least 8 stages per split) whose grid fits in one wave of one
// CTA per SM: the fastest measured split on the Llama-7B shapes at
// M = 40 / 80 / 160 within that limit.
template <int MP>
int choose_splits(int dev, int tiles, int nst) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
    int best = 1;
    for (int sp = 2; sp <= kMaxSplits && sp <= nst / 8; ++sp)
        if ((long long)tiles * sp <= sms) best = sp;
    return best;
}

template <int MP>
cudaError_t launch_mp(const CUtensorMap& wmap, const CUtensorMap& xmap, TcParams P, int tiles, cudaStream_t s) {
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
    return cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<MP>, wmap, xmap, P);
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
    if (mp < 16 || mp > 160) return cudaErrorInvalidValue;
    // x as a 2D bf16 tensor [M][K]: one box = 64 inputs (128 bytes) x MP rows,
    // 128-byte swizzle (the K-major SW128 layout of the MMA's B operand); rows
    // past M read as zero
    CUtensorMap xmap;
    std::memset(&xmap, 0, sizeof xmap);
    const cuuint64_t xdim[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t xstride[1] = {(cuuint64_t)K * 2};
    const cuuint32_t xbox[2] = {kStageK, (cuuint32_t)mp};
    if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), xdim, xstride, xbox, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    switch (mp) {
        case 16: return launch_mp<16>(wmap, xmap, P, tiles, s);
        case 32: return launch_mp<32>(wmap, xmap, P, tiles, s);
        case 48: return launch_mp<48>(wmap, xmap, P, tiles, s);
        case 64: return launch_mp<64>(wmap, xmap, P, tiles, s);
        case 80: return launch_mp<80>(wmap, xmap, P, tiles, s);
        case 96: return launch_mp<96>(wmap, xmap, P, tiles, s);
        case 112: return launch_mp<112>(wmap, xmap, P, tiles, s);
        case 128: return launch_mp<128>(wmap, xmap, P, tiles, s);
        case 144: return launch_mp<144>(wmap, xmap, P, tiles, s);
        default: return launch_mp<160>(wmap, xmap, P, tiles, s);
    }
}

}  // namespace sd
