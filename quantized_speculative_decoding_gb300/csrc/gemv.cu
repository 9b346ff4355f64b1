// CUDA-core weight-only GEMV for small M (M <= 8): y = x . W'^T.
//
// The decode-time linear layers of "When Do Quantized Drafts Help Speculative
// Decoding?" (pilot setup: draft at M = 1; target verification at
// M = batch * (gamma + 1) = 5) in the three draft precisions it compares:
// GPTQ INT4 (group 128, fp16 scale and zero), GPTQ INT8 (per-channel fp16
// scale) and BF16.
//
// Mapping: a warp owns R consecutive weight rows and a slice of K; each lane
// streams one 16-byte weight chunk per row per step (32 lanes = 512 contiguous
// bytes of a row, coalesced, no L1 allocation), double-buffered so that 2R
// loads are in flight per lane.  x is staged in shared memory one K segment at
// a time (at most 32 KB, XOR-swizzled so that the lanes' 16-byte reads are
// conflict-free) and shared by every warp of the CTA.  INT4 is dequantised
// exactly in fp32: with f = 1 + q/16 built by a
// mantissa insert, (q - z) s = f * 16s - (16 + z) s in one FMA with exact
// operands.  Accumulation is fp32; the K-slices of a row are combined by warp
// shuffles and then across warps in shared memory; the output is rounded to
// bf16 (nearest even).
#include "device_common.cuh"
#include "launch.cuh"
#include "sd_internal.h"

namespace sd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// elements per 16-byte weight chunk
template <int FMT> struct Fmt;
template <> struct Fmt<0> { static constexpr int kElems = 32; };  // uint4 nibbles
template <> struct Fmt<1> { static constexpr int kElems = 16; };  // int8
template <> struct Fmt<2> { static constexpr int kElems = 8; };   // bf16

// f = 1 + q/16 for nibble j of w (q placed in mantissa bits 19..22).
template <int J>
__device__ __forceinline__ float nibble_plus16(uint32_t w) {
    uint32_t b;
    if constexpr (J <= 4) b = (w << (19 - 4 * J)) & 0x00780000u;
    else b = (w >> (4 * J - 19)) & 0x00780000u;
    return __uint_as_float(b | 0x3f800000u);
}

// signed byte j of w as an exact float: (byte ^ 0x80) + 2^23 + ... - (2^23 + 128)
template <int J>
__device__ __forceinline__ float sbyte_to_float(uint32_t w) {
    return __uint_as_float(((w >> (8 * J)) & 0xffu) ^ 0x4b000080u) - 8388736.0f;
}

// x staged in shared memory, one K segment at a time.  Within a segment the
// 16-byte piece p of 32-element chunk c of row m sits at piece position
// p ^ ((c >> 1) & 3): the 8 lanes of a quarter-warp (consecutive c, same p)
// then hit 8 distinct 16-byte bank groups.
template <int M>
__device__ __forceinline__ void load_x8_smem(const uint4* __restrict__ xs, int seg_chunks32,
                                             int c32, int p, float (&xf)[M][8]) {
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 v = xs[((size_t)m * seg_chunks32 + c32) * 4 + (p ^ ((c32 >> 1) & 3))];
        xf[m][0] = bf16lo_to_float(v.x); xf[m][1] = bf16hi_to_float(v.x);
        xf[m][2] = bf16lo_to_float(v.y); xf[m][3] = bf16hi_to_float(v.y);
        xf[m][4] = bf16lo_to_float(v.z); xf[m][5] = bf16hi_to_float(v.z);
        xf[m][6] = bf16lo_to_float(v.w); xf[m][7] = bf16hi_to_float(v.w);
    }
}

template <int M, int R>
__device__ __forceinline__ void fma8(float (&acc)[R][M], int r, const float (&xf)[M][8],
                                     const float (&wd)[8]) {
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[r][m] = fmaf(xf[m][j], wd[j], acc[r][m]);
}

// K elements per x segment held in shared memory (M * kSegK * 2 bytes <= 32 KB)
template <int M>
struct Seg {
    static constexpr int kSegK = M == 1 ? 16384 : M == 2 ? 8192 : M <= 4 ? 4096 : 2048;
};

template <int FMT, int M, int R>
__global__ void __launch_bounds__(kThreads)
gemv_kernel(const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ w,
            const __half* __restrict__ scales, const __half* __restrict__ zeros, int N, int K,
            int ks, __nv_bfloat16* __restrict__ out) {
    constexpr int E = Fmt<FMT>::kElems;
    constexpr int SEGK = Seg<M>::kSegK;
    __shared__ uint4 xs[M * SEGK / 8];
    // programmatic dependent launch: let the next kernel be scheduled, then
    // wait for the previous one before touching global memory
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = warp / ks, split = warp - rg * ks;
    const int n0 = (blockIdx.x * (kWarps / ks) + rg) * R;
    const size_t row_bytes = (size_t)(K / E) * 16;
    const int G = K / 128;

    float acc[R][M];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

    const uint8_t* wrow[R];
#pragma unroll
    for (int r = 0; r < R; ++r) wrow[r] = w + (size_t)min(n0 + r, N - 1) * row_bytes;

    for (int seg0 = 0; seg0 < K; seg0 += SEGK) {
        const int segk = min(SEGK, K - seg0);  // multiple of 8 (K % 8 == 0)
        const int seg32 = (segk + 31) >> 5;      // 32-element chunks (last may be partial)
        // stage x[:, seg0 : seg0 + segk] (16-byte pieces; pieces past segk are not read)
        __syncthreads();
        for (int i = threadIdx.x; i < M * seg32 * 4; i += kThreads) {
            const int m = i / (seg32 * 4);
            const int rem = i - m * seg32 * 4;
            const int c32 = rem >> 2, p = rem & 3;
            const int k = c32 * 32 + p * 8;
            if (k < segk)
                xs[((size_t)m * seg32 + c32) * 4 + (p ^ ((c32 >> 1) & 3))] =
                    __ldg(reinterpret_cast<const uint4*>(x + (size_t)m * K + seg0 + k));
        }
        __syncthreads();
        if (n0 < N) {
            const int nch = segk / E;          // weight chunks in this segment
            const int cbase = seg0 / E;
            const int step = 32 * ks;
            int c = split * 32 + lane;
            uint4 cur[R], nxt[R];
            if (c < nch) {
#pragma unroll
                for (int r = 0; r < R; ++r) cur[r] = ld_stream_u4(wrow[r] + (size_t)(cbase + c) * 16);
            }
            while (c < nch) {
                const int cn = c + step;
                if (cn < nch) {
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        nxt[r] = ld_stream_u4(wrow[r] + (size_t)(cbase + cn) * 16);
                }
                const int kl = c * E;  // segment-relative first k of this chunk
                if constexpr (FMT == 0) {
                    float s16[R], c0[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int n = min(n0 + r, N - 1);
                        const int g = (seg0 + kl) >> 7;
                        const float sc = __half2float(__ldg(scales + (size_t)n * G + g));
                        const float z = __half2float(__ldg(zeros + (size_t)n * G + g));
                        s16[r] = 16.f * sc;
                        c0[r] = -(16.f + z) * sc;
                    }
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        float xf[M][8];
                        load_x8_smem<M>(xs, seg32, kl >> 5, p, xf);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t wv = p == 0 ? cur[r].x : p == 1 ? cur[r].y : p == 2 ? cur[r].z : cur[r].w;
                            float wd[8];
                            wd[0] = fmaf(nibble_plus16<0>(wv), s16[r], c0[r]);
                            wd[1] = fmaf(nibble_plus16<1>(wv), s16[r], c0[r]);
                            wd[2] = fmaf(nibble_plus16<2>(wv), s16[r], c0[r]);
                            wd[3] = fmaf(nibble_plus16<3>(wv), s16[r], c0[r]);
                            wd[4] = fmaf(nibble_plus16<4>(wv), s16[r], c0[r]);
                            wd[5] = fmaf(nibble_plus16<5>(wv), s16[r], c0[r]);
                            wd[6] = fmaf(nibble_plus16<6>(wv), s16[r], c0[r]);
                            wd[7] = fmaf(nibble_plus16<7>(wv), s16[r], c0[r]);
                            fma8<M, R>(acc, r, xf, wd);
                        }
                    }
                } else if constexpr (FMT == 1) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // 16-element chunk = half of a 32-element x chunk
                        float xf[M][8];
                        load_x8_smem<M>(xs, seg32, kl >> 5, ((kl >> 3) & 3) + h, xf);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t a = h == 0 ? cur[r].x : cur[r].z;
                            const uint32_t b = h == 0 ? cur[r].y : cur[r].w;
                            float wd[8];
                            wd[0] = sbyte_to_float<0>(a); wd[1] = sbyte_to_float<1>(a);
                            wd[2] = sbyte_to_float<2>(a); wd[3] = sbyte_to_float<3>(a);
                            wd[4] = sbyte_to_float<0>(b); wd[5] = sbyte_to_float<1>(b);
                            wd[6] = sbyte_to_float<2>(b); wd[7] = sbyte_to_float<3>(b);
                            fma8<M, R>(acc, r, xf, wd);
                        }
                    }
                } else {
                    float xf[M][8];
                    load_x8_smem<M>(xs, seg32, kl >> 5, (kl >> 3) & 3, xf);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float wd[8];
                        wd[0] = bf16lo_to_float(cur[r].x); wd[1] = bf16hi_to_float(cur[r].x);
                        wd[2] = bf16lo_to_float(cur[r].y); wd[3] = bf16hi_to_float(cur[r].y);
                        wd[4] = bf16lo_to_float(cur[r].z); wd[5] = bf16hi_to_float(cur[r].z);
                        wd[6] = bf16lo_to_float(cur[r].w); wd[7] = bf16hi_to_float(cur[r].w);
                        fma8<M, R>(acc, r, xf, wd);
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r) cur[r] = nxt[r];
                c = cn;
            }
        }
    }

    // reduce over the lanes of the warp, then over the ks warps of a row group
    __shared__ float red[kWarps][R * M];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float v = acc[r][m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[warp][r * M + m] = v;
        }
    __syncthreads();
    if (split == 0 && lane < R * M) {
        const int r = lane / M, m = lane - r * M;
        const int n = n0 + r;
        if (n < N) {
            float v = 0.f;
            for (int s = 0; s < ks; ++s) v += red[rg * ks + s][lane];
            if constexpr (FMT == 1) v *= __half2float(scales[n]);
            out[(size_t)m * N + n] = __float2bfloat16_rn(v);
        }
    }
}

template <int FMT, int M>
cudaError_t launch_m(const void* x, const void* w, const void* scales, const void* zeros, int N,
                     int K, void* out, cudaStream_t s) {
    constexpr int R = M <= 2 ? 4 : 2;
    const int nchunks = K / Fmt<FMT>::kElems;
    int dev = 0;
    cudaGetDevice(&dev);
    const int target = 2 * num_sms(dev);
    int ks = 1;
    while (ks < kWarps) {
        const int rows_per_cta = (kWarps / ks) * R;
        const int ctas = (N + rows_per_cta - 1) / rows_per_cta;
        if (ctas >= target || nchunks < 64 * ks) break;
        ks *= 2;
    }
    const int rows_per_cta = (kWarps / ks) * R;
    const int grid = (N + rows_per_cta - 1) / rows_per_cta;
    return launch_pdl(gemv_kernel<FMT, M, R>, dim3(grid), dim3(kThreads), 0, s,
                      static_cast<const __nv_bfloat16*>(x), static_cast<const uint8_t*>(w),
                      static_cast<const __half*>(scales), static_cast<const __half*>(zeros), N, K,
                      ks, static_cast<__nv_bfloat16*>(out));
}

template <int FMT>
cudaError_t launch_fmt(const void* x, const void* w, const void* scales, const void* zeros, int M,
                       int N, int K, void* out, cudaStream_t s) {
    switch (M) {
        case 1: return launch_m<FMT, 1>(x, w, scales, zeros, N, K, out, s);
        case 2: return launch_m<FMT, 2>(x, w, scales, zeros, N, K, out, s);
        case 3: return launch_m<FMT, 3>(x, w, scales, zeros, N, K, out, s);
        case 4: return launch_m<FMT, 4>(x, w, scales, zeros, N, K, out, s);
        case 5: return launch_m<FMT, 5>(x, w, scales, zeros, N, K, out, s);
        case 6: return launch_m<FMT, 6>(x, w, scales, zeros, N, K, out, s);
        case 7: return launch_m<FMT, 7>(x, w, scales, zeros, N, K, out, s);
        case 8: return launch_m<FMT, 8>(x, w, scales, zeros, N, K, out, s);
        default: return cudaErrorInvalidValue;
    }
}

__global__ void w4_unpack_kernel(const uint32_t* __restrict__ qweight, size_t words,
                                 uint8_t* __restrict__ q) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < words;
         i += (size_t)gridDim.x * blockDim.x) {
        const uint32_t v = qweight[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) q[i * 8 + j] = (uint8_t)((v >> (4 * j)) & 0xfu);
    }
}

__global__ void philox_kernel(const uint4* __restrict__ ctr, uint32_t k0, uint32_t k1, int n,
                              uint4* __restrict__ out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = philox4x32_10(ctr[i], k0, k1);
}

}  // namespace

cudaError_t launch_gemv(int fmt, const void* x, const void* w, const void* scales,
                        const void* zeros, int M, int N, int K, void* out, cudaStream_t s) {
    // M > 8 runs as consecutive blocks of at most 8 rows of x and y.
    const size_t xb = (size_t)K * 2, yb = (size_t)N * 2;
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mb = M - m0 < 8 ? M - m0 : 8;
        const void* xm = static_cast<const char*>(x) + (size_t)m0 * xb;
        void* ym = static_cast<char*>(out) + (size_t)m0 * yb;
        cudaError_t e;
        if (fmt == 0) e = launch_fmt<0>(xm, w, scales, zeros, mb, N, K, ym, s);
        else if (fmt == 1) e = launch_fmt<1>(xm, w, scales, zeros, mb, N, K, ym, s);
        else e = launch_fmt<2>(xm, w, scales, zeros, mb, N, K, ym, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_w4_unpack(const uint32_t* qweight, int N, int K, uint8_t* q, cudaStream_t s) {
    const size_t words = (size_t)N * (K / 8);
    int dev = 0;
    cudaGetDevice(&dev);
    size_t blocks = (words + 255) / 256;
    const size_t cap = (size_t)num_sms(dev) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    w4_unpack_kernel<<<(unsigned)blocks, 256, 0, s>>>(qweight, words, q);
    return cudaGetLastError();
}

cudaError_t launch_philox(const uint32_t* ctr, uint32_t k0, uint32_t k1, int n, uint32_t* out,
                          cudaStream_t s) {
    philox_kernel<<<(n + 255) / 256, 256, 0, s>>>(reinterpret_cast<const uint4*>(ctr), k0, k1, n,
                                                   reinterpret_cast<uint4*>(out));
    return cudaGetLastError();
}

}  // namespace sd
