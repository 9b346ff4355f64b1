// Device helpers shared by the sm_103a kernels of libsd.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sd {

// Error codes written into the per-device error word (values of sd_status).
constexpr int kDevErrInvalidArg = 1;
constexpr int kDevErrTimeout = 4;

__device__ __forceinline__ void record_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// bf16 pair (one 32-bit word, element k in the low half) -> two floats.
__device__ __forceinline__ float bf16lo_to_float(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_float(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Streaming 16-byte global load that does not allocate in L1 (weights are
// read exactly once per call).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of
//   (c0,c1,c2,c3) <- (hi(B*c2)^c1^k0, lo(B*c2), hi(A*c0)^c3^k1, lo(A*c0)),
// A = 0xD2511F53, B = 0xCD9E8D57, key bumped by (0x9E3779B9, 0xBB67AE85)
// after every round.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a_hi = __umulhi(0xD2511F53u, c.x);
        const uint32_t a_lo = 0xD2511F53u * c.x;
        const uint32_t b_hi = __umulhi(0xCD9E8D57u, c.z);
        const uint32_t b_lo = 0xCD9E8D57u * c.z;
        c = make_uint4(b_hi ^ c.y ^ k0, b_lo, a_hi ^ c.w ^ k1, a_lo);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Exponential variate of the race from one Philox word w:
// t = (w + 1/2) 2^-32, E = -ln(1 - t).  Each branch evaluates the form that is
// accurate there; the fp32 operands are single roundings of the exact t and
// 1 - t.
__device__ __forceinline__ float race_exponential(uint32_t w) {
    if (w < 0x80000000u) {
        const float t = fmaf((float)(w >> 8), 0x1p-24f, ((float)(w & 255u) + 0.5f) * 0x1p-32f);
        return -log1pf(-t);
    }
    const uint32_t c = ~w;  // 1 - t = (c + 1/2) 2^-32
    const float omt = fmaf((float)(c >> 8), 0x1p-24f, ((float)(c & 255u) + 0.5f) * 0x1p-32f);
    return -logf(omt);
}

}  // namespace sd
