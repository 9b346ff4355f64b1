// Diagnostic kernel for the bounded device waits of the tensor-core kernels
// (test hook sd_test_wait_expiry): one CTA waits, with the same bounded wait
// routine the pipelines of w4a16_tc.cu use, on an mbarrier that nothing ever
// arrives on.  The wait must give up after `limit` cycles and record
// SD_ERR_TIMEOUT in the device error word; no copy or MMA is in flight, so the
// CTA exits cleanly and the context stays usable.
#include "device_common.cuh"
#include "sd_internal.h"
#include "tcgen05.cuh"

namespace sd {
namespace {

__global__ void wait_expiry_kernel(long long limit, int* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc::smem_u32(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait_bounded(&bar, 0, limit)) record_error(err, kDevErrTimeout);
}

}  // namespace

cudaError_t launch_wait_expiry(long long cycles, int* err, cudaStream_t s) {
    wait_expiry_kernel<<<1, 32, 0, s>>>(cycles, err);
    return cudaGetLastError();
}

}  // namespace sd
