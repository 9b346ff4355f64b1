// Kernel launch with programmatic dependent launch (PDL) allowed.
//
// A kernel launched this way may start while the previous kernel on the
// stream is still finishing.  Every kernel of libsd.so therefore follows two
// rules: it calls griddep_launch_dependents() early (so that the next kernel
// may be scheduled as soon as SMs free up), and it calls griddep_wait()
// before it reads anything an earlier kernel may have written (activations,
// logits, workspaces) and before it writes anything (outputs, workspaces).
// Constant inputs (packed weights, scales, zeros) may be read before the
// wait, which is what lets a linear layer stream its weights while the
// previous layer drains.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace sd {

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace sd
