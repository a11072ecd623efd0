// pdl.cuh -- programmatic dependent launch for the kernels of a forward.
#pragma once

#include <cuda_runtime.h>

namespace ssd {

// ---- programmatic dependent launch ------------------------------------------
// The plan and the kernels of a forward are launched with programmatic stream
// serialisation (launch_after_prev): such a kernel may be scheduled while the
// stream's previous kernel still runs, once every CTA of that kernel has called
// pdl_launch_dependents or exited.  Every thread of it calls pdl_wait before its
// first global-memory access; the wait returns once the previous kernels have
// completed and their writes are visible.  Only shared-memory and TMEM set-up
// runs before it.  The plan (one CTA) calls pdl_launch_dependents at its start,
// so the forward's first kernel is resident when the plan ends; the forward's
// kernels signal by exiting (an early signal from the segment-state pre-pass let
// the next kernel's waiting CTAs sit beside it and made a long request's forward
// about 1 % slower).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_after_prev(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace ssd
