// launch.h -- kernel launches with programmatic dependent launch (PDL), for
// the CUDA sources of libzero.
//
// Every kernel of the library is launched with programmatic stream
// serialization allowed, and every kernel begins with pdl_enter(): it waits
// until the previous kernel in the stream has completed and its writes are
// visible (griddepcontrol.wait), then lets the next kernel of the stream begin
// launching (griddepcontrol.launch_dependents).  No global memory is read or
// written before the wait, so the stream order of the step is kept exactly;
// what overlaps is the next kernel's launch and CTA start-up with the
// previous kernel's last CTAs.  A dependent grid launches only after every
// CTA of the previous grid has started and passed pdl_enter(), so waiting
// dependents can never keep a CTA of the grid they wait for off the SMs.  A
// kernel launched without the attribute (or after a non-kernel stream
// operation) finds the wait already satisfied.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace zk {

#ifdef __CUDACC__
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace zk
