// Programmatic dependent launch for the per-step kernels (decode, spec-verify, fused tail):
// back-to-back calls on one stream overlap one grid's tail with the next grid's launch.
#pragma once

#include <utility>

#include <cuda_runtime.h>

namespace kda {

// First statement of a kernel launched with launch_pdl: wait until the kernel before it in
// the stream has completed and its writes are visible (every global read comes after
// this), then let the next grid launch once every CTA of this one has started; that grid's
// own wait still orders it after this one.
__device__ __forceinline__ void pdl_wait_then_release()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` with programmatic stream serialization. After a kernel that never
// releases its dependents early, this is an ordinary stream-ordered launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args)
{
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

}  // namespace kda
