// launch.h -- kernel launch with programmatic dependent launch enabled.
//
// Every kernel of this library starts with griddepcontrol.wait before it
// touches global memory, so it may be scheduled while the previous kernel in
// the stream drains; this hides the launch gap between the short kernels of a
// draft step.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace wm {

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
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

}  // namespace wm
