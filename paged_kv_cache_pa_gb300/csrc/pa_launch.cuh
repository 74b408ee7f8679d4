// pa_launch.cuh -- host helper: launch a kernel on a stream with programmatic
// dependent launch allowed, so its launch overlaps the tail of the previous
// kernel on the stream.  Every kernel launched this way calls
// griddepcontrol.wait (pa::pdl_wait) before it touches global memory that
// earlier work may write or read.
#pragma once

#include <cuda_runtime.h>

namespace pa {

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
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

}  // namespace pa
