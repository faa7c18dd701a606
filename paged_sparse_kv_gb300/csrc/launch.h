// launch.h -- host-side launchers behind the libpsk C ABI (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace psk {

// Launch with programmatic stream serialisation (PDL): the kernel may begin
// while its predecessor on the stream finishes; it calls pdl_wait() before
// touching global memory.  Inside a CUDA graph this becomes a programmatic
// edge.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
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

// Number of SMs on the current device (queried once per device).
int sm_count();

}  // namespace psk
