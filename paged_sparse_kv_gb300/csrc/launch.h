// launch.h -- host-side launchers behind the libpsk C ABI (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
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

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to the device, so each call site keeps one
// `done` mask (bit d: set on device d) and the attribute is set once per
// device; device ids past 63 set it on every call.  Safe to call from several
// host threads (setting it twice is harmless).
template <typename... KArgs>
cudaError_t set_smem_limit_per_device(void (*kernel)(KArgs...), int bytes,
                                      std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
    return e;
}

}  // namespace psk
