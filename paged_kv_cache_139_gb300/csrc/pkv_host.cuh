// Host-side launch helpers shared by the CUDA translation units.
#pragma once

#include <cuda_runtime.h>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// The status word of the current device (its device address).
DeviceStatus *status_ptr();
// Streaming multiprocessors of the current device.
int sm_count();

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous grid in the stream finishes, and every kernel of this library
// calls pdl_wait() before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
inline int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) r++;
    return r;
}

}  // namespace pkv
