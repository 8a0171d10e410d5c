// launch.cuh -- host-side kernel launch used by every launcher of the library: programmatic
// dependent launch on (the kernels wait for their predecessor with griddepcontrol.wait), an
// optional thread-block cluster along x.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace moe {

// Raises `kernel`'s dynamic shared memory limit to at least `bytes` on the current device
// (static plus dynamic shared memory above 48 KB needs it); remembered per device and kernel.
cudaError_t ensure_dynamic_smem(const void *kernel, size_t bytes);

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, int cluster_x, Args &&...args)
{
    if (smem > 0) {
        const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kernel), smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    int n = 0;
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = (unsigned)cluster_x;
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = at;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe
