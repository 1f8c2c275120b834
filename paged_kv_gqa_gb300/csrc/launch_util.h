// launch_util.h -- kernel launches with optional programmatic dependent launch (PDL).
//
// With PDL enabled (pkv_set_programmatic_launch), every launch carries the
// programmatic-stream-serialization attribute: the grid may begin launching while the
// previous kernel in the stream is still running (once that kernel has triggered, or
// finished), and each kernel of this library waits in griddepcontrol.wait before it
// reads an input, so results do not change; the launch latency overlaps the previous
// kernel instead of following it (Atlas "CUDA Kernel Engineering", "CUDA graphs": the
// launch gaps of a decode step).
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace pkv {

bool pdl_enabled();  // defined in api.cu

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
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
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// launch_kernel with the grid's blocks grouped into thread-block clusters of
// (1, cluster_y, 1) blocks.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                  unsigned cluster_y, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = cluster_y;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Whether clusters of (1, cluster_y, 1) blocks of `kern` with `smem` bytes of dynamic shared
// memory can be resident on the current device at all.
template <typename... KArgs>
bool cluster_fits(void (*kern)(KArgs...), dim3 block, size_t smem, unsigned cluster_y)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, cluster_y, 1);
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = cluster_y;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    return cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0;
}

}  // namespace pkv
