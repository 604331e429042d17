// mq_launch.cuh -- kernel launches with programmatic stream serialization:
// the launched kernel may begin while the previous kernel on the stream
// finishes (its prologue and the loads that do not depend on that kernel
// overlap the previous kernel's last blocks); inside, grid_dep_wait()
// (mq_ptx.cuh) orders everything that does depend on it.  Environment
// variable MQ_PDL=0 turns the attribute off (plain stream order).
#pragma once

#include <cuda_runtime.h>
#include <utility>

namespace mq {

bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args &&...args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (pdl_enabled()) {
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace mq
