// fused.cu -- fused dequant-in-GEMM (in progress).
#include "mq_internal.h"

namespace mq {

cudaError_t launch_gemm_fused(const CUtensorMap &, const GemmArgs &, const GemmPlan &, cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace mq
