// step_chained.cu -- the MQ_STEP_CHAINED form of the persistent step kernel
// (mq_step_kernel.cuh): every phase stages its input from its producer's
// output records.
#include "mq_step_kernel.cuh"

namespace mq {

cudaError_t launch_step_kernel_chained(const cudaLaunchConfig_t& cfg, const mq_layer_desc* layers, const StepPlan& sp,
                                       int ncols, unsigned* status, unsigned* ws)
{
    switch (ncols) {
#define MQ_CASE(N) \
    case N: return cudaLaunchKernelEx(&cfg, step_kernel<N, true>, layers, sp, status, ws);
        MQ_CASE(1) MQ_CASE(2) MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t set_step_chained_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
#define MQ_SET(N) \
    if (e == cudaSuccess) e = set_max_dyn_smem(reinterpret_cast<const void*>(step_kernel<N, true>), max_smem);
    MQ_SET(1) MQ_SET(2) MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
#undef MQ_SET
    return e;
}

}  // namespace mq
