// step.cu -- launches of the persistent step kernel (mq_step_kernel.cuh) in its
// default form; step_chained.cu holds the MQ_STEP_CHAINED form, compiled on
// its own so the two build in parallel.
#include "mq_step_kernel.cuh"

namespace mq {

cudaError_t launch_step_kernel_chained(const cudaLaunchConfig_t& cfg, const mq_layer_desc* layers, const StepPlan& sp,
                                       int ncols, unsigned* status, unsigned* ws);
cudaError_t set_step_chained_attributes(int max_smem);

cudaError_t launch_step(const mq_layer_desc* layers, const StepPlan& sp, int ncols, unsigned* status, unsigned* ws,
                        cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(ws, 0, sp.ws_bytes, s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sp.grid);
    cfg.blockDim = dim3(32 * (sp.nwc + 1));
    cfg.dynamicSmemBytes = sp.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident at once: the phase waits need it
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (sp.chained) return launch_step_kernel_chained(cfg, layers, sp, ncols, status, ws);
    switch (ncols) {
#define MQ_CASE(N) \
    case N: return cudaLaunchKernelEx(&cfg, step_kernel<N, false>, layers, sp, status, ws);
        MQ_CASE(1) MQ_CASE(2) MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t set_step_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
#define MQ_SET(N) \
    if (e == cudaSuccess) e = set_max_dyn_smem(reinterpret_cast<const void*>(step_kernel<N, false>), max_smem);
    MQ_SET(1) MQ_SET(2) MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
#undef MQ_SET
    if (e == cudaSuccess) e = set_step_chained_attributes(max_smem);
    return e;
}

}  // namespace mq
