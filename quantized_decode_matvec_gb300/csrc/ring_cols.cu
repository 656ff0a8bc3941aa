// ring_cols.cu -- the q4_K ring kernels built for column lanes (3..8
// activation columns, every column's activation in registers; see
// ring_consume_cols), in a translation unit of their own.
#include "mq_ring_kernel.cuh"

namespace mq {

template <int KIND>
static cudaError_t launch_cols_kind(const void* desc, int a, int b, int ncols, const MvPlan& p, unsigned* status,
                                    cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(p.block);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (ncols) {
#define MQ_CASE(N) \
    case N: return cudaLaunchKernelEx(&cfg, ring_kernel<N, KIND, FmtQ4K, true>, desc, a, b, p, status);
        MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_ring_cols(const void* desc, int kind, int a, int b, int ncols, const MvPlan& p, unsigned* status,
                             cudaStream_t s, bool pdl)
{
    if (ncols < 3 || p.block > 32 * ring_max_warps<3, true>()) return cudaErrorInvalidConfiguration;
    switch (kind) {
        case KIND_MV: return launch_cols_kind<KIND_MV>(desc, a, b, ncols, p, status, s, pdl);
        case KIND_DOWN: return launch_cols_kind<KIND_DOWN>(desc, a, b, ncols, p, status, s, pdl);
        case KIND_GU: return launch_cols_kind<KIND_GU>(desc, a, b, ncols, p, status, s, pdl);
    }
    return cudaErrorInvalidValue;
}

cudaError_t set_ring_cols_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
#define MQ_SET(N)                                                                                               \
    if (e == cudaSuccess)                                                                                       \
        e = set_max_dyn_smem(reinterpret_cast<const void*>(ring_kernel<N, KIND_MV, FmtQ4K, true>), max_smem);   \
    if (e == cudaSuccess)                                                                                       \
        e = set_max_dyn_smem(reinterpret_cast<const void*>(ring_kernel<N, KIND_DOWN, FmtQ4K, true>), max_smem); \
    if (e == cudaSuccess)                                                                                       \
        e = set_max_dyn_smem(reinterpret_cast<const void*>(ring_kernel<N, KIND_GU, FmtQ4K, true>), max_smem);
    MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
#undef MQ_SET
    return e;
}

}  // namespace mq
