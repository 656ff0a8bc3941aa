// wtypes.cu -- the matvec for q4_0 and q8_0 weights (the weight types of the
// pages' other models) against q8_0 activations: the bulk-copy ring kernel
// with the FmtQ4_0 / FmtQ8_0 unit formats, same staging, reduction and
// combine as the q4_K matvec.
#include "mq_ring_kernel.cuh"

namespace mq {

template <class Fmt, int MODE>
static cudaError_t launch_wring_fmt(const void* desc, int rows, int K, int ncols, const MvPlan& p, unsigned* status,
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
    case N: return cudaLaunchKernelEx(&cfg, ring_kernel<N, KIND_MV, Fmt, (N <= 2 ? 0 : MODE)>, desc, rows, K, p, status);
        MQ_CASE(1) MQ_CASE(2) MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_wring(const void* desc, int wtype, int rows, int K, int ncols, const MvPlan& p, unsigned* status,
                         cudaStream_t s, bool pdl)
{
    if (p.variant != 1) return cudaErrorInvalidConfiguration;
    if (p.block > 32 * ring_max_warps<1>() || p.cmap) return cudaErrorInvalidConfiguration;
    const bool wide = ncols >= 3 && p.block > 32 * ring_max_warps<3>();  // 3..8 columns beyond 8 warps
    if (wtype == MQ_TYPE_Q4_0)
        return wide ? launch_wring_fmt<FmtQ4_0, 2>(desc, rows, K, ncols, p, status, s, pdl)
                    : launch_wring_fmt<FmtQ4_0, 0>(desc, rows, K, ncols, p, status, s, pdl);
    if (wtype == MQ_TYPE_Q8_0)
        return wide ? launch_wring_fmt<FmtQ8_0, 2>(desc, rows, K, ncols, p, status, s, pdl)
                    : launch_wring_fmt<FmtQ8_0, 0>(desc, rows, K, ncols, p, status, s, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t set_wring_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
#define MQ_SET1(N, F, M) \
    if (e == cudaSuccess) e = set_max_dyn_smem(reinterpret_cast<const void*>(ring_kernel<N, KIND_MV, F, M>), max_smem);
#define MQ_SET(N) MQ_SET1(N, FmtQ4_0, 0) MQ_SET1(N, FmtQ8_0, 0) MQ_SET1(N, FmtQ4_0, (N <= 2 ? 0 : 2)) \
    MQ_SET1(N, FmtQ8_0, (N <= 2 ? 0 : 2))
    MQ_SET(1) MQ_SET(2) MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
#undef MQ_SET
#undef MQ_SET1
    return e;
}

}  // namespace mq
