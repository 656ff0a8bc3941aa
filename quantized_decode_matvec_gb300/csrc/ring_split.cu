// ring_split.cu -- the ring kernel instances for one part of a K split (matvec
// and down projections whose whole activation does not fit beside a ring):
// each streams a range of whole super-blocks of every row, stages only that
// part of the activation and, after the first part, adds its sums to y.
#include "mq_ring_kernel.cuh"

namespace mq {

template <int KIND, int MODE>
static cudaError_t launch_split_kind(const void* desc, int a, int b, int ncols, const MvPlan& p, unsigned* status,
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
    if constexpr (MODE == 0) {
        switch (ncols) {
            case 1: return cudaLaunchKernelEx(&cfg, ring_kernel<1, KIND, FmtQ4K, 0, true>, desc, a, b, p, status);
            case 2: return cudaLaunchKernelEx(&cfg, ring_kernel<2, KIND, FmtQ4K, 0, true>, desc, a, b, p, status);
        }
    } else {
        switch (ncols) {
#define MQ_CASE(N) \
    case N: return cudaLaunchKernelEx(&cfg, ring_kernel<N, KIND, FmtQ4K, MODE, true>, desc, a, b, p, status);
            MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
        }
    }
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_ring_split(const void* desc, int kind, int a, int b, int ncols, const MvPlan& p, unsigned* status,
                              cudaStream_t s, bool pdl)
{
    if (kind != KIND_MV && kind != KIND_DOWN) return cudaErrorInvalidValue;
    const bool mv = kind == KIND_MV;
    if (ncols <= 2) {
        if (p.block > 32 * ring_max_warps<1>()) return cudaErrorInvalidConfiguration;
        return mv ? launch_split_kind<KIND_MV, 0>(desc, a, b, ncols, p, status, s, pdl)
                  : launch_split_kind<KIND_DOWN, 0>(desc, a, b, ncols, p, status, s, pdl);
    }
    // 3..8 columns: the 16-warp instances (column groups, column lanes or unit lanes)
    if (p.block > 32 * ring_max_warps<3, 1>()) return cudaErrorInvalidConfiguration;
    if (p.hu) {
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
        if (ncols == 4)
            return mv ? cudaLaunchKernelEx(&cfg, ring_kernel<4, KIND_MV, FmtQ4K, 4, true>, desc, a, b, p, status)
                      : cudaLaunchKernelEx(&cfg, ring_kernel<4, KIND_DOWN, FmtQ4K, 4, true>, desc, a, b, p, status);
        if (ncols == 8)
            return mv ? cudaLaunchKernelEx(&cfg, ring_kernel<8, KIND_MV, FmtQ4K, 4, true>, desc, a, b, p, status)
                      : cudaLaunchKernelEx(&cfg, ring_kernel<8, KIND_DOWN, FmtQ4K, 4, true>, desc, a, b, p, status);
        return cudaErrorInvalidConfiguration;
    }
    if (p.cgw)
        return mv ? launch_split_kind<KIND_MV, 3>(desc, a, b, ncols, p, status, s, pdl)
                  : launch_split_kind<KIND_DOWN, 3>(desc, a, b, ncols, p, status, s, pdl);
    if (p.cmap)
        return mv ? launch_split_kind<KIND_MV, 1>(desc, a, b, ncols, p, status, s, pdl)
                  : launch_split_kind<KIND_DOWN, 1>(desc, a, b, ncols, p, status, s, pdl);
    return mv ? launch_split_kind<KIND_MV, 2>(desc, a, b, ncols, p, status, s, pdl)
              : launch_split_kind<KIND_DOWN, 2>(desc, a, b, ncols, p, status, s, pdl);
}

cudaError_t set_ring_split_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
#define MQ_SET1(N, K, M)  \
    if (e == cudaSuccess) \
        e = set_max_dyn_smem(reinterpret_cast<const void*>(ring_kernel<N, K, FmtQ4K, M, true>), max_smem);
    MQ_SET1(1, KIND_MV, 0) MQ_SET1(1, KIND_DOWN, 0) MQ_SET1(2, KIND_MV, 0) MQ_SET1(2, KIND_DOWN, 0)
#define MQ_SET(N)                                                                                       \
    MQ_SET1(N, KIND_MV, 1) MQ_SET1(N, KIND_DOWN, 1) MQ_SET1(N, KIND_MV, 2) MQ_SET1(N, KIND_DOWN, 2) \
        MQ_SET1(N, KIND_MV, 3) MQ_SET1(N, KIND_DOWN, 3)
    MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
    MQ_SET1(4, KIND_MV, 4) MQ_SET1(4, KIND_DOWN, 4) MQ_SET1(8, KIND_MV, 4) MQ_SET1(8, KIND_DOWN, 4)
#undef MQ_SET
#undef MQ_SET1
    return e;
}

}  // namespace mq
