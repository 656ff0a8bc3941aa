// ring_cols.cu -- the q4_K ring kernels for 3..8 activation columns, all with
// 16 warps: half-unit lanes (kMode 4, 4 or 8 columns, four columns per warp
// group with their activation in registers; see ring_consume_half), column
// groups (kMode 3, two columns per warp group; see ring_consume_groups),
// column lanes (kMode 1, every column's activation in registers; see
// ring_consume_cols) or unit lanes (kMode 2), in a translation unit of their
// own.
#include "mq_ring_kernel.cuh"

namespace mq {

template <int KIND, int MODE>
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
    case N: return cudaLaunchKernelEx(&cfg, ring_kernel<N, KIND, FmtQ4K, MODE>, desc, a, b, p, status);
        MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
    }
    return cudaErrorInvalidValue;
}

// half-unit lanes: 4 or 8 columns only
template <int KIND>
static cudaError_t launch_half_kind(const void* desc, int a, int b, int ncols, const MvPlan& p, unsigned* status,
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
    if (ncols == 4) return cudaLaunchKernelEx(&cfg, ring_kernel<4, KIND, FmtQ4K, 4>, desc, a, b, p, status);
    if (ncols == 8) return cudaLaunchKernelEx(&cfg, ring_kernel<8, KIND, FmtQ4K, 4>, desc, a, b, p, status);
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_ring_cols(const void* desc, int kind, int a, int b, int ncols, const MvPlan& p, unsigned* status,
                             cudaStream_t s, bool pdl)
{
    if (ncols < 3 || p.block > 32 * ring_max_warps<3, 1>()) return cudaErrorInvalidConfiguration;
    if (p.hu) {
        switch (kind) {
            case KIND_MV: return launch_half_kind<KIND_MV>(desc, a, b, ncols, p, status, s, pdl);
            case KIND_DOWN: return launch_half_kind<KIND_DOWN>(desc, a, b, ncols, p, status, s, pdl);
            case KIND_GU: return launch_half_kind<KIND_GU>(desc, a, b, ncols, p, status, s, pdl);
        }
    } else if (p.cgw) {
        switch (kind) {
            case KIND_MV: return launch_cols_kind<KIND_MV, 3>(desc, a, b, ncols, p, status, s, pdl);
            case KIND_DOWN: return launch_cols_kind<KIND_DOWN, 3>(desc, a, b, ncols, p, status, s, pdl);
            case KIND_GU: return launch_cols_kind<KIND_GU, 3>(desc, a, b, ncols, p, status, s, pdl);
        }
    } else if (p.cmap) {
        switch (kind) {
            case KIND_MV: return launch_cols_kind<KIND_MV, 1>(desc, a, b, ncols, p, status, s, pdl);
            case KIND_DOWN: return launch_cols_kind<KIND_DOWN, 1>(desc, a, b, ncols, p, status, s, pdl);
            case KIND_GU: return launch_cols_kind<KIND_GU, 1>(desc, a, b, ncols, p, status, s, pdl);
        }
    } else {
        switch (kind) {
            case KIND_MV: return launch_cols_kind<KIND_MV, 2>(desc, a, b, ncols, p, status, s, pdl);
            case KIND_DOWN: return launch_cols_kind<KIND_DOWN, 2>(desc, a, b, ncols, p, status, s, pdl);
            case KIND_GU: return launch_cols_kind<KIND_GU, 2>(desc, a, b, ncols, p, status, s, pdl);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t set_ring_cols_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
#define MQ_SET1(N, K, M) \
    if (e == cudaSuccess) e = set_max_dyn_smem(reinterpret_cast<const void*>(ring_kernel<N, K, FmtQ4K, M>), max_smem);
#define MQ_SET(N)                                                                              \
    MQ_SET1(N, KIND_MV, 1) MQ_SET1(N, KIND_DOWN, 1) MQ_SET1(N, KIND_GU, 1) MQ_SET1(N, KIND_MV, 2) \
        MQ_SET1(N, KIND_DOWN, 2) MQ_SET1(N, KIND_GU, 2) MQ_SET1(N, KIND_MV, 3) MQ_SET1(N, KIND_DOWN, 3) \
            MQ_SET1(N, KIND_GU, 3)
    MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
    MQ_SET1(4, KIND_MV, 4) MQ_SET1(4, KIND_DOWN, 4) MQ_SET1(4, KIND_GU, 4)
    MQ_SET1(8, KIND_MV, 4) MQ_SET1(8, KIND_DOWN, 4) MQ_SET1(8, KIND_GU, 4)
#undef MQ_SET
#undef MQ_SET1
    return e;
}

}  // namespace mq
