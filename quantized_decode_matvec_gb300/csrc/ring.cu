// ring.cu -- host side of the bulk-copy (TMA) ring kernels for q4_K weights
// (matvec, down, gate/up); the kernel itself is in mq_ring_kernel.cuh.
#include "mq_ring_kernel.cuh"

namespace mq {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// 3..8 columns with 16 warps (column lanes, or unit lanes beyond 8 warps), in ring_cols.cu
cudaError_t launch_ring_cols(const void* desc, int kind, int a, int b, int ncols, const MvPlan& p, unsigned* status,
                             cudaStream_t s, bool pdl);

template <int KIND>
static cudaError_t launch_ring_kind(const void* desc, int a, int b, int ncols, const MvPlan& p, unsigned* status,
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
    case N: return cudaLaunchKernelEx(&cfg, ring_kernel<N, KIND>, desc, a, b, p, status);
        MQ_CASE(1) MQ_CASE(2) MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
    }
    return cudaErrorInvalidValue;
}

// one part of a K split (matvec and down), in ring_split.cu
cudaError_t launch_ring_split(const void* desc, int kind, int a, int b, int ncols, const MvPlan& p, unsigned* status,
                              cudaStream_t s, bool pdl);

cudaError_t launch_ring(const void* desc, int kind, int a, int b, int ncols, const MvPlan& p, unsigned* status,
                        cudaStream_t s, bool pdl)
{
    if (p.kpn) return launch_ring_split(desc, kind, a, b, ncols, p, status, s, pdl);
    // 3..8 columns beyond 8 consumer warps: the 16-warp instances
    if (ncols >= 3 && (p.cmap || p.cgw || p.block > 32 * ring_max_warps<3>()))
        return launch_ring_cols(desc, kind, a, b, ncols, p, status, s, pdl);
    if (p.block > 32 * (ncols <= 2 ? ring_max_warps<1>() : ring_max_warps<3>())) return cudaErrorInvalidConfiguration;
    switch (kind) {
        case KIND_MV: return launch_ring_kind<KIND_MV>(desc, a, b, ncols, p, status, s, pdl);
        case KIND_DOWN: return launch_ring_kind<KIND_DOWN>(desc, a, b, ncols, p, status, s, pdl);
        case KIND_GU: return launch_ring_kind<KIND_GU>(desc, a, b, ncols, p, status, s, pdl);
    }
    return cudaErrorInvalidValue;
}

cudaError_t set_ring_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
#define MQ_SET(N)                                                                                               \
    if (e == cudaSuccess)                                                                                       \
        e = set_max_dyn_smem(reinterpret_cast<const void*>(ring_kernel<N, KIND_MV>), max_smem); \
    if (e == cudaSuccess)                                                                                       \
        e = set_max_dyn_smem(reinterpret_cast<const void*>(ring_kernel<N, KIND_DOWN>), max_smem); \
    if (e == cudaSuccess)                                                                                       \
        e = set_max_dyn_smem(reinterpret_cast<const void*>(ring_kernel<N, KIND_GU>), max_smem);
    MQ_SET(1) MQ_SET(2) MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
#undef MQ_SET
    return e;
}

}  // namespace mq
