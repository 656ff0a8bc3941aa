// ffn.cu -- gate/up matvec over the concatenated ffn_gu weight with the
// SwiGLU product and the q8_0 re-quantization of h fused into the epilogue
// (register-streaming variant; the bulk-copy ring variant is in ring.cu).
//
// "04 . 8o -- Killing the CPU stall at decode start", sections 1 and 3.1:
// gate and up weights are concatenated row-wise into ffn_gu (gate rows
// first), so one pass over ffn_gu produces both.  A CTA owns whole q8_0 blocks
// of h: 32*k consecutive intermediate indices i, i.e. gate rows i and up rows
// I+i, so SiLU(g)*u and the amax of each 32-block of h are formed in shared
// memory and h leaves the kernel already as q8_0 for the down projection.
#include "mq_epilogue.cuh"
#include "mq_job.cuh"
#include "mq_stream.cuh"

namespace mq {

template <int NC>
__global__ void __launch_bounds__(512, 1)
    gu_kernel(const mq_ffn_desc* __restrict__ d, int H_h, int I_h, MvPlan p, unsigned* status)
{
    griddep_wait();
    extern __shared__ uint4 smem[];
    const unsigned bad = check_ffn_gu(d, H_h, I_h, NC);
    if (bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, bad);
        return;
    }
    const uint8_t* W = static_cast<const uint8_t*>(d->W_gu);
    const float* x = d->x;
    const uint8_t* xq = static_cast<const uint8_t*>(d->xq);
    const int H = d->H, I = d->I;
    const int G = gridDim.x;
    const int nblk = I / kQK8;
    const int b0 = int(int64_t(blockIdx.x) * nblk / G), b1 = int(int64_t(blockIdx.x + 1) * nblk / G);
    const int i0 = b0 * kQK8, n = (b1 - b0) * kQK8;
    const int nrows = 2 * n;
    ActSmem act{smem, reinterpret_cast<float4*>(smem + size_t(NC) * 4 * p.C), p.C};
    float* part = reinterpret_cast<float*>(act.scales + size_t(NC) * p.C);
    float* vals = part + size_t(p.rows_per_cta) * p.nseg * NC;  // [NC][2n]: g then u
    const size_t row_bytes = size_t(H / kQK) * kQ4KBytes;

    mv_stream<NC, 2>(
        W, row_bytes, [=](int lr) { return lr < n ? i0 + lr : I + i0 + (lr - n); }, nrows, p, act, part, [&]() {
            if (x)
                stage_x_quantize<NC>(x, H, act, nullptr, threadIdx.x, blockDim.x);
            else
                stage_q8_global<NC>(xq, H, act, nullptr, threadIdx.x, blockDim.x);
        });
    __syncthreads();
    griddep_launch_dependents();
    gu_epilogue<NC>(part, vals, p.nseg, n, i0, I, static_cast<uint8_t*>(d->h_q8), d->gu_dbg, d->h_dbg);
}

cudaError_t launch_gu(const mq_ffn_desc* d, int H, int I, int ncols, const MvPlan& p, unsigned* status,
                      cudaStream_t s, bool pdl)
{
    if (p.variant == 1) return launch_ring(d, KIND_GU, H, I, ncols, p, status, s, pdl);
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
    case N: return cudaLaunchKernelEx(&cfg, gu_kernel<N>, d, H, I, p, status);
        MQ_CASE(1) MQ_CASE(2) MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t set_gu_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
#define MQ_SET(N) \
    if (e == cudaSuccess) e = set_max_dyn_smem(reinterpret_cast<const void*>(gu_kernel<N>), max_smem);
    MQ_SET(1) MQ_SET(2) MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
#undef MQ_SET
    return e;
}

}  // namespace mq
