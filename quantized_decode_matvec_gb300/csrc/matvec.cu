// matvec.cu -- q4_K x q8_0 decode matvec kernels (sm_103a).
//
// MMVQ of "07 . R3 -- Small-model per-token overhead", section 1: q4_K
// weight rows times a q8_0-quantized activation with dp4a integer dot
// products and per-32-block int32 sums, fp32 scaling and row reduction.
// GB300 design: persistent grid of one CTA per SM (rows split evenly), 16-byte
// read-only streaming loads two batches ahead, activation staged in shared
// memory in a bank-conflict-free layout, deterministic segment combine.
#include "mq_epilogue.cuh"
#include "mq_job.cuh"
#include "mq_stream.cuh"
#include "mq_unit.cuh"

namespace mq {

template <int NC, int KIND>
__global__ void __launch_bounds__(512, 1)
    mv_kernel(const void* __restrict__ desc, int rows_h, int K_h, MvPlan p, unsigned* status)
{
    griddep_wait();
    extern __shared__ uint4 smem[];
    const MvJob j = read_job<KIND>(desc);
    const unsigned bad = check_job(j, rows_h, K_h, NC);
    if (bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, bad);
        return;
    }
    const int G = gridDim.x;
    const int r0 = int(int64_t(blockIdx.x) * j.rows / G);
    const int r1 = int(int64_t(blockIdx.x + 1) * j.rows / G);
    const int nrows = r1 - r0;
    ActSmem act{smem, reinterpret_cast<float4*>(smem + size_t(NC) * 4 * p.C), p.C};
    float* part = reinterpret_cast<float*>(act.scales + size_t(NC) * p.C);
    const size_t row_bytes = size_t(j.K / kQK) * kQ4KBytes;

    mv_stream<NC, 2>(
        j.W, row_bytes, [r0](int lr) { return r0 + lr; }, nrows, p, act, part, [&]() {
            if (j.x)
                stage_x_quantize<NC>(j.x, j.K, act, blockIdx.x == 0 ? j.xq_out : nullptr, threadIdx.x, blockDim.x);
            else
                stage_q8_global<NC>(j.xq, j.K, act, nullptr, threadIdx.x, blockDim.x);
        });
    __syncthreads();
    griddep_launch_dependents();
    mv_epilogue<NC>(part, p.nseg, nrows, r0, j.y, j.y_ld, threadIdx.x, blockDim.x);
}

// Test export: the per-32-block int32 sums, through the same staging and
// unit_dot as the bulk-copy ring kernels.  One CTA per row.
template <int NC>
__global__ void __launch_bounds__(256)
    block_sums_kernel(const mq_mv_desc* __restrict__ desc, int rows_h, int K_h, int32_t* __restrict__ sumi,
                      int32_t* __restrict__ sumq, unsigned* status)
{
    griddep_wait();
    extern __shared__ uint4 smem[];
    const MvJob j = read_job<KIND_MV>(desc);
    const unsigned bad = check_job(j, rows_h, K_h, NC);
    if (bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, bad);
        return;
    }
    const int U = j.K / kUnitElems, nq = j.K / kQK8;
    UnitAct act{smem, reinterpret_cast<float4*>(smem + size_t(NC) * 8 * U), U};
    int32_t* sq_smem = reinterpret_cast<int32_t*>(act.scales + size_t(NC) * U * 2);
    if (j.x)
        stage_units_x<NC>(j.x, j.K, act, nullptr, sq_smem, threadIdx.x, blockDim.x);
    else
        stage_units_q8<NC>(j.xq, j.K, act, sq_smem, threadIdx.x, blockDim.x);
    __syncthreads();
    if (blockIdx.x == 0)
        for (int t = threadIdx.x; t < NC * nq; t += blockDim.x) sumq[t] = sq_smem[t];
    const int r = blockIdx.x;
    const uint8_t* row = j.W + size_t(r) * (j.K / kQK) * kQ4KBytes;
    for (int u = threadIdx.x; u < U; u += blockDim.x) {
        UnitW w;
        const uint8_t* sb = row + size_t(u >> 1) * kQ4KBytes;
        const uint8_t* q = sb + 16 + 64 * (u & 1);
        w.h = ldg16(sb);
        w.qa0 = ldg16(q);
        w.qb0 = ldg16(q + 16);
        w.qa1 = ldg16(q + 32);
        w.qb1 = ldg16(q + 48);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            uint4 A[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) A[k] = act.planes[size_t(c * 8 + k) * U + u];
            int sd[4];
            unit_dot(w, A, sd);
            int32_t* o = sumi + (size_t(c) * j.rows + r) * nq + 4 * u;
            o[0] = sd[0];
            o[1] = sd[1] >> 4;  // exact: multiples of 16 (high nibbles in place)
            o[2] = sd[2];
            o[3] = sd[3] >> 4;
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int KIND>
static cudaError_t launch_mv_kind(const void* desc, int rows, int K, int ncols, const MvPlan& p, unsigned* status,
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
    case N: return cudaLaunchKernelEx(&cfg, mv_kernel<N, KIND>, desc, rows, K, p, status);
        MQ_CASE(1) MQ_CASE(2) MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_mv(const void* desc, int kind, int rows, int K, int ncols, const MvPlan& p, unsigned* status,
                      cudaStream_t s, bool pdl)
{
    if (p.variant == 1 && p.ksplit > 1) {
        // K split: the parts in stream order, each after its predecessor's
        // grid-dependency wait (programmatic dependent launch), the later ones
        // adding to y
        for (int i = 0; i < p.ksplit; ++i) {
            MvPlan pi = p;
            pi.kp0 = i * p.kpn;
            pi.kacc = i > 0 ? 1 : 0;
            const cudaError_t e = launch_ring(desc, kind, rows, K, ncols, pi, status, s, i > 0 || pdl);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (p.variant == 1) return launch_ring(desc, kind, rows, K, ncols, p, status, s, pdl);
    if (kind == KIND_MV) return launch_mv_kind<KIND_MV>(desc, rows, K, ncols, p, status, s, pdl);
    return launch_mv_kind<KIND_DOWN>(desc, rows, K, ncols, p, status, s, pdl);
}

cudaError_t launch_block_sums(const mq_mv_desc* d, int rows, int K, int ncols, int32_t* sumi, int32_t* sumq,
                              int smem, unsigned* status, cudaStream_t s)
{
    switch (ncols) {
#define MQ_CASE(N)                                                                        \
    case N:                                                                               \
        block_sums_kernel<N><<<rows, 256, smem, s>>>(d, rows, K, sumi, sumq, status);     \
        return cudaGetLastError();
        MQ_CASE(1) MQ_CASE(2) MQ_CASE(3) MQ_CASE(4) MQ_CASE(5) MQ_CASE(6) MQ_CASE(7) MQ_CASE(8)
#undef MQ_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t set_mv_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
#define MQ_SET(N)                                                                                           \
    if (e == cudaSuccess) e = set_max_dyn_smem(reinterpret_cast<const void*>(mv_kernel<N, KIND_MV>), max_smem);   \
    if (e == cudaSuccess) e = set_max_dyn_smem(reinterpret_cast<const void*>(mv_kernel<N, KIND_DOWN>), max_smem); \
    if (e == cudaSuccess) e = set_max_dyn_smem(reinterpret_cast<const void*>(block_sums_kernel<N>), max_smem);
    MQ_SET(1) MQ_SET(2) MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
#undef MQ_SET
    return e;
}

}  // namespace mq
