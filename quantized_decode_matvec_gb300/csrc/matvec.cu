// matvec.cu -- q4_K x q8_0 decode matvec kernels (sm_103a).
//
// MMVQ of "07 . R3 -- Small-model per-token overhead", section 1: q4_K
// weight rows times a q8_0-quantized activation with dp4a integer dot
// products and per-32-block int32 sums, fp32 scaling and row reduction.
// GB300 design: persistent grid of one CTA per SM (rows split evenly), 16-byte
// read-only streaming loads two batches ahead, activation staged in shared
// memory in a bank-conflict-free layout, deterministic segment combine.
#include "mq_stream.cuh"

namespace mq {

struct MvJob {
    const uint8_t* W;
    const float* x;
    const uint8_t* xq;
    uint8_t* xq_out;
    float* y;
    int rows, K, ncols, y_ld;
};

template <int KIND>
__device__ __forceinline__ MvJob read_job(const void* desc)
{
    MvJob j;
    if (KIND == KIND_MV) {
        const mq_mv_desc* d = static_cast<const mq_mv_desc*>(desc);
        j.W = static_cast<const uint8_t*>(d->W);
        j.x = d->x;
        j.xq = static_cast<const uint8_t*>(d->xq);
        j.xq_out = static_cast<uint8_t*>(d->xq_out);
        j.y = d->y;
        j.rows = d->rows;
        j.K = d->K;
        j.ncols = d->ncols;
        j.y_ld = d->y_ld;
    } else {  // the down projection of an FFN descriptor: y = W_down . h_q8
        const mq_ffn_desc* d = static_cast<const mq_ffn_desc*>(desc);
        j.W = static_cast<const uint8_t*>(d->W_down);
        j.x = nullptr;
        j.xq = static_cast<const uint8_t*>(d->h_q8);
        j.xq_out = nullptr;
        j.y = d->y;
        j.rows = d->H;
        j.K = d->I;
        j.ncols = d->ncols;
        j.y_ld = d->y_ld;
    }
    return j;
}

// device-side re-check of the descriptor against the launch shape; returns
// the status bits to record (0 = fine)
__device__ __forceinline__ unsigned check_job(const MvJob& j, int rows_h, int K_h, int nc)
{
    unsigned bad = 0;
    if (j.rows != rows_h || j.K != K_h || j.ncols != nc || j.y_ld < j.rows) bad |= MQ_DEV_DESC_MISMATCH;
    if ((reinterpret_cast<uintptr_t>(j.W) & 15) || (reinterpret_cast<uintptr_t>(j.y) & 3) ||
        (j.x && (reinterpret_cast<uintptr_t>(j.x) & 3)) || (!j.x && (reinterpret_cast<uintptr_t>(j.xq) & 1)) ||
        (reinterpret_cast<uintptr_t>(j.xq_out) & 1) || !j.W || !j.y || (!j.x && !j.xq))
        bad |= MQ_DEV_DESC_ALIGN;
    return bad;
}

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
                stage_x_quantize<NC>(j.x, j.K, act, blockIdx.x == 0 ? j.xq_out : nullptr);
            else
                stage_q8_global<NC>(j.xq, j.K, act, nullptr);
        });
    __syncthreads();
    griddep_launch_dependents();
    for (int t = threadIdx.x; t < NC * nrows; t += blockDim.x) {
        const int c = t / nrows, lr = t - c * nrows;
        float s = 0.0f;
        for (int g = 0; g < p.nseg; ++g) s += part[(lr * p.nseg + g) * NC + c];
        j.y[size_t(c) * j.y_ld + r0 + lr] = s;
    }
}

// Test export: the per-32-block int32 sums, through the same chunk_dot as
// the matvec kernel.  One CTA per row.
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
    const int C = j.K / kChunkElems, nq = j.K / kQK8;
    ActSmem act{smem, reinterpret_cast<float4*>(smem + size_t(NC) * 4 * C), C};
    int32_t* sq_smem = reinterpret_cast<int32_t*>(act.scales + size_t(NC) * C);
    if (j.x) {
        stage_x_quantize<NC>(j.x, j.K, act, nullptr);
        __syncthreads();
        // block sums of the codes, from the staged planes
        for (int t = threadIdx.x; t < NC * nq; t += blockDim.x) {
            const int c = t / nq, J = t - c * nq, ch = J >> 1, half = J & 1;
            const uint4 lo = act.planes[size_t(c * 4 + 2 * half) * C + ch];
            const uint4 hi = act.planes[size_t(c * 4 + 2 * half + 1) * C + ch];
            int s = 0;
            s = __dp4a(int(lo.x), 0x01010101, s);
            s = __dp4a(int(lo.y), 0x01010101, s);
            s = __dp4a(int(lo.z), 0x01010101, s);
            s = __dp4a(int(lo.w), 0x01010101, s);
            s = __dp4a(int(hi.x), 0x01010101, s);
            s = __dp4a(int(hi.y), 0x01010101, s);
            s = __dp4a(int(hi.z), 0x01010101, s);
            s = __dp4a(int(hi.w), 0x01010101, s);
            sq_smem[t] = s;
        }
    } else {
        stage_q8_global<NC>(j.xq, j.K, act, sq_smem);
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int t = threadIdx.x; t < NC * nq; t += blockDim.x) sumq[t] = sq_smem[t];
    const int r = blockIdx.x;
    const uint8_t* row = j.W + size_t(r) * (j.K / kQK) * kQ4KBytes;
    for (int ch = threadIdx.x; ch < C; ch += blockDim.x) {
        Chunk k;
        load_chunk(k, row + size_t(ch >> 2) * kQ4KBytes, ch & 3);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4* P = act.planes + size_t(c * 4) * C + ch;
            int s0, s1;
            chunk_dot(k, P[0], P[C], P[2 * C], P[3 * C], s0, s1);
            int32_t* o = sumi + (size_t(c) * j.rows + r) * nq + 2 * ch;
            o[0] = s0;
            o[1] = s1;
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
    if (e == cudaSuccess) e = cudaFuncSetAttribute(mv_kernel<N, KIND_MV>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);   \
    if (e == cudaSuccess) e = cudaFuncSetAttribute(mv_kernel<N, KIND_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem); \
    if (e == cudaSuccess) e = cudaFuncSetAttribute(block_sums_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    MQ_SET(1) MQ_SET(2) MQ_SET(3) MQ_SET(4) MQ_SET(5) MQ_SET(6) MQ_SET(7) MQ_SET(8)
#undef MQ_SET
    return e;
}

}  // namespace mq
