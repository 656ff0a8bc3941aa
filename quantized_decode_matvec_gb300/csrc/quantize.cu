// quantize.cu -- stand-alone fp32 -> q8_0 quantizer.
//
// q8_0 is the activation format of the MMVQ path ("07 . R3 --
// Small-model per-token overhead", section 1); its amax scan is a max over
// magnitudes and therefore exactly order-independent ("Part 4 . Lecture 08 --
// Graph-Resident Decode", section 8), which is why the warp-wide max below is
// bit-identical to any serial scan.  One warp per 32-value block; x is viewed
// as a flat run of ncols*K/32 blocks (K % 32 == 0, so no block straddles two
// columns).
#include "mq_stream.cuh"

namespace mq {

__global__ void __launch_bounds__(256)
    quantize_kernel(const float* __restrict__ x, uint8_t* __restrict__ xq, int64_t nblocks)
{
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t b = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblocks; b += nwarps) {
        const float v = __ldg(x + b * kQK8 + lane);
        float d;
        const int q = q8_quantize_lane(v, &d);
        uint8_t* ob = xq + b * kQ8Bytes;
        if (lane == 0) *reinterpret_cast<uint16_t*>(ob) = __half_as_ushort(__float2half_rn(d));
        ob[2 + lane] = uint8_t(int8_t(q));
    }
}

cudaError_t launch_quantize(const float* x, void* xq, int64_t nblocks, cudaStream_t s)
{
    const int per_cta = 8;  // warps (blocks) per CTA
    int64_t grid = (nblocks + per_cta - 1) / per_cta;
    if (grid > 65535) grid = 65535;
    quantize_kernel<<<unsigned(grid), 32 * per_cta, 0, s>>>(x, static_cast<uint8_t*>(xq), nblocks);
    return cudaGetLastError();
}

}  // namespace mq
