// dequant.cu -- the operands of the prefill GEMM: the resident f16 copy of a
// q4_K weight matrix ("07 . R3 -- Small-model per-token overhead", section 1:
// the prefill GEMM reads a resident f16 weight cache built once from the
// quantized weights) and the f16 copy of the fp32 activations.
//
// A weight is d*sc*q - dmin*m; both products are exact in fp64 (at most 21
// and 17 significant bits) and so is their difference for every finite f16
// d and dmin, so the value is formed in fp64 and rounded once to f16
// (round to nearest, ties to even).  The activations are rounded from fp32 to
// f16 the same way.
#include <cuda_fp16.h>

#include "mq_internal.h"

namespace mq {

// One warp per super-block (256 weights, 144 bytes): lane l writes weights
// 8l .. 8l+7, which sit in sub-block j = l/4, i.e. quant bytes 32*(j/2) +
// 8*(l%4) .. +7, low nibbles for even j, high nibbles for odd j.
__global__ void dequant_q4K_f16_kernel(const uint8_t* __restrict__ W, __half* __restrict__ out, int64_t nblocks)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t b = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblocks; b += warps) {
        const uint8_t* blk = W + b * 144;
        const int j = lane >> 2;
        // the block's scales: d, dmin (f16), then 12 bytes of 6-bit scale/min pairs
        const double d = __half2float(__ushort_as_half(uint16_t(blk[0] | (blk[1] << 8))));
        const double dmin = __half2float(__ushort_as_half(uint16_t(blk[2] | (blk[3] << 8))));
        const uint8_t* S = blk + 4;
        int sc, m;
        if (j < 4) {
            sc = S[j] & 63;
            m = S[j + 4] & 63;
        } else {
            sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4);
            m = (S[j + 4] >> 4) | ((S[j] >> 6) << 4);
        }
        const double ds = d * sc, dm = dmin * m;
        const uint8_t* qb = blk + 16 + 32 * (j >> 1) + 8 * (lane & 3);
        const int shift = (j & 1) ? 4 : 0;
        __align__(16) __half h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = __double2half(ds * double((qb[i] >> shift) & 15) - dm);
        *reinterpret_cast<uint4*>(out + b * 256 + 8 * lane) = *reinterpret_cast<const uint4*>(h);
    }
}

__global__ void f32_to_f16_kernel(const float* __restrict__ x, __half* __restrict__ y, int64_t n)
{
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) y[i] = __float2half_rn(x[i]);
}

cudaError_t launch_dequant_q4K_f16(const void* W, void* W16, int64_t nblocks, int num_sms, cudaStream_t s)
{
    const int64_t want = (nblocks + 7) / 8;  // 8 warps per CTA
    const int grid = int(want < int64_t(num_sms) * 16 ? want : int64_t(num_sms) * 16);
    dequant_q4K_f16_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(W), static_cast<__half*>(W16), nblocks);
    return cudaGetLastError();
}

cudaError_t launch_f32_to_f16(const float* x, void* y, int64_t n, int num_sms, cudaStream_t s)
{
    const int64_t want = (n + 255) / 256;
    const int grid = int(want < int64_t(num_sms) * 32 ? want : int64_t(num_sms) * 32);
    f32_to_f16_kernel<<<grid, 256, 0, s>>>(x, static_cast<__half*>(y), n);
    return cudaGetLastError();
}

}  // namespace mq
