// mq_epilogue.cuh -- what a CTA does after its rows are streamed: the fixed-
// order combine of the per-segment partial sums, and for the gate/up kernel
// the SwiGLU product and the q8_0 re-quantization of h.
#pragma once

#include "mq_device.cuh"

namespace mq {

// y[c][r0 + lr] = sum over segments, in segment order, of part[(lr*nseg+seg)*NC + c]
// rec (nullable): each output also as a tagged record rec[c*R + r0 + lr] (the
// value's bits and `tag` in one 8-byte store), for a reader in the same launch
// acc: y += the sum (a later part of a K split; y holds the earlier parts' sum)
template <int NC>
__device__ __forceinline__ void mv_epilogue(const float* __restrict__ part, int nseg, int nrows, int r0,
                                            float* __restrict__ y, int y_ld, int tid, int nthr,
                                            uint64_t* __restrict__ rec = nullptr, int R = 0, uint32_t tag = 0,
                                            bool acc = false)
{
    if (acc) {  // a loop of its own: the plain store below must not wait on a load of y
        for (int t = tid; t < NC * nrows; t += nthr) {
            const int c = t / nrows, lr = t - c * nrows;
            float s = 0.0f;
            for (int g = 0; g < nseg; ++g) s += part[(lr * nseg + g) * NC + c];
            y[size_t(c) * y_ld + r0 + lr] += s;
        }
        return;
    }
    for (int t = tid; t < NC * nrows; t += nthr) {
        const int c = t / nrows, lr = t - c * nrows;
        float s = 0.0f;
        for (int g = 0; g < nseg; ++g) s += part[(lr * nseg + g) * NC + c];
        y[size_t(c) * y_ld + r0 + lr] = s;
        if (rec) st_tagged(rec + size_t(c) * R + r0 + lr, __float_as_uint(s), tag);
    }
}

// Gate/up epilogue ("04 . 8o", sections 1 and 3.1: gate rows first in ffn_gu).
// Local rows 0..n-1 are gate rows i0.., rows n..2n-1 the up rows I+i0..; n is a
// multiple of 32, so the CTA owns whole q8_0 blocks of h (block indices
// b0 .. b0 + n/32 - 1 of each column).  Called by all threads of the CTA.
// Runs on threads tid = 0..nthr-1 (whole warps); `sync` is a barrier over
// exactly those threads.
//
// rec (nullable): h also as tagged records in the activation's unit layout,
// for a reader in the same launch: per column 40 * (I/128) records, record r
// carrying word r of the unit layout (code planes, then dq and dq*sumq per
// block) with `tag` in its upper half; one 8-byte store per record, so a
// reader that sees the tag sees the word with it.
template <int NC, typename SyncFn>
__device__ __forceinline__ void gu_epilogue_on(const float* __restrict__ part, float* __restrict__ vals, int nseg,
                                               int n, int i0, int I, uint8_t* __restrict__ hq,
                                               float* __restrict__ gu_dbg, float* __restrict__ h_dbg, int tid,
                                               int nthr, SyncFn sync, uint64_t* __restrict__ rec = nullptr,
                                               uint32_t tag = 0)
{
    const int nrows = 2 * n;
    const int nblk = I / kQK8, b0 = i0 / kQK8;
    for (int t = tid; t < NC * nrows; t += nthr) {
        const int c = t / nrows, lr = t - c * nrows;
        float s = 0.0f;
        for (int g = 0; g < nseg; ++g) s += part[(lr * nseg + g) * NC + c];
        vals[t] = s;
        if (gu_dbg) gu_dbg[size_t(c) * 2 * I + (lr < n ? i0 + lr : I + i0 + (lr - n))] = s;
    }
    sync();
    // h = SiLU(g) * u = g / (1 + exp(-g)) * u, then q8_0 per 32 indices
    const int lane = tid & 31, warp = tid >> 5, NW = nthr >> 5;
    const int nb = n / kQK8;
    for (int t = warp; t < NC * nb; t += NW) {
        const int c = t / nb, k = t - c * nb;
        const int i = k * kQK8 + lane;
        const float g = vals[size_t(c) * nrows + i];
        const float u = vals[size_t(c) * nrows + n + i];
        const float h = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
        float dd;
        const int q = q8_quantize_lane(h, &dd);
        const __half dh = __float2half_rn(dd);
        uint8_t* ob = hq + (size_t(c) * nblk + b0 + k) * kQ8Bytes;
        if (lane == 0) *reinterpret_cast<uint16_t*>(ob) = __half_as_ushort(dh);
        ob[2 + lane] = uint8_t(int8_t(q));
        if (h_dbg) h_dbg[size_t(c) * I + i0 + i] = h;
        if (rec) {
            // block j = unit j/4, slot j%4: codes 16k..16k+15 of the unit are plane k
            // (four words), so this block's 32 codes are planes 2*slot and 2*slot+1
            const int j = b0 + k, uh = j >> 2, slot = j & 3, Uh = I / 128;
            const uint32_t byte = uint32_t(q) & 0xffu;
            const uint32_t w = byte | (__shfl_down_sync(0xffffffffu, byte, 1) << 8) |
                               (__shfl_down_sync(0xffffffffu, byte, 2) << 16) |
                               (__shfl_down_sync(0xffffffffu, byte, 3) << 24);
            const int sq = __reduce_add_sync(0xffffffffu, q);
            if ((lane & 3) == 0)
                st_tagged(rec + ((size_t(c) * 8 + 2 * slot + (lane >> 4)) * Uh + uh) * 4 + ((lane & 15) >> 2), w, tag);
            if (lane == 0) {
                const float dq = __half2float(dh);
                uint64_t* sr = rec + size_t(NC) * 32 * Uh + (size_t(c) * Uh + uh) * 8;
                st_tagged(sr + slot, __float_as_uint(dq), tag);
                st_tagged(sr + 4 + slot, __float_as_uint(dq * float(sq)), tag);
            }
        }
    }
}

// the whole CTA
template <int NC>
__device__ __forceinline__ void gu_epilogue(const float* __restrict__ part, float* __restrict__ vals, int nseg,
                                            int n, int i0, int I, uint8_t* __restrict__ hq,
                                            float* __restrict__ gu_dbg, float* __restrict__ h_dbg)
{
    gu_epilogue_on<NC>(part, vals, nseg, n, i0, I, hq, gu_dbg, h_dbg, threadIdx.x, blockDim.x,
                       []() { __syncthreads(); });
}

}  // namespace mq
