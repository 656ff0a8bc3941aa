// mq_stream.cuh -- the weight-streaming loop shared by the matvec, down and
// gate/up kernels.
//
// A CTA owns a set of rows ("local rows" 0..nrows-1, mapped to matrix rows by
// a row function).  Each row is cut into nseg segments of at most S chunks; a
// (row, segment) pair is a work item, handled by L lanes of one warp, one
// chunk per lane.  Segments start on super-block boundaries (S % 4 == 0).  A warp takes 32/L items per step; steps are handed out
// round-robin over the warps.  Loads run two batches of U steps ahead of the
// arithmetic (register double-buffering), and the first batch is issued
// before the activation is staged, so the weight stream starts at once.
// Each item's partial sum goes to shared memory (part[(lr*nseg+seg)*NC+c]);
// the caller sums the segments of a row in a fixed order, so results do not
// depend on timing (no atomics).
#pragma once

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {

struct ItemCursor {
    int lr, seg;
    __device__ __forceinline__ void advance(int dq, int dr, int nseg)
    {
        seg += dr;
        lr += dq;
        if (seg >= nseg) {
            seg -= nseg;
            ++lr;
        }
    }
};

// programmatic dependent launch: wait for the preceding kernel's writes
// (a no-op when the kernel was launched without the attribute)
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int NC, int U, typename RowFn, typename StageFn>
__device__ __forceinline__ void mv_stream(const uint8_t* __restrict__ W, size_t row_bytes, RowFn rowfn,
                                          int nrows, const MvPlan& p, const ActSmem& act,
                                          float* __restrict__ part, StageFn stage)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, NW = blockDim.x >> 5;
    const int L = p.L, nseg = p.nseg, S = p.S, C = p.C;
    const int ipw = 32 / L, sub = lane / L, l = lane - sub * L;
    const int n_items = nrows * nseg;
    const int per_step = NW * ipw;
    const int nsteps = (n_items + per_step - 1) / per_step;
    const int dq = per_step / nseg, dr = per_step - dq * nseg;

    ItemCursor lc;
    {
        const int t0 = warp * ipw + sub;
        lc.lr = t0 / nseg;
        lc.seg = t0 - lc.lr * nseg;
    }
    ItemCursor cc = lc;

    auto load = [&](Chunk& k, const ItemCursor& cur) {
        const int ch = cur.seg * S + l;
        if (cur.lr < nrows && l < S && ch < C) {
            const uint8_t* sb = W + size_t(rowfn(cur.lr)) * row_bytes + size_t(ch >> 2) * kQ4KBytes;
            load_chunk(k, sb, ch & 3);
        }
    };
    auto compute = [&](const Chunk& k, const ItemCursor& cur) {
        float acc[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c] = 0.0f;
        const int ch = cur.seg * S + l;
        if (cur.lr < nrows && l < S && ch < C) chunk_accumulate<NC>(k, ch & 3, ch, act, acc);
#pragma unroll
        for (int c = 0; c < NC; ++c)
            for (int off = L >> 1; off > 0; off >>= 1) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], off);
        if (l == 0 && cur.lr < nrows) {
#pragma unroll
            for (int c = 0; c < NC; ++c) part[(cur.lr * nseg + cur.seg) * NC + c] = acc[c];
        }
    };

    Chunk A[U], B[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (u < nsteps) load(A[u], lc);
        lc.advance(dq, dr, nseg);
    }
    stage();
    __syncthreads();

    for (int s = 0; s < nsteps; s += 2 * U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (s + U + u < nsteps) load(B[u], lc);
            lc.advance(dq, dr, nseg);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (s + u < nsteps) compute(A[u], cc);
            cc.advance(dq, dr, nseg);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (s + 2 * U + u < nsteps) load(A[u], lc);
            lc.advance(dq, dr, nseg);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (s + U + u < nsteps) compute(B[u], cc);
            cc.advance(dq, dr, nseg);
        }
    }
}

}  // namespace mq
