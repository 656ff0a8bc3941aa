// mq_job.cuh -- reading and re-checking a kernel's device descriptor.
//
// Shapes and pointers live in device memory ("Part 4 . Lecture 08 --
// Graph-Resident Decode", section 2); the host passes only the shapes it sized
// the grid for, and every kernel re-checks the descriptor against them before
// touching anything.
#pragma once

#include "mq_device.cuh"
#include "mq_internal.h"

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

// device-side re-check of an FFN descriptor for the gate/up launch
__device__ __forceinline__ unsigned check_ffn_gu(const mq_ffn_desc* d, int H_h, int I_h, int nc)
{
    unsigned bad = 0;
    if (d->H != H_h || d->I != I_h || d->ncols != nc) bad |= MQ_DEV_DESC_MISMATCH;
    const uintptr_t W = reinterpret_cast<uintptr_t>(d->W_gu), hq = reinterpret_cast<uintptr_t>(d->h_q8);
    const uintptr_t x = reinterpret_cast<uintptr_t>(d->x), xq = reinterpret_cast<uintptr_t>(d->xq);
    if ((W & 15) || (hq & 1) || !W || !hq || (x && (x & 3)) || (!x && (!xq || (xq & 1))) ||
        (reinterpret_cast<uintptr_t>(d->gu_dbg) & 3) || (reinterpret_cast<uintptr_t>(d->h_dbg) & 3))
        bad |= MQ_DEV_DESC_ALIGN;
    return bad;
}

}  // namespace mq
