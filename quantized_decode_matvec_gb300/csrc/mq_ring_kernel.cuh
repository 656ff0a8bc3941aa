// mq_ring_kernel.cuh -- the bulk-copy (TMA) ring kernel of the matvec, down and
// gate/up launches for sm_103a, templated on the weight format (q4_K; the
// matvec also for q4_0 and q8_0 weights).
//
// Same arithmetic as the register-streaming kernels (MMVQ of "07 . R3 --
// Small-model per-token overhead", section 1; the fused ffn_gu epilogue of
// "04 . 8o", sections 1 and 3.1), different data movement:
//
// * One producer warp per CTA streams the CTA's rows, tile by tile, into a
//   ring of shared-memory stages with cp.async.bulk (one elected lane, one or
//   two bulk copies per tile, completion counted on a per-stage mbarrier).
//   Bytes in flight per SM = stages x stage size, independent of registers.
// * Consumer warps are segment-stationary: warp w always handles K-segment
//   w % nseg, so each lane always works on the same half-super-block unit
//   (128 weights) of every row and keeps that unit's 128 q8_0 codes and
//   scales in registers (ncols <= 2).  A consumer reads its unit from the
//   stage with five conflict-free 16-byte shared loads, reduces over its
//   lanes, writes one partial per (row, segment) and releases the stage on
//   its "empty" mbarrier.
// * Weights are never written by any kernel, so the producer issues the
//   first ring's worth of tiles before the grid-dependency wait: under
//   programmatic dependent launch the weight stream of a kernel starts while
//   its predecessor drains ("Part 4 . Lecture 08", section 7), and every
//   thread still waits before it touches memory the predecessor wrote.
// * Every mbarrier wait is bounded in time; on a timeout the CTA records
//   MQ_DEV_TIMEOUT, stops, drains its own copies in flight and writes nothing.
#pragma once

#include "mq_epilogue.cuh"
#include "mq_job.cuh"
#include "mq_stream.cuh"
#include "mq_tma.cuh"
#include "mq_unit.cuh"
#include "mq_ring.cuh"

namespace mq {

// ring tiles a CTA issues before its dependency wait (the rest follow the
// activation); 1 or 3 measured slower for the down projection, equal elsewhere
constexpr int kEarlyTiles = 2;
// each CTA prefetches its share of the activation's lines into L2 before the wait
constexpr bool kPrefetchAct = true;

// kSplit: the instance for one part of a K split (p.kp0, p.kpn; a separate
// instance, so the whole-row kernels carry none of its code)
template <int NC, int KIND, class Fmt = FmtQ4K, int kMode = 0, bool kSplit = false>
__global__ void __launch_bounds__(32 * ring_max_warps<NC, kMode>(), 1)
    ring_kernel(const void* __restrict__ desc, int a_h, int b_h, MvPlan p, unsigned* status)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ volatile int abort_flag;

    // ---- descriptor: never written by a kernel, so it may be read before the grid-dependency wait
    const uint8_t* W;
    const float* x;
    const uint8_t* xq;
    uint8_t* xq_out = nullptr;
    float* y = nullptr;
    int y_ld = 0, K, R;  // R: rows (matvec/down) or I (gate/up)
    const mq_ffn_desc* fd = nullptr;
    unsigned bad;
    if constexpr (KIND == KIND_GU) {
        fd = static_cast<const mq_ffn_desc*>(desc);
        bad = check_ffn_gu(fd, a_h, b_h, NC);
        W = static_cast<const uint8_t*>(fd->W_gu);
        x = fd->x;
        xq = static_cast<const uint8_t*>(fd->xq);
        K = fd->H;
        R = fd->I;
    } else {
        const MvJob j = read_job<KIND>(desc);
        bad = check_job(j, a_h, b_h, NC);
        W = j.W;
        x = j.x;
        xq = j.xq;
        xq_out = j.xq_out;
        y = j.y;
        y_ld = j.y_ld;
        K = j.K;
        R = j.rows;
    }
    if (bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, bad);
        return;
    }

    // ---- this CTA's rows: local row lr maps to matrix row rowmap(lr)
    const int G = gridDim.x;
    int nrows, r0 = 0, i0 = 0, n = 0;
    if constexpr (KIND == KIND_GU) {
        const int nblk = R / kQK8;
        const int b0 = int(int64_t(blockIdx.x) * nblk / G), b1 = int(int64_t(blockIdx.x + 1) * nblk / G);
        i0 = b0 * kQK8;
        n = (b1 - b0) * kQK8;
        nrows = 2 * n;
    } else {
        r0 = int(int64_t(blockIdx.x) * R / G);
        nrows = int(int64_t(blockIdx.x + 1) * R / G) - r0;
    }
    auto rowmap = [&](int lr) -> int64_t {
        if constexpr (KIND == KIND_GU)
            return lr < n ? int64_t(i0) + lr : int64_t(R) + i0 + (lr - n);
        else
            return int64_t(r0) + lr;
    };
    const size_t row_bytes = Fmt::row_bytes(K / kUnitElems);
    // K split: this launch streams super-blocks [sb0, sb0 + nsb) of every row,
    // one bulk copy per row into tile rows of tile_row bytes
    const int sb0 = kSplit ? p.kp0 : 0;
    const size_t tile_row = kSplit ? Fmt::row_bytes(2 * p.kpn) : row_bytes;
    const size_t src_off = kSplit ? Fmt::row_bytes(2 * sb0) : 0;
    const int ntiles = (nrows + p.T - 1) / p.T;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + p.ns;
    uint8_t* ring = smem + p.off_ring;
    const UnitAct act{reinterpret_cast<uint4*>(smem + p.off_act),
                      reinterpret_cast<float4*>(smem + p.off_act + size_t(NC) * 8 * p.C * 16), p.C};
    float* part = reinterpret_cast<float*>(smem + p.off_part);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t limit_ns = uint64_t(p.wait_ms) * 1000000ull;
    // test-only fault: the producer never delivers the CTA's last tile
    const int withheld = (p.fault == FAULT_WITHHOLD_TILE) ? ntiles - 1 : -1;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < p.ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], p.nwc);
        }
        fence_barrier_init();
    }
    __syncthreads();
    griddep_launch_dependents();

    int issued = 0;  // tiles issued (producer lane 0)
    if (warp == p.nwc) {
        // ---- producer; each weight byte is read once: evict-first in L2
        const uint64_t wpolicy = l2_policy_evict_first();
        auto issue = [&](int i) {
            if (i == withheld) return;
            const int s = i % p.ns;
            const int lr0 = i * p.T, tn = min(p.T, nrows - lr0);
            mbar_arrive_expect_tx(&full[s], uint32_t(size_t(tn) * tile_row));
            uint8_t* dst = ring + size_t(s) * p.stage_bytes;
            int a = lr0;
            const int e = lr0 + tn;
            if constexpr (kSplit) {  // part of each row: one copy per row
                for (; a < e; ++a)
                    bulk_copy_g2s_evict_first(dst + size_t(a - lr0) * tile_row, W + size_t(rowmap(a)) * row_bytes + src_off,
                                              uint32_t(tile_row), &full[s], wpolicy);
            }
            while (a < e) {  // one copy per run of contiguous matrix rows (gate/up: at most two)
                int stop = e;
                if (KIND == KIND_GU && a < n && e > n) stop = n;
                bulk_copy_g2s_evict_first(dst + size_t(a - lr0) * row_bytes, W + size_t(rowmap(a)) * row_bytes,
                                          uint32_t(size_t(stop - a) * row_bytes), &full[s], wpolicy);
                a = stop;
            }
        };
        // A few tiles before the dependency wait; the rest only once the
        // consumers have staged the activation, so the activation's loads are not
        // queued behind a ring's worth of weight bytes on their way into this SM.
        if (lane == 0)
            for (; issued < ntiles && issued < kEarlyTiles && issued < p.ns; ++issued) issue(issued);
        if (kPrefetchAct && lane == 1) {  // the activation into L2 (a hint), each line by one CTA
            const char* a = x ? reinterpret_cast<const char*>(x) : reinterpret_cast<const char*>(xq);
            const size_t abytes = x ? size_t(NC) * K * 4 : size_t(NC) * (K / kQK8) * kQ8Bytes;
            for (size_t o = size_t(blockIdx.x) * 128; o < abytes; o += size_t(gridDim.x) * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a + o));
        }
        __syncwarp();
        griddep_wait();
        named_barrier_sync(2, (p.nwc + 1) * 32);  // the consumers' staging is done
        if (lane == 0) {
            for (; issued < ntiles && issued < p.ns; ++issued) issue(issued);
            for (; issued < ntiles; ++issued) {
                const int s = issued % p.ns;
                if (abort_flag || !mbar_wait_bounded(&empty[s], uint32_t(issued / p.ns - 1) & 1u, limit_ns)) {
                    abort_flag = 1;
                    break;
                }
                issue(issued);
            }
        }
    } else {
        // ---- consumers: activation first (it may come from the predecessor), then the ring
        griddep_wait();
        const int ctid = threadIdx.x, cthr = p.nwc * 32;
        if constexpr (kSplit) {
            uint8_t* const xo = (KIND == KIND_MV && blockIdx.x == 0) ? xq_out : nullptr;
            if (x)
                stage_units_x_range<NC>(x, K, sb0 * kQK, p.kpn * kQK, act, xo, ctid, cthr);
            else
                stage_q8_range<NC>(xq, K / kQK8, sb0 * (kQK / kQK8), p.kpn * (kQK / kQK8), act, ctid, cthr);
        } else {
            if (x)
                stage_units_x<NC>(x, K, act, (KIND == KIND_MV && blockIdx.x == 0) ? xq_out : nullptr, nullptr, ctid,
                                  cthr);
            else
                stage_units_q8<NC>(xq, K, act, nullptr, ctid, cthr);
        }
        named_barrier_sync(1, cthr);
        named_barrier_arrive(2, cthr + 32);  // release the producer's remaining ring tiles
        if (!ring_consume<NC, Fmt, kMode>(p, nrows, 0, p.nwc, ring, full, empty, act, part, limit_ns) && lane == 0)
            abort_flag = 1;
    }
    __syncthreads();
    if (abort_flag) {
        if (threadIdx.x == 0) atomicOr(status, MQ_DEV_TIMEOUT);
        if (warp == p.nwc && lane == 0)  // drain this CTA's copies that may still be in flight
            for (int t = issued > p.ns ? issued - p.ns : 0; t < issued; ++t)
                if (t != withheld) (void)mbar_wait_bounded(&full[t % p.ns], uint32_t(t / p.ns) & 1u, limit_ns);
        return;
    }
    if constexpr (KIND == KIND_GU) {
        float* vals = reinterpret_cast<float*>(smem + p.off_vals);
        gu_epilogue<NC>(part, vals, p.nseg, n, i0, R, static_cast<uint8_t*>(fd->h_q8), fd->gu_dbg, fd->h_dbg);
    } else {
        if constexpr (kSplit)
            mv_epilogue<NC>(part, p.nseg, nrows, r0, y, y_ld, threadIdx.x, blockDim.x, nullptr, 0, 0, p.kacc != 0);
        else
            mv_epilogue<NC>(part, p.nseg, nrows, r0, y, y_ld, threadIdx.x, blockDim.x);
    }
}

}  // namespace mq
