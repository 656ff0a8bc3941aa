// mq_step_kernel.cuh -- the whole decode step of a layer stack as one persistent
// kernel (device code; step.cu and step_chained.cu instantiate and launch it).
//
// "Part 4 . Lecture 08 -- Graph-Resident Decode" captures a decode step as one
// graph (section 1) and names a single resident kernel as the endpoint of
// that road; PDL (section 7) attacks the device-side gap between kernels.
// Here that gap is removed outright: one cooperative CTA per SM runs every
// matrix of every layer (phases qkv, o, ffn_gu + SiLU*mul + q8_0(h), down, in
// that order), and
//
// * the producer warp streams the CTA's rows of all phases, back to back,
//   through one bulk-copy ring, so the weights of phase p+1 are already in
//   shared memory while phase p finishes: weights are never written by any
//   kernel, so fetching them early is always correct;
// * consumers follow the dependency chain a real decode has: before a
//   phase stages its activation they wait until every CTA has written the
//   previous phase's outputs.  The down projection really reads the h written
//   by the gate/up phase: that phase also writes h as tagged records (a word
//   of the activation's unit layout and the phase, in one 8-byte store), and
//   the down phase copies them into shared memory once every tag is there.
//   By default the other inputs stand for results of the previous phase:
//   after a phase's outputs are written each CTA adds one to a phase
//   counter, and the next phase waits until the counter shows every CTA.  In a chained step (a real
//   decode chain: each phase reads the previous phase's output) every fp32
//   output is also written as tagged records and the next phase stages its
//   input from them.  No fence sits on either path: the records carry their
//   own readiness, and the counter only orders phases whose inputs no CTA of
//   this launch writes (the kernel checks that first);
// * every wait (ring mbarriers, phase counter, records) is bounded in time;
//   on a timeout a CTA records MQ_DEV_TIMEOUT, raises the step's abort word so
//   the other CTAs stop too, drains its own copies in flight and returns.
//
// Arithmetic, segment split and combine order per matrix are those of the
// per-matrix ring kernels, so the outputs are bit-identical to mq_step's
// multi-kernel path.
#pragma once

#include <type_traits>

#include "mq_epilogue.cuh"
#include "mq_job.cuh"
#include "mq_ring.cuh"
#include "mq_stream.cuh"

namespace mq {

// record pairs a staging thread loads per round
constexpr int kRecBatch = 8;

// Dependency points on the step workspace (zeroed by the host before each
// launch): word 1 is the abort word, word 2 the phase counter (CTAs x phases
// finished), then the h records.  Tags are "phase number + 1", so zero means
// "not yet".

// Wait until the phase counter (workspace word 2; every CTA adds one per
// finished phase) reaches `target`.  Warp 0 polls the one word (its lanes' loads
// of one address are one request); the other warps go on, and the barrier
// after the activation staging holds them.  A counter instead of one flag per
// CTA: 152 CTAs polling 152 flags put ~23K loads per round on five L2 lines.
// False on a timeout or when another CTA aborted.
__device__ __forceinline__ bool wait_count(const unsigned* count, unsigned target, const unsigned* abort_word,
                                           uint64_t limit_ns, int tid)
{
    if (tid >= 32) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (ld_relaxed_u32(count) >= target) return true;
        if ((it & 15u) == 15u && (ld_relaxed_u32(abort_word) != 0 || global_timer_ns() - t0 > limit_ns))
            return false;
    }
}

// The down phase's activation: the h records that this launch's gate/up phase
// wrote with `tag`, copied word for word into the unit layout (record r is
// word r of the planes-then-scales area).  Each thread loads its share of
// record pairs and reads again the ones whose tag is not there yet, bounded
// in time.  False on a timeout or when another CTA aborted.
template <int NC>
__device__ __forceinline__ bool stage_units_rec(const uint64_t* rec, int U, UnitAct s, uint32_t tag,
                                                const unsigned* abort_word, uint64_t limit_ns, int tid, int nthr)
{
    uint32_t* dst = reinterpret_cast<uint32_t*>(s.planes);
    const int npair = NC * 20 * U;  // 40 * U words per column, two per load
    constexpr int B = kRecBatch;
    for (int p0 = tid; p0 < npair; p0 += B * nthr) {
        uint64_t a[B], b[B];
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int i = p0 + k * nthr;
            a[k] = b[k] = uint64_t(tag) << 32;  // pairs past the end count as there
            if (i < npair) ld_tagged2(rec + 2 * size_t(i), a[k], b[k]);
        }
        uint64_t t0 = 0;
        for (uint32_t it = 0;; ++it) {
            bool all = true;
#pragma unroll
            for (int k = 0; k < B; ++k)
                if (uint32_t(a[k] >> 32) != tag || uint32_t(b[k] >> 32) != tag) {
                    all = false;
                    ld_tagged2(rec + 2 * size_t(p0 + k * nthr), a[k], b[k]);
                }
            if (all) break;
            if (it == 0)
                t0 = global_timer_ns();
            else if ((it & 15u) == 0 && (ld_relaxed_u32(abort_word) != 0 || global_timer_ns() - t0 > limit_ns))
                return false;
        }
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int i = p0 + k * nthr;
            if (i < npair) *reinterpret_cast<uint2*>(dst + 2 * i) = make_uint2(uint32_t(a[k]), uint32_t(b[k]));
        }
    }
    return true;
}

// phase views of a layer descriptor
struct PhaseJob {
    const uint8_t* W;
    const float* x;
    const uint8_t* xq;
    uint8_t* xq_out;
    float* y;
    int y_ld;
    const mq_ffn_desc* ffn;
};

__device__ __forceinline__ PhaseJob phase_job(const mq_layer_desc* L, int ph)
{
    PhaseJob j{};
    if (ph == 0 || ph == 1) {
        const mq_mv_desc* d = ph == 0 ? &L->qkv : &L->o;
        j.W = static_cast<const uint8_t*>(d->W);
        j.x = d->x;
        j.xq = static_cast<const uint8_t*>(d->xq);
        j.xq_out = static_cast<uint8_t*>(d->xq_out);
        j.y = d->y;
        j.y_ld = d->y_ld;
    } else if (ph == 2) {
        j.ffn = &L->ffn;
        j.W = static_cast<const uint8_t*>(L->ffn.W_gu);
        j.x = L->ffn.x;
        j.xq = static_cast<const uint8_t*>(L->ffn.xq);
    } else {
        j.ffn = &L->ffn;
        j.W = static_cast<const uint8_t*>(L->ffn.W_down);
        j.xq = static_cast<const uint8_t*>(L->ffn.h_q8);
        j.y = L->ffn.y;
        j.y_ld = L->ffn.y_ld;
    }
    return j;
}

// rows of matrix phase ph owned by CTA b of G: local row lr -> matrix row
struct PhaseRows {
    int nrows, r0, i0, n, R;
    bool gu;
    __device__ __forceinline__ int64_t map(int lr) const
    {
        return gu ? (lr < n ? int64_t(i0) + lr : int64_t(R) + i0 + (lr - n)) : int64_t(r0) + lr;
    }
};

__device__ __forceinline__ PhaseRows phase_rows(const StepPlan& sp, int ph, int b, int G)
{
    PhaseRows r{};
    r.R = sp.R[ph];
    r.gu = (ph == 2);
    if (r.gu) {
        const int nblk = r.R / kQK8;
        const int b0 = int(int64_t(b) * nblk / G), b1 = int(int64_t(b + 1) * nblk / G);
        r.i0 = b0 * kQK8;
        r.n = (b1 - b0) * kQK8;
        r.nrows = 2 * r.n;
    } else {
        r.r0 = int(int64_t(b) * r.R / G);
        r.nrows = int(int64_t(b + 1) * r.R / G) - r.r0;
    }
    return r;
}

// plan values of a phase known only at run time, without indexing the plan
// (a run-time index into the parameter struct would copy it to local memory)
__device__ __forceinline__ int sel4(int ph, int a, int b, int c, int d)
{
    return ph == 0 ? a : (ph == 1 ? b : (ph == 2 ? c : d));
}

// The producer's L2 prefetcher: walks the CTA's tile sequence (layer, phase,
// tile) ahead of the ring, so HBM keeps streaming while the ring is full
// (barrier waits, staging, epilogues).  A prefetch is only a hint: it moves
// data from HBM into L2 and changes nothing else.
struct TileWalker {
    int l, ph, t, ntiles, T;
    int64_t g;  // position in the ring's tile sequence
    PhaseRows pr;
    const uint8_t* W;
    uint32_t row_bytes;
    bool done;

    // settle on the first phase at or after (l, ph) that has tiles
    __device__ __forceinline__ void enter(const mq_layer_desc* layers, const StepPlan& sp, int b, int G, int nc)
    {
        for (;;) {
            if (l >= sp.n_layers) {
                done = true;
                return;
            }
            T = sel4(ph, sp.ph[0].T, sp.ph[1].T, sp.ph[2].T, sp.ph[3].T);
            const int K = sel4(ph, sp.K[0], sp.K[1], sp.K[2], sp.K[3]);
            const int R = sel4(ph, sp.R[0], sp.R[1], sp.R[2], sp.R[3]);
            pr = PhaseRows{};
            pr.R = R;
            pr.gu = (ph == 2);
            if (pr.gu) {
                const int nblk = R / kQK8;
                const int b0 = int(int64_t(b) * nblk / G), b1 = int(int64_t(b + 1) * nblk / G);
                pr.i0 = b0 * kQK8;
                pr.n = (b1 - b0) * kQK8;
                pr.nrows = 2 * pr.n;
            } else {
                pr.r0 = int(int64_t(b) * R / G);
                pr.nrows = int(int64_t(b + 1) * R / G) - pr.r0;
            }
            const PhaseJob j = phase_job(&layers[l], ph);
            W = j.W;
            row_bytes = uint32_t(K / kQK) * kQ4KBytes;
            ntiles = (pr.nrows + T - 1) / T;
            t = 0;
            // the phase's activation too, where it is an fp32 input on a 16-byte boundary
            // that no phase of this launch writes
            if (ntiles > 0 && ph < 3 && !sp.chained && j.x && (reinterpret_cast<uintptr_t>(j.x) & 15) == 0)
                prefetch_l2(j.x, uint32_t(nc) * K * 4);
            if (ntiles > 0) return;
            if (++ph == 4) {
                ph = 0;
                ++l;
            }
        }
    }

    // prefetch the current tile and step to the next
    __device__ __forceinline__ void step(const mq_layer_desc* layers, const StepPlan& sp, int b, int G, int nc)
    {
        const int lr0 = t * T, e = min(lr0 + T, pr.nrows);
        int a = lr0;
        while (a < e) {
            int stop = e;
            if (pr.gu && a < pr.n && e > pr.n) stop = pr.n;
            prefetch_l2(W + size_t(pr.map(a)) * row_bytes, uint32_t(stop - a) * row_bytes);
            a = stop;
        }
        ++g;
        if (++t == ntiles) {
            if (++ph == 4) {
                ph = 0;
                ++l;
            }
            enter(layers, sp, b, G, nc);
        }
    }
};

// The phase whose fp32 output phase (l, ph) reads in a chained step: the
// closest earlier phase with an fp32 output (qkv, o or down; gate/up writes
// h, which only down reads) that is not left out.  False for the launch's
// first such phase, which reads the caller's input.
__device__ __forceinline__ bool chain_producer(const StepPlan& sp, int l, int ph, int* lp, int* php)
{
    for (;;) {
        if (ph == 0) {
            if (l == 0) return false;
            --l;
            ph = 3;
        } else {
            ph = ph == 3 ? 1 : ph - 1;
        }
        if (ph != 2 && sel4(ph, sp.R[0], sp.R[1], sp.R[2], sp.R[3]) > 0) {
            *lp = l;
            *php = ph;
            return true;
        }
    }
}

// fp32 output of phase ph of layer L: pointer, column stride and rows
__device__ __forceinline__ void phase_y(const mq_layer_desc& L, int ph, const float** y, int* ld)
{
    if (ph == 0) {
        *y = L.qkv.y;
        *ld = L.qkv.y_ld;
    } else if (ph == 1) {
        *y = L.o.y;
        *ld = L.o.y_ld;
    } else {
        *y = L.ffn.y;
        *ld = L.ffn.y_ld;
    }
}

// device-side re-check of every layer descriptor against the step plan; in a
// chained step also the chain: every qkv, o and FFN input after the first is
// the fp32 output of its producer phase (same pointer, a column stride equal
// to its K when ncols > 1, at least K rows)
static __device__ __noinline__ unsigned check_layers(const mq_layer_desc* layers, const StepPlan sp, int nc)
{
    unsigned bad = 0;
    for (int l = 0; l < sp.n_layers; ++l) {
        const mq_layer_desc& L = layers[l];
        if (sp.R[0] > 0) bad |= check_job(read_job<KIND_MV>(&L.qkv), sp.R[0], sp.K[0], nc);
        if (sp.R[1] > 0) bad |= check_job(read_job<KIND_MV>(&L.o), sp.R[1], sp.K[1], nc);
        bad |= check_ffn_gu(&L.ffn, sp.K[2], sp.R[2], nc);
        MvJob dn = read_job<KIND_DOWN>(&L.ffn);
        bad |= check_job(dn, sp.R[3], sp.K[3], nc);
        if (!sp.chained) continue;
        for (int ph = 0; ph < 3; ++ph) {
            const int K = sel4(ph, sp.K[0], sp.K[1], sp.K[2], sp.K[3]);
            if (sel4(ph, sp.R[0], sp.R[1], sp.R[2], sp.R[3]) == 0) continue;
            int lp, php;
            if (!chain_producer(sp, l, ph, &lp, &php)) continue;
            const float* x = ph == 0 ? L.qkv.x : (ph == 1 ? L.o.x : L.ffn.x);
            const float* y;
            int ld;
            phase_y(layers[lp], php, &y, &ld);
            if (x != y || (nc > 1 && ld != K) || K > sel4(php, sp.R[0], sp.R[1], sp.R[2], sp.R[3]))
                bad |= MQ_DEV_DESC_MISMATCH;
        }
    }
    return bad;
}

// Byte range [lo, hi) of range `kind` of layer l (lo == hi: none):
// outputs 0 qkv.y, 1 qkv.xq_out, 2 o.y, 3 o.xq_out, 4 h_q8, 5 gu_dbg, 6 h_dbg,
// 7 ffn.y; inputs 8 qkv.W, 9 qkv input, 10 o.W, 11 o input, 12 W_gu, 13
// W_down, 14 FFN input (a chained phase's input is its producer's output and
// is not counted again); 15 the step's workspace.
struct ByteRange {
    uintptr_t lo, hi;
};

__device__ __forceinline__ ByteRange range_of(const mq_layer_desc& L, const StepPlan& sp, int nc, int l, int kind,
                                              const void* ws)
{
    auto r = [](const void* p, size_t n) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        return p ? ByteRange{a, a + n} : ByteRange{a, a};
    };
    auto act_in = [&](const float* x, const void* xq, int K) {
        return x ? r(x, size_t(nc) * K * 4) : r(xq, size_t(nc) * (K / kQK8) * kQ8Bytes);
    };
    auto chained_in = [&](int ph) {
        int lp, php;
        return sp.chained && chain_producer(sp, l, ph, &lp, &php);
    };
    const size_t wrow3 = size_t(sp.K[3] / kQK) * kQ4KBytes;  // down row bytes
    switch (kind) {
        case 0: return sp.R[0] ? r(L.qkv.y, (size_t(nc - 1) * L.qkv.y_ld + sp.R[0]) * 4) : ByteRange{0, 0};
        case 1: return sp.R[0] && L.qkv.x ? r(L.qkv.xq_out, size_t(nc) * (sp.K[0] / kQK8) * kQ8Bytes) : ByteRange{0, 0};
        case 2: return sp.R[1] ? r(L.o.y, (size_t(nc - 1) * L.o.y_ld + sp.R[1]) * 4) : ByteRange{0, 0};
        case 3: return sp.R[1] && L.o.x ? r(L.o.xq_out, size_t(nc) * (sp.K[1] / kQK8) * kQ8Bytes) : ByteRange{0, 0};
        case 4: return r(L.ffn.h_q8, size_t(nc) * (sp.R[2] / kQK8) * kQ8Bytes);
        case 5: return r(L.ffn.gu_dbg, size_t(nc) * 2 * sp.R[2] * 4);
        case 6: return r(L.ffn.h_dbg, size_t(nc) * sp.R[2] * 4);
        case 7: return r(L.ffn.y, (size_t(nc - 1) * L.ffn.y_ld + sp.R[3]) * 4);
        case 8: return sp.R[0] ? r(L.qkv.W, size_t(sp.R[0]) * (sp.K[0] / kQK) * kQ4KBytes) : ByteRange{0, 0};
        case 9: return sp.R[0] && !chained_in(0) ? act_in(L.qkv.x, L.qkv.xq, sp.K[0]) : ByteRange{0, 0};
        case 10: return sp.R[1] ? r(L.o.W, size_t(sp.R[1]) * (sp.K[1] / kQK) * kQ4KBytes) : ByteRange{0, 0};
        case 11: return sp.R[1] && !chained_in(1) ? act_in(L.o.x, L.o.xq, sp.K[1]) : ByteRange{0, 0};
        case 12: return r(L.ffn.W_gu, size_t(2) * sp.R[2] * (sp.K[2] / kQK) * kQ4KBytes);
        case 13: return r(L.ffn.W_down, size_t(sp.R[3]) * wrow3);
        case 14: return !chained_in(2) ? act_in(L.ffn.x, L.ffn.xq, sp.K[2]) : ByteRange{0, 0};
        default: return r(ws, sp.ws_bytes);
    }
}

// True if two ranges of the launch overlap where they must not: any output
// with any other output or any input, the workspace with anything, within a
// layer and between neighbouring layers (inputs may overlap each other: they
// are only read).  The ranges are computed once into `tab` (shared memory,
// n_layers * 16 entries), then every thread of the CTA tests its share of the
// pairs; every CTA reaches the same verdict.  Overlaps between layers further
// apart are not looked for.
static __device__ __noinline__ bool find_alias(const mq_layer_desc* layers, const StepPlan sp, int nc, const void* ws,
                                        ByteRange* tab)
{
    const int nl = sp.n_layers;
    for (int i = threadIdx.x; i < nl * 16; i += blockDim.x) tab[i] = range_of(layers[i >> 4], sp, nc, i >> 4, i & 15, ws);
    __syncthreads();
    int found = 0;
    for (int q = threadIdx.x; q < nl * 512; q += blockDim.x) {
        const int l = q >> 9, dl = (q >> 8) & 1, a = (q >> 4) & 15, b = q & 15;
        if (l + dl >= nl) continue;
        if (a >= 8 && a < 15 && b >= 8 && b < 15) continue;  // two inputs
        if (dl == 0 ? a >= b : (a == 15 || b == 15)) continue;
        const ByteRange x = tab[(l << 4) + a], y = tab[((l + dl) << 4) + b];
        if (x.lo < x.hi && y.lo < y.hi && x.lo < y.hi && y.lo < x.hi) found = 1;
    }
    return __syncthreads_or(found) != 0;
}

// staging of a chained phase's input from its producer's output records (not
// inlined: one copy serves every phase, and the default path carries no code
// for it)
template <int NC>
__device__ __noinline__ bool stage_from_yrec(const uint64_t* yr, int ld, int K, UnitAct act, uint8_t* xq_out,
                                             uint32_t tag, const unsigned* abort_word, uint64_t limit_ns, int tid,
                                             int nthr)
{
    return stage_units_yrec<NC>(yr, ld, K, act, xq_out, tag, abort_word, limit_ns, tid, nthr);
}

// kChained: the MQ_STEP_CHAINED form (inputs staged from the producers'
// output records, outputs also written as records); the default form has no
// code for it
template <int NC, bool kChained>
__global__ void __launch_bounds__(32 * ring_max_warps<NC, 1>(), 1)
    step_kernel(const mq_layer_desc* __restrict__ layers, StepPlan sp, unsigned* status, unsigned* ws)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ volatile int abort_flag;
    const MvPlan& P0 = sp.ph[0];  // ring geometry and shared-memory offsets are common to all phases
    const int G = gridDim.x, b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwc = sp.nwc;
    const uint64_t limit_ns = uint64_t(P0.wait_ms) * 1000000ull;
    unsigned* const count = ws + kWsCountWord;
    // what a CTA adds per finished phase (test-only fault: the last CTA adds nothing)
    const unsigned count_inc = (P0.fault == FAULT_WITHHOLD_COUNT && b == G - 1) ? 0u : 1u;
    uint64_t* const rec = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ws) + kWsRecOff);

    {
        const unsigned bad = check_layers(layers, sp, NC);  // every CTA reaches the same verdict
        if (bad) {
            if (b == 0 && threadIdx.x == 0) atomicOr(status, bad);
            return;
        }
        // overlapping inputs and outputs: the ring's shared memory is free until the producer starts
        if (find_alias(layers, sp, NC, ws, reinterpret_cast<ByteRange*>(smem + P0.off_ring))) {
            if (b == 0 && threadIdx.x == 0) atomicOr(status, MQ_DEV_ALIAS);
            return;
        }
    }
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + P0.ns;
    uint8_t* ring = smem + P0.off_ring;
    float* part = reinterpret_cast<float*>(smem + P0.off_part);
    float* vals = reinterpret_cast<float*>(smem + P0.off_vals);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < P0.ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nwc);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // Phases run in a fixed order per layer; the phase index is a compile-time
    // constant everywhere (run-time indexing of the plan in parameter space
    // would copy it to local memory).
    using P0c = std::integral_constant<int, 0>;
    using P1c = std::integral_constant<int, 1>;
    using P2c = std::integral_constant<int, 2>;
    using P3c = std::integral_constant<int, 3>;
    const int nphase = sp.n_layers * 4;
    int issued = 0;  // tiles issued by the producer (lane 0 of the producer warp)
    if (warp == nwc) {
        // ---- producer: all phases' tiles, back to back
        TileWalker pf{};
        if (lane == 0) pf.enter(layers, sp, b, G, NC);
        // each weight byte is read once per step: its ring copy marks it evict-first
        // in L2, so prefetched tiles and activations stay
        const uint64_t wpolicy = l2_policy_evict_first();
        auto produce = [&](auto phc, int l) -> bool {
            constexpr int ph = decltype(phc)::value;
            const MvPlan& P = sp.ph[ph];
            const PhaseJob j = phase_job(&layers[l], ph);
            const PhaseRows pr = phase_rows(sp, ph, b, G);
            const size_t row_bytes = size_t(sp.K[ph] / kQK) * kQ4KBytes;
            const int ntiles = (pr.nrows + P.T - 1) / P.T;
            for (int t = 0; t < ntiles; ++t, ++issued) {
                const int s = issued % P0.ns;
                // keep the L2 prefetch window pf_tiles ahead of this copy (it also
                // runs ahead while the wait below blocks)
                while (!pf.done && pf.g < int64_t(issued) + sp.pf_tiles) pf.step(layers, sp, b, G, NC);
                if (issued >= P0.ns && !mbar_wait_bounded(&empty[s], uint32_t(issued / P0.ns - 1) & 1u, limit_ns))
                    return false;
                const int lr0 = t * P.T, tn = min(P.T, pr.nrows - lr0);
                mbar_arrive_expect_tx(&full[s], uint32_t(size_t(tn) * row_bytes));
                uint8_t* dst = ring + size_t(s) * P0.stage_bytes;
                int a = lr0;
                const int e = lr0 + tn;
                while (a < e) {
                    int stop = e;
                    if (pr.gu && a < pr.n && e > pr.n) stop = pr.n;
                    bulk_copy_g2s_evict_first(dst + size_t(a - lr0) * row_bytes, j.W + size_t(pr.map(a)) * row_bytes,
                                              uint32_t(size_t(stop - a) * row_bytes), &full[s], wpolicy);
                    a = stop;
                }
            }
            return true;
        };
        if (lane == 0) {
            for (int l = 0; l < sp.n_layers && !abort_flag; ++l) {
                if (!produce(P0c{}, l) || !produce(P1c{}, l) || !produce(P2c{}, l) || !produce(P3c{}, l)) {
                    abort_flag = 1;
                    break;
                }
            }
        }
    } else {
        // ---- consumers
        const int ctid = threadIdx.x, cthr = nwc * 32;
        int gi = 0;  // tile index of the ring sequence at the start of the phase
        auto consume = [&](auto phc, int l) -> bool {
            constexpr int ph = decltype(phc)::value;
            const int k = 4 * l + ph;  // phase number within the launch
            if (sp.R[ph] == 0) {  // a phase left out: only its flag moves on
                if (ctid == 0 && k + 1 < nphase) red_relaxed_add_u32(count, count_inc);
                return true;
            }
            const MvPlan& P = sp.ph[ph];
            const PhaseJob j = phase_job(&layers[l], ph);
            const PhaseRows pr = phase_rows(sp, ph, b, G);
            const int K = sp.K[ph];
            // the input of a chained phase: its producer's output records
            int lp = 0, php = 0;
            const bool from_rec = kChained && ph != 3 && chain_producer(sp, l, ph, &lp, &php);
            // wait until every CTA has written the previous phase's outputs: the
            // down phase, and a chained phase, read their input itself as tagged
            // records; the other phases, whose inputs are separate buffers standing
            // for the previous phase's results, wait for every CTA's flag of that
            // phase
            if (k > 0 && ph != 3 && !from_rec && !wait_count(count, unsigned(G) * unsigned(k), ws + 1, limit_ns, ctid) &&
                lane == 0)
                abort_flag = 1;
            const UnitAct act{reinterpret_cast<uint4*>(smem + P0.off_act),
                              reinterpret_cast<float4*>(smem + P0.off_act + size_t(NC) * 8 * P.C * 16), P.C};
            if (ph == 3) {
                if (!stage_units_rec<NC>(rec, P.C, act, unsigned(k), ws + 1, limit_ns, ctid, cthr)) abort_flag = 1;
            } else if (kChained && from_rec) {
                const int64_t off = php == 0 ? sp.yrec_off[0] : (php == 1 ? sp.yrec_off[1] : sp.yrec_off[3]);
                const int ld = php == 0 ? sp.R[0] : (php == 1 ? sp.R[1] : sp.R[3]);
                const uint64_t* yr = reinterpret_cast<const uint64_t*>(reinterpret_cast<const uint8_t*>(ws) + off);
                if (!stage_from_yrec<NC>(yr, ld, K, act, (ph <= 1 && b == 0) ? j.xq_out : nullptr,
                                         unsigned(4 * lp + php + 1), ws + 1, limit_ns, ctid, cthr))
                    abort_flag = 1;
            } else if (j.x) {
                stage_units_x<NC>(j.x, K, act, (ph <= 1 && b == 0) ? j.xq_out : nullptr, nullptr, ctid, cthr);
            } else {
                stage_units_q8<NC>(j.xq, K, act, nullptr, ctid, cthr);
            }
            named_barrier_sync(1, cthr);
            if (abort_flag) return false;
            bool ok;
            if (NC % 4 == 0 && P.hu)  // the same split as the per-matrix kernel of this shape
                ok = ring_consume<NC, FmtQ4K, 4>(P, pr.nrows, gi, P.nwc, ring, full, empty, act, part, limit_ns);
            else if (NC >= 3 && P.cgw)
                ok = ring_consume<NC, FmtQ4K, 3>(P, pr.nrows, gi, P.nwc, ring, full, empty, act, part, limit_ns);
            else if (NC >= 3 && P.cmap)
                ok = ring_consume<NC, FmtQ4K, 1>(P, pr.nrows, gi, P.nwc, ring, full, empty, act, part, limit_ns);
            else
                ok = ring_consume<NC>(P, pr.nrows, gi, P.nwc, ring, full, empty, act, part, limit_ns);
            gi += (pr.nrows + P.T - 1) / P.T;
            if (!ok && lane == 0) abort_flag = 1;
            named_barrier_sync(1, cthr);
            if (abort_flag) return false;
            if (ph == 2) {
                gu_epilogue_on<NC>(part, vals, P.nseg, pr.n, pr.i0, pr.R, static_cast<uint8_t*>(j.ffn->h_q8),
                                   j.ffn->gu_dbg, j.ffn->h_dbg, ctid, cthr, [cthr]() { named_barrier_sync(1, cthr); },
                                   (P.fault == FAULT_WITHHOLD_RECORDS && b == G - 1) ? nullptr : rec, unsigned(k + 1));
            } else {
                if (kChained && sp.yrec_off[ph] >= 0)
                    mv_epilogue<NC>(part, P.nseg, pr.nrows, pr.r0, j.y, j.y_ld, ctid, cthr,
                                    reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ws) + sp.yrec_off[ph]),
                                    pr.R, unsigned(k + 1));
                else
                    mv_epilogue<NC>(part, P.nseg, pr.nrows, pr.r0, j.y, j.y_ld, ctid, cthr);
            }
            named_barrier_sync(1, cthr);  // this CTA's outputs of phase k are written
            if (ctid == 0 && k + 1 < nphase) red_relaxed_add_u32(count, count_inc);
            return true;
        };
        for (int l = 0; l < sp.n_layers; ++l)
            if (!consume(P0c{}, l) || !consume(P1c{}, l) || !consume(P2c{}, l) || !consume(P3c{}, l)) break;
        if (abort_flag && ctid == 0) atomicExch(ws + 1, 1u);  // let the other CTAs stop early
    }
    __syncthreads();
    if (abort_flag) {
        if (threadIdx.x == 0) atomicOr(status, MQ_DEV_TIMEOUT);
        if (warp == nwc && lane == 0)  // drain this CTA's copies that may still be in flight
            for (int t = issued > P0.ns ? issued - P0.ns : 0; t < issued; ++t)
                (void)mbar_wait_bounded(&full[t % P0.ns], uint32_t(t / P0.ns) & 1u, limit_ns);
    }
}


}  // namespace mq
