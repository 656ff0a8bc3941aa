// mq_ring.cuh -- consumer side of the bulk-copy weight ring, shared by the
// per-matrix ring kernels (ring.cu) and the persistent step kernel (step.cu).
#pragma once

#include "mq_internal.h"
#include "mq_tma.cuh"
#include "mq_unit.cuh"

namespace mq {

// consumer warps + the producer warp: 15 + 1 for one or two columns; 8 + 1 for more
// columns, which need more registers per thread (activation and
// accumulators).  The register file is split between the SM's four
// schedulers, so the busiest scheduler's warp count sets the per-thread
// budget: 16 warps (4 per scheduler) allow 128 registers, 17 only 96.
// kMode: 0 = unit lanes, the kernel built for 1..2 columns (16 warps) or the
// 9-warp form; 1 = column lanes (16 warps); 2 = unit lanes for 3..8 columns
// with 16 warps (activation columns read from shared memory per row pair)
// 3 = column groups (16 warps; see ring_consume_groups)
template <int NC, int kMode = 0>
__host__ __device__ constexpr int ring_max_warps()
{
    return (NC <= 2 || kMode != 0) ? 16 : 9;
}

// Column lanes (3..8 columns): lane = (unit-lane ul, column c) with c the low
// bits; cols_group columns per group (4 or 8), 32/cols_group unit-lanes per
// item.
template <int NC>
__host__ __device__ constexpr int cols_group()
{
    return NC <= 4 ? 4 : 8;
}

// Sum of v over the L lanes of each lane group, into every lane of the group.
template <int L>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int off = L >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Two rows' partials a, b reduced over the L lanes of each group in one tree:
// afterwards lanes l < L/2 hold row a's sum, lanes l >= L/2 row b's.
template <int L>
__device__ __forceinline__ float group_sum2(float a, float b, int l)
{
    const bool upper = l >= (L >> 1);
    float keep = upper ? b : a;
    const float send = upper ? a : b;
    keep += __shfl_xor_sync(0xffffffffu, send, L >> 1);
#pragma unroll
    for (int off = L >> 2; off > 0; off >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, off);
    return keep;
}

// Consumer side of the ring, for L lanes per item.  A lane always works on the
// same unit u of every row (segment-stationary warps), so its 128 activation
// codes and scales stay in registers (ncols <= 2; from shared memory above).
// Each iteration takes two rows of the tile (r + sub and r + rg + sub): two
// independent dp4a chains per lane and one shuffle tree for both rows.
// Returns false if a wait timed out.
// What a consumer needs of a ring plan, by value: a non-inlined callee that
// took the plan by reference would read it through local memory.
struct ConsumeArgs {
    int C, L, nseg, S, rg, T, ns, stage_bytes;
    int nrows;      // the CTA's rows of this matrix
    int tile_base;  // ring position of the matrix's first tile
    int nwc_used;   // consumer warps with work (the others only hand tiles back)
    // partials: part[(row * nseg + seg) * pcols + pc0 + c] for the consumer's
    // columns c; warps are numbered from warp0 (a column group's first warp)
    int pcols, pc0, warp0;
};

__device__ __forceinline__ ConsumeArgs consume_args(const MvPlan& p, int nrows, int tile_base, int nwc_used, int pcols)
{
    return ConsumeArgs{p.C, p.L, p.nseg, p.S, p.rg, p.T, p.ns, p.stage_bytes, nrows, tile_base, nwc_used, pcols, 0, 0};
}

// (not inlined: called once per matrix, it keeps its own register allocation
// instead of adding to the caller's)
template <int NC, int L, class Fmt = FmtQ4K>
__device__ __noinline__ bool ring_consume_L(const ConsumeArgs p, const uint8_t* ring, uint64_t* full,
                                            uint64_t* empty, const UnitAct act, float* __restrict__ part,
                                            uint64_t limit_ns)
{
    const int nrows = p.nrows, nwc_used = p.nwc_used;
    const int warp = (threadIdx.x >> 5) - p.warp0, lane = threadIdx.x & 31;
    const int nseg = p.nseg;
    const int seg = warp % nseg, jj = warp / nseg;
    constexpr int ipw = 32 / L;
    const int sub = lane / L, l = lane - sub * L;
    const int rho0 = jj * ipw;  // first row-lane of this warp
    const int rg = p.rg;
    const int u = seg * p.S + l;  // this lane's unit of every row
    // warps beyond nwc_used have no work in this matrix but still take part in
    // every tile's full/empty handshake, so the stage counts stay exact
    const bool warp_active = warp < nwc_used;
    const bool on = warp_active && (l < p.S) && (u < p.C);
    const uint32_t row_bytes = Fmt::row_bytes(p.C);
    // 1..2 columns: a lane without a unit computes on unit 0 and drops the
    // result, and rows past the tile's end are clamped to its last row, so the
    // row loop has no divergent branch, only selects and predicated stores.
    const int uu = on ? u : 0;
    const typename Fmt::Off off = Fmt::offsets(uu);

    constexpr bool kRegAct = NC <= 2;
    uint4 A[NC][8];
    float4 DQ[NC], DQSQ[NC];
    auto load_act = [&](int c, int slot) {  // column c's codes and scales into A[slot], DQ[slot], DQSQ[slot]
#pragma unroll
        for (int k = 0; k < 8; ++k) A[slot][k] = act.planes[size_t(c * 8 + k) * act.U + uu];
        DQ[slot] = act.scales[(size_t(c) * act.U + uu) * 2];
        DQSQ[slot] = act.scales[(size_t(c) * act.U + uu) * 2 + 1];
    };
    if (kRegAct) {
#pragma unroll
        for (int c = 0; c < NC; ++c) load_act(c, c);
    }

    // the partial this lane stores: lane 0 of an item holds row r + sub's sum,
    // lane L/2 row r + rg + sub's (group_sum2); one pointer, advanced per step
    const bool storer = l == 0 || l == (L >> 1);
    const int srow = sub + (l == 0 ? 0 : rg);
    const int pstep = 2 * rg * nseg * p.pcols;

    int s = p.tile_base % p.ns;  // ring stage and its parity, advanced per tile
    uint32_t par = uint32_t(p.tile_base / p.ns) & 1u;
    for (int tr0 = 0; tr0 < nrows; tr0 += p.T) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], par, limit_ns));
        if (!ok) return false;
        const uint8_t* stage = ring + uint32_t(s) * uint32_t(p.stage_bytes);
        const int tn = min(p.T, nrows - tr0);
        float* pq = part + (size_t(tr0 + rho0 + srow) * nseg + seg) * p.pcols + p.pc0;
        for (int r = warp_active ? rho0 : tn; r < tn; r += 2 * rg, pq += pstep) {  // r is warp-uniform
            const int ra = r + sub, rb = r + rg + sub;
            const bool st = storer && r + srow < tn;
            const bool va = on && ra < tn, vb = on && rb < tn;
            float xa[NC], xb[NC];
            if constexpr (kRegAct) {
                typename Fmt::W wa, wb;
                Fmt::load(stage + uint32_t(min(ra, tn - 1)) * row_bytes, off, wa);
                Fmt::load(stage + uint32_t(min(rb, tn - 1)) * row_bytes, off, wb);
                const typename Fmt::S ka = Fmt::prep(wa, off), kb = Fmt::prep(wb, off);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    xa[c] = Fmt::column(wa, ka, A[c], DQ[c], DQSQ[c]);
                    xb[c] = Fmt::column(wb, kb, A[c], DQ[c], DQSQ[c]);
                }
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    xa[c] = va ? xa[c] : 0.0f;
                    xb[c] = vb ? xb[c] : 0.0f;
                }
            } else {
                // 3..8 columns (activation read from shared memory per row pair):
                // branches keep fewer values live than computing every lane
#pragma unroll
                for (int c = 0; c < NC; ++c) xa[c] = xb[c] = 0.0f;
                if (va || vb) {
                    typename Fmt::W wa, wb;
                    Fmt::load(stage + uint32_t(va ? ra : rb) * row_bytes, off, wa);
                    Fmt::load(stage + uint32_t(vb ? rb : ra) * row_bytes, off, wb);
                    const typename Fmt::S ka = Fmt::prep(wa, off), kb = Fmt::prep(wb, off);
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        load_act(c, 0);
                        if (va) xa[c] = Fmt::column(wa, ka, A[0], DQ[0], DQSQ[0]);
                        if (vb) xb[c] = Fmt::column(wb, kb, A[0], DQ[0], DQSQ[0]);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const float t = group_sum2<L>(xa[c], xb[c], l);
                if (st) pq[c] = t;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == p.ns) {
            s = 0;
            par ^= 1u;
        }
    }
    return true;
}

// Consumer side for 3..8 columns with column lanes: lane (ul, c) keeps the
// codes and scales of unit seg*S + ul of column c in registers (so every
// column's activation stays in registers, whatever the column count), loads
// that unit's weights of each row (the lanes of one unit read the same bytes:
// shared-memory broadcast) and reduces over its unit-lanes per column.  The
// warp <-> (segment, row-lane) split, tiles, partials and combine order are
// those of ring_consume_L with one item per warp.
template <int NC, class Fmt = FmtQ4K>
__device__ __noinline__ bool ring_consume_cols(const ConsumeArgs p, const uint8_t* ring, uint64_t* full,
                                               uint64_t* empty, const UnitAct act, float* __restrict__ part,
                                               uint64_t limit_ns)
{
    constexpr int CP = cols_group<NC>();
    const int nrows = p.nrows, tile_base = p.tile_base, nwc_used = p.nwc_used;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nseg = p.nseg;
    const int seg = warp % nseg, jj = warp / nseg;
    const int c = lane % CP, ul = lane / CP;
    const int rg = p.rg;
    const int u = seg * p.S + ul;
    const bool warp_active = warp < nwc_used;
    const bool on = warp_active && (ul < p.S) && (u < p.C) && (c < NC);
    const uint32_t row_bytes = Fmt::row_bytes(p.C);
    const typename Fmt::Off off = Fmt::offsets(on ? u : 0);
    uint4 A[8];
    float4 DQ = make_float4(0.f, 0.f, 0.f, 0.f), DQSQ = DQ;
    if (on) {
#pragma unroll
        for (int k = 0; k < 8; ++k) A[k] = act.planes[size_t(c * 8 + k) * act.U + u];
        DQ = act.scales[(size_t(c) * act.U + u) * 2];
        DQSQ = act.scales[(size_t(c) * act.U + u) * 2 + 1];
    }
    const int ntiles = (nrows + p.T - 1) / p.T;
    for (int i = 0; i < ntiles; ++i) {
        const int gi = tile_base + i;
        const int s = gi % p.ns;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], uint32_t(gi / p.ns) & 1u, limit_ns));
        if (!ok) return false;
        const uint8_t* stage = ring + uint32_t(s) * uint32_t(p.stage_bytes);
        const int tr0 = i * p.T, tn = min(p.T, nrows - tr0);
        for (int r = warp_active ? jj : tn; r < tn; r += 2 * rg) {
            const int ra = r, rb = r + rg;
            const bool va = on && ra < tn, vb = on && rb < tn;
            float acc_a = 0.0f, acc_b = 0.0f;
            if (va || vb) {
                typename Fmt::W wa, wb;
                Fmt::load(stage + uint32_t(va ? ra : rb) * row_bytes, off, wa);
                Fmt::load(stage + uint32_t(vb ? rb : ra) * row_bytes, off, wb);
                const typename Fmt::S ka = Fmt::prep(wa, off), kb = Fmt::prep(wb, off);
                if (va) acc_a = Fmt::column(wa, ka, A, DQ, DQSQ);
                if (vb) acc_b = Fmt::column(wb, kb, A, DQ, DQSQ);
            }
#pragma unroll
            for (int o = CP; o < 32; o <<= 1) {
                acc_a += __shfl_xor_sync(0xffffffffu, acc_a, o);
                acc_b += __shfl_xor_sync(0xffffffffu, acc_b, o);
            }
            if (ul == 0 && c < NC) {
                if (ra < tn) part[((tr0 + ra) * nseg + seg) * NC + c] = acc_a;
                if (rb < tn) part[((tr0 + rb) * nseg + seg) * NC + c] = acc_b;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    return true;
}

// Half-unit lanes (3..8 columns, q4_K weights): lane l of a (row, segment)
// item works on half-unit v = seg*S + l of every row: 64 weights, the two
// sub-blocks 2hh, 2hh+1 (hh = v & 1) of unit v >> 1, i.e. 32 quant bytes and
// the super-block's header.  Its activation is 16 code words and two scale
// pairs per column, so a lane holds up to four columns in registers and
// unpacks each weight once for them.  Warps form groups of four columns (as
// ring_consume_groups does for two); the unit split counts half-units.
template <int NCW, int L>
__device__ __noinline__ bool ring_consume_half(const ConsumeArgs p, const uint8_t* ring, uint64_t* full,
                                               uint64_t* empty, const UnitAct act, float* __restrict__ part,
                                               uint64_t limit_ns)
{
    const int nrows = p.nrows, nwc_used = p.nwc_used;
    const int warp = (threadIdx.x >> 5) - p.warp0, lane = threadIdx.x & 31;
    const int nseg = p.nseg;
    const int seg = warp % nseg, jj = warp / nseg;
    constexpr int ipw = 32 / L;
    const int sub = lane / L, l = lane - sub * L;
    const int rho0 = jj * ipw;
    const int rg = p.rg;
    const int v = seg * p.S + l;
    const bool warp_active = warp < nwc_used;
    const bool on = warp_active && (l < p.S) && (v < 2 * p.C);
    const int vv = on ? v : 0;
    const int u = vv >> 1, hh = vv & 1;
    const bool upper = (u & 1) != 0;
    const uint32_t row_bytes = uint32_t(p.C / 2) * kQ4KBytes;
    const uint32_t off_h = uint32_t(u >> 1) * kQ4KBytes;
    const uint32_t off_q = off_h + 16 + 64 * uint32_t(u & 1) + 32 * uint32_t(hh);
    const uint32_t j0 = 2 * uint32_t(hh);  // the half's low-nibble sub-block within the unit
    uint4 A[NCW][4];
    float dq0[NCW], dq1[NCW], dqs0[NCW], dqs1[NCW];
#pragma unroll
    for (int c = 0; c < NCW; ++c) {
#pragma unroll
        for (int i = 0; i < 4; ++i) A[c][i] = act.planes[size_t(c * 8 + 4 * hh + i) * act.U + u];
        const float4 d4 = act.scales[(size_t(c) * act.U + u) * 2], s4 = act.scales[(size_t(c) * act.U + u) * 2 + 1];
        dq0[c] = hh ? d4.z : d4.x;
        dq1[c] = (hh ? d4.w : d4.y) * 0.0625f;  // high nibbles are used as 16*q
        dqs0[c] = hh ? s4.z : s4.x;
        dqs1[c] = hh ? s4.w : s4.y;
    }
    const bool storer = l == 0 || l == (L >> 1);
    const int srow = sub + (l == 0 ? 0 : rg);
    const int pstep = 2 * rg * nseg * p.pcols;
    // one row's contribution per column
    auto row = [&](const uint8_t* stage, int r, float (&x)[NCW]) {
        const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(stage)) + uint32_t(r) * row_bytes;
        uint4 hd, q0, q1;
        lds128(hd, a + off_h);
        lds128(q0, a + off_q);
        lds128(q1, a + off_q + 16);
        const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
        const uint32_t S0 = hd.y, S1 = hd.z, S2 = hd.w;
        const uint32_t mlo = upper ? 0x0f0f0f0fu : 0x3f3f3f3fu;
        const uint32_t mhi = upper ? 0x30303030u : 0u;
        const uint32_t scw = ((upper ? S2 : S0) & mlo) | ((S0 >> 2) & mhi);
        const uint32_t mw = ((upper ? (S2 >> 4) : S1) & mlo) | ((S1 >> 2) & mhi);
        const int sc0 = int(__byte_perm(scw, 0u, 0x4440u | j0)), sc1 = int(__byte_perm(scw, 0u, 0x4440u | (j0 + 1)));
        const float m0 = __int_as_float(__byte_perm(mw, 0x4B000000u, 0x7540u | j0)) - 8388608.0f;
        const float m1 = __int_as_float(__byte_perm(mw, 0x4B000000u, 0x7540u | (j0 + 1))) - 8388608.0f;
#pragma unroll
        for (int c = 0; c < NCW; ++c) {
            const int s0 = dot16_lo(q1, A[c][1], dot16_lo(q0, A[c][0], 0));
            const int s1 = dot16_hi(q1, A[c][3], dot16_hi(q0, A[c][2], 0));
            const float t = fmaf(dq1[c], float(sc1 * s1), dq0[c] * float(sc0 * s0));
            const float um = fmaf(m1, dqs1[c], m0 * dqs0[c]);
            x[c] = fmaf(-dd.y, um, dd.x * t);
        }
    };
    int s = p.tile_base % p.ns;
    uint32_t par = uint32_t(p.tile_base / p.ns) & 1u;
    for (int tr0 = 0; tr0 < nrows; tr0 += p.T) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], par, limit_ns));
        if (!ok) return false;
        const uint8_t* stage = ring + uint32_t(s) * uint32_t(p.stage_bytes);
        const int tn = min(p.T, nrows - tr0);
        float* pq = part + (size_t(tr0 + rho0 + srow) * nseg + seg) * p.pcols + p.pc0;
        for (int r = warp_active ? rho0 : tn; r < tn; r += 2 * rg, pq += pstep) {  // r is warp-uniform
            const int ra = r + sub, rb = r + rg + sub;
            const bool st = storer && r + srow < tn;
            const bool va = on && ra < tn, vb = on && rb < tn;
            float xa[NCW], xb[NCW];
            row(stage, min(ra, tn - 1), xa);
            row(stage, min(rb, tn - 1), xb);
#pragma unroll
            for (int c = 0; c < NCW; ++c) {
                const float t = group_sum2<L>(va ? xa[c] : 0.0f, vb ? xb[c] : 0.0f, l);
                if (st) pq[c] = t;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == p.ns) {
            s = 0;
            par ^= 1u;
        }
    }
    return true;
}

// Column groups (3..8 columns): the consumer warps split into groups of
// p.cgw warps; group g runs the one- or two-column consumer (activation in
// registers, the row loop without branches) on columns 2g and 2g+1 of every
// tile, so each group reads and unpacks the tile's weights once for its
// columns.  Warps past the last group only hand the tiles back.  The unit
// split, partials and combine order are those of the plan (the same for every
// group).
template <int NC, class Fmt>
__device__ __forceinline__ bool ring_consume_groups(ConsumeArgs a, int cgw, const uint8_t* ring, uint64_t* full,
                                                    uint64_t* empty, const UnitAct& act, float* __restrict__ part,
                                                    uint64_t limit_ns)
{
    constexpr int NG = (NC + 1) / 2;
    const int g = (int(threadIdx.x) >> 5) / cgw;
    const int c0 = 2 * g;
    a.pc0 = c0;
    a.warp0 = g * cgw;
    if (g >= NG) a.nwc_used = 0;
    // the group's columns as a view of the activation (each column's planes and
    // scales are contiguous in the unit layout)
    const int gc = g < NG ? c0 : 0;
    const UnitAct v{act.planes + size_t(gc) * 8 * act.U, act.scales + size_t(gc) * act.U * 2, act.U};
    const bool two = g < NG && c0 + 1 < NC;
#define MQ_GROUP_L(LL)                                                                      \
    return two ? ring_consume_L<2, LL, Fmt>(a, ring, full, empty, v, part, limit_ns)        \
               : ring_consume_L<1, LL, Fmt>(a, ring, full, empty, v, part, limit_ns);
    if (a.L == 32) { MQ_GROUP_L(32) }
    if (a.L == 16) { MQ_GROUP_L(16) }
    if (a.L == 8) { MQ_GROUP_L(8) }
    MQ_GROUP_L(4)
#undef MQ_GROUP_L
}

// Groups of four columns on half-unit lanes (4 or 8 columns): group g on
// columns 4g..4g+3.
template <int NC>
__device__ __forceinline__ bool ring_consume_half_groups(ConsumeArgs a, int cgw, const uint8_t* ring, uint64_t* full,
                                                         uint64_t* empty, const UnitAct& act,
                                                         float* __restrict__ part, uint64_t limit_ns)
{
    static_assert(NC % 4 == 0, "half-unit lanes take groups of four columns");
    constexpr int NG = NC / 4;
    const int g = (int(threadIdx.x) >> 5) / cgw;
    a.pc0 = 4 * g;
    a.warp0 = g * cgw;
    if (g >= NG) a.nwc_used = 0;
    const int gc = g < NG ? 4 * g : 0;
    const UnitAct v{act.planes + size_t(gc) * 8 * act.U, act.scales + size_t(gc) * act.U * 2, act.U};
    if (a.L == 32) return ring_consume_half<4, 32>(a, ring, full, empty, v, part, limit_ns);
    if (a.L == 16) return ring_consume_half<4, 16>(a, ring, full, empty, v, part, limit_ns);
    if (a.L == 8) return ring_consume_half<4, 8>(a, ring, full, empty, v, part, limit_ns);
    return ring_consume_half<4, 4>(a, ring, full, empty, v, part, limit_ns);
}

// kMode 1: the kernel was built for column lanes (its plans all have cmap = 1);
// kMode 3: for column groups (cgw > 0); kMode 4: for half-unit lanes (hu = 1)
template <int NC, class Fmt = FmtQ4K, int kMode = 0>
__device__ __forceinline__ bool ring_consume(const MvPlan& p, int nrows, int tile_base, int nwc_used,
                                             const uint8_t* ring, uint64_t* full, uint64_t* empty,
                                             const UnitAct& act, float* __restrict__ part, uint64_t limit_ns)
{
    const ConsumeArgs a = consume_args(p, nrows, tile_base, nwc_used, NC);
    if constexpr (kMode == 3) {
        ConsumeArgs ag = consume_args(p, nrows, tile_base, p.cgu, NC);
        return ring_consume_groups<NC, Fmt>(ag, p.cgw, ring, full, empty, act, part, limit_ns);
    }
    if constexpr (kMode == 4) {
        if constexpr (NC % 4 == 0) {
            ConsumeArgs ag = consume_args(p, nrows, tile_base, p.cgu, NC);
            return ring_consume_half_groups<NC>(ag, p.cgw, ring, full, empty, act, part, limit_ns);
        }
        return false;
    }
    if constexpr (kMode == 1) return ring_consume_cols<NC, Fmt>(a, ring, full, empty, act, part, limit_ns);
    if (p.L == 32) return ring_consume_L<NC, 32, Fmt>(a, ring, full, empty, act, part, limit_ns);
    if (p.L == 16) return ring_consume_L<NC, 16, Fmt>(a, ring, full, empty, act, part, limit_ns);
    if (NC <= 2 && p.L == 4) return ring_consume_L<NC, 4, Fmt>(a, ring, full, empty, act, part, limit_ns);
    return ring_consume_L<NC, 8, Fmt>(a, ring, full, empty, act, part, limit_ns);
}

}  // namespace mq
