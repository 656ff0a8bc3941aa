// mq_unit.cuh -- the half-super-block work unit of the bulk-copy ring kernels.
//
// A unit is half of a q4_K super-block: 128 weights = sub-blocks 4h..4h+3
// (h = 0 or 1), i.e. quant bytes 64h..64h+63 of the block plus the shared
// 16-byte header.  Unit u of a row covers activation elements [128u,
// 128u+128): four q8_0 blocks, 128 codes, in element order.  Per unit a lane
// does five 16-byte loads, one scale unpack for four sub-blocks (the lane's h
// is fixed, so it needs one of the two scale forms, picked by a select) and
// 32 dp4a: half the per-weight overhead of a 64-weight unit.
//
// Activation staging layout (shared memory), per column c, U = K/128 units:
//   planes[(c*8 + k)*U + u]  = codes 16k..16k+15 of unit u   (uint4)
//   scales[(c*U + u)*2 + 0]  = {dq_0, dq_1, dq_2, dq_3}       (float4)
//   scales[(c*U + u)*2 + 1]  = {dq_j * sumq_j}                (float4)
// with dq the stored binary16 scale of each of the unit's four q8_0 blocks.
// Eight consecutive lanes reading consecutive units touch 128 consecutive
// bytes of a plane, so reads are free of bank conflicts.
#pragma once

#include "mq_device.cuh"
#include "mq_tma.cuh"

namespace mq {

constexpr int kUnitElems = 128;
// q8_0 activations staged from global memory one thread per block (true) or
// one warp per unit (fp32 activations: always one warp per unit, which
// measured faster for them)
constexpr bool kBlockStaging = true;

struct UnitAct {
    uint4* planes;
    float4* scales;
    int U;  // units per row = K/128
};

// Staging works one warp per unit: lane l holds codes 4l..4l+3 of the unit,
// i.e. values 4g..4g+3 (g = l % 8) of the unit's q8_0 block l / 8, which is
// one 32-bit word of plane l / 4.  The eight lanes of a block reduce its
// amax / code sum with three xor-shuffles.  tid = 0..nthr-1 are whole warps.

// Where one lane's results of unit u go: its code word in plane l / 4, and
// (lanes g == 0) its block's scale pair.  Lane constants, so the per-unit
// address is one multiply-add.
struct UnitLaneOut {
    uint32_t* code;  // + 4u words
    float* scale;    // + 8u floats: [slot] = dq, [4 + slot] = dq*sumq
    __device__ __forceinline__ UnitLaneOut(UnitAct s, int c, int lane)
    {
        code = reinterpret_cast<uint32_t*>(s.planes + size_t(c * 8 + (lane >> 2)) * s.U) + (lane & 3);
        scale = reinterpret_cast<float*>(s.scales + size_t(c) * s.U * 2) + (lane >> 3);
    }
    __device__ __forceinline__ void put(int u, int lane, uint32_t codes, float dq, int sq) const
    {
        code[4 * u] = codes;
        if ((lane & 7) == 0) {
            scale[8 * u] = dq;
            scale[8 * u + 4] = dq * float(sq);
        }
    }
};

__device__ __forceinline__ int group8_sum(int v)
{
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v + __shfl_xor_sync(0xffffffffu, v, 4);
}

// One q8_0 block's place in the unit layout: block J of column c is slot J % 4
// of unit J / 4; its 32 codes are planes 2*slot and 2*slot + 1 of that unit.
__device__ __forceinline__ void put_block(UnitAct s, int c, int J, const uint32_t (&w)[8], float dq, int sq)
{
    const int u = J >> 2, slot = J & 3;
    s.planes[size_t(c * 8 + 2 * slot) * s.U + u] = make_uint4(w[0], w[1], w[2], w[3]);
    s.planes[size_t(c * 8 + 2 * slot + 1) * s.U + u] = make_uint4(w[4], w[5], w[6], w[7]);
    float* S = reinterpret_cast<float*>(s.scales + (size_t(c) * s.U + u) * 2);
    S[slot] = dq;
    S[4 + slot] = dq * float(sq);
}

// From q8_0 blocks in global memory, one thread per block (xq 4-byte aligned,
// K % 256 == 0): block J of a column starts at byte 34J, i.e. on a word
// boundary (J even) or two bytes past one (J odd); nine aligned words hold it
// either way.  A thread's blocks are loaded before any is used.
// sumq_out (nullable, test export): int32 [NC][K/32].  (Not inlined: it keeps
// its own register allocation, apart from the kernels' hot loops.)
// Blocks [j0, j0 + nqr) of each column of nq_all blocks (K split: one part of
// every row; otherwise j0 = 0, nqr = nq_all), staged as units 0 .. nqr/4 - 1.
template <int NC>
__device__ __noinline__ void stage_blocks_q8(const uint8_t* __restrict__ xq, int nq_all, int j0, int nqr, UnitAct s,
                                                int32_t* sumq_out, int tid, int nthr)
{
    const int nq = nqr, total = NC * nq;
    constexpr int B = 2;
    for (int t0 = tid; t0 < total; t0 += B * nthr) {
        uint32_t w[B][9];
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int t = t0 + k * nthr;
            if (t < total) {
                const int c = t / nq;
                const size_t tg = size_t(c) * nq_all + j0 + (t - c * nq);  // the block's index in xq
                const uint32_t* p = reinterpret_cast<const uint32_t*>(xq + (tg * kQ8Bytes & ~size_t(3)));
#pragma unroll
                for (int i = 0; i < 9; ++i) w[k][i] = __ldg(p + i);
            }
        }
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int t = t0 + k * nthr;
            if (t >= total) break;
            const int c = t / nq, J = t - c * nq;
            const bool odd = ((size_t(c) * nq_all + j0 + J) & 1) != 0;
            uint32_t cw[8];
            int sq = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                cw[i] = odd ? w[k][i + 1] : __funnelshift_r(w[k][i], w[k][i + 1], 16);
                sq = __dp4a(int(cw[i]), 0x01010101, sq);
            }
            const float dq = __half2float(__ushort_as_half(uint16_t(odd ? w[k][0] >> 16 : w[k][0])));
            put_block(s, c, J, cw, dq, sq);
            if (sumq_out) sumq_out[t] = sq;
        }
    }
}

// q8_0 blocks, one thread per block: the form for a 2-byte aligned xq.
template <int NC>
__device__ __forceinline__ void stage_units_q8_by_block(const uint8_t* __restrict__ xq, int nq_all, int j0, int nqr,
                                                        UnitAct s, int32_t* sumq_out, int tid, int nthr)
{
    const int nq = nqr;
    for (int t = tid; t < NC * nq; t += nthr) {
        const int c = t / nq, J = t - c * nq;
        const uint16_t* h = reinterpret_cast<const uint16_t*>(xq + (size_t(c) * nq_all + j0 + J) * kQ8Bytes);
        uint16_t v[17];
#pragma unroll
        for (int k = 0; k < 17; ++k) v[k] = __ldg(h + k);
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = uint32_t(v[1 + 2 * k]) | (uint32_t(v[2 + 2 * k]) << 16);
        const float dq = __half2float(__ushort_as_half(v[0]));
        int sq = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) sq = __dp4a(int(w[k]), 0x01010101, sq);
        const int u = J >> 2, slot = J & 3;
        s.planes[size_t(c * 8 + 2 * slot) * s.U + u] = make_uint4(w[0], w[1], w[2], w[3]);
        s.planes[size_t(c * 8 + 2 * slot + 1) * s.U + u] = make_uint4(w[4], w[5], w[6], w[7]);
        float* S = reinterpret_cast<float*>(s.scales + (size_t(c) * s.U + u) * 2);
        S[slot] = dq;
        S[4 + slot] = dq * float(sq);
        if (sumq_out) sumq_out[size_t(c) * nq + J] = sq;
    }
}

// From q8_0 blocks in global memory (34-byte blocks; column c starts at byte
// c*K/32*34).  sumq_out (nullable, test export): int32 [NC][K/32].
// A unit's four blocks are 136 contiguous bytes at byte 136u of its column,
// 34 words when xq is 4-byte aligned (K % 256 == 0 keeps every column and
// unit on a word boundary): lanes load words 0..31 and lanes 0, 1 words 32,
// 33, and each lane gathers its four codes and its block's scale by shuffles.
template <int NC>
__device__ __forceinline__ void stage_units_q8(const uint8_t* __restrict__ xq, int K, UnitAct s, int32_t* sumq_out,
                                               int tid, int nthr)
{
    if (reinterpret_cast<uintptr_t>(xq) & 3) {
        stage_units_q8_by_block<NC>(xq, K / kQK8, 0, K / kQK8, s, sumq_out, tid, nthr);
        return;
    }
    if (kBlockStaging) {
        stage_blocks_q8<NC>(xq, K / kQK8, 0, K / kQK8, s, sumq_out, tid, nthr);
        return;
    }
    const int lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    const int nq = K / kQK8, U = s.U;
    const int slot = lane >> 3, g = lane & 7;
    const int cb = 34 * slot + 2 + 4 * g;                   // byte of my first code within the unit
    const int cw = cb >> 2, cw1 = min(cw + 1, 33), csh = (cb & 3) * 8;
    const int sw = (34 * slot) >> 2, ssh = ((34 * slot) & 3) * 8;  // the block's f16 scale
    auto unit = [&](uint32_t w0, uint32_t w1, uint32_t& codes, float& dq) {
        const uint32_t a0 = __shfl_sync(0xffffffffu, w0, cw & 31), a1 = __shfl_sync(0xffffffffu, w1, cw & 31);
        const uint32_t b0 = __shfl_sync(0xffffffffu, w0, cw1 & 31), b1 = __shfl_sync(0xffffffffu, w1, cw1 & 31);
        const uint32_t s0 = __shfl_sync(0xffffffffu, w0, sw);
        const uint32_t lo = cw < 32 ? a0 : a1, hi = cw1 < 32 ? b0 : b1;
        codes = csh ? __funnelshift_r(lo, hi, csh) : lo;
        dq = __half2float(__ushort_as_half(uint16_t(s0 >> ssh)));
    };
    for (int c = 0; c < NC; ++c) {
        const uint32_t* col = reinterpret_cast<const uint32_t*>(xq + size_t(c) * nq * kQ8Bytes);
        const UnitLaneOut out(s, c, lane);
        // two units per step, both loads first (a warp's last step may repeat its unit)
        for (int u = warp; u < U; u += 2 * nw) {
            const int u2 = u + nw < U ? u + nw : u;
            const uint32_t* p = col + size_t(u) * 34;
            const uint32_t* p2 = col + size_t(u2) * 34;
            const uint32_t w0 = __ldg(p + lane), v0 = __ldg(p2 + lane);
            const uint32_t w1 = lane < 2 ? __ldg(p + 32 + lane) : 0u;
            const uint32_t v1 = lane < 2 ? __ldg(p2 + 32 + lane) : 0u;
            uint32_t ca, cb2;
            float da, db;
            unit(w0, w1, ca, da);
            unit(v0, v1, cb2, db);
            int sa = __dp4a(int(ca), 0x01010101, 0), sb = __dp4a(int(cb2), 0x01010101, 0);
            sa += __shfl_xor_sync(0xffffffffu, sa, 1);
            sb += __shfl_xor_sync(0xffffffffu, sb, 1);
            sa += __shfl_xor_sync(0xffffffffu, sa, 2);
            sb += __shfl_xor_sync(0xffffffffu, sb, 2);
            sa += __shfl_xor_sync(0xffffffffu, sa, 4);
            sb += __shfl_xor_sync(0xffffffffu, sb, 4);
            out.put(u, lane, ca, da, sa);
            if (u2 != u) out.put(u2, lane, cb2, db, sb);
            if (sumq_out && g == 0) {
                sumq_out[size_t(c) * nq + 4 * u + slot] = sa;
                if (u2 != u) sumq_out[size_t(c) * nq + 4 * u2 + slot] = sb;
            }
        }
    }
}

// From fp32 values: q8_0 quantization straight into the unit layout (the same
// quantizer as the stand-alone kernel, hence bit-identical).  Optionally also
// writes the q8_0 blocks to xq_out (2-byte aligned) and the code sums to
// sumq_out.  `load(c, u)` gives this lane's values 4l..4l+3 of unit u of
// column c (lane l = tid & 31).
// kPair: the loader fetches a step's two units together, load.pair(c, u, u2,
// va, vb) (a polling loader then waits for both in one loop)
template <int NC, typename Loader, bool kPair = false>
__device__ __forceinline__ void stage_units_f32(Loader load, int K, UnitAct s, uint8_t* __restrict__ xq_out,
                                                int32_t* sumq_out, int tid, int nthr, int xq_ld = 0)
{
    // xq_out: block j of column c at block c*xq_ld + j (xq_ld = 0: K/32)
    const int lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    const int nq = K / kQK8, U = s.U;
    const int slot = lane >> 3, g = lane & 7;
    auto amax8 = [](float4 v) {  // max |x| over the lane's 4 values, then its block's 8 lanes
        float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        return fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    };
    // the lane's four codes, packed (code 4g in the low byte), and their sum
    auto codes4 = [](float4 v, const Q8Scale& sc, uint32_t& codes, int& qs) {
        int q0, q1, q2, q3;
        bool ok = q8_code_fast(v.x, sc, &q0);
        ok &= q8_code_fast(v.y, sc, &q1);
        ok &= q8_code_fast(v.z, sc, &q2);
        ok &= q8_code_fast(v.w, sc, &q3);
        if (!ok) {  // rare: the IEEE division decides
            q0 = q8_code_exact(v.x, sc.d);
            q1 = q8_code_exact(v.y, sc.d);
            q2 = q8_code_exact(v.z, sc.d);
            q3 = q8_code_exact(v.w, sc.d);
        }
        codes = (uint32_t(q0) & 0xffu) | ((uint32_t(q1) & 0xffu) << 8) | ((uint32_t(q2) & 0xffu) << 16) |
                (uint32_t(q3) << 24);
        qs = q0 + q1 + q2 + q3;
    };
    for (int c = 0; c < NC; ++c) {
        const UnitLaneOut out(s, c, lane);
        // two units per step, both loads first (a warp's last step may repeat its unit)
        for (int u = warp; u < U; u += 2 * nw) {
            const int u2 = u + nw < U ? u + nw : u;
            float4 va, vb;
            if constexpr (kPair) {
                load.pair(c, u, u2, va, vb);
            } else {
                va = load(c, u);
                vb = load(c, u2);
            }
            const float ma = amax8(va), mb = amax8(vb);
            const Q8Scale sa = q8_scale_of(ma), sb = q8_scale_of(mb);
            uint32_t ca, cb2;
            int qa, qb;
            codes4(va, sa, ca, qa);
            codes4(vb, sb, cb2, qb);
            qa += __shfl_xor_sync(0xffffffffu, qa, 1);
            qb += __shfl_xor_sync(0xffffffffu, qb, 1);
            qa += __shfl_xor_sync(0xffffffffu, qa, 2);
            qb += __shfl_xor_sync(0xffffffffu, qb, 2);
            qa += __shfl_xor_sync(0xffffffffu, qa, 4);
            qb += __shfl_xor_sync(0xffffffffu, qb, 4);
            const __half ha = __float2half_rn(sa.d), hb = __float2half_rn(sb.d);
            out.put(u, lane, ca, __half2float(ha), qa);
            if (u2 != u) out.put(u2, lane, cb2, __half2float(hb), qb);
            if (sumq_out && g == 0) {
                sumq_out[size_t(c) * nq + 4 * u + slot] = qa;
                if (u2 != u) sumq_out[size_t(c) * nq + 4 * u2 + slot] = qb;
            }
            if (xq_out) {
                auto put_q8 = [&](int uu, __half h, uint32_t cd) {
                    uint8_t* ob = xq_out + (size_t(c) * (xq_ld ? xq_ld : nq) + 4 * uu + slot) * kQ8Bytes;
                    if (g == 0) *reinterpret_cast<uint16_t*>(ob) = __half_as_ushort(h);
                    uint16_t* o = reinterpret_cast<uint16_t*>(ob + 2 + 4 * g);
                    o[0] = uint16_t(cd);
                    o[1] = uint16_t(cd >> 16);
                };
                put_q8(u, ha, ca);
                if (u2 != u) put_q8(u2, hb, cb2);
            }
        }
    }
}

// From fp32 x [NC][K] in global memory (one 16-byte load per lane and unit
// when x is 16-byte aligned).
template <int NC>
__device__ __forceinline__ void stage_units_x(const float* __restrict__ x, int K, UnitAct s,
                                              uint8_t* __restrict__ xq_out, int32_t* sumq_out, int tid, int nthr)
{
    const int lane = tid & 31;
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    auto load = [&](int c, int u) {
        const float* p = x + size_t(c) * K + size_t(u) * kUnitElems + 4 * lane;
        return vec ? __ldg(reinterpret_cast<const float4*>(p))
                   : make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
    };
    stage_units_f32<NC>(load, K, s, xq_out, sumq_out, tid, nthr);
}

// From fp32 x [NC][ld] in global memory, elements [k0, k0 + Kr) of every
// column (one part of a K split; k0 and Kr multiples of 256); xq_out (nullable)
// gets the q8_0 blocks of that range at their place in [NC][ld/32] blocks.
// (Not inlined, like stage_q8_range: code that only a K split runs stays out
// of the kernels' bodies.)
template <int NC>
__device__ __noinline__ void stage_units_x_range(const float* __restrict__ x, int ld, int k0, int Kr, UnitAct s,
                                                    uint8_t* __restrict__ xq_out, int tid, int nthr)
{
    const int lane = tid & 31;
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (ld & 3) == 0;
    if (vec) {
        // many columns of a long row: one thread per q8_0 block (its 32 values
        // loaded at once) takes fewer rounds than one warp per unit
        const int nqr = Kr / kQK8, total = NC * nqr, nq_all = ld / kQK8, j0 = k0 / kQK8;
        for (int t = tid; t < total; t += nthr) {
            const int c = t / nqr, J = t - c * nqr;
            const float4* p = reinterpret_cast<const float4*>(x + size_t(c) * ld + k0) + size_t(J) * 8;
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __ldg(p + i);
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
            const Q8Scale sc = q8_scale_of(m);
            int q[32];
            bool ok = true;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                ok &= q8_code_fast(v[i].x, sc, &q[4 * i]);
                ok &= q8_code_fast(v[i].y, sc, &q[4 * i + 1]);
                ok &= q8_code_fast(v[i].z, sc, &q[4 * i + 2]);
                ok &= q8_code_fast(v[i].w, sc, &q[4 * i + 3]);
            }
            if (!ok) {  // rare: the IEEE division decides
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    q[4 * i] = q8_code_exact(v[i].x, sc.d);
                    q[4 * i + 1] = q8_code_exact(v[i].y, sc.d);
                    q[4 * i + 2] = q8_code_exact(v[i].z, sc.d);
                    q[4 * i + 3] = q8_code_exact(v[i].w, sc.d);
                }
            }
            uint32_t cw[8];
            int sq = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                cw[i] = (uint32_t(q[4 * i]) & 0xffu) | ((uint32_t(q[4 * i + 1]) & 0xffu) << 8) |
                        ((uint32_t(q[4 * i + 2]) & 0xffu) << 16) | (uint32_t(q[4 * i + 3]) << 24);
                sq += q[4 * i] + q[4 * i + 1] + q[4 * i + 2] + q[4 * i + 3];
            }
            const __half hd = __float2half_rn(sc.d);
            put_block(s, c, J, cw, __half2float(hd), sq);
            if (xq_out) {
                uint16_t* o = reinterpret_cast<uint16_t*>(xq_out + (size_t(c) * nq_all + j0 + J) * kQ8Bytes);
                o[0] = __half_as_ushort(hd);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[1 + 2 * i] = uint16_t(cw[i]);
                    o[2 + 2 * i] = uint16_t(cw[i] >> 16);
                }
            }
        }
        return;
    }
    auto load = [&](int c, int u) {
        const float* p = x + size_t(c) * ld + k0 + size_t(u) * kUnitElems + 4 * lane;
        return vec ? __ldg(reinterpret_cast<const float4*>(p))
                   : make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
    };
    stage_units_f32<NC>(load, Kr, s, xq_out ? xq_out + size_t(k0 / kQK8) * kQ8Bytes : nullptr, nullptr, tid, nthr,
                        ld / kQK8);
}

// q8_0 blocks [j0, j0 + nqr) of each column of nq_all blocks (one part of a K split)
template <int NC>
__device__ __noinline__ void stage_q8_range(const uint8_t* __restrict__ xq, int nq_all, int j0, int nqr, UnitAct s,
                                               int tid, int nthr)
{
    if (reinterpret_cast<uintptr_t>(xq) & 3)
        stage_units_q8_by_block<NC>(xq, nq_all, j0, nqr, s, nullptr, tid, nthr);
    else
        stage_blocks_q8<NC>(xq, nq_all, j0, nqr, s, nullptr, tid, nthr);
}

// From fp32 values written earlier in the same launch as tagged records
// (value bits in the low half, the writer's tag in the high half; record
// c*ld + i holds element i of column c; rec 32-byte aligned, ld % 4 == 0).
// A lane loads its four records with two 16-byte loads and reads again until
// all four carry `tag`, bounded in time: one load both reads a value and
// proves it written.  False (on every lane of the warp) after a timeout or
// when another CTA raised the abort word; the staged values are then garbage.
template <int NC>
__device__ __forceinline__ bool stage_units_yrec(const uint64_t* __restrict__ rec, int ld, int K, UnitAct s,
                                                 uint8_t* __restrict__ xq_out, uint32_t tag,
                                                 const unsigned* abort_word, uint64_t limit_ns, int tid, int nthr)
{
    // a step's two units are read and polled together: one round trip per
    // poll for both, not one after the other
    struct PairLoader {
        const uint64_t* rec;
        int ld, lane;
        uint32_t tag;
        const unsigned* abort_word;
        uint64_t limit_ns;
        bool bad;
        __device__ __forceinline__ void pair(int c, int u, int u2, float4& va, float4& vb)
        {
            const uint64_t* p = rec + size_t(c) * ld + size_t(u) * kUnitElems + 4 * lane;
            const uint64_t* q = rec + size_t(c) * ld + size_t(u2) * kUnitElems + 4 * lane;
            uint64_t r[8];
            ld_tagged2(p, r[0], r[1]);
            ld_tagged2(p + 2, r[2], r[3]);
            ld_tagged2(q, r[4], r[5]);
            ld_tagged2(q + 2, r[6], r[7]);
            uint64_t t0 = 0;
            for (uint32_t it = 0; !bad; ++it) {
                bool ok = true;
#pragma unroll
                for (int i = 0; i < 8; ++i) ok &= uint32_t(r[i] >> 32) == tag;
                if (ok) break;
                if (it == 0)
                    t0 = global_timer_ns();
                else if ((it & 15u) == 0 && (ld_relaxed_u32(abort_word) != 0 || global_timer_ns() - t0 > limit_ns))
                    bad = true;
                if (uint32_t(r[0] >> 32) != tag || uint32_t(r[1] >> 32) != tag) ld_tagged2(p, r[0], r[1]);
                if (uint32_t(r[2] >> 32) != tag || uint32_t(r[3] >> 32) != tag) ld_tagged2(p + 2, r[2], r[3]);
                if (uint32_t(r[4] >> 32) != tag || uint32_t(r[5] >> 32) != tag) ld_tagged2(q, r[4], r[5]);
                if (uint32_t(r[6] >> 32) != tag || uint32_t(r[7] >> 32) != tag) ld_tagged2(q + 2, r[6], r[7]);
            }
            va = make_float4(__uint_as_float(uint32_t(r[0])), __uint_as_float(uint32_t(r[1])),
                             __uint_as_float(uint32_t(r[2])), __uint_as_float(uint32_t(r[3])));
            vb = make_float4(__uint_as_float(uint32_t(r[4])), __uint_as_float(uint32_t(r[5])),
                             __uint_as_float(uint32_t(r[6])), __uint_as_float(uint32_t(r[7])));
        }
    };
    PairLoader load{rec, ld, tid & 31, tag, abort_word, limit_ns, false};
    stage_units_f32<NC, PairLoader&, true>(load, K, s, xq_out, nullptr, tid, nthr);
    return !__any_sync(0xffffffffu, load.bad);
}

// 16 bytes from shared memory (the ring's stages are written by the bulk-copy
// engine and published by the mbarrier wait that precedes every read)
__device__ __forceinline__ void lds128(uint4& v, uint32_t addr)
{
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
}

// The unit's weight bytes: header and 64 quant bytes (four 16-byte words).
struct UnitW {
    uint4 h;                   // d, dmin, s[0..11]
    uint4 qa0, qb0, qa1, qb1;  // quant bytes 64h + 0, 16, 32, 48
};

// byte b of w as an exact float: 2^23 + b, read as float, minus 2^23
__device__ __forceinline__ float byte_as_float(uint32_t w, int b)
{
    return __int_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | uint32_t(b))) - 8388608.0f;
}

// Scales of the unit's four sub-blocks j = 4h..4h+3: sc[j] as integers, m[j]
// as floats, and the block's d and dmin.
//   h = 0: sc_j = s[j] & 63, m_j = s[j+4] & 63                     (j = 0..3)
//   h = 1: sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
//          m_j  = (s[j+4] >> 4) | (s[j] >> 6) << 4                  (j = 4..7)
struct UnitScales {
    int sc[4];  // 0..63
    float m[4];
    float d, dmin;
};

__device__ __forceinline__ UnitScales unit_scales(const uint4& hd, bool upper)
{
    UnitScales r;
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
    const uint32_t S0 = hd.y, S1 = hd.z, S2 = hd.w;
    const uint32_t mlo = upper ? 0x0f0f0f0fu : 0x3f3f3f3fu;
    const uint32_t mhi = upper ? 0x30303030u : 0u;
    const uint32_t sc = ((upper ? S2 : S0) & mlo) | ((S0 >> 2) & mhi);
    const uint32_t m = ((upper ? (S2 >> 4) : S1) & mlo) | ((S1 >> 2) & mhi);
#pragma unroll
    for (int b = 0; b < 4; ++b) r.sc[b] = int(__byte_perm(sc, 0u, 0x4440u | uint32_t(b)));
#pragma unroll
    for (int b = 0; b < 4; ++b) r.m[b] = byte_as_float(m, b);
    r.d = dd.x;
    r.dmin = dd.y;
    return r;
}

__device__ __forceinline__ int dot16_lo(const uint4& w, const uint4& a, int acc)
{
    const uint32_t lo = 0x0f0f0f0fu;
    acc = dp4a_us(w.x & lo, a.x, acc);
    acc = dp4a_us(w.y & lo, a.y, acc);
    acc = dp4a_us(w.z & lo, a.z, acc);
    acc = dp4a_us(w.w & lo, a.w, acc);
    return acc;
}

__device__ __forceinline__ int dot16_hi(const uint4& w, const uint4& a, int acc)
{
    const uint32_t hi = 0xf0f0f0f0u;
    acc = dp4a_us(w.x & hi, a.x, acc);
    acc = dp4a_us(w.y & hi, a.y, acc);
    acc = dp4a_us(w.z & hi, a.z, acc);
    acc = dp4a_us(w.w & hi, a.w, acc);
    return acc;
}

// Exact int32 sums of the unit's four sub-blocks with the activation codes
// A[0..7] (unit layout): s[0], s[2] plain, s[1], s[3] times 16 (high
// nibbles used in place).
__device__ __forceinline__ void unit_dot(const UnitW& w, const uint4 (&A)[8], int s[4])
{
    s[0] = dot16_lo(w.qb0, A[1], dot16_lo(w.qa0, A[0], 0));
    s[1] = dot16_hi(w.qb0, A[3], dot16_hi(w.qa0, A[2], 0));
    s[2] = dot16_lo(w.qb1, A[5], dot16_lo(w.qa1, A[4], 0));
    s[3] = dot16_hi(w.qb1, A[7], dot16_hi(w.qa1, A[6], 0));
}

// acc + the unit's contribution for one column:
// sum_j dq_j*(d*sc_j*s_j - dmin*m_j*sumq_j)
//   = d * sum_j dq_j*(sc_j*s_j) - dmin * sum_j m_j*(dq_j*sumq_j)
__device__ __forceinline__ float unit_column(const UnitW& w, const UnitScales& k, const uint4 (&A)[8],
                                             const float4& dq, const float4& dqsq, float acc)
{
    int s[4];
    unit_dot(w, A, s);
    // sc_j * s_j in int32 (|s_j| < 2^20 with the high nibbles in place, sc_j < 64);
    // the high nibbles' factor 16 comes off dq_j (exact: a power of two)
    float t = dq.x * float(k.sc[0] * s[0]);
    t = fmaf(dq.y * 0.0625f, float(k.sc[1] * s[1]), t);
    t = fmaf(dq.z, float(k.sc[2] * s[2]), t);
    t = fmaf(dq.w * 0.0625f, float(k.sc[3] * s[3]), t);
    float u = k.m[0] * dqsq.x;
    u = fmaf(k.m[1], dqsq.y, u);
    u = fmaf(k.m[2], dqsq.z, u);
    u = fmaf(k.m[3], dqsq.w, u);
    acc = fmaf(k.d, t, acc);
    return fmaf(-k.dmin, u, acc);
}

// ---------------------------------------------------------------------------
// Weight formats of the ring consumer.  A format gives, for the 128-weight
// unit u of a row: the row's bytes per unit, where the unit's bytes sit, how a
// lane loads them from a ring stage, what it derives once per unit (scales),
// and the unit's contribution for one activation column (unit layout above).
// ---------------------------------------------------------------------------

// q4_K: half a super-block, 72 bytes of row per unit
struct FmtQ4K {
    using W = UnitW;
    using S = UnitScales;
    struct Off {
        uint32_t h, q;
        bool upper;
    };
    __device__ __forceinline__ static uint32_t row_bytes(int U) { return uint32_t(U / 2) * kQ4KBytes; }
    __device__ __forceinline__ static Off offsets(int u)
    {
        const uint32_t h = uint32_t(u >> 1) * kQ4KBytes;
        return Off{h, h + 16 + 64 * uint32_t(u & 1), (u & 1) != 0};
    }
    __device__ __forceinline__ static void load(const uint8_t* row, const Off& o, W& w)
    {
        // explicit shared-memory loads on a 32-bit address: the ring is shared
        // memory, and the generic pointer's conversion stays out of the row loop
        const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(row));
        lds128(w.h, a + o.h);
        lds128(w.qa0, a + o.q);
        lds128(w.qb0, a + o.q + 16);
        lds128(w.qa1, a + o.q + 32);
        lds128(w.qb1, a + o.q + 48);
    }
    __device__ __forceinline__ static S prep(const W& w, const Off& o) { return unit_scales(w.h, o.upper); }
    __device__ __forceinline__ static float column(const W& w, const S& k, const uint4 (&A)[8], const float4& dq,
                                                   const float4& dqsq)
    {
        return unit_column(w, k, A, dq, dqsq, 0.0f);
    }
};

__device__ __forceinline__ float f16_bits_to_float(uint32_t bits)
{
    return __half2float(__ushort_as_half(uint16_t(bits)));
}

// q4_0 weights ("32 weights in 18 bytes: f16 d, then 16 bytes; byte i holds
// weight i in its low nibble and weight i+16 in its high nibble; w = d(q-8)"):
// a unit is 4 blocks, 72 bytes at byte 72u of the row (8-byte aligned: rows
// are 16-byte aligned when K % 256 == 0).  Block j's scale and quants sit at
// bytes 18j and 18j+2: words 0, 4(hi), 9, 13(hi) and quants from word
// offsets 0.5, 5, 9.5, 14 (a half-word offset is undone by a funnel shift).
// Low nibbles meet codes 0..15 of the block (plane 2j), high nibbles codes
// 16..31 (plane 2j+1); the -8 comes off through the block's code sum:
// d*(dq*sum(q*a) - 8*dq*sum(a)).
struct FmtQ4_0 {
    struct W {
        uint32_t w[18];
    };
    struct S {
        float d[4];
    };
    struct Off {
        uint32_t o;
    };
    __device__ __forceinline__ static uint32_t row_bytes(int U) { return uint32_t(U) * 72; }
    __device__ __forceinline__ static Off offsets(int u) { return Off{uint32_t(u) * 72}; }
    __device__ __forceinline__ static void load(const uint8_t* row, const Off& o, W& w)
    {
        const uint2* p = reinterpret_cast<const uint2*>(row + o.o);
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            const uint2 v = p[k];
            w.w[2 * k] = v.x;
            w.w[2 * k + 1] = v.y;
        }
    }
    __device__ __forceinline__ static S prep(const W& w, const Off&)
    {
        return S{{f16_bits_to_float(w.w[0]), f16_bits_to_float(w.w[4] >> 16), f16_bits_to_float(w.w[9]),
                  f16_bits_to_float(w.w[13] >> 16)}};
    }
    // sum over the block's 32 weights of q * code, q in 0..15
    __device__ __forceinline__ static int block_dot(uint32_t q0, uint32_t q1, uint32_t q2, uint32_t q3, const uint4& lo,
                                                    const uint4& hi)
    {
        const uint32_t m = 0x0f0f0f0fu;
        int s = dp4a_us(q0 & m, lo.x, 0);
        s = dp4a_us(q1 & m, lo.y, s);
        s = dp4a_us(q2 & m, lo.z, s);
        s = dp4a_us(q3 & m, lo.w, s);
        s = dp4a_us((q0 >> 4) & m, hi.x, s);
        s = dp4a_us((q1 >> 4) & m, hi.y, s);
        s = dp4a_us((q2 >> 4) & m, hi.z, s);
        return dp4a_us((q3 >> 4) & m, hi.w, s);
    }
    __device__ __forceinline__ static float column(const W& w, const S& k, const uint4 (&A)[8], const float4& dq,
                                                   const float4& dqsq)
    {
        const uint32_t* v = w.w;
        const int s0 = block_dot(__funnelshift_r(v[0], v[1], 16), __funnelshift_r(v[1], v[2], 16),
                                 __funnelshift_r(v[2], v[3], 16), __funnelshift_r(v[3], v[4], 16), A[0], A[1]);
        const int s1 = block_dot(v[5], v[6], v[7], v[8], A[2], A[3]);
        const int s2 = block_dot(__funnelshift_r(v[9], v[10], 16), __funnelshift_r(v[10], v[11], 16),
                                 __funnelshift_r(v[11], v[12], 16), __funnelshift_r(v[12], v[13], 16), A[4], A[5]);
        const int s3 = block_dot(v[14], v[15], v[16], v[17], A[6], A[7]);
        float t = k.d[0] * fmaf(dq.x, float(s0), -8.0f * dqsq.x);
        t = fmaf(k.d[1], fmaf(dq.y, float(s1), -8.0f * dqsq.y), t);
        t = fmaf(k.d[2], fmaf(dq.z, float(s2), -8.0f * dqsq.z), t);
        return fmaf(k.d[3], fmaf(dq.w, float(s3), -8.0f * dqsq.w), t);
    }
};

// q8_0 weights (the activation's own block format, w = d*q): a unit is 4
// blocks, 136 bytes at byte 136u of the row (8-byte aligned).  Block j's scale
// and quants sit at bytes 34j and 34j+2: scale words 0, 8(hi), 17, 25(hi) and
// quants from word offsets 0.5, 9, 17.5, 26.
struct FmtQ8_0 {
    struct W {
        uint32_t w[34];
    };
    struct S {
        float d[4];
    };
    struct Off {
        uint32_t o;
    };
    __device__ __forceinline__ static uint32_t row_bytes(int U) { return uint32_t(U) * 136; }
    __device__ __forceinline__ static Off offsets(int u) { return Off{uint32_t(u) * 136}; }
    __device__ __forceinline__ static void load(const uint8_t* row, const Off& o, W& w)
    {
        const uint2* p = reinterpret_cast<const uint2*>(row + o.o);
#pragma unroll
        for (int k = 0; k < 17; ++k) {
            const uint2 v = p[k];
            w.w[2 * k] = v.x;
            w.w[2 * k + 1] = v.y;
        }
    }
    __device__ __forceinline__ static S prep(const W& w, const Off&)
    {
        return S{{f16_bits_to_float(w.w[0]), f16_bits_to_float(w.w[8] >> 16), f16_bits_to_float(w.w[17]),
                  f16_bits_to_float(w.w[25] >> 16)}};
    }
    // sum over the block's 32 weights of q * code, q signed; words at v[0..8]
    // with half-word offset `shift` (0 or 16)
    template <int kShift>
    __device__ __forceinline__ static int block_dot(const uint32_t* v, const uint4& lo, const uint4& hi)
    {
        auto word = [&](int i) -> int {
            return kShift ? int(__funnelshift_r(v[i], v[i + 1], kShift)) : int(v[i]);
        };
        int s = __dp4a(word(0), int(lo.x), 0);
        s = __dp4a(word(1), int(lo.y), s);
        s = __dp4a(word(2), int(lo.z), s);
        s = __dp4a(word(3), int(lo.w), s);
        s = __dp4a(word(4), int(hi.x), s);
        s = __dp4a(word(5), int(hi.y), s);
        s = __dp4a(word(6), int(hi.z), s);
        return __dp4a(word(7), int(hi.w), s);
    }
    __device__ __forceinline__ static float column(const W& w, const S& k, const uint4 (&A)[8], const float4& dq,
                                                   const float4&)
    {
        const int s0 = block_dot<16>(w.w + 0, A[0], A[1]);
        const int s1 = block_dot<0>(w.w + 9, A[2], A[3]);
        const int s2 = block_dot<16>(w.w + 17, A[4], A[5]);
        const int s3 = block_dot<0>(w.w + 26, A[6], A[7]);
        float t = k.d[0] * (dq.x * float(s0));
        t = fmaf(k.d[1], dq.y * float(s1), t);
        t = fmaf(k.d[2], dq.z * float(s2), t);
        return fmaf(k.d[3], dq.w * float(s3), t);
    }
};

}  // namespace mq
