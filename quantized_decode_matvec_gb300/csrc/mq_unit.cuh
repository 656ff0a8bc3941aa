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

namespace mq {

constexpr int kUnitElems = 128;

struct UnitAct {
    uint4* planes;
    float4* scales;
    int U;  // units per row = K/128
};

// From q8_0 blocks in global memory (34-byte blocks, 2-byte aligned), threads
// tid = 0..nthr-1.  sumq_out (nullable, test export): int32 [NC][K/32].
// kL2Only: read through L2 only (ld.global.cg), for blocks written earlier in
// the same kernel by other CTAs (the read-only path may hold stale lines).
template <int NC, bool kL2Only = false>
__device__ __forceinline__ void stage_units_q8(const uint8_t* __restrict__ xq, int K, UnitAct s, int32_t* sumq_out,
                                               int tid, int nthr)
{
    const int nq = K / kQK8;
    for (int t = tid; t < NC * nq; t += nthr) {
        const int c = t / nq, J = t - c * nq;
        const uint16_t* h = reinterpret_cast<const uint16_t*>(xq + (size_t(c) * nq + J) * kQ8Bytes);
        uint16_t v[17];
#pragma unroll
        for (int k = 0; k < 17; ++k) v[k] = kL2Only ? __ldcg(h + k) : __ldg(h + k);
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

// From fp32 x: q8_0 quantization (the same warp-level quantizer halves as the
// stand-alone kernel, hence bit-identical) straight into the unit layout.
// Whole warps tid = 0..nthr-1.  Each warp takes B blocks at a time and runs
// their quantizations in lockstep (independent chains), since a single
// block's amax -> divide -> round -> sum chain is mostly latency.
template <int NC>
__device__ __forceinline__ void stage_units_x(const float* __restrict__ x, int K, UnitAct s,
                                              uint8_t* __restrict__ xq_out, int32_t* sumq_out, int tid, int nthr)
{
    constexpr int B = 8;
    const int nq = K / kQK8;
    const int lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
    const int total = NC * nq;
    for (int t0 = warp * B; t0 < total; t0 += nw * B) {
        float v[B], d[B];
        int q[B], sq[B];
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int t = t0 + b;
            v[b] = 0.0f;
            if (t < total) {
                const int c = t / nq, J = t - c * nq;
                v[b] = __ldg(x + size_t(c) * K + size_t(J) * kQK8 + lane);
            }
        }
#pragma unroll
        for (int b = 0; b < B; ++b) d[b] = q8_block_scale(v[b]);
#pragma unroll
        for (int b = 0; b < B; ++b) q[b] = q8_code(v[b], d[b]);
#pragma unroll
        for (int b = 0; b < B; ++b) sq[b] = __reduce_add_sync(0xffffffffu, q[b]);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int t = t0 + b;
            if (t < total) {
                const int c = t / nq, J = t - c * nq;
                const __half dh = __float2half_rn(d[b]);
                const float dq = __half2float(dh);
                const int u = J >> 2, slot = J & 3;
                uint8_t* P = reinterpret_cast<uint8_t*>(s.planes + size_t(c * 8 + 2 * slot + (lane >> 4)) * s.U + u);
                P[lane & 15] = uint8_t(int8_t(q[b]));
                if (lane == 0) {
                    float* S = reinterpret_cast<float*>(s.scales + (size_t(c) * s.U + u) * 2);
                    S[slot] = dq;
                    S[4 + slot] = dq * float(sq[b]);
                    if (sumq_out) sumq_out[size_t(c) * nq + J] = sq[b];
                }
                if (xq_out) {
                    uint8_t* ob = xq_out + (size_t(c) * nq + J) * kQ8Bytes;
                    if (lane == 0) *reinterpret_cast<uint16_t*>(ob) = __half_as_ushort(dh);
                    ob[2 + lane] = uint8_t(int8_t(q[b]));
                }
            }
        }
    }
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

// Scales of the unit's four sub-blocks j = 4h..4h+3 as floats: sc[j], m[j]
// (sc[1], sc[3] pre-divided by 16, exact, to match the in-place high nibbles
// of unit_dot), and the block's d and dmin.
//   h = 0: sc_j = s[j] & 63, m_j = s[j+4] & 63                     (j = 0..3)
//   h = 1: sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
//          m_j  = (s[j+4] >> 4) | (s[j] >> 6) << 4                  (j = 4..7)
struct UnitScales {
    float sc[4], m[4];
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
    r.sc[0] = byte_as_float(sc, 0);
    r.sc[1] = 0.0625f * byte_as_float(sc, 1);
    r.sc[2] = byte_as_float(sc, 2);
    r.sc[3] = 0.0625f * byte_as_float(sc, 3);
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
//   = d * sum_j sc_j*(dq_j*s_j) - dmin * sum_j m_j*(dq_j*sumq_j)
__device__ __forceinline__ float unit_column(const UnitW& w, const UnitScales& k, const uint4 (&A)[8],
                                             const float4& dq, const float4& dqsq, float acc)
{
    int s[4];
    unit_dot(w, A, s);
    float t = k.sc[0] * (dq.x * float(s[0]));
    t = fmaf(k.sc[1], dq.y * float(s[1]), t);
    t = fmaf(k.sc[2], dq.z * float(s[2]), t);
    t = fmaf(k.sc[3], dq.w * float(s[3]), t);
    float u = k.m[0] * dqsq.x;
    u = fmaf(k.m[1], dqsq.y, u);
    u = fmaf(k.m[2], dqsq.z, u);
    u = fmaf(k.m[3], dqsq.w, u);
    acc = fmaf(k.d, t, acc);
    return fmaf(-k.dmin, u, acc);
}

}  // namespace mq
