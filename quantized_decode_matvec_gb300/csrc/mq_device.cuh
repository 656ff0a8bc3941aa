// mq_device.cuh -- device building blocks shared by the libmq kernels.
//
// q4_K x q8_0 decode matvec ("07 . R3 -- Small-model per-token overhead",
// section 1: MMVQ, dp4a over q4_K weights and q8_0 activations).
//
// Work unit: a "chunk" = 32 bytes of q4_K quants = 64 weights = two q8_0
// blocks.  Chunk ch of a row covers activation elements [64ch, 64ch+64):
// super-block ch/4, quant bytes 32*(ch%4) .. +32, sub-blocks j0 = 2*(ch%4)
// (low nibbles) and j1 = j0+1 (high nibbles).  A lane streams one chunk with
// three 16-byte loads (the super-block header and the two quant halves).
//
// The q8_0 activation is staged once per CTA in shared memory, re-laid out
// so that 8 consecutive lanes reading consecutive chunks touch 128
// consecutive bytes (no bank conflicts):
//   plane p (0..3) of column c: uint4 per chunk = elements 16p..16p+15 of
//     the chunk (p = 0,1: block j0 halves; p = 2,3: block j1 halves)
//   scale of column c: float4 per chunk = {dq_j0, dq_j1, dq_j0*sumq_j0,
//     dq_j1*sumq_j1} with dq the stored binary16 scale as fp32.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace mq {

constexpr int kQK = 256;         // weights per q4_K super-block
constexpr int kQ4KBytes = 144;   // bytes per q4_K super-block
constexpr int kQK8 = 32;         // values per q8_0 block
constexpr int kQ8Bytes = 34;     // bytes per q8_0 block
constexpr int kChunkElems = 64;  // weights per chunk

// ---------------------------------------------------------------------------
// loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg16(const uint8_t* p)
{
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------------------
// q8_0 quantization of one 32-value block held one value per lane.
// amax = max |x| over the warp: for non-negative floats the bit pattern
// orders like the value, so an unsigned max-reduction is exact and
// order-free.  d = amax/127 and x/d by IEEE division, round half away from
// zero, clamp to +-127.  Returns this lane's code; *d_out is the fp32 d.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int q8_quantize_lane(float x, float* d_out)
{
    const unsigned ab = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(x)));
    const float amax = __uint_as_float(ab);
    const float d = __fdiv_rn(amax, 127.0f);
    int q = 0;
    if (d != 0.0f) {
        float r = roundf(__fdiv_rn(x, d));
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        q = static_cast<int>(r);
    }
    *d_out = d;
    return q;
}

// ---------------------------------------------------------------------------
// Activation staging.  Layout in shared memory (see the file header):
//   planes: NC*4*C uint4, plane (c, p) starts at (c*4 + p)*C
//   scales: NC*C float4, column c starts at c*C
// ---------------------------------------------------------------------------
struct ActSmem {
    uint4* planes;
    float4* scales;
    int C;  // chunks per row = K/64
};

// From q8_0 blocks in global memory (34-byte blocks, 2-byte aligned).
// sumq_out (nullable, test export): int32 [NC][K/32] block sums of the codes.
template <int NC>
__device__ __forceinline__ void stage_q8_global(const uint8_t* __restrict__ xq, int K, ActSmem s,
                                                int32_t* sumq_out)
{
    const int nq = K / kQK8;
    for (int t = threadIdx.x; t < NC * nq; t += blockDim.x) {
        const int c = t / nq, J = t - c * nq;
        const uint16_t* h = reinterpret_cast<const uint16_t*>(xq + (size_t(c) * nq + J) * kQ8Bytes);
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
        const int ch = J >> 1, half = J & 1;
        uint4* P = s.planes + size_t(c * 4 + 2 * half) * s.C + ch;
        P[0] = make_uint4(w[0], w[1], w[2], w[3]);
        P[s.C] = make_uint4(w[4], w[5], w[6], w[7]);
        float* S = reinterpret_cast<float*>(s.scales + size_t(c) * s.C + ch);
        S[half] = dq;
        S[2 + half] = dq * float(sq);
        if (sumq_out) sumq_out[size_t(c) * nq + J] = sq;
    }
}

// From fp32 x in global memory: quantize to q8_0 (bit-identical to the
// stand-alone quantizer) straight into shared memory.  One warp per block;
// each warp first issues the loads of up to 8 blocks, then quantizes them,
// so the L2 latency is paid once per 8 blocks.  xq_out (nullable) receives
// the 34-byte blocks.
template <int NC>
__device__ __forceinline__ void stage_x_quantize(const float* __restrict__ x, int K, ActSmem s,
                                                 uint8_t* __restrict__ xq_out)
{
    constexpr int B = 8;
    const int nq = K / kQK8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int total = NC * nq;
    for (int t0 = warp * B; t0 < total; t0 += nw * B) {
        float v[B];
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
        for (int b = 0; b < B; ++b) {
            const int t = t0 + b;
            if (t >= total) break;  // warp-uniform
            const int c = t / nq, J = t - c * nq;
            float d;
            const int q = q8_quantize_lane(v[b], &d);
            const __half dh = __float2half_rn(d);
            const float dq = __half2float(dh);
            const int sq = __reduce_add_sync(0xffffffffu, q);
            const int ch = J >> 1, half = J & 1;
            uint8_t* P = reinterpret_cast<uint8_t*>(s.planes + size_t(c * 4 + 2 * half + (lane >> 4)) * s.C + ch);
            P[lane & 15] = uint8_t(int8_t(q));
            if (lane == 0) {
                float* S = reinterpret_cast<float*>(s.scales + size_t(c) * s.C + ch);
                S[half] = dq;
                S[2 + half] = dq * float(sq);
            }
            if (xq_out) {
                uint8_t* ob = xq_out + (size_t(c) * nq + J) * kQ8Bytes;
                if (lane == 0) *reinterpret_cast<uint16_t*>(ob) = __half_as_ushort(dh);
                ob[2 + lane] = uint8_t(int8_t(q));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// q4_K chunk: the super-block header (d, dmin, 12 scale bytes) and 32 quant
// bytes.  c4 = chunk index within the super-block (0..3).
// ---------------------------------------------------------------------------
struct Chunk {
    uint4 h;  // bytes 0..15 of the super-block
    uint4 a;  // quant bytes 32*c4 .. +16  (elements 0..15 of j0 low / j1 high)
    uint4 b;  // quant bytes 32*c4+16 .. +16 (elements 16..31)
};

__device__ __forceinline__ void load_chunk(Chunk& k, const uint8_t* sb, int c4)
{
    k.h = ldg16(sb);
    k.a = ldg16(sb + 16 + 32 * c4);
    k.b = ldg16(sb + 32 + 32 * c4);
}

// Float scales of the chunk's two sub-blocks: fd = d*sc, fm = dmin*m.
// Scale bytes s[0..11] are h.y (s0..s3), h.z (s4..s7), h.w (s8..s11).
// j < 4: sc = s[j] & 63, m = s[j+4] & 63.
// j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4.
__device__ __forceinline__ void chunk_scales(const uint4& h, int c4, float& fd0, float& fd1, float& fm0,
                                             float& fm1)
{
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
    uint32_t scw, mw;
    if (c4 < 2) {
        scw = h.y & 0x3f3f3f3fu;
        mw = h.z & 0x3f3f3f3fu;
    } else {
        scw = (h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u);
        mw = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
    }
    const int sh = (c4 & 1) * 16;
    fd0 = dd.x * float((scw >> sh) & 0xffu);
    fd1 = dd.x * float((scw >> (sh + 8)) & 0xffu);
    fm0 = dd.y * float((mw >> sh) & 0xffu);
    fm1 = dd.y * float((mw >> (sh + 8)) & 0xffu);
}

// Exact int32 dot products of the chunk's quants with the activation codes:
// s0 = sum over the 32 elements of block j0 of q4 * q8, s1 likewise for j1.
// p0..p3 are the four activation planes of this chunk.
__device__ __forceinline__ void chunk_dot(const Chunk& k, const uint4& p0, const uint4& p1, const uint4& p2,
                                          const uint4& p3, int& s0, int& s1)
{
    const uint32_t m4 = 0x0f0f0f0fu;
    int a = 0, b = 0;
    a = __dp4a(int(k.a.x & m4), int(p0.x), a);
    a = __dp4a(int(k.a.y & m4), int(p0.y), a);
    a = __dp4a(int(k.a.z & m4), int(p0.z), a);
    a = __dp4a(int(k.a.w & m4), int(p0.w), a);
    a = __dp4a(int(k.b.x & m4), int(p1.x), a);
    a = __dp4a(int(k.b.y & m4), int(p1.y), a);
    a = __dp4a(int(k.b.z & m4), int(p1.z), a);
    a = __dp4a(int(k.b.w & m4), int(p1.w), a);
    b = __dp4a(int((k.a.x >> 4) & m4), int(p2.x), b);
    b = __dp4a(int((k.a.y >> 4) & m4), int(p2.y), b);
    b = __dp4a(int((k.a.z >> 4) & m4), int(p2.z), b);
    b = __dp4a(int((k.a.w >> 4) & m4), int(p2.w), b);
    b = __dp4a(int((k.b.x >> 4) & m4), int(p3.x), b);
    b = __dp4a(int((k.b.y >> 4) & m4), int(p3.y), b);
    b = __dp4a(int((k.b.z >> 4) & m4), int(p3.z), b);
    b = __dp4a(int((k.b.w >> 4) & m4), int(p3.w), b);
    s0 = a;
    s1 = b;
}

// acc[c] += this chunk's contribution for every column:
// dq_j0*(d*sc_j0*s0 - dmin*m_j0*sumq_j0) + (same for j1).
template <int NC>
__device__ __forceinline__ void chunk_accumulate(const Chunk& k, int c4, int ch, const ActSmem& s, float acc[NC])
{
    float fd0, fd1, fm0, fm1;
    chunk_scales(k.h, c4, fd0, fd1, fm0, fm1);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4* P = s.planes + size_t(c * 4) * s.C + ch;
        const uint4 p0 = P[0], p1 = P[s.C], p2 = P[2 * s.C], p3 = P[3 * s.C];
        const float4 sc = s.scales[size_t(c) * s.C + ch];
        int s0, s1;
        chunk_dot(k, p0, p1, p2, p3, s0, s1);
        float t = acc[c];
        t = fmaf(fd0, sc.x * float(s0), t);
        t = fmaf(fd1, sc.y * float(s1), t);
        t = fmaf(-fm0, sc.z, t);
        t = fmaf(-fm1, sc.w, t);
        acc[c] = t;
    }
}

}  // namespace mq
