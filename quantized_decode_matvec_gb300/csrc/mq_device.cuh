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
// q8_0 quantization.  The definition: amax = max |x| over the 32 values,
// d = amax/127 and code = round_half_away(x/d) clamped to +-127, both
// divisions correctly rounded fp32.  The common path computes exactly the
// same numbers without an IEEE division:
//  * d: Markstein's correction step (P. Markstein, IBM J. Res. Dev. 34(1),
//    1990; the division chapter of Muller et al., "Handbook of Floating-Point
//    Arithmetic").  With y = RN(1/127) and q0 = RN(amax*y) within one ulp of
//    amax/127, the residual r = amax - 127*q0 is exact in one FMA, and
//    RN(q0 + r*y) = RN(amax/127) as long as nothing under- or overflows;
//    outside [2^-100, 2^100] the division itself is used.
//  * code: the quotient matters only through the integer it rounds to.  The
//    approximate quotient x*rcp(d) is within 2^-22 relative (2^-15 absolute,
//    since |x/d| <= 127.0001) of x/d, and RN(x/d) within 2^-17 of it, so
//    both round to the same integer unless the fractional part lies within
//    2^-14 of 1/2; there (about one value in 8000) the exact division is
//    taken.
// Both were checked bit for bit against the IEEE divisions on a GB300: the
// scale for every finite non-negative float, the code for every x of a dozen
// scales spanning 1e-20 .. 3e15 and for random and near-tie samples of 200000
// more.  For non-negative floats the bit pattern orders like the value, so
// amax is an unsigned max over the bits (exact, order-free).
// ---------------------------------------------------------------------------
constexpr float kInv127 = 1.0f / 127.0f;  // RN(1/127), folded by the compiler

__device__ __forceinline__ float rcp_approx(float d)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(d));
    return y;
}

struct Q8Scale {
    float d;     // fp32 scale amax/127
    float rd;    // approximate 1/d (fast path only)
    bool exact;  // take the IEEE division for every code of the block
};

__device__ __forceinline__ Q8Scale q8_scale_of(float amax)
{
    Q8Scale s;
    if (amax >= 0x1p-100f && amax <= 0x1p+100f) {
        const float q0 = amax * kInv127;
        s.d = fmaf(fmaf(-q0, 127.0f, amax), kInv127, q0);
        s.rd = rcp_approx(s.d);
        s.exact = false;
    } else {  // zero, tiny, huge or not finite
        s.d = __fdiv_rn(amax, 127.0f);
        s.rd = 0.0f;
        s.exact = true;
    }
    return s;
}

__device__ __forceinline__ int q8_code_exact(float x, float d)
{
    if (d == 0.0f) return 0;
    const float r = roundf(__fdiv_rn(x, d));
    return static_cast<int>(fminf(fmaxf(r, -127.0f), 127.0f));
}

// The code from the approximate quotient; false where it cannot be trusted
// (then the caller takes q8_code_exact).  Away from a tie, adding +-1/2 and
// truncating rounds half away from zero exactly (the sum cannot land on an
// integer), and |x/d| <= 127.0001 keeps the result within +-127.
__device__ __forceinline__ bool q8_code_fast(float x, const Q8Scale& s, int* q)
{
    const float qa = x * s.rd;
    const float a = fabsf(qa);
    *q = __float2int_rz(qa + copysignf(0.5f, qa));
    return !s.exact && fabsf(a - floorf(a) - 0.5f) > 0x1p-14f;
}

// One 32-value block held one value per lane of the warp: returns this
// lane's code; *d_out is the fp32 d.
__device__ __forceinline__ int q8_quantize_lane(float x, float* d_out)
{
    const unsigned ab = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(x)));
    const Q8Scale s = q8_scale_of(__uint_as_float(ab));
    *d_out = s.d;
    int q;
    if (!q8_code_fast(x, s, &q)) q = q8_code_exact(x, s.d);
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

// From q8_0 blocks in global memory (34-byte blocks, 2-byte aligned), by
// threads tid = 0..nthr-1.  sumq_out (nullable, test export): int32
// [NC][K/32] block sums of the codes.
template <int NC>
__device__ __forceinline__ void stage_q8_global(const uint8_t* __restrict__ xq, int K, ActSmem s,
                                                int32_t* sumq_out, int tid, int nthr)
{
    const int nq = K / kQK8;
    for (int t = tid; t < NC * nq; t += nthr) {
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
// the 34-byte blocks.  Run by whole warps tid = 0..nthr-1 (nthr % 32 == 0).
template <int NC>
__device__ __forceinline__ void stage_x_quantize(const float* __restrict__ x, int K, ActSmem s,
                                                 uint8_t* __restrict__ xq_out, int tid, int nthr)
{
    constexpr int B = 8;
    const int nq = K / kQK8;
    const int lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
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
// Branch-free (c4 differs across the lanes of a warp): both forms are
// computed and one is selected.  fd1 comes out divided by 16 (exact, a power
// of two) to match chunk_dot's s1x16.
__device__ __forceinline__ void chunk_scales(const uint4& h, int c4, float& fd0, float& fd1, float& fm0,
                                             float& fm1)
{
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
    const uint32_t sc_lo = h.y & 0x3f3f3f3fu;
    const uint32_t m_lo = h.z & 0x3f3f3f3fu;
    const uint32_t sc_hi = (h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
    const bool upper = c4 >= 2;
    const uint32_t scw = upper ? sc_hi : sc_lo;
    const uint32_t mw = upper ? m_hi : m_lo;
    // bytes j0 and j1 of the selected words (j0 = 2*(c4 & 1) within the word)
    const uint32_t sel = (c4 & 1) ? 0x4442u : 0x4440u;  // byte_perm: byte 2 or 0 into byte 0, zero elsewhere
    const uint32_t sel1 = (c4 & 1) ? 0x4443u : 0x4441u;
    fd0 = dd.x * float(__byte_perm(scw, 0u, sel));
    fd1 = (dd.x * 0.0625f) * float(__byte_perm(scw, 0u, sel1));
    fm0 = dd.y * float(__byte_perm(mw, 0u, sel));
    fm1 = dd.y * float(__byte_perm(mw, 0u, sel1));
}

// unsigned bytes of a times signed bytes of b, summed into c (PTX dp4a.u32.s32)
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Exact int32 dot products of the chunk's quants with the activation codes:
// s0 = sum over the 32 elements of block j0 of q4 * q8 (low nibbles), and
// s1x16 = 16 * (the same for j1): the high nibbles are used in place, masked
// but not shifted, as unsigned bytes (16*q), so s1 = s1x16 / 16 exactly.
// Two accumulators per block keep the dependent dp4a chains short.
// p0..p3 are the four activation planes of this chunk.
__device__ __forceinline__ void chunk_dot(const Chunk& k, const uint4& p0, const uint4& p1, const uint4& p2,
                                          const uint4& p3, int& s0, int& s1x16)
{
    const uint32_t lo = 0x0f0f0f0fu, hi = 0xf0f0f0f0u;
    int a0 = 0, a1 = 0, b0 = 0, b1 = 0;
    a0 = dp4a_us(k.a.x & lo, p0.x, a0);
    a1 = dp4a_us(k.b.x & lo, p1.x, a1);
    b0 = dp4a_us(k.a.x & hi, p2.x, b0);
    b1 = dp4a_us(k.b.x & hi, p3.x, b1);
    a0 = dp4a_us(k.a.y & lo, p0.y, a0);
    a1 = dp4a_us(k.b.y & lo, p1.y, a1);
    b0 = dp4a_us(k.a.y & hi, p2.y, b0);
    b1 = dp4a_us(k.b.y & hi, p3.y, b1);
    a0 = dp4a_us(k.a.z & lo, p0.z, a0);
    a1 = dp4a_us(k.b.z & lo, p1.z, a1);
    b0 = dp4a_us(k.a.z & hi, p2.z, b0);
    b1 = dp4a_us(k.b.z & hi, p3.z, b1);
    a0 = dp4a_us(k.a.w & lo, p0.w, a0);
    a1 = dp4a_us(k.b.w & lo, p1.w, a1);
    b0 = dp4a_us(k.a.w & hi, p2.w, b0);
    b1 = dp4a_us(k.b.w & hi, p3.w, b1);
    s0 = a0 + a1;
    s1x16 = b0 + b1;
}

// One column's contribution of a chunk:
// dq_j0*(d*sc_j0*s0 - dmin*m_j0*sumq_j0) + (same for j1), with fd0..fm1 from
// chunk_scales (fd1 pre-divided by 16 for s1x16).
__device__ __forceinline__ float chunk_column(const Chunk& k, float fd0, float fd1, float fm0, float fm1,
                                              const uint4& p0, const uint4& p1, const uint4& p2, const uint4& p3,
                                              const float4& sc, float acc)
{
    int s0, s1x16;
    chunk_dot(k, p0, p1, p2, p3, s0, s1x16);
    acc = fmaf(fd0, sc.x * float(s0), acc);
    acc = fmaf(fd1, sc.y * float(s1x16), acc);  // fd1 carries the 1/16
    acc = fmaf(-fm0, sc.z, acc);
    acc = fmaf(-fm1, sc.w, acc);
    return acc;
}

// acc[c] += this chunk's contribution for every column, activation from shared memory
template <int NC>
__device__ __forceinline__ void chunk_accumulate(const Chunk& k, int c4, int ch, const ActSmem& s, float acc[NC])
{
    float fd0, fd1, fm0, fm1;
    chunk_scales(k.h, c4, fd0, fd1, fm0, fm1);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4* P = s.planes + size_t(c * 4) * s.C + ch;
        acc[c] = chunk_column(k, fd0, fd1, fm0, fm1, P[0], P[s.C], P[2 * s.C], P[3 * s.C],
                              s.scales[size_t(c) * s.C + ch], acc[c]);
    }
}

// the same with this chunk's activation held in registers (one lane, fixed chunk)
template <int NC>
__device__ __forceinline__ void chunk_accumulate_regs(const Chunk& k, int c4, const uint4 (&P)[NC][4],
                                                      const float4 (&SC)[NC], float acc[NC])
{
    float fd0, fd1, fm0, fm1;
    chunk_scales(k.h, c4, fd0, fd1, fm0, fm1);
#pragma unroll
    for (int c = 0; c < NC; ++c)
        acc[c] = chunk_column(k, fd0, fd1, fm0, fm1, P[c][0], P[c][1], P[c][2], P[c][3], SC[c], acc[c]);
}

// Tagged records: a 32-bit word and a 32-bit tag written by one 8-byte
// relaxed store at GPU scope.  An aligned 8-byte access is single-copy atomic,
// so a relaxed load at GPU scope of the same record returns the word together
// with the tag it was stored with: a reader that sees the tag it expects has
// the word, with no fence on either side.
__device__ __forceinline__ void st_tagged(uint64_t* p, uint32_t word, uint32_t tag)
{
    const uint64_t v = uint64_t(word) | (uint64_t(tag) << 32);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// two consecutive records (16-byte aligned); each 8-byte element is atomic
__device__ __forceinline__ void ld_tagged2(const uint64_t* p, uint64_t& a, uint64_t& b)
{
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// relaxed atomic add at GPU scope, no value returned
__device__ __forceinline__ void red_relaxed_add_u32(unsigned* p, unsigned v)
{
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

}  // namespace mq
