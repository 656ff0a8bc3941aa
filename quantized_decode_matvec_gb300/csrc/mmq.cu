// mmq.cu -- the q4_K x q8_0 matmul for 9..64 activation columns on the 5th-
// generation tensor cores ("07 . R3 -- Small-model per-token overhead",
// section 5: past the decode matvec, the "MMQ" work for more tokens).
//
// Beyond a few columns the matvec becomes a contraction, and the dp4a work of
// the decode kernels grows with the columns while the weight stream does not.
// Here the integer dot products run on tcgen05.mma of kind::f16 with operands
// that are exact in binary16:
//   A = the weights' 4-bit quants q (0..15; the high nibbles as 16*q),
//   B = the activation's q8_0 codes (-127..127),
// so every product is an integer and every 32-element sub-block sum
//   S[r][j][c] = sum over the sub-block of q * code   (|S| < 2^20)
// is exact in the fp32 accumulator.  Each sub-block has its own accumulator
// slot in tensor memory (the weights' scale sc_j and the activation's dq_j
// change every 32 elements), and the epilogue applies the scales per
// sub-block as the decode kernels do:
//   y[r][c] += d*sc_j * (dq_jc * S) - dmin*m_j * (dq_jc * sumq_jc)
//
// Launches: (1) the activation is quantized to q8_0 (the same quantizer as
// every other path) and laid out for the MMA: codes as f16 in the 128-byte-
// swizzled K-major image of each 256-element step, with (dq, dq*sumq) per
// block and column; (2) the matmul; (3) for matrices with few row tiles, the
// K range is split over CTAs and a fixed-order sum combines the partials.
//
// The matmul CTA (persistent over its work items, 14 warps):
//   warp 0      each step's 128 weight rows (144 bytes each) by 16-byte
//               asynchronous copies spread over the lanes, the step's
//               activation image and its scales by two bulk copies (TMA), into
//               a ring of stages
//   warp 1      TMEM allocation; one lane issues two MMAs (M=128, N=ncols
//               rounded up to 16, K=16) per sub-block into the sub-block's slot
//   warps 2-9   convert the rows' quants to the f16 A image (thread = row;
//               warps 2-5 the first half of each step, 6-9 the second), into a
//               ring of half-step buffers, so conversion overlaps the MMAs
//   warps 10-13 epilogue (thread = row = TMEM lane): per sub-block, read the
//               slot, apply the scales into fp32 registers (packed f32x2
//               arithmetic), free the slot
// Every wait is bounded in time; a timeout records MQ_DEV_TIMEOUT and the
// roles stop (the producer waits, bounded, for its copies in flight).
#include <cuda_fp16.h>

#include "mq_job.cuh"
#include "mq_umma.cuh"

namespace mq {

constexpr int kMmqBM = 128;                          // weight rows per tile
constexpr int kMmqThreads = 448;
constexpr int kMmqAtom = kMmqBM * 128;               // one 128 x 64 f16 swizzled atom: 16 KB
constexpr int kMmqAHalf = 2 * kMmqAtom;              // half a step of A (128 K): 32 KB
constexpr int kMmqRaw = kMmqBM * kQ4KBytes;          // 128 rows x 144 bytes
constexpr uint32_t kMmqTmemCols = 512;

__host__ __device__ constexpr int mmq_np(int nc) { return (nc + 15) / 16 * 16; }
// stage: raw weights | activation image (4 atoms of NP rows x 128 B) | scales [8][2][NP] (dq, dq*sumq)
__host__ __device__ constexpr int mmq_stage_bytes(int NP) { return kMmqRaw + NP * 512 + 8 * NP * 8; }
__host__ __device__ constexpr int mmq_round1k(int b) { return (b + 1023) / 1024 * 1024; }

struct MmqArgs {
    int R, K, ncols;
    int m_tiles, ksplit, nkb;
    int stages;
    int nab;                  // half-step A buffers
    int stage_bytes;          // 1024-aligned
    const uint8_t* bimg;      // activation images, nkb x NP*512 bytes
    const float* sc;          // [K/32][2][NP]: dq, then dq*sumq
    float* part;              // [ksplit][ncols][R] partial sums (ksplit > 1)
    uint64_t limit_ns;
};

// ---- (1) activation: q8_0, then the MMA image -----------------------------------------
// One warp per (column, 32-block); lane l is element 32J + l.
template <int NP>
__global__ void mmq_stage_act_kernel(const mq_mv_desc* __restrict__ desc, int rows_h, int K_h, int nc_h,
                                     uint8_t* __restrict__ bimg, float* __restrict__ sc, unsigned* status)
{
    const MvJob j = read_job<KIND_MV>(desc);
    const unsigned bad = check_job(j, rows_h, K_h, nc_h);
    if (bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, bad);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int nq = K_h / kQK8;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t w = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < int64_t(NP) * nq;
         w += nwarps) {
        const int c = int(w / nq), J = int(w - int64_t(c) * nq);
        int q = 0;
        float dq = 0.0f;
        if (c < nc_h) {
            if (j.x) {
                float d;
                q = q8_quantize_lane(j.x[size_t(c) * K_h + size_t(J) * kQK8 + lane], &d);
                const __half dh = __float2half_rn(d);
                dq = __half2float(dh);
                if (j.xq_out) {  // the q8_0 blocks too, for the bit-exact check
                    uint8_t* ob = j.xq_out + (size_t(c) * nq + J) * kQ8Bytes;
                    if (lane == 0) *reinterpret_cast<uint16_t*>(ob) = __half_as_ushort(dh);
                    ob[2 + lane] = uint8_t(int8_t(q));
                }
            } else {
                const uint8_t* blk = j.xq + (size_t(c) * nq + J) * kQ8Bytes;
                dq = __half2float(__ushort_as_half(uint16_t(blk[0] | (blk[1] << 8))));
                q = int(int8_t(blk[2 + lane]));
            }
        }
        const int sq = __reduce_add_sync(0xffffffffu, q);
        const int k = J * kQK8 + lane, kb = k >> 8, a = (k >> 6) & 3, e = k & 63;
        const size_t off = size_t(kb) * (NP * 512) + size_t(a) * (NP * 128) + size_t(c) * 128 +
                           size_t(((e >> 3) ^ (c & 7)) << 4) + size_t(e & 7) * 2;
        *reinterpret_cast<__half*>(bimg + off) = __int2half_rn(q);
        if (lane == 0) {
            sc[size_t(2 * J) * NP + c] = dq;
            sc[size_t(2 * J + 1) * NP + c] = dq * float(sq);
        }
    }
}

// ---- (2) the matmul ------------------------------------------------------------------------
// quants -> f16 pairs: bytes (b0, b1) of w selected by sel into the two
// halves, the low nibbles as 1024 + n or the high nibbles as 1024 + 16n
// (exact binary16), minus 1024
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, uint32_t sel, uint32_t mask)
{
    uint32_t u = (__byte_perm(w, 0u, sel) & mask) | 0x64006400u;
    __half2 h = *reinterpret_cast<__half2*>(&u);
    h = __hsub2(h, __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 16 bytes global -> shared, through L2 only; completion tracked per thread
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// the mbarrier receives one arrival (counted in its expected count) once every
// cp.async this thread issued before has completed
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// packed fp32 pairs: (lo, hi) in one 64-bit register for the f32x2 instructions
__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    return uint64_t(__float_as_uint(lo)) | (uint64_t(__float_as_uint(hi)) << 32);
}

// y += ds * (dq * S) - dm * dqs on two columns at once (each lane of the pair
// rounds exactly as the scalar fmaf chain would)
__device__ __forceinline__ void epi2(uint64_t& y, uint64_t S, uint64_t dq, uint64_t dqs, uint64_t ds2, uint64_t ndm2)
{
    uint64_t t;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(dq), "l"(S));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(y) : "l"(ds2), "l"(t));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(y) : "l"(ndm2), "l"(dqs));
}

template <int NP>
__global__ void __launch_bounds__(kMmqThreads, 1)
    mmq_kernel(const mq_mv_desc* __restrict__ desc, const MmqArgs a, unsigned* status)
{
    constexpr int NSLOT = int(kMmqTmemCols) / NP;  // accumulator slots of NP columns
    constexpr int NGRP = NSLOT / 8;                   // steps whose eight slots fit at once
    extern __shared__ uint8_t msm_raw[];
    __shared__ __align__(8) uint64_t full[4], empty[4], a_full[4], a_free[4], acc_full[4], slot_free[32];
    __shared__ uint32_t tmem_base;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t raw_addr = smem_u32(msm_raw);
    uint8_t* const sm = msm_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* const abuf = sm;                                     // a.nab x 32 KB, 1024-aligned
    uint8_t* const stages = sm + size_t(a.nab) * kMmqAHalf;       // a.stages x a.stage_bytes
    {
        // the activation launch checked the descriptor too; a bad one stops this launch as well
        const unsigned bad = check_job(read_job<KIND_MV>(desc), a.R, a.K, a.ncols);
        if (bad) return;
    }
    const uint8_t* W = static_cast<const uint8_t*>(desc->W);
    float* Y = desc->y;
    const int y_ld = desc->y_ld;
    const size_t row_bytes = size_t(a.nkb) * kQ4KBytes;
    const int nitems = a.m_tiles * a.ksplit;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 32 + 1);      // the producer's lanes' row copies, and its activation copies
            mbar_init(&empty[s], 8 + 1 + 4);  // converter warps, the MMA commit, epilogue warps
        }
        for (int b = 0; b < a.nab; ++b) {
            mbar_init(&a_full[b], 4);  // the four warps of a half's converter group
            mbar_init(&a_free[b], 1);  // MMA commit
        }
        for (int i = 0; i < NGRP; ++i) mbar_init(&acc_full[i], 1);  // MMA commit, once per step
        for (int i = 0; i < NSLOT; ++i) mbar_init(&slot_free[i], 4);  // epilogue warps, per slot
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, kMmqTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    // the SB range of work item it: tile m, K split ks
    auto item = [&](int it, int& m, int& kb0, int& kb1) {
        m = it / a.ksplit;
        const int ks = it - m * a.ksplit;
        kb0 = int(int64_t(ks) * a.nkb / a.ksplit);
        kb1 = int(int64_t(ks + 1) * a.nkb / a.ksplit);
    };

    if (warp == 0) {
        // ---- producer: every lane issues row copies; lane 0 the barrier and the activation
        int g = 0;
        for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
            if (__shfl_sync(0xffffffffu, abort_flag, 0)) break;  // one decision for the whole warp
            int m, kb0, kb1;
            item(it, m, kb0, kb1);
            const int r0 = m * kMmqBM, nrow = min(kMmqBM, a.R - r0);
            for (int kb = kb0; kb < kb1; ++kb, ++g) {
                const int s = g % a.stages;
                bool ok = true;
                if (lane == 0 && g >= a.stages)
                    ok = mbar_wait_bounded(&empty[s], uint32_t(g / a.stages - 1) & 1u, a.limit_ns);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                    if (lane == 0) abort_flag = 1;
                    break;
                }
                uint8_t* st = stages + size_t(s) * a.stage_bytes;
                if (lane == 0) {  // the activation image and its scales: two bulk copies
                    mbar_arrive_expect_tx(&full[s], uint32_t(NP * 512 + 8 * NP * 8));
                    bulk_copy_g2s(st + kMmqRaw, a.bimg + size_t(kb) * (NP * 512), NP * 512, &full[s]);
                    bulk_copy_g2s(st + kMmqRaw + NP * 512, a.sc + size_t(kb) * 16 * NP, 8 * NP * 8, &full[s]);
                }
                // the rows' 144-byte blocks: nine 16-byte chunks each, consecutive chunks on
                // consecutive lanes (one bulk copy per row would queue 128 small copies on the
                // copy engine, which handles them one after another)
                const uint8_t* src = W + size_t(r0) * row_bytes + size_t(kb) * kQ4KBytes;
                const uint32_t dst = smem_u32(st);
                for (int i = lane; i < nrow * 9; i += 32) {
                    const int r = i / 9, c = i - r * 9;
                    cp_async16(dst + uint32_t(i) * 16, src + size_t(r) * row_bytes + 16 * c);
                }
                cp_async_arrive_noinc(&full[s]);  // arrives once this lane's copies have landed
            }
        }
        if (lane == 0)  // copies still in flight land before the CTA exits
            for (int j = g > a.stages ? g - a.stages : 0; j < g; ++j)
                (void)mbar_wait_bounded(&full[j % a.stages], uint32_t(j / a.stages) & 1u, a.limit_ns);
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16_f32(kMmqBM, NP);
            const uint32_t aaddr = smem_u32(abuf);
            int g = 0, v = 0;  // steps and slot uses so far
            bool ok = true;
            for (int it = blockIdx.x; it < nitems && ok && !abort_flag; it += gridDim.x) {
                int m, kb0, kb1;
                item(it, m, kb0, kb1);
                for (int kb = kb0; kb < kb1 && ok; ++kb, ++g) {
                    const int s = g % a.stages;
                    ok = mbar_wait_bounded(&full[s], uint32_t(g / a.stages) & 1u, a.limit_ns);
                    const uint32_t baddr = smem_u32(stages + size_t(s) * a.stage_bytes + kMmqRaw);
                    for (int h = 0; h < 2 && ok; ++h) {
                        const int u = 2 * g + h, b = u % a.nab;
                        ok = mbar_wait_bounded(&a_full[b], uint32_t(u / a.nab) & 1u, a.limit_ns);
                        tc_fence_after();
                        const uint32_t ah = aaddr + uint32_t(b) * kMmqAHalf;
                        // the half's four slots free, then one fence for its eight MMAs
                        for (int jj = 0; jj < 4 && ok; ++jj) {
                            const int vv = v + jj;
                            if (vv >= NSLOT)
                                ok = mbar_wait_bounded(&slot_free[vv % NSLOT], uint32_t(vv / NSLOT - 1) & 1u,
                                                       a.limit_ns);
                        }
                        if (!ok) break;
                        tc_fence_after();
                        for (int jj = 0; jj < 4; ++jj, ++v) {
                            const int j = 4 * h + jj;  // sub-block of the step
                            const int slot = v % NSLOT;
                            const uint32_t koff = uint32_t(j & 1) * 64;
                            const uint32_t ab = ah + uint32_t(jj >> 1) * kMmqAtom + koff;
                            const uint32_t bb = baddr + uint32_t(j >> 1) * (NP * 128) + koff;
                            const uint32_t d = tmem + uint32_t(slot * NP);
                            umma_f16(d, umma_desc_sw128(ab), umma_desc_sw128(bb), idesc, false);
                            umma_f16(d, umma_desc_sw128(ab + 32), umma_desc_sw128(bb + 32), idesc, true);
                        }
                        if (ok) umma_commit(&a_free[b]);  // this half's A buffer may be rewritten
                    }
                    if (ok) {
                        // one commit per step for its eight slots (a commit per sub-block
                        // serialized the issue of these small MMAs), and the stage
                        umma_commit(&acc_full[g % NGRP]);
                        umma_commit(&empty[s]);  // this step's activation image has been read
                    }
                }
            }
            if (!ok) abort_flag = 1;
            if (g > 0)  // the last MMAs complete before TMEM is freed
                (void)mbar_wait_bounded(&acc_full[(g - 1) % NGRP], uint32_t((g - 1) / NGRP) & 1u, a.limit_ns);
        }
    } else if (warp < 10) {
        // ---- converters: thread = row r of the tile; group h converts half h of every step
        // (quant bytes 64h..64h+63: sub-blocks 4h..4h+3) into the half-step buffer
        const int h = (warp - 2) >> 2;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t sw = uint32_t(r & 7);
        int g = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x) {
            int m, kb0, kb1;
            item(it, m, kb0, kb1);
            const bool live = m * kMmqBM + r < a.R;
            for (int kb = kb0; kb < kb1; ++kb, ++g) {
                const int s = g % a.stages;
                const int u = 2 * g + h, b = u % a.nab, n = u / a.nab;
                bool w = mbar_wait_bounded(&full[s], uint32_t(g / a.stages) & 1u, a.limit_ns);
                if (w && n > 0) w = mbar_wait_bounded(&a_free[b], uint32_t(n - 1) & 1u, a.limit_ns);
                ok = __all_sync(0xffffffffu, w && !abort_flag);  // one decision for the whole warp
                if (!ok) break;
                const uint8_t* raw = stages + size_t(s) * a.stage_bytes + size_t(r) * kQ4KBytes;
                const uint32_t arow = smem_u32(abuf) + uint32_t(b) * kMmqAHalf + uint32_t(r) * 128;
#pragma unroll
                for (int ca = 0; ca < 2; ++ca) {
                    const int cc = 2 * h + ca;  // quant bytes 32cc..32cc+31: sub-blocks 2cc (low), 2cc+1 (high)
                    uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
                    if (live) {
                        q0 = *reinterpret_cast<const uint4*>(raw + 16 + 32 * cc);
                        q1 = *reinterpret_cast<const uint4*>(raw + 32 + 32 * cc);
                    }
                    const uint32_t wq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                    const uint32_t atom = arow + uint32_t(ca) * kMmqAtom;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        // chunk c: elements 8c..8c+7 of the atom's 64: low nibbles of bytes
                        // 8c.. (c < 4) or high nibbles of bytes 8(c-4).. (c >= 4)
                        const uint32_t m4 = c < 4 ? 0x000F000Fu : 0x00F000F0u;
                        const uint32_t w0 = wq[2 * (c & 3)], w1 = wq[2 * (c & 3) + 1];
                        sts128(atom + ((uint32_t(c) ^ sw) << 4), nib_pair(w0, 0x4140u, m4), nib_pair(w0, 0x4342u, m4),
                               nib_pair(w1, 0x4140u, m4), nib_pair(w1, 0x4342u, m4));
                    }
                }
                fence_proxy_async_smem();  // the A image is read by the tensor cores
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&a_full[b]);
                    mbar_arrive(&empty[s]);
                }
            }
        }
        if (!ok && lane == 0) abort_flag = 1;
    } else {
        // ---- epilogue: thread = TMEM lane = row r of the tile
        const int q = warp & 3, r = q * 32 + lane;
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        int g = 0, v = 0;
        bool stop = false;
        for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
            int m, kb0, kb1;
            item(it, m, kb0, kb1);
            const int row = m * kMmqBM + r;
            uint64_t y2[NP / 2];  // column pairs (2c, 2c+1)
#pragma unroll
            for (int c = 0; c < NP / 2; ++c) y2[c] = 0;
            for (int kb = kb0; kb < kb1 && !stop; ++kb, ++g) {
                const int s = g % a.stages;
                const uint8_t* st = stages + size_t(s) * a.stage_bytes;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], uint32_t(g / a.stages) & 1u, a.limit_ns))) {
                    stop = true;
                    break;
                }
                // this row's scales from its super-block header (rows past the end: zeros)
                float ds[8], dm[8];
                {
                    uint4 hd = make_uint4(0, 0, 0, 0);
                    if (row < a.R) hd = *reinterpret_cast<const uint4*>(st + size_t(r) * kQ4KBytes);
                    const float d = __half2float(__ushort_as_half(uint16_t(hd.x)));
                    const float dmin = __half2float(__ushort_as_half(uint16_t(hd.x >> 16)));
                    const uint32_t S[3] = {hd.y, hd.z, hd.w};
                    auto byte = [&](int i) { return int((S[i >> 2] >> (8 * (i & 3))) & 0xffu); };
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        int scv, mv;
                        if (jj < 4) {
                            scv = byte(jj) & 63;
                            mv = byte(jj + 4) & 63;
                        } else {
                            scv = (byte(jj + 4) & 15) | ((byte(jj - 4) >> 6) << 4);
                            mv = (byte(jj + 4) >> 4) | ((byte(jj) >> 6) << 4);
                        }
                        // odd sub-blocks come from the high nibbles, taken as 16*q
                        ds[jj] = d * float(scv) * ((jj & 1) ? 0.0625f : 1.0f);
                        dm[jj] = dmin * float(mv);
                    }
                }
                const float4* scj = reinterpret_cast<const float4*>(st + kMmqRaw + NP * 512);
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(&acc_full[g % NGRP], uint32_t(g / NGRP) & 1u, a.limit_ns))) {
                    stop = true;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int jj = 0; jj < 8; ++jj, ++v) {
                    const int slot = v % NSLOT;
                    const uint64_t ds2 = pack2(ds[jj], ds[jj]), ndm2 = pack2(-dm[jj], -dm[jj]);
                    const float4* dqv = scj + (2 * jj) * (NP / 4);       // dq of the sub-block's columns
                    const float4* dqsv = scj + (2 * jj + 1) * (NP / 4);  // dq*sumq
#pragma unroll
                    for (int c0 = 0; c0 < NP; c0 += 16) {
                        float t[16];
                        tmem_ld16(tmem + lane_base + uint32_t(slot * NP + c0), t);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            const float4 dq = dqv[(c0 + i) >> 2], dqs = dqsv[(c0 + i) >> 2];
                            epi2(y2[(c0 + i) >> 1], pack2(t[i], t[i + 1]), pack2(dq.x, dq.y), pack2(dqs.x, dqs.y), ds2,
                                 ndm2);
                            epi2(y2[((c0 + i) >> 1) + 1], pack2(t[i + 2], t[i + 3]), pack2(dq.z, dq.w),
                                 pack2(dqs.z, dqs.w), ds2, ndm2);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&slot_free[slot]);
                }
                __syncwarp();
                if (lane == 0 && !stop) mbar_arrive(&empty[s]);
            }
            if (stop) break;
            if (row < a.R) {
                const int ks = it - m * a.ksplit;
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    if (c >= a.ncols) break;
                    const float yc = __uint_as_float(uint32_t(y2[c >> 1] >> (32 * (c & 1))));
                    if (a.ksplit == 1)
                        Y[size_t(c) * y_ld + row] = yc;
                    else
                        a.part[(size_t(ks) * a.ncols + c) * a.R + row] = yc;
                }
            }
        }
        if (stop && lane == 0) abort_flag = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (abort_flag && threadIdx.x == 0) atomicOr(status, MQ_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kMmqTmemCols);
    }
}

// ---- (3) fixed-order sum of the K-split partials ---------------------------------------------
__global__ void mmq_reduce_kernel(const mq_mv_desc* __restrict__ desc, const float* __restrict__ part, int ksplit,
                                  int R, int ncols)
{
    float* Y = desc->y;
    const int y_ld = desc->y_ld;
    const int64_t n = int64_t(ncols) * R;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        const int c = int(i / R), r = int(i - int64_t(c) * R);
        float s = 0.0f;
        for (int ks = 0; ks < ksplit; ++ks) s += part[(size_t(ks) * ncols + c) * R + r];
        Y[size_t(c) * y_ld + r] = s;
    }
}

// ---- host side ----------------------------------------------------------------------------------
MmqPlan plan_mmq(int rows, int K, int ncols, int num_sms, int max_smem)
{
    MmqPlan p{};
    p.np = mmq_np(ncols);
    p.nkb = K / kQK;
    p.m_tiles = (rows + kMmqBM - 1) / kMmqBM;
    int ks = num_sms / p.m_tiles;
    p.ksplit = ks < 1 ? 1 : (ks > p.nkb ? p.nkb : ks);
    p.stage_bytes = mmq_round1k(mmq_stage_bytes(p.np));
    // the most half-step A buffers (4, 3, 2) that still leave two stages; up to 4 stages
    // (the kernel's static shared memory, under 2 KB, comes off the opt-in maximum)
    p.stages = 0;
    for (int nab = 4; nab >= 2 && p.stages < 2; --nab) {
        const int st = (max_smem - 2048 - 1024 - nab * kMmqAHalf) / p.stage_bytes;
        p.nab = nab;
        p.stages = st > 4 ? 4 : st;
    }
    p.smem = 1024 + p.nab * kMmqAHalf + p.stages * p.stage_bytes;
    const int items = p.m_tiles * p.ksplit;
    p.grid = items < num_sms ? items : num_sms;
    p.bimg_bytes = (size_t(p.nkb) * p.np * 512 + 127) / 128 * 128;
    p.sc_bytes = (size_t(K / kQK8) * p.np * 8 + 127) / 128 * 128;
    p.part_bytes = p.ksplit > 1 ? size_t(p.ksplit) * ncols * rows * 4 : 0;
    p.ws_bytes = p.bimg_bytes + p.sc_bytes + p.part_bytes;
    return p;
}

template <int NP>
static cudaError_t launch_mmq_np(const mq_mv_desc* d, int rows, int K, int ncols, const MmqPlan& p, uint8_t* ws,
                                 int num_sms, unsigned* status, cudaStream_t s)
{
    uint8_t* bimg = ws;
    float* sc = reinterpret_cast<float*>(ws + p.bimg_bytes);
    float* part = reinterpret_cast<float*>(ws + p.bimg_bytes + p.sc_bytes);
    const int64_t warps = int64_t(NP) * (K / kQK8);
    const int64_t want = (warps + 7) / 8;
    const int g1 = int(want < int64_t(num_sms) * 16 ? want : int64_t(num_sms) * 16);
    mmq_stage_act_kernel<NP><<<g1, 256, 0, s>>>(d, rows, K, ncols, bimg, sc, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    MmqArgs a;
    a.R = rows;
    a.K = K;
    a.ncols = ncols;
    a.m_tiles = p.m_tiles;
    a.ksplit = p.ksplit;
    a.nkb = p.nkb;
    a.stages = p.stages;
    a.nab = p.nab;
    a.stage_bytes = p.stage_bytes;
    a.bimg = bimg;
    a.sc = sc;
    a.part = part;
    a.limit_ns = uint64_t(fault_policy() == FAULT_NONE ? 2000 : 50) * 1000000ull;
    mmq_kernel<NP><<<p.grid, kMmqThreads, p.smem, s>>>(d, a, status);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.ksplit == 1) return e;
    const int64_t n = int64_t(ncols) * rows;
    const int64_t w2 = (n + 255) / 256;
    mmq_reduce_kernel<<<int(w2 < int64_t(num_sms) * 8 ? w2 : int64_t(num_sms) * 8), 256, 0, s>>>(d, part, p.ksplit,
                                                                                                rows, ncols);
    return cudaGetLastError();
}

cudaError_t launch_mmq(const mq_mv_desc* d, int rows, int K, int ncols, const MmqPlan& p, void* ws, int num_sms,
                       unsigned* status, cudaStream_t s)
{
    uint8_t* w = static_cast<uint8_t*>(ws);
    switch (p.np) {
        case 16: return launch_mmq_np<16>(d, rows, K, ncols, p, w, num_sms, status, s);
        case 32: return launch_mmq_np<32>(d, rows, K, ncols, p, w, num_sms, status, s);
        case 48: return launch_mmq_np<48>(d, rows, K, ncols, p, w, num_sms, status, s);
        case 64: return launch_mmq_np<64>(d, rows, K, ncols, p, w, num_sms, status, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t set_mmq_attributes(int max_smem)
{
    cudaError_t e = cudaSuccess;
    const void* k[4] = {reinterpret_cast<const void*>(mmq_kernel<16>), reinterpret_cast<const void*>(mmq_kernel<32>),
                        reinterpret_cast<const void*>(mmq_kernel<48>), reinterpret_cast<const void*>(mmq_kernel<64>)};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i) e = set_max_dyn_smem(k[i], max_smem);
    return e;
}

}  // namespace mq
