// gemm.cu -- the prefill GEMM on the 5th-generation tensor cores.
//
// "07 . R3 -- Small-model per-token overhead", section 1: prefill of the 7B
// model at 2K tokens runs a half-precision tensor-core GEMM over a resident
// f16 copy of the weights (the quantized weights dequantized once).  Here:
//
//   Y[t][r] = sum_k X[t][k] * W[r][k]      X f16 [T][K], W f16 [R][K], Y fp32 [T][R]
//
// with fp32 accumulation in tensor memory.  One CTA per SM walks output tiles
// of 128 weight rows x BN tokens, BN = 256 (128 for at most 128 tokens),
// persistent, static round robin, a last wave that would leave half the CTAs
// idle split into BN/2-token tiles; tiles that
// share a weight block run at the same time, so each block comes from HBM
// about once and from L2 for the other token tiles.  Per CTA:
//
// * warp 0, one lane: TMA loads of 128x64 weight and BNx64 activation tiles
//   (128-byte swizzle) into a ring of shared-memory stages, tracked by
//   mbarriers;
// * warp 1: allocates 2*BN TMEM columns (two 128xBN fp32 accumulators); one
//   lane issues four tcgen05.mma (M=128, N=BN, K=16) per stage and commits
//   each stage back to the producer, and each finished tile to the epilogue;
// * warps 2..5: the epilogue reads its 32 TMEM lanes (32 weight rows) with
//   tcgen05.ld and stores fp32 Y, coalesced across the rows, while the MMAs
//   of the next tile fill the other accumulator.
//
// Every wait is bounded in time: on a timeout the CTA records MQ_DEV_TIMEOUT,
// the roles stop, the producer waits (bounded) for its copies in flight and
// TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mq_internal.h"
#include "mq_umma.cuh"

namespace mq {

constexpr int kGemmBM = 128;                          // weight rows per tile (TMEM lanes)
constexpr int kGemmBK = 64;                           // f16 per 128-byte swizzled row
constexpr int kGemmATile = kGemmBM * kGemmBK * 2;     // 16 KB
constexpr int kGemmThreads = 192;

// tokens per tile BN (256, or 128 where 256-token tiles would leave the last
// wave of CTAs mostly idle); a stage holds one A and one B tile
template <int BN>
struct GemmTile {
    static constexpr int kBTile = BN * kGemmBK * 2;
    static constexpr int kStage = kGemmATile + kBTile;
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
    static constexpr int kSmem = kStages * kStage + 1024;  // + alignment slack
};

struct GemmArgs {
    int R, K, T;
    int m_tiles, n_tiles, k_steps;
    // the last wave of BN-token tiles split in two BN/2-token tiles when that
    // fills at most a wave of CTAs: tiles [0, full_tiles) are BN wide, the
    // ntiles - full_tiles after them BN/2 wide (full_tiles = ntiles: no split)
    int full_tiles, ntiles;
    uint64_t limit_ns;
};

// output tile t: weight-row block m, first token tok0, width bn
struct GemmTileAt {
    int m, tok0, bn;
};

template <int BN>
__device__ __forceinline__ GemmTileAt gemm_tile_at(int t, const GemmArgs& a)
{
    if (t < a.full_tiles) {
        const int m = t / a.n_tiles;
        return GemmTileAt{m, (t - m * a.n_tiles) * BN, BN};
    }
    const int u = t - a.full_tiles, t2 = a.full_tiles + (u >> 1);  // the BN tile it halves
    const int m = t2 / a.n_tiles;
    return GemmTileAt{m, (t2 - m * a.n_tiles) * BN + (u & 1) * (BN / 2), BN / 2};
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_f16_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmXh, float* __restrict__ Y, const GemmArgs a,
                    unsigned* status)
{
    using G = GemmTile<BN>;
    constexpr int kGemmBN = BN, kGemmStages = G::kStages, kGemmStage = G::kStage;
    constexpr uint32_t kGemmTmemCols = G::kTmemCols;
    extern __shared__ uint8_t gsm_raw[];
    __shared__ __align__(8) uint64_t full[kGemmStages], empty[kGemmStages], accf[2], acce[2];
    __shared__ uint32_t tmem_base;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the swizzled tiles want 1024-byte alignment
    const uint32_t raw = smem_u32(gsm_raw);
    uint8_t* const gsm = gsm_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int ntiles = a.ntiles;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 4 * 32);
        }
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        if (a.full_tiles < a.ntiles) tma_prefetch_desc(&tmXh);
    }
    if (warp == 1) tmem_alloc(&tmem_base, kGemmTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0) {
        // ---- TMA producer
        if (lane == 0) {
            int it = 0;
            for (int t = blockIdx.x; t < ntiles && !abort_flag; t += gridDim.x) {
                const GemmTileAt ti = gemm_tile_at<BN>(t, a);
                const bool half = ti.bn != BN;
                for (int kk = 0; kk < a.k_steps; ++kk, ++it) {
                    const int s = it % kGemmStages;
                    if (it >= kGemmStages &&
                        !mbar_wait_bounded(&empty[s], uint32_t(it / kGemmStages - 1) & 1u, a.limit_ns)) {
                        abort_flag = 1;
                        break;
                    }
                    uint8_t* sa = gsm + s * kGemmStage;
                    mbar_arrive_expect_tx(&full[s], uint32_t(kGemmATile + ti.bn * kGemmBK * 2));
                    tma_load_2d(sa, &tmW, kk * kGemmBK, ti.m * kGemmBM, &full[s]);
                    tma_load_2d(sa + kGemmATile, half ? &tmXh : &tmX, kk * kGemmBK, ti.tok0, &full[s]);
                }
            }
            // copies still in flight land before the CTA can exit
            for (int j = it > kGemmStages ? it - kGemmStages : 0; j < it; ++j)
                (void)mbar_wait_bounded(&full[j % kGemmStages], uint32_t(j / kGemmStages) & 1u, a.limit_ns);
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_full = umma_idesc_f16_f32(kGemmBM, kGemmBN);
            constexpr uint32_t idesc_half = umma_idesc_f16_f32(kGemmBM, kGemmBN / 2);
            int it = 0, tl = 0;
            for (int t = blockIdx.x; t < ntiles && !abort_flag; t += gridDim.x, ++tl) {
                const uint32_t idesc = t < a.full_tiles ? idesc_full : idesc_half;
                const int b = tl & 1;
                if (tl >= 2 && !mbar_wait_bounded(&acce[b], uint32_t(tl / 2 - 1) & 1u, a.limit_ns)) {
                    abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + uint32_t(b * kGemmBN);
                bool ok = true;
                for (int kk = 0; kk < a.k_steps; ++kk, ++it) {
                    const int s = it % kGemmStages;
                    if (!mbar_wait_bounded(&full[s], uint32_t(it / kGemmStages) & 1u, a.limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(gsm + s * kGemmStage);
#pragma unroll
                    for (int k4 = 0; k4 < kGemmBK / 16; ++k4)
                        umma_f16(d, umma_desc_sw128(sa + 32u * k4), umma_desc_sw128(sa + kGemmATile + 32u * k4), idesc,
                                 kk > 0 || k4 > 0);
                    umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
                }
                if (!ok) {
                    abort_flag = 1;
                    break;
                }
                umma_commit(&accf[b]);  // the tile's accumulator is complete
            }
            // the last commits land before TMEM is freed
            if (it > 0) {
                const int j = it - 1;
                (void)mbar_wait_bounded(&empty[j % kGemmStages], uint32_t(j / kGemmStages) & 1u, a.limit_ns);
            }
        }
    } else {
        // ---- epilogue: TMEM lanes 32*(warp%4) .. +31 = weight rows of the tile
        const int q = warp & 3;
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        int tl = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tl) {
            const int b = tl & 1;
            // one decision for the whole warp
            const bool ok = __all_sync(0xffffffffu,
                                       mbar_wait_bounded(&accf[b], uint32_t(tl / 2) & 1u, a.limit_ns) && !abort_flag);
            if (!ok) {
                if (lane == 0) abort_flag = 1;
                break;
            }
            tc_fence_after();
            const GemmTileAt ti = gemm_tile_at<BN>(t, a);
            const int r = ti.m * kGemmBM + q * 32 + lane;
            const int t0 = ti.tok0;
#pragma unroll 1
            for (int c0 = 0; c0 < ti.bn; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + uint32_t(b * kGemmBN + c0), v);
                tmem_ld_wait();
                if (r < a.R) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = t0 + c0 + j;
                        if (tok < a.T) Y[size_t(tok) * a.R + r] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acce[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (abort_flag && threadIdx.x == 0) atomicOr(status, MQ_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kGemmTmemCols);
    }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D tensor map of a row-major f16 matrix [rows][K], box {64, box_rows}, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kGemmBK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t set_gemm_attributes(int max_smem)
{
    (void)max_smem;
    cudaError_t e = cudaFuncSetAttribute(gemm_f16_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GemmTile<256>::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_f16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 GemmTile<128>::kSmem);
    return e;
}


// returns cudaErrorInvalidValue when the tensor maps cannot be built
cudaError_t launch_gemm_f16(const void* W16, const void* X16, float* Y, int R, int K, int T, int num_sms,
                            unsigned* status, cudaStream_t s)
{
    const int m_tiles = (R + kGemmBM - 1) / kGemmBM;
    // 256-token tiles (128-token tiles, which fill the last wave of CTAs better for
    // the 3584-row matrices at 2048 tokens, measured slower there on GB300: o
    // 63 against 48 us, down 275 against 219 us); 128 only for at most 128 tokens
    const int BN = T <= 128 ? 128 : 256;
    CUtensorMap tmW, tmX, tmXh;
    if (!make_map(&tmW, W16, R, K, kGemmBM) || !make_map(&tmX, X16, T, K, BN) || !make_map(&tmXh, X16, T, K, BN / 2))
        return cudaErrorInvalidValue;
    GemmArgs a;
    a.R = R;
    a.K = K;
    a.T = T;
    a.m_tiles = m_tiles;
    a.n_tiles = (T + BN - 1) / BN;
    a.k_steps = K / kGemmBK;
    a.limit_ns = uint64_t(fault_policy() == FAULT_NONE ? 2000 : 50) * 1000000ull;
    const int tiles = a.m_tiles * a.n_tiles;
    const int grid = tiles < num_sms ? tiles : num_sms;
    // a last wave that fills at most half the CTAs runs as twice as many
    // half-width tiles: 224 tiles on 152 CTAs take 1.5 tile times, not 2
    const int rem = tiles % grid;
    a.full_tiles = tiles;
    a.ntiles = tiles;
    if (BN == 256 && tiles > grid && rem > 0 && 2 * rem <= grid) {
        a.full_tiles = tiles - rem;
        a.ntiles = a.full_tiles + 2 * rem;
    }
    if (BN == 256)
        gemm_f16_kernel<256><<<grid, kGemmThreads, GemmTile<256>::kSmem, s>>>(tmW, tmX, tmXh, Y, a, status);
    else
        gemm_f16_kernel<128><<<grid, kGemmThreads, GemmTile<128>::kSmem, s>>>(tmW, tmX, tmXh, Y, a, status);
    return cudaGetLastError();
}

}  // namespace mq
