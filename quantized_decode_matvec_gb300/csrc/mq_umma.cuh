// mq_umma.cuh -- inline-PTX helpers for the 5th-generation tensor cores of
// sm_103a: tensor-memory (TMEM) allocation, tcgen05.mma of kind::f16 with
// both operands in shared memory, its commit to an mbarrier, tcgen05.ld of
// the fp32 accumulator, and tiled TMA loads (cp.async.bulk.tensor).
//
// Operand layout: K-major tiles with the 128-byte swizzle, as a tiled TMA
// load with CU_TENSOR_MAP_SWIZZLE_128B writes them: a tile of rows x 64 f16
// (128 bytes per row), row r at byte 128r, its 16-byte chunk c at chunk
// position c ^ (r % 8), the tile 1024-byte aligned.  The matrix descriptor
// of such a tile has stride-dimension offset 1024 bytes (eight rows); a
// K-step of 16 elements inside the 128-byte row advances the start address
// by 32 bytes (the swizzle is a function of the address bits, so the offset
// start keeps the pattern).
#pragma once

#include <stdint.h>

#include "mq_tma.cuh"

namespace mq {

// ---- shared-memory matrix descriptor (64 bits) -------------------------------------
//   [0,14) start address >> 4, [16,30) leading-dimension byte offset >> 4,
//   [32,46) stride-dimension byte offset >> 4, [46,48) version (1),
//   [49,52) base offset, [52] LBO mode, [61,64) layout (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= uint64_t((smem_addr >> 4) & 0x3FFFu);
    d |= uint64_t(1u) << 16;              // leading-dimension offset: unused for a swizzled K-major tile
    d |= uint64_t(1024u >> 4) << 32;      // stride-dimension offset: eight 128-byte rows
    d |= uint64_t(1u) << 46;              // descriptor version of this architecture
    d |= uint64_t(2u) << 61;              // 128-byte swizzle
    return d;
}

// ---- instruction descriptor of kind::f16 (32 bits) ----------------------------------
//   [4,6) D format (1 = f32), [7,10) A format (0 = f16), [10,13) B format
//   (0 = f16), [15] A major (0 = K), [16] B major (0 = K), [17,23) N >> 3,
//   [24,29) M >> 4
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32(int M, int N)
{
    return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// ---- tensor memory ----------------------------------------------------------------------
// allocate ncols columns (a power of two >= 32) for this CTA; one whole warp
// calls it; the base address is written to *dst (shared memory)
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one MMA of M x N x 16 (issued by one thread)
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// the mbarrier completes (one arrival) once every tcgen05 operation this
// thread issued before has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes
// 32*(w%4) .. +31; taddr carries the lane base in its upper half)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- tiled TMA ---------------------------------------------------------------------------
// 2-D tile {x (inner, elements), y (rows)} of the tensor map into shared
// memory, completion counted on bar.  x * element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

}  // namespace mq
