// mq_internal.h -- host-side plan and launcher declarations shared by the
// libmq translation units.  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mq.h"

namespace mq {

// Launch plan of one streaming matvec kernel.  Computed on the host from the
// shapes alone, so it is a pure function of the capture key ("Part 4 .
// Lecture 08 -- Graph-Resident Decode", section 2: grid sizes are decided on
// the host by one function, shared by the launcher and any probe).
struct MvPlan {
    int C;             // chunks (64 weights) per row = K/64
    int L;             // lanes per work item: 8, 16 or 32
    int nseg;          // K segments per row (one work item = one row segment)
    int S;             // chunks per segment (<= L, a multiple of 4)
    int rows_per_cta;  // max rows handled by one CTA
    int grid;          // CTAs
    int block;         // threads per CTA
    int smem;          // dynamic shared memory bytes
    // bulk-copy ring variant (variant == 1)
    int variant;       // 0: register-streaming kernels, 1: bulk-copy ring kernels
    int nwc;           // consumer warps (one more warp is the producer)
    int rg;            // row-lanes per segment: consumer rows advance by rg
    int T;             // rows per tile (a multiple of rg)
    int ns;            // ring stages
    int stage_bytes;   // bytes per stage (128-byte multiple)
    int off_ring, off_act, off_part, off_vals;  // shared-memory offsets
    int fault;         // test-only: FAULT_* injected by the ring kernels (0 = none)
    int wait_ms;       // limit of every mbarrier wait of the ring kernels
    int cmap;          // 1: column lanes (3..8 columns, ring_consume_cols), 0: unit lanes
    // column groups (3..8 columns, q4_K): the consumer warps form groups of cgw
    // warps, group g on columns 2g, 2g+1 with their activation in registers (the
    // one- and two-column consumer), cgu of each group's warps with work; 0: off
    int cgw, cgu;
    // half-unit lanes (4 or 8 columns): the unit split above counts half-units
    // and the groups take four columns each (cgw, cgu as for column groups)
    int hu;
    // K split (matvec and down, q4_K, when one launch cannot stage the whole
    // activation): ksplit launches in stream order, each over kpn super-blocks
    // of every row starting at super-block kp0; launch i > 0 adds its sums to y
    // (kacc = 1), so y = ((part 0) + part 1) + ... in that order.  kpn = 0: the
    // whole row in one launch.
    int ksplit, kp0, kpn, kacc;
};

// Plan of the persistent step kernel: one ring plan per phase (qkv, o, gate/up,
// down) sharing the ring geometry and shared-memory layout of the phases.
// Persistent-step workspace (bytes): [0, 256) control words (word 1: abort,
// word 2: the phase counter), [256, 4352) reserved (one u32 per CTA), then the
// h records: per column
// 40 * (I/128) records of 8 bytes (a 32-bit word of the activation's unit
// layout and the phase that wrote it); for a chained step, then the output
// records of the qkv, o and down phases: per phase ncols * rows records of 8
// bytes (an fp32 output and the phase that wrote it), column-major, each
// phase's area rounded up to 32 bytes.
constexpr int kWsCountWord = 2;  // the phase counter: every CTA adds one per finished phase
constexpr int kWsFlagsOff = 256;
constexpr int kWsMaxCtas = 1024;
constexpr int kWsRecOff = kWsFlagsOff + 4 * kWsMaxCtas;
static_assert(kWsRecOff == MQ_STEP_WORKSPACE_BYTES, "workspace layout and header disagree");

struct StepWorkspace {
    size_t bytes;
    int64_t yrec_off[4];  // byte offset of phase ph's output records (-1: none; gate/up never has any)
};

inline StepWorkspace step_workspace(const mq_step_shape& h)
{
    StepWorkspace w;
    size_t off = size_t(kWsRecOff) + size_t(h.ncols) * (h.I / 128) * 40 * 8;
    const int64_t rows[4] = {h.qkv_rows, h.o_rows, 0, h.H};
    for (int ph = 0; ph < 4; ++ph) {
        w.yrec_off[ph] = -1;
        if ((h.flags & MQ_STEP_CHAINED) && rows[ph] > 0) {
            w.yrec_off[ph] = int64_t(off);
            off += (size_t(h.ncols) * size_t(rows[ph]) * 8 + 31) / 32 * 32;  // records are read 16 bytes at a time
        }
    }
    w.bytes = off;
    return w;
}

struct StepPlan {
    size_t ws_bytes;  // workspace the launch zeroes and uses
    MvPlan ph[4];
    int K[4];      // reduction length per phase
    int R[4];      // rows per phase (gate/up: I); 0 = phase left out
    int n_layers;
    int pf_tiles;  // tiles the producer prefetches into L2 beyond its next ring copy
    int nwc;       // consumer warps of the kernel (phases may use fewer)
    int grid;
    int smem;
    int chained;              // MQ_STEP_CHAINED: inputs are the previous phase's output records
    int64_t yrec_off[4];      // byte offsets of the output records in the workspace (-1: none)
};

// test-only fault injection (mq_debug_set_fault)
enum Fault { FAULT_NONE = 0, FAULT_WITHHOLD_TILE = 1, FAULT_WITHHOLD_RECORDS = 2, FAULT_WITHHOLD_COUNT = 3 };
int fault_policy();

enum Kind { KIND_MV = 0, KIND_DOWN = 1, KIND_GU = 2 };

// kernel family selection (test hook; 0 = automatic)
enum VariantPolicy { VARIANT_AUTO = 0, VARIANT_FORCE_REGISTER = 1 };
int variant_policy();

struct DeviceInfo {
    int num_sms = 0;
    int max_smem_optin = 0;
    int l2_bytes = 0;
    unsigned* status = nullptr;  // device status word
    bool ready = false;
};

// the calling thread's current device, initialised by mq_init (nullptr otherwise)
const DeviceInfo* current_device_info();
// records e for mq_last_cuda_error on the calling thread; returns MQ_ERR_CUDA
mq_status record_cuda_error(cudaError_t e);

// returns false if the shapes cannot be planned within the device limits
// unit_bytes: row bytes per 128 weights (72 for q4_K and q4_0, 136 for q8_0 weights)
// ring_only: plan the bulk-copy ring kernels whatever the variant policy
bool plan_mv(int64_t rows, int K, int ncols, int kind, int I, const DeviceInfo& dev, MvPlan* p, int unit_bytes = 72,
             bool ring_only = false);

cudaError_t launch_quantize(const float* x, void* xq, int64_t nblocks, cudaStream_t s);
// launch_mv / launch_gu dispatch on p.variant
cudaError_t launch_mv(const void* desc, int kind, int rows, int K, int ncols, const MvPlan& p,
                      unsigned* status, cudaStream_t s, bool pdl);
cudaError_t launch_gu(const mq_ffn_desc* d, int H, int I, int ncols, const MvPlan& p, unsigned* status,
                      cudaStream_t s, bool pdl);
cudaError_t launch_ring(const void* desc, int kind, int a, int b, int ncols, const MvPlan& p, unsigned* status,
                        cudaStream_t s, bool pdl);
// the matvec for q4_0 / q8_0 weights (wtype MQ_TYPE_Q4_0 or MQ_TYPE_Q8_0), ring plans only
cudaError_t launch_wring(const void* desc, int wtype, int rows, int K, int ncols, const MvPlan& p, unsigned* status,
                         cudaStream_t s, bool pdl);
bool plan_step(const mq_step_shape& h, const DeviceInfo& dev, StepPlan* sp);
cudaError_t launch_step(const mq_layer_desc* layers, const StepPlan& sp, int ncols, unsigned* status, unsigned* ws,
                        cudaStream_t s);
cudaError_t launch_block_sums(const mq_mv_desc* d, int rows, int K, int ncols, int32_t* sumi, int32_t* sumq,
                              int smem, unsigned* status, cudaStream_t s);
// raises the dynamic shared memory limit of every kernel on the current device
cudaError_t set_kernel_attributes(int max_smem);
// small-batch matmul on the tensor cores (mmq.cu)
struct MmqPlan {
    int np;           // columns rounded up to 16 (the MMA's N)
    int nkb;          // super-blocks per row
    int m_tiles;      // 128-row tiles
    int ksplit;       // K ranges per tile (partials summed in a fixed order)
    int stages, stage_bytes, smem, grid;
    int nab;          // half-step A buffers
    size_t bimg_bytes, sc_bytes, part_bytes, ws_bytes;  // workspace: activation image, scales, partials
};
MmqPlan plan_mmq(int rows, int K, int ncols, int num_sms, int max_smem);
cudaError_t launch_mmq(const mq_mv_desc* d, int rows, int K, int ncols, const MmqPlan& p, void* ws, int num_sms,
                       unsigned* status, cudaStream_t s);
// prefill operands and GEMM (dequant.cu, gemm.cu)
cudaError_t launch_dequant_q4K_f16(const void* W, void* W16, int64_t nblocks, int num_sms, cudaStream_t s);
cudaError_t launch_f32_to_f16(const float* x, void* y, int64_t n, int num_sms, cudaStream_t s);
cudaError_t launch_gemm_f16(const void* W16, const void* X16, float* Y, int R, int K, int T, int num_sms,
                            unsigned* status, cudaStream_t s);
// looks up the device address of the no-alloc FFN's fixed scratch on device
// `dev` (current) and caches it
cudaError_t noalloc_setup(int dev);

}  // namespace mq

namespace mq {
// Raise a kernel's dynamic shared-memory limit to the device's opt-in maximum
// minus the kernel's own static shared memory.
inline cudaError_t set_max_dyn_smem(const void* func, int max_optin)
{
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, func);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin - int(a.sharedSizeBytes));
}
}  // namespace mq
