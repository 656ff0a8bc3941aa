// api.cu -- the extern "C" boundary of libmq (declared in include/mq.h):
// argument validation, launch planning and launches.  No allocation after
// mq_init, no synchronization and no host read of device memory inside a
// compute call, so every compute call can be captured into a CUDA graph.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "mq.h"
#include "mq_internal.h"

namespace mq {
cudaError_t set_mv_attributes(int max_smem);
cudaError_t set_gu_attributes(int max_smem);
cudaError_t set_ring_attributes(int max_smem);
cudaError_t set_step_attributes(int max_smem);
cudaError_t set_wring_attributes(int max_smem);
cudaError_t set_ring_cols_attributes(int max_smem);
cudaError_t set_ring_split_attributes(int max_smem);
cudaError_t set_gemm_attributes(int max_smem);
cudaError_t set_mmq_attributes(int max_smem);
void plan_ring(MvPlan& q, int64_t units, int kind, int nc, const DeviceInfo& dev, int64_t unit_bytes,
               bool allow_cols);
}  // namespace mq

namespace {

constexpr int kMaxDevices = 64;
mq::DeviceInfo g_dev[kMaxDevices];
thread_local int g_last_cuda_error = 0;
int g_variant_policy = mq::VARIANT_AUTO;  // set only through mq_debug_set_variant (tests)
int g_fault_policy = mq::FAULT_NONE;       // set only through mq_debug_set_fault (tests)

// Device status word (one per device that loads the library): kernels OR in
// MQ_DEV_* bits when their device descriptor disagrees with their launch.
__device__ unsigned g_status_word;

mq_status cuda_fail(cudaError_t e)
{
    g_last_cuda_error = int(e);
    return MQ_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

mq_status current_dev(const mq::DeviceInfo** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices || !g_dev[dev].ready) return MQ_ERR_NOT_INITIALIZED;
    *out = &g_dev[dev];
    return MQ_OK;
}

mq_status check_mv_shape(int64_t rows, int64_t K, int64_t ncols)
{
    if (rows < 0 || ncols < 0 || K < 0) return MQ_ERR_SHAPE;
    if (ncols > MQ_MAX_NCOLS) return MQ_ERR_SHAPE;
    if (K == 0 || K % 256) return MQ_ERR_SHAPE;
    if (K > MQ_MAX_K || K * ncols > MQ_MAX_K_TIMES_NCOLS || rows > INT32_MAX) return MQ_ERR_UNSUPPORTED;
    return MQ_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

namespace mq {

const DeviceInfo* current_device_info()
{
    const DeviceInfo* d = nullptr;
    return current_dev(&d) == MQ_OK ? d : nullptr;
}

mq_status record_cuda_error(cudaError_t e) { return cuda_fail(e); }

int variant_policy() { return g_variant_policy; }
int fault_policy() { return g_fault_policy; }

bool plan_mv(int64_t rows, int K, int nc, int kind, int I, const DeviceInfo& dev, MvPlan* p, int unit_bytes,
             bool ring_only)
{
    MvPlan q = {};
    q.C = K / 64;
    if (q.C <= 8) {
        q.L = 8;
        q.nseg = 1;
    } else if (q.C <= 16) {
        q.L = 16;
        q.nseg = 1;
    } else {
        q.L = 32;
        q.nseg = (q.C + 31) / 32;
    }
    // segments of whole super-blocks (4 chunks), at most L chunks
    q.S = ((q.C + q.nseg - 1) / q.nseg + 3) / 4 * 4;
    q.nseg = (q.C + q.S - 1) / q.S;
    // distribution unit: a row, or for the gate/up kernel a 32-index block of h
    const int64_t units = (kind == KIND_GU) ? I / 32 : rows;
    if (units <= 0) return false;
    int64_t G = units < dev.num_sms ? units : dev.num_sms;
    int64_t rpc = 0, smem = 0;
    for (;;) {
        const int64_t upc = (units + G - 1) / G;
        rpc = (kind == KIND_GU) ? upc * 64 : upc;
        smem = int64_t(nc) * q.C * 80 + rpc * q.nseg * nc * 4 + ((kind == KIND_GU) ? int64_t(nc) * rpc * 4 : 0);
        if (smem <= dev.max_smem_optin) break;
        if (upc == 1) return false;
        G = (G + dev.num_sms < units) ? G + dev.num_sms : units;
    }
    const int ipw = 32 / q.L;
    int64_t nw = (rpc * q.nseg + ipw - 1) / ipw;
    if (nw < 4) nw = 4;
    if (nw > 16) nw = 16;
    q.rows_per_cta = int(rpc);
    q.grid = int(G);
    q.block = int(32 * nw);
    q.smem = int(smem);
    q.variant = 0;
    q.ksplit = 1;
    if (ring_only || variant_policy() != VARIANT_FORCE_REGISTER)
        plan_ring(q, units, kind, nc, dev, unit_bytes, !ring_only);  // column lanes: q4_K only
    if (q.variant == 0 && !ring_only && kind != KIND_GU && variant_policy() != VARIANT_FORCE_REGISTER) {
        // the whole activation does not fit beside a ring (e.g. eight columns of
        // K = 18944): split K into 2..4 equal parts of whole super-blocks, one
        // ring launch each, one CTA per SM
        const int sb = K / 256;  // super-blocks per row
        for (int ks = 2; ks <= 4; ++ks) {
            if (sb % ks) continue;
            MvPlan qs = q;
            qs.C = (K / ks) / 64;
            qs.grid = int(units < dev.num_sms ? units : dev.num_sms);
            qs.rows_per_cta = int((units + qs.grid - 1) / qs.grid);
            plan_ring(qs, units, kind, nc, dev, unit_bytes, true);
            if (qs.variant == 1) {
                qs.ksplit = ks;
                qs.kpn = sb / ks;
                q = qs;
                break;
            }
        }
    }
    *p = q;
    return true;
}

// How the consumer warps split a row of C units (128 weights each) for nc
// columns, shared by the per-matrix and the persistent plans so that both
// reduce in the same order (bit-identical results):
//  * unit lanes (1..4 columns, or 5..8 when column lanes do not fit): L lanes
//    per (row, segment) item, lane l on unit seg*S + l, nseg segments of S <= L
//    units, up to 15 consumer warps (1..2 columns: the L of 32, 16, 8, 4 with
//    the fewest idle lanes and warps; 3..8 columns: 8 warps when they divide
//    evenly);
//  * column lanes (5..8 columns, q4_K, when the segments fit in 15 warps):
//    one item per warp, lane = (unit-lane, column), 4 unit-lanes per item, 15
//    consumer warps.  (Measured on GB300: faster than unit lanes from 5
//    columns up, slower at 3 and 4, where the unit lanes' once-per-unit scale
//    unpacking wins.)
// Returns false when the segments do not fit in the warps.
// 3..8 columns of q4_K weights as column groups where the split fits
constexpr bool kColumnGroups = true;
// 4 or 8 columns of q4_K weights on half-unit lanes where the split fits
constexpr bool kHalfUnits = true;

static bool unit_split(int C, int nc, bool allow_cols, MvPlan& q)
{
    q.cmap = 0;
    q.cgw = q.cgu = 0;
    q.hu = 0;
    if ((nc == 4 || nc == 8) && allow_cols && kHalfUnits) {
        // half-unit lanes, groups of four columns: the split counts 2C half-units
        const int ng = nc / 4, wpg = 15 / ng, CH = 2 * C;
        double best = 0.0;
        for (const int L : {32, 16, 8, 4}) {
            int nseg = (CH + L - 1) / L;
            const int S = (CH + nseg - 1) / nseg;
            nseg = (CH + S - 1) / S;
            if (nseg > wpg) continue;
            const int used = nseg * (wpg / nseg);
            const double score = double(CH) / double(nseg * L) * double(used) / double(wpg);
            if (score > best + 1e-9) {
                best = score;
                q.L = L;
                q.nseg = nseg;
                q.S = S;
                q.cgu = used;
            }
        }
        if (best > 0.0) {
            q.hu = 1;
            q.cgw = wpg;
            q.nwc = ng * wpg;
            q.rg = (q.cgu / q.nseg) * (32 / q.L);
            return true;
        }
        q.cgu = 0;
    }
    if (nc >= 3 && allow_cols && kColumnGroups) {
        // column groups: (nc+1)/2 groups of 15/groups warps, each group split as
        // the two-column consumer would split its warps
        const int ng = (nc + 1) / 2, wpg = 15 / ng;
        double best = 0.0;
        for (const int L : {32, 16, 8, 4}) {
            int nseg = (C + L - 1) / L;
            const int S = (C + nseg - 1) / nseg;
            nseg = (C + S - 1) / S;
            if (nseg > wpg) continue;
            const int used = nseg * (wpg / nseg);
            const double score = double(C) / double(nseg * L) * double(used) / double(wpg);
            if (score > best + 1e-9) {
                best = score;
                q.L = L;
                q.nseg = nseg;
                q.S = S;
                q.cgu = used;
            }
        }
        if (best > 0.0) {
            q.cgw = wpg;
            q.nwc = ng * wpg;
            q.rg = (q.cgu / q.nseg) * (32 / q.L);
            return true;
        }
        q.cgu = 0;
    }
    if (nc >= 5 && allow_cols) {
        const int lu = 32 / (nc <= 4 ? 4 : 8);
        int nseg = (C + lu - 1) / lu;
        const int S = (C + nseg - 1) / nseg;
        nseg = (C + S - 1) / S;
        if (nseg <= 15) {
            q.cmap = 1;
            q.L = 32;  // one item per warp
            q.nseg = nseg;
            q.S = S;
            q.nwc = nseg * (15 / nseg);
            q.rg = q.nwc / nseg;
            return true;
        }
    }
    if (nc <= 2) {
        // Unit lanes, 1..2 columns: the consumers are issue-bound, so pick the
        // items of L lanes (32, 16, 8 or 4) that leave the fewest lanes and
        // warps idle; ties go to the longer items (fewer partials per row).
        // K = 3584, 28 units: 7 segments of 4 units on 4-lane items in 14 warps
        // (every lane busy) instead of one segment of 28 on 32 lanes.
        double best = 0.0;
        for (const int L : {32, 16, 8, 4}) {
            int nseg = (C + L - 1) / L;
            const int S = (C + nseg - 1) / nseg;
            nseg = (C + S - 1) / S;
            if (nseg > 15) continue;
            const int nwc = nseg * (15 / nseg);
            const double score = double(C) / double(nseg * L) * double(nwc) / 15.0;
            if (score > best + 1e-9) {
                best = score;
                q.L = L;
                q.nseg = nseg;
                q.S = S;
                q.nwc = nwc;
            }
        }
        if (best <= 0.0) return false;
        q.rg = (q.nwc / q.nseg) * (32 / q.L);
        return true;
    }
    if (C <= 8) {
        q.L = 8;
        q.nseg = 1;
    } else if (C <= 16) {
        q.L = 16;
        q.nseg = 1;
    } else {
        q.L = 32;
        q.nseg = (C + 31) / 32;
    }
    q.S = (C + q.nseg - 1) / q.nseg;
    q.nseg = (C + q.S - 1) / q.S;
    if (q.nseg > 15) return false;
    // 3..8 columns: 8 warps (9-warp kernel, more registers per thread) when the
    // segments fill them, else up to 15 (16-warp kernel): long rows split into
    // 3, 5, 6, 7 ... segments would leave most of the 8 warps idle
    const int w8 = (q.nseg <= 8) ? q.nseg * (8 / q.nseg) : 0;
    q.nwc = (nc >= 3 && w8 == 8) ? 8 : q.nseg * (15 / q.nseg);
    q.rg = (q.nwc / q.nseg) * (32 / q.L);
    return true;
}

// Bulk-copy ring plan on top of a register-streaming plan q (same rows per CTA,
// same segments).  Leaves q unchanged when the ring does not apply.
//  * consumers: nwc warps from unit_split, segment-stationary,
//    rg = warps per segment * items per warp row-lanes;
//  * tiles of T = 2*rg*m rows (about 24 KB), at most the CTA's rows rounded up;
//  * 2..8 stages, within ~110 KB of shared memory when possible so that the
//    next kernel's CTA fits beside this one under programmatic dependent launch.
void plan_ring(MvPlan& q0, int64_t units, int kind, int nc, const DeviceInfo& dev, int64_t unit_bytes,
               bool allow_cols)
{
    // work unit: half a super-block (128 weights); C counts units per row here
    MvPlan q = q0;
    q.C = q0.C / 2;
    if (!unit_split(q.C, nc, allow_cols, q)) return;
    const int nwc = q.nwc;
    const int rg = q.rg;
    const int64_t row_bytes = int64_t(q.C) * unit_bytes;  // q.C units of 128 weights
    // tiles of whole row pairs per row-lane (consumers take two rows per step)
    const int64_t unit = 2 * rg * row_bytes;
    int64_t m = (24576 + unit / 2) / unit;
    if (m < 1) m = 1;
    int64_t T = 2 * rg * m;
    // tiles of at most ~64 KB (wide rows, e.g. q8_0 weights: fewer rows than a
    // full step of the row-lanes; the consumers handle any tile height)
    if (T * row_bytes > 65536) T = 65536 / row_bytes > 1 ? 65536 / row_bytes : 1;
    // no tile beyond the CTA's rows; a CTA's few rows beyond one tile (q|k|v:
    // 31 rows, tiles of 30) ride in that tile rather than in a tile of their own
    if (T > q.rows_per_cta || (q.rows_per_cta * row_bytes <= 65536)) T = q.rows_per_cta;
    const int64_t stage = (T * row_bytes + 127) / 128 * 128;
    const int64_t act = int64_t(nc) * q.C * 160;
    const int64_t part = int64_t(q.rows_per_cta) * q.nseg * nc * 4;
    const int64_t vals = (kind == KIND_GU) ? int64_t(nc) * q.rows_per_cta * 4 : 0;
    const int64_t fixed = 256 + act + (part + 15) / 16 * 16 + vals;
    const int64_t pair_budget = 110 * 1024;
    // (the ring kernel also has a few bytes of static shared memory)
    const int64_t budget = (fixed + 4 * stage <= pair_budget) ? pair_budget : dev.max_smem_optin - 256;
    int64_t ns = (budget - fixed) / stage;
    if (ns > 8) ns = 8;
    if (ns < 2) return;
    (void)units;
    q.variant = 1;
    q.fault = fault_policy();
    q.wait_ms = q.fault == FAULT_NONE ? 2000 : 50;
    q.nwc = nwc;
    q.rg = rg;
    q.T = int(T);
    q.ns = int(ns);
    q.stage_bytes = int(stage);
    q.off_ring = 256;
    q.off_act = int(q.off_ring + ns * stage);
    q.off_part = int(q.off_act + act);
    q.off_vals = int(q.off_part + (part + 15) / 16 * 16);
    q.smem = int(q.off_vals + vals);
    q.block = 32 * (nwc + 1);
    q0 = q;
}

// Plan of the persistent step kernel.  Per phase the same unit split as the
// per-matrix ring kernels (so results are bit-identical); one ring shared by
// all phases: stages as large as the largest phase tile (about 64 KB: two rows
// per row-lane), as many as fit beside the largest activation, partial and
// gate/up buffers.
bool plan_step(const mq_step_shape& h, const DeviceInfo& dev, StepPlan* out)
{
    StepPlan sp = {};
    const int nc = h.ncols;
    int nwc_max = 1;  // consumer warps of the kernel: the most any phase uses
    const int64_t G = dev.num_sms;
    const int kinds[4] = {KIND_MV, KIND_MV, KIND_GU, KIND_DOWN};
    const int64_t Ks[4] = {h.H, h.o_K, h.H, h.I};
    const int64_t Rs[4] = {h.qkv_rows, h.o_rows, h.I, h.H};
    int64_t stage = 0, act = 0, part = 0, vals = 0;
    for (int ph = 0; ph < 4; ++ph) {
        MvPlan q = {};
        if (Rs[ph] == 0) {  // a projection left out: no tiles, no staging
            q.T = 1;
            sp.ph[ph] = q;
            continue;
        }
        q.C = int(Ks[ph] / 128);
        if (!unit_split(q.C, nc, true, q)) return false;
        if (q.nwc > nwc_max) nwc_max = q.nwc;
        const bool gu = kinds[ph] == KIND_GU;
        const int64_t units = gu ? Rs[ph] / 32 : Rs[ph];
        const int64_t upc = (units + G - 1) / G;
        const int64_t rpc = gu ? upc * 64 : upc;
        const int64_t row_bytes = int64_t(q.C / 2) * 144;
        const int64_t unit2 = 2 * int64_t(q.rg) * row_bytes;
        int64_t m = 65536 / unit2;
        if (m < 1) m = 1;
        int64_t T = 2 * int64_t(q.rg) * m;
        const int64_t rpc_round = (rpc + 2 * q.rg - 1) / (2 * q.rg) * (2 * q.rg);
        if (T > rpc_round) T = rpc_round;
        if (rpc > T && rpc * row_bytes <= 65536) T = rpc;  // a few rows beyond one tile ride in it
        q.T = int(T);
        q.rows_per_cta = int(rpc);
        q.variant = 1;
        const int64_t st = (T * row_bytes + 127) / 128 * 128;
        if (st > stage) stage = st;
        if (int64_t(nc) * q.C * 160 > act) act = int64_t(nc) * q.C * 160;
        if (rpc * q.nseg * nc * 4 > part) part = rpc * q.nseg * nc * 4;
        if (gu) vals = int64_t(nc) * rpc * 4;
        sp.ph[ph] = q;
        sp.K[ph] = int(Ks[ph]);
        sp.R[ph] = int(Rs[ph]);
    }
    const int64_t fixed = 256 + act + (part + 15) / 16 * 16 + vals;
    int64_t ns = (dev.max_smem_optin - 256 - fixed) / stage;  // the kernel has a few static bytes too
    if (ns > 8) ns = 8;
    if (ns < 2) return false;
    // the input/output overlap check keeps 16 byte ranges per layer in the ring's memory
    if (int64_t(h.n_layers) * 16 * 16 > ns * stage) return false;
    const int off_ring = 256, off_act = int(256 + ns * stage), off_part = int(off_act + act);
    const int off_vals = int(off_part + (part + 15) / 16 * 16);
    for (int ph = 0; ph < 4; ++ph) {
        MvPlan& q = sp.ph[ph];
        q.ns = int(ns);
        q.stage_bytes = int(stage);
        q.off_ring = off_ring;
        q.off_act = off_act;
        q.off_part = off_part;
        q.off_vals = off_vals;
        q.grid = int(G);
        q.fault = fault_policy();
        q.wait_ms = q.fault == FAULT_NONE ? 2000 : 50;
    }
    sp.n_layers = h.n_layers;
    // L2 prefetch window: the whole grid's prefetched tiles take at most a
    // third of the L2 (wider windows measured slower on GB300: they evict
    // prefetched tiles before use and crowd the critical path's loads)
    int64_t pf = int64_t(dev.l2_bytes) / 3 / (G * stage);
    sp.pf_tiles = int(pf < 0 ? 0 : (pf > 16 ? 16 : pf));
    sp.nwc = nwc_max;
    sp.grid = int(G);
    if (sp.grid > kWsMaxCtas) return false;  // the workspace reserves one word per CTA
    sp.smem = int(off_vals + vals);
    const StepWorkspace w = step_workspace(h);
    sp.ws_bytes = w.bytes;
    sp.chained = (h.flags & MQ_STEP_CHAINED) != 0;
    for (int ph = 0; ph < 4; ++ph) sp.yrec_off[ph] = w.yrec_off[ph];
    *out = sp;
    return true;
}

cudaError_t set_kernel_attributes(int max_smem)
{
    cudaError_t e = set_mv_attributes(max_smem);
    if (e == cudaSuccess) e = set_gu_attributes(max_smem);
    if (e == cudaSuccess) e = set_ring_attributes(max_smem);
    if (e == cudaSuccess) e = set_step_attributes(max_smem);
    if (e == cudaSuccess) e = set_wring_attributes(max_smem);
    if (e == cudaSuccess) e = set_ring_cols_attributes(max_smem);
    if (e == cudaSuccess) e = set_ring_split_attributes(max_smem);
    if (e == cudaSuccess) e = set_gemm_attributes(max_smem);
    if (e == cudaSuccess) e = set_mmq_attributes(max_smem);
    return e;
}

}  // namespace mq

extern "C" {

const char* mq_status_string(mq_status s)
{
    switch (s) {
        case MQ_OK: return "ok";
        case MQ_ERR_INVALID_ARG: return "invalid argument";
        case MQ_ERR_SHAPE: return "invalid shape";
        case MQ_ERR_ALIGN: return "misaligned pointer";
        case MQ_ERR_CUDA: return "CUDA error";
        case MQ_ERR_UNSUPPORTED: return "size beyond the library's limits";
        case MQ_ERR_NOT_INITIALIZED: return "mq_init was not called for this device";
        default: return "unknown status";
    }
}

int mq_abi_version(void) { return MQ_ABI_VERSION; }

mq_status mq_debug_set_fault(int32_t fault)
{
    if (fault != mq::FAULT_NONE && fault != mq::FAULT_WITHHOLD_TILE && fault != mq::FAULT_WITHHOLD_RECORDS &&
        fault != mq::FAULT_WITHHOLD_COUNT)
        return MQ_ERR_INVALID_ARG;
    g_fault_policy = fault;
    return MQ_OK;
}

mq_status mq_debug_set_variant(int32_t policy)
{
    if (policy != mq::VARIANT_AUTO && policy != mq::VARIANT_FORCE_REGISTER) return MQ_ERR_INVALID_ARG;
    g_variant_policy = policy;
    return MQ_OK;
}

int mq_last_cuda_error(void) { return g_last_cuda_error; }

mq_status mq_init(int device)
{
    if (device < 0 || device >= kMaxDevices) return MQ_ERR_INVALID_ARG;
    int prev = 0;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((e = cudaSetDevice(device)) != cudaSuccess) return cuda_fail(e);
    mq::DeviceInfo info;
    mq_status st = MQ_OK;
    do {
        if ((e = cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess) break;
        if ((e = cudaDeviceGetAttribute(&info.l2_bytes, cudaDevAttrL2CacheSize, device)) != cudaSuccess) break;
        if ((e = cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device)) !=
            cudaSuccess)
            break;
        if ((e = mq::set_kernel_attributes(info.max_smem_optin)) != cudaSuccess) break;
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) break;
        info.status = static_cast<unsigned*>(p);
        if ((e = cudaMemset(info.status, 0, sizeof(unsigned))) != cudaSuccess) break;
        if ((e = mq::noalloc_setup(device)) != cudaSuccess) break;
        if ((e = cudaDeviceSynchronize()) != cudaSuccess) break;
        info.ready = true;
    } while (0);
    if (e != cudaSuccess) st = cuda_fail(e);
    cudaSetDevice(prev);
    if (st == MQ_OK) g_dev[device] = info;
    return st;
}

mq_status mq_read_device_status(uint32_t* bits, void* stream)
{
    if (!bits) return MQ_ERR_INVALID_ARG;
    const mq::DeviceInfo* dev = nullptr;
    mq_status st = current_dev(&dev);
    if (st != MQ_OK) return st;
    cudaError_t e;
    unsigned v = 0;
    if ((e = cudaMemcpyAsync(&v, dev->status, sizeof(unsigned), cudaMemcpyDeviceToHost, as_stream(stream))) !=
        cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaMemsetAsync(dev->status, 0, sizeof(unsigned), as_stream(stream))) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamSynchronize(as_stream(stream))) != cudaSuccess) return cuda_fail(e);
    *bits = v;
    return MQ_OK;
}

size_t mq_q4K_row_bytes(int64_t K) { return (K < 0 || K % 256) ? 0 : size_t(K / 256) * 144; }

size_t mq_q8_0_bytes(int64_t K) { return (K < 0 || K % 32) ? 0 : size_t(K / 32) * 34; }

int mq_quant_block_elems(int32_t ttype)
{
    return ttype == MQ_TYPE_Q4_K ? 256 : (ttype == MQ_TYPE_Q8_0 || ttype == MQ_TYPE_Q4_0) ? 32 : 0;
}

int mq_quant_block_bytes(int32_t ttype)
{
    return ttype == MQ_TYPE_Q4_K ? 144 : ttype == MQ_TYPE_Q8_0 ? 34 : ttype == MQ_TYPE_Q4_0 ? 18 : 0;
}

// Mirrors mq_concat_rows' preconditions clause by clause ("04 . 8o",
// section 3.2): at least two tensors, one type, one ne0 that is a multiple of
// the block size, and each tensor's bytes == rows * row bytes.
int mq_concat_rows_feasible(int32_t n, const int32_t* ttype, const int64_t* ne0, const int64_t* ne1,
                            const uint64_t* nbytes)
{
    if (n < 2 || !ttype || !ne0 || !ne1 || !nbytes) return 0;
    const int32_t tt = ttype[0];
    for (int32_t i = 0; i < n; ++i)
        if (ttype[i] != tt) return 0;
    const int bq = mq_quant_block_elems(tt), bb = mq_quant_block_bytes(tt);
    if (bb == 0) return 0;
    const int64_t k = ne0[0];
    for (int32_t i = 0; i < n; ++i)
        if (ne0[i] != k) return 0;
    if (k <= 0 || k % bq) return 0;
    const uint64_t row = uint64_t(k / bq) * uint64_t(bb);
    for (int32_t i = 0; i < n; ++i)
        if (ne1[i] < 0 || nbytes[i] != row * uint64_t(ne1[i])) return 0;
    return 1;
}

mq_status mq_concat_rows(void* dst, const void* const* srcs, const int64_t* rows, int32_t n, int32_t ttype,
                         int64_t ne0, void* stream)
{
    if (!dst || !srcs || !rows || n < 2) return MQ_ERR_INVALID_ARG;
    const int bq = mq_quant_block_elems(ttype), bb = mq_quant_block_bytes(ttype);
    if (bb == 0) return MQ_ERR_INVALID_ARG;
    if (ne0 <= 0 || ne0 % bq) return MQ_ERR_SHAPE;
    const size_t row = size_t(ne0 / bq) * size_t(bb);
    for (int32_t i = 0; i < n; ++i) {
        if (rows[i] < 0) return MQ_ERR_SHAPE;
        if (!srcs[i] && rows[i] > 0) return MQ_ERR_INVALID_ARG;
    }
    uint8_t* out = static_cast<uint8_t*>(dst);
    for (int32_t i = 0; i < n; ++i) {
        const size_t bytes = row * size_t(rows[i]);
        if (bytes) {
            cudaError_t e = cudaMemcpyAsync(out, srcs[i], bytes, cudaMemcpyDeviceToDevice, as_stream(stream));
            if (e != cudaSuccess) return cuda_fail(e);
        }
        out += bytes;
    }
    return MQ_OK;
}

mq_status mq_quantize_q8_0(const float* x, void* xq, int64_t K, int32_t ncols, void* stream)
{
    if (K < 0 || ncols < 0 || K % 32) return MQ_ERR_SHAPE;
    if (K == 0 || ncols == 0) return MQ_OK;
    if (!x || !xq) return MQ_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(xq, 2)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    mq_status st = current_dev(&dev);
    if (st != MQ_OK) return st;
    cudaError_t e = mq::launch_quantize(x, xq, K / 32 * int64_t(ncols), as_stream(stream));
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

mq_status mq_check_mv_desc(const mq_mv_desc* h)
{
    if (!h) return MQ_ERR_INVALID_ARG;
    mq_status st = check_mv_shape(h->rows, h->K, h->ncols);
    if (st != MQ_OK) return st;
    if (h->y_ld < h->rows) return MQ_ERR_SHAPE;
    if (h->rows == 0 || h->ncols == 0) return MQ_OK;
    if (!h->W || !h->y || (!h->x && !h->xq)) return MQ_ERR_INVALID_ARG;
    if (!aligned(h->W, 16) || !aligned(h->y, 4) || (h->x && !aligned(h->x, 4)) || (!h->x && !aligned(h->xq, 2)) ||
        !aligned(h->xq_out, 2))
        return MQ_ERR_ALIGN;
    return MQ_OK;
}

static mq_status launch_matvec(const void* d_desc, int kind, int32_t rows, int32_t K, int32_t ncols,
                               const mq::DeviceInfo* dev, cudaStream_t s, bool pdl)
{
    mq::MvPlan p;
    if (!mq::plan_mv(rows, K, ncols, kind, 0, *dev, &p)) return MQ_ERR_UNSUPPORTED;
    cudaError_t e = mq::launch_mv(d_desc, kind, rows, K, ncols, p, dev->status, s, pdl);
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

mq_status mq_matvec_q4K_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols, void* stream)
{
    mq_status st = check_mv_shape(rows, K, ncols);
    if (st != MQ_OK) return st;
    if (rows == 0 || ncols == 0) return MQ_OK;
    if (!d_desc) return MQ_ERR_INVALID_ARG;
    if (!aligned(d_desc, 8)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    if ((st = current_dev(&dev)) != MQ_OK) return st;
    return launch_matvec(d_desc, mq::KIND_MV, rows, K, ncols, dev, as_stream(stream), false);
}

// q4_0 / q8_0 weights: the same checks and descriptor, the ring kernel with
// that type's unit format (there is no register-streaming fallback for them)
static mq_status matvec_wtype(int wtype, const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols,
                              void* stream)
{
    mq_status st = check_mv_shape(rows, K, ncols);
    if (st != MQ_OK) return st;
    if (rows == 0 || ncols == 0) return MQ_OK;
    if (!d_desc) return MQ_ERR_INVALID_ARG;
    if (!aligned(d_desc, 8)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    if ((st = current_dev(&dev)) != MQ_OK) return st;
    mq::MvPlan p;
    const int unit_bytes = wtype == MQ_TYPE_Q4_0 ? 72 : 136;  // four 32-weight blocks
    if (!mq::plan_mv(rows, K, ncols, mq::KIND_MV, 0, *dev, &p, unit_bytes, true) || p.variant != 1)
        return MQ_ERR_UNSUPPORTED;
    cudaError_t e = mq::launch_wring(d_desc, wtype, rows, K, ncols, p, dev->status, as_stream(stream), false);
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

mq_status mq_matvec_q4_0_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols, void* stream)
{
    return matvec_wtype(MQ_TYPE_Q4_0, d_desc, rows, K, ncols, stream);
}

mq_status mq_matvec_q8_0_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols, void* stream)
{
    return matvec_wtype(MQ_TYPE_Q8_0, d_desc, rows, K, ncols, stream);
}

static mq_status check_ffn_shape(int64_t H, int64_t I, int64_t ncols)
{
    if (H < 0 || I < 0 || ncols < 0 || ncols > MQ_MAX_NCOLS) return MQ_ERR_SHAPE;
    if (H == 0 || I == 0 || H % 256 || I % 256) return MQ_ERR_SHAPE;
    if (H > MQ_MAX_K || I > MQ_MAX_K || H * ncols > MQ_MAX_K_TIMES_NCOLS || I * ncols > MQ_MAX_K_TIMES_NCOLS)
        return MQ_ERR_UNSUPPORTED;
    return MQ_OK;
}

mq_status mq_check_ffn_desc(const mq_ffn_desc* h)
{
    if (!h) return MQ_ERR_INVALID_ARG;
    mq_status st = check_ffn_shape(h->H, h->I, h->ncols);
    if (st != MQ_OK) return st;
    if (h->y_ld < h->H) return MQ_ERR_SHAPE;
    if (h->ncols == 0) return MQ_OK;
    if (!h->W_gu || !h->W_down || !h->h_q8 || !h->y || (!h->x && !h->xq)) return MQ_ERR_INVALID_ARG;
    if (!aligned(h->W_gu, 16) || !aligned(h->W_down, 16) || !aligned(h->h_q8, 2) || !aligned(h->y, 4) ||
        (h->x && !aligned(h->x, 4)) || (!h->x && !aligned(h->xq, 2)) || !aligned(h->gu_dbg, 4) ||
        !aligned(h->h_dbg, 4))
        return MQ_ERR_ALIGN;
    return MQ_OK;
}

static mq_status launch_ffn(const mq_ffn_desc* d_desc, int32_t H, int32_t I, int32_t ncols,
                            const mq::DeviceInfo* dev, cudaStream_t s, bool pdl)
{
    mq::MvPlan pg, pd;
    if (!mq::plan_mv(2 * int64_t(I), H, ncols, mq::KIND_GU, I, *dev, &pg)) return MQ_ERR_UNSUPPORTED;
    if (!mq::plan_mv(H, I, ncols, mq::KIND_DOWN, 0, *dev, &pd)) return MQ_ERR_UNSUPPORTED;
    cudaError_t e = mq::launch_gu(d_desc, H, I, ncols, pg, dev->status, s, pdl);
    if (e != cudaSuccess) return cuda_fail(e);
    // the down launch always under programmatic dependent launch: its weight
    // copies start while gate/up drains, and it reads h only after its
    // grid-dependency wait
    e = mq::launch_mv(d_desc, mq::KIND_DOWN, H, I, ncols, pd, dev->status, s, true);
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

mq_status mq_ffn_gu_silu_down(const mq_ffn_desc* d_desc, int32_t H, int32_t I, int32_t ncols, void* stream)
{
    mq_status st = check_ffn_shape(H, I, ncols);
    if (st != MQ_OK) return st;
    if (ncols == 0) return MQ_OK;
    if (!d_desc) return MQ_ERR_INVALID_ARG;
    if (!aligned(d_desc, 8)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    if ((st = current_dev(&dev)) != MQ_OK) return st;
    return launch_ffn(d_desc, H, I, ncols, dev, as_stream(stream), false);
}

mq_status mq_ffn_gate_up(const mq_ffn_desc* d_desc, int32_t H, int32_t I, int32_t ncols, void* stream)
{
    mq_status st = check_ffn_shape(H, I, ncols);
    if (st != MQ_OK) return st;
    if (ncols == 0) return MQ_OK;
    if (!d_desc) return MQ_ERR_INVALID_ARG;
    if (!aligned(d_desc, 8)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    if ((st = current_dev(&dev)) != MQ_OK) return st;
    mq::MvPlan pg;
    if (!mq::plan_mv(2 * int64_t(I), H, ncols, mq::KIND_GU, I, *dev, &pg)) return MQ_ERR_UNSUPPORTED;
    cudaError_t e = mq::launch_gu(d_desc, H, I, ncols, pg, dev->status, as_stream(stream), false);
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

// the shapes of a step: q|k|v and o may be left out (zero rows), the FFN may not
static mq_status check_step_shape(const mq_step_shape* h)
{
    if (h->n_layers < 0 || h->ncols < 0 || h->qkv_rows < 0 || h->o_rows < 0) return MQ_ERR_SHAPE;
    if (h->flags & ~uint32_t(MQ_STEP_PDL | MQ_STEP_PERSISTENT | MQ_STEP_CHAINED)) return MQ_ERR_INVALID_ARG;
    mq_status st;
    if (h->qkv_rows > 0 && (st = check_mv_shape(h->qkv_rows, h->H, h->ncols)) != MQ_OK) return st;
    if (h->o_rows > 0 && (st = check_mv_shape(h->o_rows, h->o_K, h->ncols)) != MQ_OK) return st;
    return check_ffn_shape(h->H, h->I, h->ncols);
}

mq_status mq_step_workspace_bytes(const mq_step_shape* h, size_t* bytes)
{
    if (!h || !bytes) return MQ_ERR_INVALID_ARG;
    mq_status st = check_step_shape(h);
    if (st != MQ_OK) return st;
    *bytes = mq::step_workspace(*h).bytes;
    return MQ_OK;
}

mq_status mq_step(const mq_layer_desc* d_layers, const mq_step_shape* h, void* stream)
{
    if (!h) return MQ_ERR_INVALID_ARG;
    mq_status st = check_step_shape(h);
    if (st != MQ_OK) return st;
    if (h->n_layers == 0 || h->ncols == 0) return MQ_OK;
    if (!d_layers) return MQ_ERR_INVALID_ARG;
    if (!aligned(d_layers, 8)) return MQ_ERR_ALIGN;
    if (h->flags & MQ_STEP_PERSISTENT) {
        if (!h->workspace) return MQ_ERR_INVALID_ARG;
        if (!aligned(h->workspace, 16)) return MQ_ERR_ALIGN;
    }
    const mq::DeviceInfo* dev = nullptr;
    if ((st = current_dev(&dev)) != MQ_OK) return st;
    const bool pdl = (h->flags & MQ_STEP_PDL) != 0;
    const cudaStream_t s = as_stream(stream);
    if (h->flags & MQ_STEP_PERSISTENT) {
        mq::StepPlan sp;
        if (!mq::plan_step(*h, *dev, &sp)) return MQ_ERR_UNSUPPORTED;
        cudaError_t e = mq::launch_step(d_layers, sp, h->ncols, dev->status, static_cast<unsigned*>(h->workspace), s);
        return e == cudaSuccess ? MQ_OK : cuda_fail(e);
    }
    // one plan per projection, decided once for the whole stack (none for a projection left out)
    mq::MvPlan p_qkv, p_o, p_gu, p_down;
    if ((h->qkv_rows > 0 && !mq::plan_mv(h->qkv_rows, h->H, h->ncols, mq::KIND_MV, 0, *dev, &p_qkv)) ||
        (h->o_rows > 0 && !mq::plan_mv(h->o_rows, h->o_K, h->ncols, mq::KIND_MV, 0, *dev, &p_o)) ||
        !mq::plan_mv(2 * int64_t(h->I), h->H, h->ncols, mq::KIND_GU, h->I, *dev, &p_gu) ||
        !mq::plan_mv(h->H, h->I, h->ncols, mq::KIND_DOWN, 0, *dev, &p_down))
        return MQ_ERR_UNSUPPORTED;
    for (int32_t l = 0; l < h->n_layers; ++l) {
        const mq_layer_desc* L = d_layers + l;
        cudaError_t e = cudaSuccess;
        if (h->qkv_rows > 0)
            e = mq::launch_mv(&L->qkv, mq::KIND_MV, h->qkv_rows, h->H, h->ncols, p_qkv, dev->status, s, pdl);
        if (e == cudaSuccess && h->o_rows > 0)
            e = mq::launch_mv(&L->o, mq::KIND_MV, h->o_rows, h->o_K, h->ncols, p_o, dev->status, s, pdl);
        if (e == cudaSuccess) e = mq::launch_gu(&L->ffn, h->H, h->I, h->ncols, p_gu, dev->status, s, pdl);
        if (e == cudaSuccess)
            e = mq::launch_mv(&L->ffn, mq::KIND_DOWN, h->H, h->I, h->ncols, p_down, dev->status, s, pdl);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return MQ_OK;
}

static mq_status check_mmq_shape(int64_t rows, int64_t K, int64_t ncols)
{
    if (rows < 0 || K <= 0 || ncols < 0 || K % 256 || ncols > MQ_MMQ_MAX_NCOLS) return MQ_ERR_SHAPE;
    if (K > MQ_MAX_K || rows > INT32_MAX) return MQ_ERR_UNSUPPORTED;
    return MQ_OK;
}

mq_status mq_mmq_workspace_bytes(int32_t rows, int32_t K, int32_t ncols, size_t* bytes)
{
    if (!bytes) return MQ_ERR_INVALID_ARG;
    mq_status st = check_mmq_shape(rows, K, ncols);
    if (st != MQ_OK) return st;
    const mq::DeviceInfo* dev = nullptr;
    if ((st = current_dev(&dev)) != MQ_OK) return st;
    *bytes = (rows == 0 || ncols == 0) ? 0 : mq::plan_mmq(rows, K, ncols, dev->num_sms, dev->max_smem_optin).ws_bytes;
    return MQ_OK;
}

mq_status mq_mmq_q4K_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols, void* workspace,
                          size_t ws_bytes, void* stream)
{
    mq_status st = check_mmq_shape(rows, K, ncols);
    if (st != MQ_OK) return st;
    if (rows == 0 || ncols == 0) return MQ_OK;
    if (!d_desc || !workspace) return MQ_ERR_INVALID_ARG;
    if (!aligned(d_desc, 8) || !aligned(workspace, 128)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    if ((st = current_dev(&dev)) != MQ_OK) return st;
    const mq::MmqPlan p = mq::plan_mmq(rows, K, ncols, dev->num_sms, dev->max_smem_optin);
    if (p.stages < 2) return MQ_ERR_UNSUPPORTED;
    if (ws_bytes < p.ws_bytes) return MQ_ERR_INVALID_ARG;
    cudaError_t e = mq::launch_mmq(d_desc, rows, K, ncols, p, workspace, dev->num_sms, dev->status,
                                   as_stream(stream));
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

mq_status mq_dequant_q4K_f16(const void* W, void* W16, int64_t rows, int64_t K, void* stream)
{
    if (rows < 0 || K <= 0 || K % 256) return MQ_ERR_SHAPE;
    if (rows == 0) return MQ_OK;
    if (!W || !W16) return MQ_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(W16, 16)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    mq_status st = current_dev(&dev);
    if (st != MQ_OK) return st;
    cudaError_t e = mq::launch_dequant_q4K_f16(W, W16, rows * (K / 256), dev->num_sms, as_stream(stream));
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

mq_status mq_convert_f32_f16(const float* x, void* y, int64_t n, void* stream)
{
    if (n < 0) return MQ_ERR_SHAPE;
    if (n == 0) return MQ_OK;
    if (!x || !y) return MQ_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(y, 2)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    mq_status st = current_dev(&dev);
    if (st != MQ_OK) return st;
    cudaError_t e = mq::launch_f32_to_f16(x, y, n, dev->num_sms, as_stream(stream));
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

mq_status mq_gemm_f16(const void* W16, const void* X16, float* Y, int32_t R, int32_t K, int32_t T, void* stream)
{
    if (R < 0 || T < 0 || K <= 0 || K % 64) return MQ_ERR_SHAPE;
    if (K > MQ_MAX_K) return MQ_ERR_UNSUPPORTED;
    if (R == 0 || T == 0) return MQ_OK;
    if (!W16 || !X16 || !Y) return MQ_ERR_INVALID_ARG;
    if (!aligned(W16, 16) || !aligned(X16, 16) || !aligned(Y, 4)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    mq_status st = current_dev(&dev);
    if (st != MQ_OK) return st;
    cudaError_t e = mq::launch_gemm_f16(W16, X16, Y, R, K, T, dev->num_sms, dev->status, as_stream(stream));
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

mq_status mq_debug_block_sums_q4K_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols,
                                       int32_t* sumi, int32_t* sumq, void* stream)
{
    mq_status st = check_mv_shape(rows, K, ncols);
    if (st != MQ_OK) return st;
    if (rows == 0 || ncols == 0) return MQ_OK;
    if (!d_desc || !sumi || !sumq) return MQ_ERR_INVALID_ARG;
    if (!aligned(d_desc, 8) || !aligned(sumi, 4) || !aligned(sumq, 4)) return MQ_ERR_ALIGN;
    const mq::DeviceInfo* dev = nullptr;
    if ((st = current_dev(&dev)) != MQ_OK) return st;
    const int64_t smem = int64_t(ncols) * (K / 64) * 80 + int64_t(ncols) * (K / 32) * 4;
    if (smem > dev->max_smem_optin) return MQ_ERR_UNSUPPORTED;
    cudaError_t e = mq::launch_block_sums(d_desc, rows, K, ncols, sumi, sumq, int(smem), dev->status,
                                          as_stream(stream));
    return e == cudaSuccess ? MQ_OK : cuda_fail(e);
}

// the planner's view for the test hooks below (field order as in mq.h)
static void plan_fields(const mq::MvPlan& p, int64_t* o)
{
    const int64_t v[MQ_PLAN_FIELDS] = {p.variant, p.grid,         p.block,        p.smem, p.C,   p.L,   p.S,
                                       p.nseg,    p.nwc,          p.rg,           p.T,    p.ns,  p.stage_bytes,
                                       p.rows_per_cta, p.cmap,    p.cgw,          p.cgu,  p.hu,  p.ksplit,
                                       p.kpn};
    for (int i = 0; i < MQ_PLAN_FIELDS; ++i) o[i] = v[i];
}

static bool fake_device(int32_t num_sms, int64_t l2_bytes, int32_t max_smem, mq::DeviceInfo* d)
{
    if (num_sms <= 0 || l2_bytes <= 0 || l2_bytes > INT32_MAX || max_smem <= 0) return false;
    d->num_sms = num_sms;
    d->l2_bytes = int(l2_bytes);
    d->max_smem_optin = max_smem;
    return true;
}

mq_status mq_debug_plan_mv(int32_t kind, int64_t rows, int32_t K, int32_t ncols, int32_t I, int32_t num_sms,
                           int64_t l2_bytes, int32_t max_smem, int64_t* out, int32_t n_out)
{
    mq::DeviceInfo dev;
    if (!out || n_out < MQ_PLAN_FIELDS || !fake_device(num_sms, l2_bytes, max_smem, &dev)) return MQ_ERR_INVALID_ARG;
    mq_status st;
    int mk = mq::KIND_MV;
    if (kind == MQ_PLAN_MATVEC) {
        st = check_mv_shape(rows, K, ncols);
    } else if (kind == MQ_PLAN_DOWN) {
        st = check_ffn_shape(rows, K, ncols);  // rows = H, K = I
        mk = mq::KIND_DOWN;
    } else if (kind == MQ_PLAN_GATE_UP) {
        st = (rows != 2 * int64_t(I)) ? MQ_ERR_SHAPE : check_ffn_shape(K, I, ncols);  // rows = 2I, K = H
        mk = mq::KIND_GU;
    } else {
        return MQ_ERR_INVALID_ARG;
    }
    if (st != MQ_OK) return st;
    if (rows == 0 || ncols == 0) return MQ_ERR_INVALID_ARG;  // the call would launch nothing
    mq::MvPlan p;
    if (!mq::plan_mv(rows, K, ncols, mk, mk == mq::KIND_GU ? I : 0, dev, &p)) return MQ_ERR_UNSUPPORTED;
    plan_fields(p, out);
    return MQ_OK;
}

mq_status mq_debug_plan_step(const mq_step_shape* h, int32_t num_sms, int64_t l2_bytes, int32_t max_smem,
                             int64_t* out, int32_t n_out)
{
    mq::DeviceInfo dev;
    if (!h || !out || n_out < MQ_STEP_PLAN_FIELDS + 4 * MQ_PLAN_FIELDS ||
        !fake_device(num_sms, l2_bytes, max_smem, &dev))
        return MQ_ERR_INVALID_ARG;
    mq_status st = check_step_shape(h);
    if (st != MQ_OK) return st;
    if (h->n_layers == 0 || h->ncols == 0) return MQ_ERR_INVALID_ARG;  // the call would launch nothing
    mq::StepPlan sp;
    if (!mq::plan_step(*h, dev, &sp)) return MQ_ERR_UNSUPPORTED;
    const int64_t g[MQ_STEP_PLAN_FIELDS] = {sp.grid, 32 * (sp.nwc + 1), sp.smem, sp.nwc, sp.ph[0].ns,
                                            sp.ph[0].stage_bytes, sp.pf_tiles, int64_t(sp.ws_bytes)};
    for (int i = 0; i < MQ_STEP_PLAN_FIELDS; ++i) out[i] = g[i];
    for (int ph = 0; ph < 4; ++ph) {
        mq::MvPlan q = sp.ph[ph];
        if (sp.R[ph] == 0) q = mq::MvPlan{};  // a phase left out
        q.ksplit = 1;                          // the persistent kernel takes whole rows
        plan_fields(q, out + MQ_STEP_PLAN_FIELDS + ph * MQ_PLAN_FIELDS);
    }
    return MQ_OK;
}

}  // extern "C"
