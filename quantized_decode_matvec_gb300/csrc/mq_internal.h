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
    int S;             // chunks per segment (<= L)
    int rows_per_cta;  // max rows handled by one CTA
    int grid;          // CTAs
    int block;         // threads per CTA
    int smem;          // dynamic shared memory bytes
};

enum Kind { KIND_MV = 0, KIND_DOWN = 1, KIND_GU = 2 };

struct DeviceInfo {
    int num_sms = 0;
    int max_smem_optin = 0;
    unsigned* status = nullptr;  // device status word
    bool ready = false;
};

// the calling thread's current device, initialised by mq_init (nullptr otherwise)
const DeviceInfo* current_device_info();

// returns false if the shapes cannot be planned within the device limits
bool plan_mv(int64_t rows, int K, int ncols, int kind, int I, const DeviceInfo& dev, MvPlan* p);

cudaError_t launch_quantize(const float* x, void* xq, int64_t nblocks, cudaStream_t s);
cudaError_t launch_mv(const void* desc, int kind, int rows, int K, int ncols, const MvPlan& p,
                      unsigned* status, cudaStream_t s, bool pdl);
cudaError_t launch_gu(const mq_ffn_desc* d, int H, int I, int ncols, const MvPlan& p, unsigned* status,
                      cudaStream_t s, bool pdl);
cudaError_t launch_block_sums(const mq_mv_desc* d, int rows, int K, int ncols, int32_t* sumi, int32_t* sumq,
                              int smem, unsigned* status, cudaStream_t s);
// raises the dynamic shared memory limit of every kernel on the current device
cudaError_t set_kernel_attributes(int max_smem);

}  // namespace mq
