// noalloc.cu -- mq_ffn_gu_silu_down_noalloc: the fused FFN for callers that
// cannot allocate device memory.  The descriptor and the h_q8 scratch that
// mq_ffn_gu_silu_down takes from its caller live here in a file-scope device
// array instead; the gate/up and down kernels are the same ones.
#include <atomic>
#include <mutex>

#include "mq_internal.h"

namespace {

constexpr size_t kDescSlot = 256;  // descriptor at offset 0, h_q8 from offset 256
static_assert(sizeof(mq_ffn_desc) <= kDescSlot, "descriptor slot");
constexpr size_t kScratchBytes = kDescSlot + MQ_NOALLOC_HQ8_MAX_BYTES;

// One instance per device (each CUDA context that loads the library has its
// own).  Shared by every call on that device: calls must not overlap.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
std::atomic<unsigned char*> g_scratch_addr[kMaxDevices];  // null until that device's first call

// Looks up the device address of the current device's g_noalloc_scratch once
// (the device must be current) and caches it; mq_init does this for its device.
cudaError_t lookup_scratch(int dev, unsigned char** out)
{
    unsigned char* ptr = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!ptr) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        ptr = g_scratch_addr[dev].load(std::memory_order_relaxed);
        if (!ptr) {
            const cudaError_t e = cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch);
            if (e != cudaSuccess) return e;
            g_scratch_addr[dev].store(ptr, std::memory_order_release);
        }
    }
    *out = ptr;
    return cudaSuccess;
}

// device address of this device's g_noalloc_scratch (cached by mq_init; looked
// up here if mq_init ran before this file's array was registered)
mq_status scratch_for_current_device(unsigned char** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return mq::record_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return MQ_ERR_NOT_INITIALIZED;
    e = lookup_scratch(dev, out);
    return e == cudaSuccess ? MQ_OK : mq::record_cuda_error(e);
}

__global__ void write_ffn_desc_kernel(mq_ffn_desc* dst, mq_ffn_desc src)
{
    if (blockIdx.x == 0 && threadIdx.x == 0) *dst = src;
}

}  // namespace

namespace mq {
// called by mq_init with `dev` current
cudaError_t noalloc_setup(int dev)
{
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned char* p = nullptr;
    return lookup_scratch(dev, &p);
}
}  // namespace mq

extern "C" mq_status mq_ffn_gu_silu_down_noalloc(const void* W_gu, const void* W_down, const float* x,
                                                 const void* xq, float* y, int32_t H, int32_t I, int32_t ncols,
                                                 int32_t y_ld, void* stream)
{
    mq_ffn_desc h{};
    h.W_gu = W_gu;
    h.W_down = W_down;
    h.x = x;
    h.xq = xq;
    // stands in for the scratch address (256-byte aligned) until the device's
    // copy is looked up, so that every host check runs before device work
    h.h_q8 = reinterpret_cast<void*>(uintptr_t(kDescSlot));
    h.y = y;
    h.H = H;
    h.I = I;
    h.ncols = ncols;
    h.y_ld = y_ld;
    mq_status st = mq_check_ffn_desc(&h);
    if (st != MQ_OK) return st;
    if (int64_t(ncols) * (I / 32) * 34 > MQ_NOALLOC_HQ8_MAX_BYTES) return MQ_ERR_UNSUPPORTED;
    if (ncols == 0) return MQ_OK;

    const mq::DeviceInfo* dev = mq::current_device_info();
    if (!dev) return MQ_ERR_NOT_INITIALIZED;
    unsigned char* scratch = nullptr;
    if ((st = scratch_for_current_device(&scratch)) != MQ_OK) return st;
    mq_ffn_desc* d_desc = reinterpret_cast<mq_ffn_desc*>(scratch);
    h.h_q8 = scratch + kDescSlot;

    mq::MvPlan pg, pd;
    if (!mq::plan_mv(2 * int64_t(I), H, ncols, mq::KIND_GU, I, *dev, &pg)) return MQ_ERR_UNSUPPORTED;
    if (!mq::plan_mv(H, I, ncols, mq::KIND_DOWN, 0, *dev, &pd)) return MQ_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    write_ffn_desc_kernel<<<1, 32, 0, s>>>(d_desc, h);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return mq::record_cuda_error(e);
    e = mq::launch_gu(d_desc, H, I, ncols, pg, dev->status, s, false);
    if (e != cudaSuccess) return mq::record_cuda_error(e);
    e = mq::launch_mv(d_desc, mq::KIND_DOWN, H, I, ncols, pd, dev->status, s, false);
    return e == cudaSuccess ? MQ_OK : mq::record_cuda_error(e);
}
