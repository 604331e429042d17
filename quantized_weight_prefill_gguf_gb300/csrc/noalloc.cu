// noalloc.cu -- mq_gemm_noalloc: the cached GEMM for callers that cannot
// allocate device memory.
//
// The cached GEMM splits K over the tiles of its last, partial wave and sums
// the partial planes in a fixed order; those planes live in scratch memory.
// mq_gemm takes that scratch from a library-owned buffer that it grows with
// cudaMalloc on demand.  Here the scratch is this file-scope device array
// instead, so nothing on this path allocates or frees device memory.
//
// In host code the array's name is only a host-side stand-in for the device
// symbol, never a device address: the device address is fetched with
// cudaGetSymbolAddress once per device (with that device current) and handed
// to the kernels.  The array costs every GPU that loads this library
// kScratchBytes of device memory until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "mq.h"
#include "mq_internal.h"

namespace {

// 16 MiB: enough split-K scratch for every GEMM of the tile planner whose
// last wave has at most 128 full-K tiles' worth of parts, e.g. all of a
// Qwen2.5-7B layer except the 3584-row weights at M = 2048.
constexpr int64_t kScratchBytes = int64_t(16) << 20;

__device__ __align__(256) float g_noalloc_scratch[kScratchBytes / sizeof(float)];
__device__ __align__(16) unsigned g_noalloc_status;   // bounded-wait timeouts of these calls

__global__ void k_clear_status_bits(unsigned bits) { atomicAnd(&g_noalloc_status, ~bits); }

struct DevPtrs {
    bool ready = false;
    float *scratch = nullptr;
    unsigned *status = nullptr;
};

constexpr int kMaxDevices = 64;
DevPtrs g_ptrs[kMaxDevices];
std::mutex g_mu;

// Device addresses of the scratch array and status word on `dev` (current).
cudaError_t device_ptrs(int dev, DevPtrs **out)
{
    std::lock_guard<std::mutex> lk(g_mu);
    DevPtrs &p = g_ptrs[dev];
    if (!p.ready) {
        cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p.scratch), g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p.status), g_noalloc_status);
        if (e != cudaSuccess)
            return e;
        p.ready = true;
    }
    *out = &p;
    return cudaSuccess;
}

}  // namespace

namespace mq {

unsigned noalloc_take_status()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_ptrs[dev].ready)
            return 0;
    }
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_noalloc_status, sizeof v) != cudaSuccess)
        return 0;
    if (v != 0) {
        // Clear only the bits just read, atomically on the device: a bit that
        // a call still running on another stream sets in the meantime stays
        // set for the next read.
        k_clear_status_bits<<<1, 1>>>(v);
        if (cudaGetLastError() == cudaSuccess)
            cudaStreamSynchronize(0);
    }
    return v;
}

}  // namespace mq

extern "C" int mq_gemm_noalloc(const void *x, mq_handle w, float *y, int64_t M, void *stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return mq::set_error(MQ_ERR_NO_DEVICE, "cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices)
        return mq::set_error(MQ_ERR_NO_DEVICE, "device ordinal out of range", cudaSuccess);
    DevPtrs *p = nullptr;
    e = device_ptrs(dev, &p);
    if (e != cudaSuccess)
        return mq::set_error(MQ_ERR_CUDA, "cudaGetSymbolAddress of the static scratch", e);
    return mq::gemm_cached_into_scratch(x, w, y, M, static_cast<cudaStream_t>(stream), p->scratch, kScratchBytes,
                                        p->status);
}
