// Shared device/host helpers of libnc (types, conversions, launch bookkeeping).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <atomic>

#include "../../include/nc_api.h"

typedef __nv_bfloat16 bf16;

namespace nc {

// ------------------------------------------------------------ conversions
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ------------------------------------------------------------ host side
// Every kernel launch of the library goes through note_launch() so that the
// number of kernels a step launched can be reported.
void note_launch(int n = 1);
int set_error(int code, const char* fmt, ...);
int cuda_check(cudaError_t e, const char* what);

#define NC_TRY(expr)                     \
    do {                                 \
        int _rc = (expr);                \
        if (_rc != NC_OK) return _rc;    \
    } while (0)

#define NC_LAUNCH_CHECK(what) NC_TRY(::nc::cuda_check(cudaGetLastError(), what))

inline int ceil_div(long a, long b) { return (int)((a + b - 1) / b); }

// Runs a set-up once per device ordinal.  Kernel attributes (the dynamic
// shared-memory limit) are kept per device, so a process-wide "done" switch
// would skip the set-up on a second GPU.  Threads that race may both run it,
// so the set-up must be idempotent (setting an attribute is).
class DeviceOnce {
  public:
    template <typename F>
    int run(F&& setup) {
        int dev = 0;
        NC_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
        const uint64_t bit = dev >= 0 && dev < 64 ? 1ull << dev : 0;
        if (bit && (done_.load(std::memory_order_acquire) & bit)) return NC_OK;
        NC_TRY(setup());
        if (bit) done_.fetch_or(bit, std::memory_order_acq_rel);
        return NC_OK;
    }

  private:
    std::atomic<uint64_t> done_{0};
};

// Device flag word for kernels launched by the kernel-level entry points,
// which have no model (and so no model flag): a word in the library's own
// device memory of the current device, read and cleared by
// nc_check_kernel_flag.  Looked up once per device.
int kernel_flag(uint32_t** out);

}  // namespace nc
