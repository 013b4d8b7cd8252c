// Shared device/host helpers of libnc (types, conversions, launch bookkeeping).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

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

}  // namespace nc
