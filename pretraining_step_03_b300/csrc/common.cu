// Error reporting and launch bookkeeping shared by every libnc entry point.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace nc {

static thread_local char g_err[512] = "";
static std::atomic<uint64_t> g_launches{0};

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int set_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_check(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return NC_OK;
    return set_error(e == cudaErrorMemoryAllocation ? NC_ERR_OOM : NC_ERR_CUDA, "%s: %s", what,
                     cudaGetErrorString(e));
}

// One word per device that loads the library (4 bytes; no allocation).
static __device__ uint32_t g_kernel_flag_word;

constexpr int KF_MAX_DEVICES = 64;
static std::mutex g_kf_mu;
static uint32_t* g_kf_ptr[KF_MAX_DEVICES] = {};

int kernel_flag(uint32_t** out) {
    int dev = 0;
    NC_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
    if (dev < 0 || dev >= KF_MAX_DEVICES) return set_error(NC_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_kf_mu);
    if (!g_kf_ptr[dev]) {
        void* p = nullptr;
        NC_TRY(cuda_check(cudaGetSymbolAddress(&p, g_kernel_flag_word), "cudaGetSymbolAddress (flag)"));
        g_kf_ptr[dev] = static_cast<uint32_t*>(p);
    }
    *out = g_kf_ptr[dev];
    return NC_OK;
}

}  // namespace nc

extern "C" int nc_check_kernel_flag(void* stream, uint32_t* flags) {
    using namespace nc;
    uint32_t* word = nullptr;
    NC_TRY(kernel_flag(&word));
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t f = 0;
    NC_TRY(cuda_check(cudaMemcpyAsync(&f, word, 4, cudaMemcpyDeviceToHost, s), "D2H kernel flag"));
    NC_TRY(cuda_check(cudaMemsetAsync(word, 0, 4, s), "clear kernel flag"));
    NC_TRY(cuda_check(cudaStreamSynchronize(s), "sync"));
    if (flags) *flags = f;
    if (f) return set_error(NC_ERR_DEVICE_FLAG, "kernel flag 0x%x", f);
    return NC_OK;
}

extern "C" const char* nc_last_error(void) { return nc::g_err; }
extern "C" uint64_t nc_launch_count(void) { return nc::g_launches.load(); }
