// Error reporting and launch bookkeeping shared by every libnc entry point.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>

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

}  // namespace nc

extern "C" const char* nc_last_error(void) { return nc::g_err; }
extern "C" uint64_t nc_launch_count(void) { return nc::g_launches.load(); }
