// Failure detection, exercised without faulting the GPU: one CTA waits on an mbarrier
// that nothing arrives on, through the same bounded wait every pipeline of the library
// uses (tc::mbar_wait: %globaltimer limit, then the CTA's abort word is set and the wait
// gives up).  The kernel then records NC_FLAG_TIMEOUT in the per-device flag word, the way
// an aborted GEMM or attention CTA does, and returns; the context stays usable.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace nc {
namespace {

__global__ void wait_timeout_kernel(uint32_t* flag) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);   // one arrival expected; none is ever made
        abort_word = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    volatile int* abort = &abort_word;
    const bool landed = tc::mbar_wait_warp(&bar, 0, abort);
    __syncthreads();
    if (threadIdx.x == 0 && !landed && *abort && flag) atomicOr(flag, NC_FLAG_TIMEOUT);
}

}  // namespace
}  // namespace nc

extern "C" int nc_selftest_wait_timeout(void* stream) {
    uint32_t* flag = nullptr;
    NC_TRY(nc::kernel_flag(&flag));
    nc::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(flag);
    nc::note_launch();
    NC_LAUNCH_CHECK("wait_timeout_kernel");
    return NC_OK;
}
