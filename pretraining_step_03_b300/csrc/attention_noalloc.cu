// Attention backward for callers that cannot allocate device memory.
//
// nc_attention_backward needs a scratch buffer of B*H*T floats for the
// per-row statistics D_t = dO_t . O_t, and expects the caller to provide it.
// Some callers cannot: a host process whose device memory is owned and
// pre-reserved by another runtime (so a stray cudaMalloc would fail or break
// its accounting), or a latency-critical loop where cudaMalloc's implicit
// device-wide synchronisation is not acceptable.  This file gives them an
// entry point whose scratch lives in a fixed array compiled into the library
// instead, so no call allocates anything.
//
// The array is file-scope device memory: every GPU that loads the library
// reserves it (NC_ATTN_NOALLOC_MAX_ROWS floats, 4 MiB) until the process
// exits.  All calls share it; two calls in flight at the same time on the
// GPU (e.g. on two streams) race on it.  Its contents are whatever the last
// call left: the statistics kernel overwrites every element a call reads,
// so nothing needs clearing.
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr long NOALLOC_MAX_ROWS = 1L << 20;   // B * H * T limit (4 MiB of fp32)
static_assert(NOALLOC_MAX_ROWS == NC_ATTN_NOALLOC_MAX_ROWS, "header and implementation disagree");

// The scratch.  In host code this name is only a stand-in for the device
// symbol; the kernels get its device address from cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_delta[NOALLOC_MAX_ROWS];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
float* g_ptr[MAX_DEVICES] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
int scratch_address(float** out) {
    int dev = 0;
    NC_TRY(nc::cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
    if (dev < 0 || dev >= MAX_DEVICES) return nc::set_error(NC_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ptr[dev]) {
        void* p = nullptr;
        NC_TRY(nc::cuda_check(cudaGetSymbolAddress(&p, g_noalloc_delta), "cudaGetSymbolAddress"));
        g_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_ptr[dev];
    return NC_OK;
}

}  // namespace

extern "C" int nc_attention_backward_noalloc(const void* q, const void* k, const void* v, int ld_qkv,
                                             const void* o, const void* dout, int ld_o, const float* lse,
                                             void* dq, void* dk, void* dv, int ld_dqkv, int B, int T,
                                             int H, int D, int dtype, void* stream) {
    using namespace nc;
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv)
        return set_error(NC_ERR_ARG, "null pointer");
    if (B < 0 || T < 0 || H < 1 || D < 2 || D > 128 || D % 2 || ld_qkv < H * D || ld_o < H * D ||
        ld_dqkv < H * D)
        return set_error(NC_ERR_ARG, "bad attention shape");
    if ((long)B * H * T > NOALLOC_MAX_ROWS)
        return set_error(NC_ERR_ARG,
                         "nc_attention_backward_noalloc: B*H*T = %ld exceeds the built-in scratch of %ld rows; "
                         "use nc_attention_backward with a caller-provided workspace",
                         (long)B * H * T, NOALLOC_MAX_ROWS);
    if (dtype != NC_BF16 && dtype != NC_FP32) return set_error(NC_ERR_ARG, "dtype %d", dtype);
    float* delta = nullptr;
    NC_TRY(scratch_address(&delta));
    uint32_t* flag = nullptr;
    NC_TRY(kernel_flag(&flag));
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == NC_BF16)
        return attention_backward<bf16>((const bf16*)q, (const bf16*)k, (const bf16*)v, ld_qkv,
                                        (const bf16*)o, (const bf16*)dout, ld_o, lse, (bf16*)dq,
                                        (bf16*)dk, (bf16*)dv, ld_dqkv, delta, B, T, H, D, s, flag);
    return attention_backward<float>((const float*)q, (const float*)k, (const float*)v, ld_qkv,
                                     (const float*)o, (const float*)dout, ld_o, lse, (float*)dq,
                                     (float*)dk, (float*)dv, ld_dqkv, delta, B, T, H, D, s, flag);
}
