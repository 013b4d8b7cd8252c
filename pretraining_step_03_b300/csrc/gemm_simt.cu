// Plain CUDA-core GEMM with the epilogue menu.  It serves the fp32 compute
// mode (where tensor-core tf32 would not meet 1e-5 loss parity) and any shape
// the tensor-core path does not take.
#include "kernels.cuh"

namespace nc {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

template <typename TI>
__device__ __forceinline__ float ld_in(const void* p, long i) {
    return to_f<TI>(reinterpret_cast<const TI*>(p)[i]);
}

__device__ __forceinline__ float ld_any(const void* p, long i, int dt) {
    return dt == NC_FP32 ? reinterpret_cast<const float*>(p)[i]
                         : __bfloat162float(reinterpret_cast<const bf16*>(p)[i]);
}
__device__ __forceinline__ void st_any(void* p, long i, int dt, float v) {
    if (dt == NC_FP32) reinterpret_cast<float*>(p)[i] = v;
    else reinterpret_cast<bf16*>(p)[i] = __float2bfloat16_rn(v);
}

template <typename TI>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(Gemm g) {
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN, b = blockIdx.z;
    const char* Ab = (const char*)g.A + (long)b * g.sA * sizeof(TI);
    const char* Bb = (const char*)g.B + (long)b * g.sB * sizeof(TI);
    float acc[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += BK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int e = tid + i * NT;
            int m, k;
            if (!g.a_t) { m = e / BK; k = e % BK; } else { k = e / BM; m = e % BM; }
            int gm = m0 + m, gk = k0 + k;
            float va = 0.f;
            if (gm < g.M && gk < g.K)
                va = ld_in<TI>(Ab, g.a_t ? (long)gk * g.lda + gm : (long)gm * g.lda + gk);
            As[k][m] = va;
            int n;
            if (!g.b_t) { n = e / BK; k = e % BK; } else { k = e / BN; n = e % BN; }
            int gn = n0 + n;
            gk = k0 + k;
            float vb = 0.f;
            if (gn < g.N && gk < g.K)
                vb = ld_in<TI>(Bb, g.b_t ? (long)gk * g.ldb + gn : (long)gn * g.ldb + gk);
            Bs[k][n] = vb;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[4], bb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = As[k][ty * 4 + i]; bb[i] = Bs[k][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int m = m0 + ty * 4 + i;
        if (m >= g.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int n = n0 + tx * 4 + j;
            if (n >= g.N) continue;
            float v = g.alpha * acc[i][j];
            long ci = (long)b * g.sC + (long)m * g.ldc + n;
            long ai = (long)b * g.sAux + (long)m * g.ldaux + n;
            if (g.epi == EPI_STORE) {
                if (g.aux && g.beta != 0.f) v += g.beta * ld_any(g.aux, ai, g.aux_dtype);
                st_any(g.C, ci, g.c_dtype, v);
            } else if (g.epi == EPI_RELU2) {
                float r = fmaxf(v, 0.f);
                st_any(g.C, ci, g.c_dtype, r * r);
            } else {  // EPI_RELU2_BWD: d/dh relu(h)^2 = 2 relu(h) = 2 sqrt(a)
                float a = ld_any(g.aux, ai, g.aux_dtype);
                st_any(g.C, ci, g.c_dtype, v * 2.f * sqrtf(fmaxf(a, 0.f)));
            }
        }
    }
}

}  // namespace

int gemm_simt(const Gemm& g, cudaStream_t s) {
    if (g.M <= 0 || g.N <= 0 || g.batch <= 0) return NC_OK;
    dim3 grid(ceil_div(g.N, BN), ceil_div(g.M, BM), g.batch);
    if (grid.y > 65535 || grid.z > 65535) return set_error(NC_ERR_UNSUPPORTED, "gemm_simt: grid too large");
    if (g.in_dtype == NC_FP32) gemm_simt_kernel<float><<<grid, NT, 0, s>>>(g);
    else gemm_simt_kernel<bf16><<<grid, NT, 0, s>>>(g);
    note_launch();
    NC_LAUNCH_CHECK("gemm_simt");
    return NC_OK;
}

}  // namespace nc
