// Elementwise parts of the optimizers.
//
// Source: nanochat speedrun walkthrough (lyylswood.com), section 预搜检
// (pretraining): Muon for the block matrices, AdamW for embedding and
// unembedding.  Muon here: momentum, Nesterov look-ahead, Frobenius
// normalisation (these kernels) around the batched Newton-Schulz GEMMs
// (tensor-core GEMM kernels), then the scaled update of the fp32 master and
// its bf16 compute copy.
#include "kernels.cuh"
#include "optim.cuh"

#include <math.h>

namespace nc {
namespace {

constexpr int NT = 256;

__device__ __forceinline__ float block_sum(float v) {
    __shared__ float sh[32];
    const int lane = threadIdx.x % 32, w = threadIdx.x / 32, nw = blockDim.x / 32;
    v = warp_sum(v);
    if (lane == 0) sh[w] = v;
    __syncthreads();
    float t = lane < nw ? sh[lane] : 0.f;
    t = warp_sum(t);
    __syncthreads();
    return t;
}

// buf = mu*buf + g; g <- g + mu*buf (Nesterov) or buf; partial sums of g^2.
__global__ void __launch_bounds__(NT) muon_momentum_kernel(float* g, float* buf,
                                                           const MuonMat* mats, float mu,
                                                           int nesterov, float* partial,
                                                           int chunks) {
    const MuonMat mm = mats[blockIdx.y];
    const long n = (long)mm.rows * mm.cols;
    float* gp = g + mm.off;
    float* bp = buf + mm.off;
    float ss = 0.f;
    const long n4 = n / 4;
    for (long i = (long)blockIdx.x * NT + threadIdx.x; i < n4; i += (long)chunks * NT) {
        float4 gv = reinterpret_cast<float4*>(gp)[i];
        float4 bv = reinterpret_cast<float4*>(bp)[i];
        bv.x = mu * bv.x + gv.x; bv.y = mu * bv.y + gv.y;
        bv.z = mu * bv.z + gv.z; bv.w = mu * bv.w + gv.w;
        if (nesterov) {
            gv.x += mu * bv.x; gv.y += mu * bv.y; gv.z += mu * bv.z; gv.w += mu * bv.w;
        } else {
            gv = bv;
        }
        reinterpret_cast<float4*>(bp)[i] = bv;
        reinterpret_cast<float4*>(gp)[i] = gv;
        ss += gv.x * gv.x + gv.y * gv.y + gv.z * gv.z + gv.w * gv.w;
    }
    ss = block_sum(ss);
    if (threadIdx.x == 0) partial[blockIdx.y * chunks + blockIdx.x] = ss;
}

__device__ float matrix_inv_norm(const float* partial, int mat, int chunks) {
    __shared__ float inv;
    if (threadIdx.x == 0 && threadIdx.y == 0) {
        double s = 0.0;
        for (int c = 0; c < chunks; ++c) s += partial[mat * chunks + c];
        inv = (float)(1.0 / (sqrt(s) + 1e-7));
    }
    __syncthreads();
    return inv;
}

// 32x32 tiles through shared memory; X[j][i] = g[i][j]*inv when transposed.
template <typename T>
__global__ void muon_normalize_kernel(const float* g, const MuonMat* mats, const float* partial,
                                      int chunks, T* xbase) {
    __shared__ float tile[32][33];
    const MuonMat mm = mats[blockIdx.y];
    const float inv = matrix_inv_norm(partial, blockIdx.y, chunks);
    const float* gp = g + mm.off;
    T* x = xbase + mm.x_off;
    const int tr = mm.rows / 32, tc = mm.cols / 32;
    for (int t = blockIdx.x; t < tr * tc; t += gridDim.x) {
        const int i0 = (t / tc) * 32, j0 = (t % tc) * 32;
        if (!mm.tr) {
            for (int y = threadIdx.y; y < 32; y += 8)
                x[(long)(i0 + y) * mm.cols + j0 + threadIdx.x] =
                    from_f<T>(gp[(long)(i0 + y) * mm.cols + j0 + threadIdx.x] * inv);
        } else {
            __syncthreads();
            for (int y = threadIdx.y; y < 32; y += 8)
                tile[y][threadIdx.x] = gp[(long)(i0 + y) * mm.cols + j0 + threadIdx.x];
            __syncthreads();
            for (int y = threadIdx.y; y < 32; y += 8)
                x[(long)(j0 + y) * mm.rows + i0 + threadIdx.x] = from_f<T>(tile[threadIdx.x][y] * inv);
        }
    }
}

// W -= step * X (transposed read when tr); refresh the bf16 copy.
template <typename T>
__global__ void muon_apply_kernel(float* w, bf16* w16, const MuonMat* mats, const T* xbase,
                                  float lr) {
    __shared__ float tile[32][33];
    const MuonMat mm = mats[blockIdx.y];
    const float step = lr * mm.scale;
    float* wp = w + mm.off;
    bf16* wp16 = w16 ? w16 + mm.off : nullptr;
    const T* x = xbase + mm.x_off;
    const int tr = mm.rows / 32, tc = mm.cols / 32;
    for (int t = blockIdx.x; t < tr * tc; t += gridDim.x) {
        const int i0 = (t / tc) * 32, j0 = (t % tc) * 32;
        if (mm.tr) {
            __syncthreads();
            for (int y = threadIdx.y; y < 32; y += 8)   // X is [cols][rows]
                tile[y][threadIdx.x] = to_f<T>(x[(long)(j0 + y) * mm.rows + i0 + threadIdx.x]);
            __syncthreads();
        }
        for (int y = threadIdx.y; y < 32; y += 8) {
            const long wi = (long)(i0 + y) * mm.cols + j0 + threadIdx.x;
            const float xv = mm.tr ? tile[threadIdx.x][y] : to_f<T>(x[wi]);
            const float nw = wp[wi] - step * xv;
            wp[wi] = nw;
            if (wp16) wp16[wi] = __float2bfloat16_rn(nw);
        }
    }
}

__global__ void adamw_kernel(float* w, bf16* w16, const float* g, float* m, float* v, long n,
                             float lr, float b1, float b2, float eps, float wd, float bc1,
                             float bc2) {
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float gi = g[i];
    const float mi = b1 * m[i] + (1.f - b1) * gi;
    const float vi = b2 * v[i] + (1.f - b2) * gi * gi;
    m[i] = mi;
    v[i] = vi;
    const float mhat = mi / bc1, vhat = vi / bc2;
    const float nw = w[i] * (1.f - lr * wd) - lr * mhat / (sqrtf(vhat) + eps);
    w[i] = nw;
    if (w16) w16[i] = __float2bfloat16_rn(nw);
}

}  // namespace

int muon_momentum(float* g, float* buf, const MuonMat* mats, int nmat, float mu, int nesterov,
                  float* partial, int chunks, cudaStream_t s) {
    muon_momentum_kernel<<<dim3(chunks, nmat), NT, 0, s>>>(g, buf, mats, mu, nesterov, partial,
                                                           chunks);
    note_launch();
    NC_LAUNCH_CHECK("muon_momentum");
    return NC_OK;
}

template <typename T>
int muon_normalize(const float* g, const MuonMat* mats, int nmat, const float* partial, int chunks,
                   T* x, int blocks_per_mat, cudaStream_t s) {
    muon_normalize_kernel<T><<<dim3(blocks_per_mat, nmat), dim3(32, 8), 0, s>>>(g, mats, partial,
                                                                                chunks, x);
    note_launch();
    NC_LAUNCH_CHECK("muon_normalize");
    return NC_OK;
}

template <typename T>
int muon_apply(float* w, bf16* w16, const MuonMat* mats, int nmat, const T* x, float lr,
               int blocks_per_mat, cudaStream_t s) {
    muon_apply_kernel<T><<<dim3(blocks_per_mat, nmat), dim3(32, 8), 0, s>>>(w, w16, mats, x, lr);
    note_launch();
    NC_LAUNCH_CHECK("muon_apply");
    return NC_OK;
}

int adamw(float* w, bf16* w16, const float* g, float* m, float* v, long n, float lr, float b1,
          float b2, float eps, float wd, float bc1, float bc2, cudaStream_t s) {
    if (n <= 0) return NC_OK;
    adamw_kernel<<<ceil_div(n, 256), 256, 0, s>>>(w, w16, g, m, v, n, lr, b1, b2, eps, wd, bc1, bc2);
    note_launch();
    NC_LAUNCH_CHECK("adamw");
    return NC_OK;
}

template int muon_normalize<float>(const float*, const MuonMat*, int, const float*, int, float*, int,
                                   cudaStream_t);
template int muon_normalize<bf16>(const float*, const MuonMat*, int, const float*, int, bf16*, int,
                                  cudaStream_t);
template int muon_apply<float>(float*, bf16*, const MuonMat*, int, const float*, float, int,
                               cudaStream_t);
template int muon_apply<bf16>(float*, bf16*, const MuonMat*, int, const bf16*, float, int,
                              cudaStream_t);

}  // namespace nc
