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

// Four consecutive values to / from T (16-byte fp32 or 8-byte bf16 accesses).
__device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ void st4(bf16* p, float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const bf16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// X = g * inv, written transposed (X[j][i] = g[i][j]) for tall matrices.  Straight
// matrices are a flat vectorised scale; transposed ones go through 32x32 shared
// tiles, each thread moving one 4-vector in and one out (row t/8, quad t%8).
template <typename T>
__global__ void __launch_bounds__(NT) muon_normalize_kernel(const float* g, const MuonMat* mats,
                                                            const float* partial, int chunks, T* xbase) {
    __shared__ float tile[32][33];
    const MuonMat mm = mats[blockIdx.y];
    const float inv = matrix_inv_norm(partial, blockIdx.y, chunks);
    const float* gp = g + mm.off;
    T* x = xbase + mm.x_off;
    if (!mm.tr) {
        const long n4 = (long)mm.rows * mm.cols / 4;
#pragma unroll 4
        for (long i = (long)blockIdx.x * NT + threadIdx.x; i < n4; i += (long)gridDim.x * NT) {
            const float4 v = ld4(gp + 4 * i);
            st4(x + 4 * i, v.x * inv, v.y * inv, v.z * inv, v.w * inv);
        }
        return;
    }
    const int tr = mm.rows / 32, tc = mm.cols / 32;
    const int ty = threadIdx.x / 8, tq = threadIdx.x % 8;
    for (int t = blockIdx.x; t < tr * tc; t += gridDim.x) {
        const int i0 = (t / tc) * 32, j0 = (t % tc) * 32;
        const float4 v = ld4(gp + (long)(i0 + ty) * mm.cols + j0 + 4 * tq);
        __syncthreads();
        tile[ty][4 * tq] = v.x; tile[ty][4 * tq + 1] = v.y; tile[ty][4 * tq + 2] = v.z; tile[ty][4 * tq + 3] = v.w;
        __syncthreads();
        // X row j0 + ty, columns i0 + 4 tq ..
        st4(x + (long)(j0 + ty) * mm.rows + i0 + 4 * tq, tile[4 * tq][ty] * inv, tile[4 * tq + 1][ty] * inv,
            tile[4 * tq + 2][ty] * inv, tile[4 * tq + 3][ty] * inv);
    }
}

// W -= step * X (X read transposed for tall matrices); refresh the bf16 copy.
template <typename T>
__global__ void __launch_bounds__(NT) muon_apply_kernel(float* w, bf16* w16, const MuonMat* mats,
                                                        const T* xbase, float lr) {
    __shared__ float tile[32][33];
    const MuonMat mm = mats[blockIdx.y];
    const float step = lr * mm.scale;
    float* wp = w + mm.off;
    bf16* wp16 = w16 ? w16 + mm.off : nullptr;
    const T* x = xbase + mm.x_off;
    if (!mm.tr) {
        const long n4 = (long)mm.rows * mm.cols / 4;
#pragma unroll 4
        for (long i = (long)blockIdx.x * NT + threadIdx.x; i < n4; i += (long)gridDim.x * NT) {
            const float4 xv = ld4(x + 4 * i);
            float4 v = ld4(wp + 4 * i);
            v.x -= step * xv.x; v.y -= step * xv.y; v.z -= step * xv.z; v.w -= step * xv.w;
            st4(wp + 4 * i, v.x, v.y, v.z, v.w);
            if (wp16) st4(wp16 + 4 * i, v.x, v.y, v.z, v.w);
        }
        return;
    }
    const int tr = mm.rows / 32, tc = mm.cols / 32;
    const int ty = threadIdx.x / 8, tq = threadIdx.x % 8;
    for (int t = blockIdx.x; t < tr * tc; t += gridDim.x) {
        const int i0 = (t / tc) * 32, j0 = (t % tc) * 32;
        // X is [cols][rows]: its row j0 + ty holds W's column j0 + ty, rows i0 + 4 tq ..
        const float4 xv = ld4(x + (long)(j0 + ty) * mm.rows + i0 + 4 * tq);
        __syncthreads();
        tile[4 * tq][ty] = xv.x; tile[4 * tq + 1][ty] = xv.y; tile[4 * tq + 2][ty] = xv.z; tile[4 * tq + 3][ty] = xv.w;
        __syncthreads();
        const long wi = (long)(i0 + ty) * mm.cols + j0 + 4 * tq;
        float4 v = ld4(wp + wi);
        v.x -= step * tile[ty][4 * tq]; v.y -= step * tile[ty][4 * tq + 1];
        v.z -= step * tile[ty][4 * tq + 2]; v.w -= step * tile[ty][4 * tq + 3];
        st4(wp + wi, v.x, v.y, v.z, v.w);
        if (wp16) st4(wp16 + wi, v.x, v.y, v.z, v.w);
    }
}

__device__ __forceinline__ float adamw_one(float& w, float g, float& m, float& v, float lr, float b1, float b2,
                                           float eps, float wd, float bc1, float bc2) {
    m = b1 * m + (1.f - b1) * g;
    v = b2 * v + (1.f - b2) * g * g;
    const float mhat = m / bc1, vhat = v / bc2;
    w = w * (1.f - lr * wd) - lr * mhat / (sqrtf(vhat) + eps);
    return w;
}

// Four parameters per thread (16-byte accesses); the tail, if n is not a
// multiple of 4, one per thread.
__global__ void __launch_bounds__(NT) adamw_kernel(float* w, bf16* w16, const float* g, float* m, float* v,
                                                   long n, float lr, float b1, float b2, float eps, float wd,
                                                   float bc1, float bc2) {
    const long n4 = n / 4;
    for (long i = (long)blockIdx.x * NT + threadIdx.x; i < n4; i += (long)gridDim.x * NT) {
        float4 wv = reinterpret_cast<float4*>(w)[i], mv = reinterpret_cast<float4*>(m)[i];
        float4 vv = reinterpret_cast<float4*>(v)[i];
        const float4 gv = reinterpret_cast<const float4*>(g)[i];
        adamw_one(wv.x, gv.x, mv.x, vv.x, lr, b1, b2, eps, wd, bc1, bc2);
        adamw_one(wv.y, gv.y, mv.y, vv.y, lr, b1, b2, eps, wd, bc1, bc2);
        adamw_one(wv.z, gv.z, mv.z, vv.z, lr, b1, b2, eps, wd, bc1, bc2);
        adamw_one(wv.w, gv.w, mv.w, vv.w, lr, b1, b2, eps, wd, bc1, bc2);
        reinterpret_cast<float4*>(w)[i] = wv;
        reinterpret_cast<float4*>(m)[i] = mv;
        reinterpret_cast<float4*>(v)[i] = vv;
        if (w16) st4(w16 + 4 * i, wv.x, wv.y, wv.z, wv.w);
    }
    for (long i = 4 * n4 + (long)blockIdx.x * NT + threadIdx.x; i < n; i += (long)gridDim.x * NT) {
        float wi = w[i], mi = m[i], vi = v[i];
        adamw_one(wi, g[i], mi, vi, lr, b1, b2, eps, wd, bc1, bc2);
        w[i] = wi; m[i] = mi; v[i] = vi;
        if (w16) w16[i] = __float2bfloat16_rn(wi);
    }
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
    muon_normalize_kernel<T><<<dim3(blocks_per_mat, nmat), NT, 0, s>>>(g, mats, partial, chunks, x);
    note_launch();
    NC_LAUNCH_CHECK("muon_normalize");
    return NC_OK;
}

template <typename T>
int muon_apply(float* w, bf16* w16, const MuonMat* mats, int nmat, const T* x, float lr,
               int blocks_per_mat, cudaStream_t s) {
    muon_apply_kernel<T><<<dim3(blocks_per_mat, nmat), NT, 0, s>>>(w, w16, mats, x, lr);
    note_launch();
    NC_LAUNCH_CHECK("muon_apply");
    return NC_OK;
}

int adamw(float* w, bf16* w16, const float* g, float* m, float* v, long n, float lr, float b1,
          float b2, float eps, float wd, float bc1, float bc2, cudaStream_t s) {
    if (n <= 0) return NC_OK;
    const long blocks = ceil_div(n / 4 > 0 ? n / 4 : 1, NT);
    adamw_kernel<<<(int)(blocks < 16L * 148 ? blocks : 16L * 148), NT, 0, s>>>(w, w16, g, m, v, n, lr, b1, b2, eps,
                                                                              wd, bc1, bc2);
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
