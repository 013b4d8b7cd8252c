// Row-wise, HBM-bound kernels of the step: embedding lookup and its sorted
// segment-sum backward, parameter-free RMSNorm forward/backward, RoPE, the
// softmax cross-entropy with its bits-per-byte reduction, and casts.
//
// Source: nanochat speedrun walkthrough (lyylswood.com), section 预搜检
// (pretraining): no RMSNorm gains, no biases, validation bits per byte =
// per-token loss normalised by the bytes each token stands for.
#include "kernels.cuh"

#include <math.h>

namespace nc {
namespace {

constexpr float RMS_EPS = 1e-6f;

__device__ __forceinline__ void flag_set(uint32_t* flag, uint32_t bits) {
    if (flag) atomicOr(flag, bits);
}

template <typename T> __device__ __forceinline__ void store4(T* p, float4 v);
template <> __device__ __forceinline__ void store4<float>(float* p, float4 v) {
    *reinterpret_cast<float4*>(p) = v;
}
template <> __device__ __forceinline__ void store4<bf16>(bf16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}
template <typename T> __device__ __forceinline__ float4 load4(const T* p);
template <> __device__ __forceinline__ float4 load4<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <> __device__ __forceinline__ float4 load4<bf16>(const bf16* p) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

// ------------------------------------------------------------ embedding
template <typename T>
__global__ void embed_fwd_kernel(const int32_t* tok, const T* wte, float* x, int M, int d, int V,
                                 uint32_t* flag) {
    const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x % 32;
    if (row >= M) return;
    int t = tok[row];
    float* xr = x + (long)row * d;
    if (t < 0 || t >= V) {
        if (lane == 0) flag_set(flag, NC_FLAG_TOKEN_RANGE);
        for (int i = lane * 4; i < d; i += 128) store4<float>(xr + i, make_float4(0, 0, 0, 0));
        return;
    }
    const T* wr = wte + (long)t * d;
    for (int i = lane * 4; i < d; i += 128) store4<float>(xr + i, load4<T>(wr + i));
}

// ------------------------------------------------------------ RMSNorm
// One warp per row: y = x / sqrt(mean(x^2) + eps), r = 1 / sqrt(mean(x^2) + eps).
template <typename T>
__global__ void rmsnorm_fwd_kernel(const float* x, T* y, float* r, int M, int d) {
    const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x % 32;
    if (row >= M) return;
    const float* xr = x + (long)row * d;
    float ss = 0.f;
    for (int i = lane * 4; i < d; i += 128) {
        float4 v = load4<float>(xr + i);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = warp_sum(ss);
    float rr = 1.0f / sqrtf(ss / (float)d + RMS_EPS);
    if (lane == 0) r[row] = rr;
    T* yr = y + (long)row * d;
    for (int i = lane * 4; i < d; i += 128) {
        float4 v = load4<float>(xr + i);
        store4<T>(yr + i, make_float4(v.x * rr, v.y * rr, v.z * rr, v.w * rr));
    }
}

// g_out = g_in + r * (dy - y * mean(dy * y)) (g_in null = 0); optional low-precision copy gT.
template <typename T>
__global__ void rmsnorm_bwd_kernel(const T* dy, const T* y, const float* r, const float* g_in,
                                   float* g_out, T* gT, int M, int d) {
    const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x % 32;
    if (row >= M) return;
    const long o = (long)row * d;
    float dot = 0.f;
    for (int i = lane * 4; i < d; i += 128) {
        float4 a = load4<T>(dy + o + i), b = load4<T>(y + o + i);
        dot += a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
    }
    dot = warp_sum(dot) / (float)d;
    const float rr = r[row];
    for (int i = lane * 4; i < d; i += 128) {
        float4 a = load4<T>(dy + o + i), b = load4<T>(y + o + i);
        float4 g = g_in ? load4<float>(g_in + o + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 out = make_float4(g.x + rr * (a.x - b.x * dot), g.y + rr * (a.y - b.y * dot),
                                 g.z + rr * (a.z - b.z * dot), g.w + rr * (a.w - b.w * dot));
        store4<float>(g_out + o + i, out);
        if (gT) store4<T>(gT + o + i, out);
    }
}

// ------------------------------------------------------------ RoPE
// Rotates pairs (j, j + Dh/2) of every q and k head by sign * angle(t, j).
template <typename T>
__global__ void rope_kernel(T* qkv, long ld, int M, int T_, int H, int Dh, const float2* table,
                            int table_ld, float sign) {
    const int half = Dh / 2;
    long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    long total = (long)M * H * half;
    if (idx >= total) return;
    int j = idx % half;
    long rh = idx / half;
    int h = rh % H;
    long row = rh / H;
    int t = row % T_;
    float2 cs = table[(long)j * table_ld + t];
    float c = cs.x, sn = sign * cs.y;
    T* base = qkv + row * ld + (long)h * Dh;
#pragma unroll
    for (int part = 0; part < 2; ++part) {  // q, then k (offset H*Dh)
        T* p = base + (long)part * H * Dh;
        float x1 = to_f<T>(p[j]), x2 = to_f<T>(p[j + half]);
        p[j] = from_f<T>(x1 * c - x2 * sn);
        p[j + half] = from_f<T>(x2 * c + x1 * sn);
    }
}

// ------------------------------------------------------------ cross-entropy
constexpr int CE_THREADS = 512;

__device__ __forceinline__ float block_reduce(float v, float* sh, bool is_max) {
    const int lane = threadIdx.x % 32, w = threadIdx.x / 32, nw = blockDim.x / 32;
    v = is_max ? warp_max(v) : warp_sum(v);
    __syncthreads();
    if (lane == 0) sh[w] = v;
    __syncthreads();
    float t = lane < nw ? sh[lane] : (is_max ? -INFINITY : 0.f);
    t = is_max ? warp_max(t) : warp_sum(t);
    return t;
}

// One CTA per row: lse = logsumexp(z); nll = lse - z[target];
// z <- scale * (softmax(z) - onehot(target)) in place.
template <typename T>
__global__ void __launch_bounds__(CE_THREADS) ce_kernel(T* z, const int32_t* tgt, float* nll, int V,
                                                        float scale, int grad, uint32_t* flag, float* zdot) {
    __shared__ float sh[32];
    __shared__ float zt_s;
    const long row = blockIdx.x;
    T* zr = z + row * V;
    const int t = tgt[row];
    const bool ok = t >= 0 && t < V;
    if (threadIdx.x == 0) {
        if (!ok) flag_set(flag, NC_FLAG_TOKEN_RANGE);
        zt_s = ok ? to_f<T>(zr[t]) : 0.f;
    }
    float mx = -INFINITY;
    for (int j = threadIdx.x; j < V; j += blockDim.x) mx = fmaxf(mx, to_f<T>(zr[j]));
    mx = block_reduce(mx, sh, true);
    float se = 0.f;
    for (int j = threadIdx.x; j < V; j += blockDim.x) se += expf(to_f<T>(zr[j]) - mx);
    se = block_reduce(se, sh, false);
    const float lse = mx + logf(se);
    __syncthreads();  // zt_s was read before any thread overwrites z
    if (threadIdx.x == 0) nll[row] = ok ? lse - zt_s : 0.f;
    if (!grad) return;   // (loss only: the logits stay as they are)
    float zd = 0.f;   // sum over the row of (softmax - onehot) * z; times scale: <dz, z>
    for (int j = threadIdx.x; j < V; j += blockDim.x) {
        const float zj = to_f<T>(zr[j]);
        float p = expf(zj - lse);
        if (j == t) p -= 1.f;
        zd = fmaf(p, zj, zd);
        zr[j] = from_f<T>(p * scale);
    }
    if (zdot) {
        const float v = block_reduce(zd, sh, false);
        if (threadIdx.x == 0) zdot[row] = v * scale;
    }
}

// Same computation for bf16 logits with V a multiple of 8 * 256, in two passes
// over the row with an online max / sum-exp: the first pass reads the row from
// HBM, the second re-reads it (from L2: a row is 2V bytes and only the rows in
// flight need to stay resident) and writes the gradient in place.  No shared
// row buffer, so several rows per SM overlap their loads.
constexpr float CE_LOG2E = 1.4426950408889634f;
constexpr int CE2_THREADS = 256;

__device__ __forceinline__ void ms_combine(float& m, float& s, float m2, float s2) {
    const float mm = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * exp2f((m - mm) * CE_LOG2E)) +
        (m2 == -INFINITY ? 0.f : s2 * exp2f((m2 - mm) * CE_LOG2E));
    m = mm;
}

__global__ void __launch_bounds__(CE2_THREADS) ce_online_kernel(bf16* z, const int32_t* tgt, float* nll,
                                                                int V, float scale, int grad, uint32_t* flag,
                                                                float* zdot) {
    __shared__ float shm[32], shs[32];
    __shared__ float zt_s, lse_s;
    const long row = blockIdx.x;
    uint4* zr = reinterpret_cast<uint4*>(z + row * V);
    const int nv = V / (8 * CE2_THREADS);
    const int t = tgt[row];
    const bool ok = t >= 0 && t < V;
    if (threadIdx.x == 0) {
        if (!ok) flag_set(flag, NC_FLAG_TOKEN_RANGE);
        zt_s = ok ? __bfloat162float(z[row * V + t]) : 0.f;
    }
    float m = -INFINITY, se = 0.f;
#pragma unroll 4
    for (int k = 0; k < nv; ++k) {
        const uint4 u = zr[threadIdx.x + k * CE2_THREADS];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            f[2 * e] = x.x;
            f[2 * e + 1] = x.y;
        }
        float cm = f[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) cm = fmaxf(cm, f[e]);
        if (cm > m) {
            se = m == -INFINITY ? 0.f : se * exp2f((m - cm) * CE_LOG2E);
            m = cm;
        }
        const float ml = m * CE_LOG2E;
#pragma unroll
        for (int e = 0; e < 8; ++e) se += exp2f(fmaf(f[e], CE_LOG2E, -ml));
    }
    // (max, sum) across the block: warps by shuffles, then warp leaders
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, se, o);
        ms_combine(m, se, m2, s2);
    }
    const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
    if (lane == 0) { shm[wid] = m; shs[wid] = se; }
    __syncthreads();
    if (wid == 0) {
        float m1 = lane < CE2_THREADS / 32 ? shm[lane] : -INFINITY;
        float s1 = lane < CE2_THREADS / 32 ? shs[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m1, o), s2 = __shfl_xor_sync(0xffffffffu, s1, o);
            ms_combine(m1, s1, m2, s2);
        }
        if (lane == 0) {
            lse_s = m1 + logf(s1);
            nll[row] = ok ? lse_s - zt_s : 0.f;
        }
    }
    __syncthreads();   // zt_s was read before any thread overwrites z
    if (!grad) return;   // (loss only: the logits stay as they are)
    const float lsel = lse_s * CE_LOG2E;
    float zd = 0.f;   // sum over the row of (softmax - onehot) * z; times scale: <dz, z>
#pragma unroll 4
    for (int k = 0; k < nv; ++k) {
        const int base = (threadIdx.x + k * CE2_THREADS) * 8;
        const uint4 u = zr[threadIdx.x + k * CE2_THREADS];
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            float p0 = exp2f(fmaf(f.x, CE_LOG2E, -lsel)), p1 = exp2f(fmaf(f.y, CE_LOG2E, -lsel));
            if (base + 2 * e == t) p0 -= 1.f;
            if (base + 2 * e + 1 == t) p1 -= 1.f;
            zd = fmaf(p0, f.x, fmaf(p1, f.y, zd));
            __nv_bfloat162 h = __floats2bfloat162_rn(p0 * scale, p1 * scale);
            w[e] = *reinterpret_cast<uint32_t*>(&h);
        }
        zr[threadIdx.x + k * CE2_THREADS] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (zdot) {
        const float v = block_reduce(zd, shm, false);
        if (threadIdx.x == 0) zdot[row] = v * scale;
    }
}

// The same with the per-row (max, sum exp) partials of every 128-column group already
// left by the LM-head GEMM's epilogue: combine them (fixed order), then one pass that
// writes dlogits = scale * (softmax - onehot) over the logits in place.
__global__ void __launch_bounds__(CE2_THREADS) ce_stats_kernel(bf16* z, const float2* part, const int32_t* tgt,
                                                               float* nll, int V, float scale, int grad,
                                                               uint32_t* flag, float* zdot) {
    __shared__ float shm[32], shs[32];
    __shared__ float zt_s, lse_s;
    const long row = blockIdx.x;
    const int ng = V / 128;
    uint4* zr = reinterpret_cast<uint4*>(z + row * V);
    const int nv = V / (8 * CE2_THREADS);
    const int t = tgt[row];
    const bool ok = t >= 0 && t < V;
    if (threadIdx.x == 0) {
        if (!ok) flag_set(flag, NC_FLAG_TOKEN_RANGE);
        zt_s = ok ? __bfloat162float(z[row * V + t]) : 0.f;
    }
    float m = -INFINITY, se = 0.f;
    for (int k = threadIdx.x; k < ng; k += CE2_THREADS) {
        const float2 ps = part[row * ng + k];
        ms_combine(m, se, ps.x, ps.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, se, o);
        ms_combine(m, se, m2, s2);
    }
    const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
    if (lane == 0) { shm[wid] = m; shs[wid] = se; }
    __syncthreads();
    if (wid == 0) {
        float m1 = lane < CE2_THREADS / 32 ? shm[lane] : -INFINITY;
        float s1 = lane < CE2_THREADS / 32 ? shs[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m1, o), s2 = __shfl_xor_sync(0xffffffffu, s1, o);
            ms_combine(m1, s1, m2, s2);
        }
        if (lane == 0) {
            lse_s = m1 + logf(s1);
            nll[row] = ok ? lse_s - zt_s : 0.f;
        }
    }
    __syncthreads();   // zt_s was read before any thread overwrites z
    if (!grad) return;   // (loss only: the logits stay as they are)
    const float lsel = lse_s * CE_LOG2E;
    float zd = 0.f;   // sum over the row of (softmax - onehot) * z; times scale: <dz, z>
#pragma unroll 4
    for (int k = 0; k < nv; ++k) {
        const int base = (threadIdx.x + k * CE2_THREADS) * 8;
        const uint4 u = zr[threadIdx.x + k * CE2_THREADS];
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            float p0 = exp2f(fmaf(f.x, CE_LOG2E, -lsel)), p1 = exp2f(fmaf(f.y, CE_LOG2E, -lsel));
            if (base + 2 * e == t) p0 -= 1.f;
            if (base + 2 * e + 1 == t) p1 -= 1.f;
            zd = fmaf(p0, f.x, fmaf(p1, f.y, zd));
            __nv_bfloat162 h = __floats2bfloat162_rn(p0 * scale, p1 * scale);
            w[e] = *reinterpret_cast<uint32_t*>(&h);
        }
        zr[threadIdx.x + k * CE2_THREADS] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (zdot) {
        const float v = block_reduce(zd, shm, false);
        if (threadIdx.x == 0) zdot[row] = v * scale;
    }
}

// Single CTA, fixed summation order: loss = mean nll; bpb = sum(nll | bytes>0) / (ln2 * sum bytes).
__global__ void loss_reduce_kernel(const float* nll, const int32_t* tgt, const int32_t* tb, int M,
                                   int V, float* out, double* sums, int accumulate, uint32_t* flag) {
    __shared__ double s_nll[1024], s_pos[1024], s_bytes[1024];
    double a = 0, b = 0, c = 0;
    for (int i = threadIdx.x; i < M; i += blockDim.x) {
        double l = nll[i];
        int t = tgt[i];
        int nb = (t >= 0 && t < V) ? tb[t] : 0;
        a += l;
        if (nb > 0) { b += l; c += nb; }
    }
    s_nll[threadIdx.x] = a;
    s_pos[threadIdx.x] = b;
    s_bytes[threadIdx.x] = c;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) {
            s_nll[threadIdx.x] += s_nll[threadIdx.x + s];
            s_pos[threadIdx.x] += s_pos[threadIdx.x + s];
            s_bytes[threadIdx.x] += s_bytes[threadIdx.x + s];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        float loss = (float)(s_nll[0] / M);
        float bpb = s_bytes[0] > 0 ? (float)(s_pos[0] / (0.6931471805599453 * s_bytes[0])) : 0.f;
        if (!isfinite(loss)) flag_set(flag, NC_FLAG_NONFINITE);
        if (out) {
            out[0] = loss;
            out[1] = bpb;
        }
        if (sums) {   // running totals over batches: sum nll, sum nll where bytes > 0, sum bytes
            sums[0] = (accumulate ? sums[0] : 0.0) + s_nll[0];
            sums[1] = (accumulate ? sums[1] : 0.0) + s_pos[0];
            sums[2] = (accumulate ? sums[2] : 0.0) + s_bytes[0];
        }
    }
}

// ------------------------------------------------------------ embedding backward
// dwte[v] = sum of g rows whose token is v, summed in row order (deterministic):
// a stable counting sort of rows by token id, then fixed-size pieces of the
// sorted list are summed; runs cut by piece borders are combined in order.
constexpr int EB_CHUNK = 1024;  // rows per rank chunk
constexpr int EB_PIECE = 64;    // sorted rows per summation piece
constexpr int EB_COLS = 256;    // columns per summation CTA

__global__ void __launch_bounds__(EB_CHUNK) eb_hist_rank_kernel(const int32_t* tok, int* hist,
                                                                 int* rank, int M, int V) {
    __shared__ int st[EB_CHUNK];
    const int c = blockIdx.x, i = threadIdx.x;
    const long r = (long)c * EB_CHUNK + i;
    int t = r < M ? tok[r] : -1;
    if (t >= V) t = -1;
    st[i] = t;
    __syncthreads();
    if (t < 0) return;
    int cnt = 0;
    for (int j = 0; j < i; ++j) cnt += (st[j] == t);
    rank[r] = cnt;
    atomicAdd(&hist[(long)c * V + t], 1);
}

// Per token id v (one thread each): the column scan of the per-chunk counts, which
// turns hist[c][v] into the number of rows of token v in chunks before c; then the
// exclusive scan of the token counts within this CTA's 256 ids (offsets[v], local to
// the CTA) and the CTA's total (bsum[blockIdx.x]).
constexpr int EB_SCAN_T = 256;

__global__ void __launch_bounds__(EB_SCAN_T) eb_colscan_kernel(int* hist, int* offsets, int* bsum, int nchunks,
                                                               int V) {
    __shared__ int wsum[EB_SCAN_T / 32];
    const int v = blockIdx.x * EB_SCAN_T + threadIdx.x;
    int run = 0;
    if (v < V) {
        // 16 chunks' counts in flight at a time (the loads do not wait on the stores)
        for (int c0 = 0; c0 < nchunks; c0 += 16) {
            int h[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) h[k] = c0 + k < nchunks ? __ldcs(hist + (long)(c0 + k) * V + v) : 0;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                if (c0 + k < nchunks) hist[(long)(c0 + k) * V + v] = run;
                run += h[k];
            }
        }
    }
    // exclusive scan of run over the CTA: warp shuffles, then the warp totals
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    int before = 0;
#pragma unroll
    for (int k = 0; k < EB_SCAN_T / 32; ++k) before += k < w ? wsum[k] : 0;
    if (v < V) offsets[v] = before + x - run;
    if (threadIdx.x == EB_SCAN_T - 1) bsum[blockIdx.x] = before + x;
}

// offsets[v] += the exclusive prefix of the CTA totals of eb_colscan_kernel;
// offsets[V] = the number of rows.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) eb_scan_kernel(int* offsets, const int* bsum, int nb, int V) {
    __shared__ int pre[1024];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    // the CTA totals (nb <= a few thousand), scanned 1024 at a time
    extern __shared__ int boff[];
    for (int b0 = 0; b0 < nb; b0 += 1024) {
        const int i = b0 + threadIdx.x;
        pre[threadIdx.x] = i < nb ? bsum[i] : 0;
        __syncthreads();
        for (int o = 1; o < 1024; o <<= 1) {
            const int y = threadIdx.x >= o ? pre[threadIdx.x - o] : 0;
            __syncthreads();
            pre[threadIdx.x] += y;
            __syncthreads();
        }
        if (i < nb) boff[i] = carry + pre[threadIdx.x] - (i < nb ? bsum[i] : 0);
        __syncthreads();
        if (threadIdx.x == 1023) carry += pre[1023];
        __syncthreads();
    }
    for (int v = threadIdx.x; v < V; v += 1024) offsets[v] += boff[v / EB_SCAN_T];
    if (threadIdx.x == 0) offsets[V] = carry;
}

__global__ void eb_scatter_kernel(const int32_t* tok, const int* hist, const int* rank,
                                  const int* offsets, int* sorted, int M, int V) {
    long r = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= M) return;
    int t = tok[r];
    if (t < 0 || t >= V) return;
    long c = r / EB_CHUNK;
    sorted[offsets[t] + hist[c * V + t] + rank[r]] = (int)r;
}

// One CTA per (piece of EB_PIECE sorted rows, EB_COLS columns).  The piece's row
// indices and token ids are staged in shared memory first, so the gradient rows are
// read eight at a time with their loads in flight together; they are still added in
// sorted order.
__global__ void __launch_bounds__(EB_COLS) eb_piece_kernel(const int32_t* tok, const int* sorted,
                                                           const int* offsets, const float* g,
                                                           float* dwte, float* head, float* tail,
                                                           int d, int V, int accumulate) {
    __shared__ int s_row[EB_PIECE];
    __shared__ int s_id[EB_PIECE + 1];
    const int piece = blockIdx.x;
    const int Mv = offsets[V];
    const int p0 = piece * EB_PIECE, p1 = min(p0 + EB_PIECE, Mv);
    if (p0 >= Mv) return;
    const int n = p1 - p0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int r = sorted[p0 + i];
        s_row[i] = r;
        s_id[i] = tok[r];
    }
    if (threadIdx.x == 0) s_id[n] = -1;
    __syncthreads();
    const int col = blockIdx.y * EB_COLS + threadIdx.x;
    if (col >= d) return;
    float acc = 0.f;
    int run_start = 0;   // relative to p0
    for (int i0 = 0; i0 < n; i0 += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = i0 + u < n ? __ldcs(g + (long)s_row[i0 + u] * d + col) : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u;
            if (i >= n) break;
            acc += v[u];
            const int id = s_id[i];
            if (s_id[i + 1] != id) {   // the run of token id ends at sorted position p0 + i
                const int off = offsets[id], cnt = offsets[id + 1] - off;
                if (off >= p0 && off + cnt <= p1) {
                    float* dst = dwte + (long)id * d + col;
                    *dst = accumulate ? *dst + acc : acc;
                } else if (run_start == 0) {
                    head[(long)piece * d + col] = acc;
                } else {
                    tail[(long)piece * d + col] = acc;
                }
                acc = 0.f;
                run_start = i + 1;
            }
        }
    }
}

// dwte[v] = 0 for the ids no row holds (count offsets[v+1] - offsets[v] = 0): the
// overwrite (accumulate = 0) then writes every row of dwte exactly once, the held ids
// by the piece sums.  One warp per id, 16-byte stores.
__global__ void eb_zero_kernel(const int* offsets, float* dwte, int d, int V) {
    const long v = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (v >= V || offsets[v + 1] != offsets[v]) return;
    float4* row = reinterpret_cast<float4*>(dwte + v * d);
    for (int c = threadIdx.x % 32; c < d / 4; c += 32) row[c] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Tokens whose run of sorted rows crosses a piece border: the piece where the run
// starts adds its own part (head or tail) and the heads of the pieces it runs into,
// in order.  One CTA per (piece, 256 columns).
__global__ void eb_fixup_kernel(const int32_t* tok, const int* sorted, const int* offsets, const float* head,
                                const float* tail, float* dwte, int d, int V, int accumulate) {
    const int pa = blockIdx.x;
    const int Mv = offsets[V];
    const int p0 = pa * EB_PIECE, p1 = min(p0 + EB_PIECE, Mv);
    if (p0 >= Mv) return;
    const int id = tok[sorted[p1 - 1]];   // the last run of this piece
    const int off = offsets[id], cnt = offsets[id + 1] - off;
    if (off + cnt <= p1) return;          // ends inside this piece: written by eb_piece_kernel
    if (off < p0) return;                 // started in an earlier piece, which sums it
    const int pb = (off + cnt - 1) / EB_PIECE;
    for (int col = blockIdx.y * blockDim.x + threadIdx.x; col < d; col += gridDim.y * blockDim.x) {
        float sum = (off == p0) ? head[(long)pa * d + col] : tail[(long)pa * d + col];
        for (int p = pa + 1; p <= pb; ++p) sum += head[(long)p * d + col];
        float* dst = dwte + (long)id * d + col;
        *dst = accumulate ? *dst + sum : sum;
    }
}

__global__ void cast_kernel(const float* x, bf16* y, long n) {
    long i = ((long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i + 3 < n) {
        store4<bf16>(y + i, load4<float>(x + i));
    } else {
        for (; i < n; ++i) y[i] = __float2bfloat16_rn(x[i]);
    }
}

}  // namespace

// ------------------------------------------------------------ launchers
template <typename T>
int embed_forward(const int32_t* tok, const T* wte, float* x, int M, int d, int V, uint32_t* flag,
                  cudaStream_t s) {
    if (M <= 0) return NC_OK;
    embed_fwd_kernel<T><<<ceil_div(M, 8), 256, 0, s>>>(tok, wte, x, M, d, V, flag);
    note_launch();
    NC_LAUNCH_CHECK("embed_forward");
    return NC_OK;
}

template <typename T>
int rmsnorm_forward(const float* x, T* y, float* r, int M, int d, cudaStream_t s) {
    if (M <= 0) return NC_OK;
    rmsnorm_fwd_kernel<T><<<ceil_div(M, 8), 256, 0, s>>>(x, y, r, M, d);
    note_launch();
    NC_LAUNCH_CHECK("rmsnorm_forward");
    return NC_OK;
}

template <typename T>
int rmsnorm_backward(const T* dy, const T* y, const float* r, const float* g_in, float* g_out,
                     T* gT, int M, int d, cudaStream_t s) {
    if (M <= 0) return NC_OK;
    rmsnorm_bwd_kernel<T><<<ceil_div(M, 8), 256, 0, s>>>(dy, y, r, g_in, g_out, gT, M, d);
    note_launch();
    NC_LAUNCH_CHECK("rmsnorm_backward");
    return NC_OK;
}

template <typename T>
int rope_apply(T* qkv, long ld, int M, int T_, int H, int Dh, const float2* table, int table_ld, float sign,
               cudaStream_t s) {
    long total = (long)M * H * (Dh / 2);
    if (total <= 0) return NC_OK;
    rope_kernel<T><<<ceil_div(total, 256), 256, 0, s>>>(qkv, ld, M, T_, H, Dh, table, table_ld, sign);
    note_launch();
    NC_LAUNCH_CHECK("rope_apply");
    return NC_OK;
}

template <typename T>
int cross_entropy(T* logits, const int32_t* tgt, float* nll, int M, int V, float scale,
                  uint32_t* flag, cudaStream_t s, const float2* lse_part, bool grad, float* zdot) {
    if (M <= 0) return NC_OK;
    if constexpr (sizeof(T) == 2) {
        if (lse_part && V % (8 * CE2_THREADS) == 0 && V % 128 == 0 && (uintptr_t)logits % 16 == 0) {
            ce_stats_kernel<<<M, CE2_THREADS, 0, s>>>(logits, lse_part, tgt, nll, V, scale, grad, flag,
                                                      grad ? zdot : nullptr);
            note_launch();
            NC_LAUNCH_CHECK("cross_entropy");
            return NC_OK;
        }
        if (V % (8 * CE2_THREADS) == 0 && (uintptr_t)logits % 16 == 0) {
            ce_online_kernel<<<M, CE2_THREADS, 0, s>>>(logits, tgt, nll, V, scale, grad, flag, grad ? zdot : nullptr);
            note_launch();
            NC_LAUNCH_CHECK("cross_entropy");
            return NC_OK;
        }
    }
    ce_kernel<T><<<M, CE_THREADS, 0, s>>>(logits, tgt, nll, V, scale, grad, flag, grad ? zdot : nullptr);
    note_launch();
    NC_LAUNCH_CHECK("cross_entropy");
    return NC_OK;
}

int loss_reduce(const float* nll, const int32_t* tgt, const int32_t* token_bytes, int M, int V,
                float* out, uint32_t* flag, cudaStream_t s, double* sums, int accumulate) {
    loss_reduce_kernel<<<1, 1024, 0, s>>>(nll, tgt, token_bytes, M, V, out, sums, accumulate, flag);
    note_launch();
    NC_LAUNCH_CHECK("loss_reduce");
    return NC_OK;
}

static size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }

size_t embed_backward_ws_bytes(int M, int d, int V) {
    long nchunks = ceil_div(M, EB_CHUNK), npieces = ceil_div(M, EB_PIECE);
    return al256(nchunks * V * 4) + al256((size_t)M * 4) + al256(((size_t)V + 1) * 4) +
           al256((size_t)M * 4) + 2 * al256((size_t)npieces * d * 4) + al256((size_t)ceil_div(V, EB_SCAN_T) * 4);
}

EmbedBwdWs embed_backward_ws(void* base, int M, int d, int V) {
    long nchunks = ceil_div(M, EB_CHUNK), npieces = ceil_div(M, EB_PIECE);
    char* p = (char*)base;
    EmbedBwdWs w;
    w.hist = (int*)p;    p += al256(nchunks * V * 4);
    w.rank = (int*)p;    p += al256((size_t)M * 4);
    w.offsets = (int*)p; p += al256(((size_t)V + 1) * 4);
    w.sorted = (int*)p;  p += al256((size_t)M * 4);
    w.head = (float*)p;  p += al256((size_t)npieces * d * 4);
    w.tail = (float*)p;  p += al256((size_t)npieces * d * 4);
    w.bsum = (int*)p;
    return w;
}

int embed_backward(const int32_t* tok, const float* g, float* dwte, int M, int d, int V,
                   int accumulate, const EmbedBwdWs& ws, cudaStream_t s) {
    const int nchunks = ceil_div(M, EB_CHUNK), npieces = ceil_div(M, EB_PIECE);
    // overwrite: the ids no row holds are zeroed after the sort (below), the others are
    // written by the piece sums; without rows, or with rows not 16-byte aligned, all at once
    const bool zero_rows = !accumulate && M > 0 && d % 4 == 0 && (uintptr_t)dwte % 16 == 0;
    if (!accumulate && !zero_rows)
        NC_TRY(cuda_check(cudaMemsetAsync(dwte, 0, (size_t)V * d * 4, s), "memset dwte"));
    if (M <= 0) return NC_OK;
    NC_TRY(cuda_check(cudaMemsetAsync(ws.hist, 0, (size_t)nchunks * V * 4, s), "memset hist"));
    const int nb = ceil_div(V, EB_SCAN_T);
    if ((size_t)nb * 4 > 48 * 1024) return set_error(NC_ERR_UNSUPPORTED, "embedding backward: vocab %d too large", V);
    eb_hist_rank_kernel<<<nchunks, EB_CHUNK, 0, s>>>(tok, ws.hist, ws.rank, M, V);
    eb_colscan_kernel<<<nb, EB_SCAN_T, 0, s>>>(ws.hist, ws.offsets, ws.bsum, nchunks, V);
    eb_scan_kernel<<<1, 1024, (size_t)nb * 4, s>>>(ws.offsets, ws.bsum, nb, V);
    eb_scatter_kernel<<<ceil_div(M, 256), 256, 0, s>>>(tok, ws.hist, ws.rank, ws.offsets, ws.sorted, M, V);
    if (zero_rows) {
        eb_zero_kernel<<<ceil_div(V, 8), 256, 0, s>>>(ws.offsets, dwte, d, V);
        note_launch();
    }
    eb_piece_kernel<<<dim3(npieces, ceil_div(d, EB_COLS)), EB_COLS, 0, s>>>(
        tok, ws.sorted, ws.offsets, g, dwte, ws.head, ws.tail, d, V, accumulate);
    eb_fixup_kernel<<<dim3(npieces, ceil_div(d, 256)), 256, 0, s>>>(tok, ws.sorted, ws.offsets, ws.head, ws.tail, dwte, d, V, accumulate);
    note_launch(6);
    NC_LAUNCH_CHECK("embed_backward");
    return NC_OK;
}

int cast_f32_bf16(const float* x, bf16* y, long n, cudaStream_t s) {
    if (n <= 0) return NC_OK;
    cast_kernel<<<ceil_div(ceil_div(n, 4), 256), 256, 0, s>>>(x, y, n);
    note_launch();
    NC_LAUNCH_CHECK("cast_f32_bf16");
    return NC_OK;
}

#define NC_INST(T)                                                                              \
    template int embed_forward<T>(const int32_t*, const T*, float*, int, int, int, uint32_t*,   \
                                  cudaStream_t);                                                \
    template int rmsnorm_forward<T>(const float*, T*, float*, int, int, cudaStream_t);          \
    template int rmsnorm_backward<T>(const T*, const T*, const float*, const float*, float*, \
                                     T*, int, int, cudaStream_t);                               \
    template int rope_apply<T>(T*, long, int, int, int, int, const float2*, int, float, cudaStream_t); \
    template int cross_entropy<T>(T*, const int32_t*, float*, int, int, float, uint32_t*,       \
                                  cudaStream_t, const float2*, bool, float*);
NC_INST(float)
NC_INST(bf16)
#undef NC_INST

}  // namespace nc
