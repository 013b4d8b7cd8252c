// Inference with a KV cache: the row-level kernels of prefill and decode.
//
// nanochat speedrun walkthrough (lyylswood.com), section 预搜检, on sampling from the
// trained base model: inference runs through an Engine class that keeps a KV cache and
// implements the two usual phases, prefill (the whole prompt at once) and decode (one
// token per sequence per step).
//
// Decode works on the B sequences of a step in a transposed layout: the residual stream
// is x^T [d][Bp] (fp32) and every projection is the product W [N, K] x Y[Bp, K]^T ->
// [N][Bp], so the weight matrix, the only large operand, is the tensor-core A operand
// streamed by TMA and the few token rows are the small B operand (Bp = B rounded up to
// a multiple of 8; the extra columns stay zero).  The kernels here do the rest: the
// embedding and RMSNorm in that layout, RoPE at the step's position with the append of
// k and v to the cache, attention of one query over the cached keys (split over key
// chunks, then combined), and the greedy next token.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace nc {
namespace {

constexpr float RMS_EPS_D = 1e-6f;
constexpr float LOG2E_D = 1.4426950408889634f;

__device__ __forceinline__ void flag_or(uint32_t* flag, uint32_t bits) {
    if (flag) atomicOr(flag, bits);
}

// x^T[j][b] = wte[tok[b]][j] for b < B; zero columns B .. Bp-1
template <typename T>
__global__ void embed_t_kernel(const int32_t* tok, const T* wte, float* xt, int B, int Bp, int d, int V,
                               uint32_t* flag) {
    const int b = blockIdx.y, j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= d) return;
    float v = 0.f;
    if (b < B) {
        const int t = tok[b];
        if (t >= 0 && t < V) v = to_f<T>(wte[(long)t * d + j]);
        else if (j == 0) flag_or(flag, NC_FLAG_TOKEN_RANGE);
    }
    xt[(long)j * Bp + b] = v;
}

// y[b][j] = x^T[j][b] / sqrt(mean_j x^T[j][b]^2 + eps), one CTA per column b
template <typename T>
__global__ void rmsnorm_cols_kernel(const float* xt, T* y, int Bp, int d) {
    __shared__ float sh[32];
    const int b = blockIdx.x;
    float ss = 0.f;
    for (int j = threadIdx.x; j < d; j += blockDim.x) {
        const float v = xt[(long)j * Bp + b];
        ss += v * v;
    }
    ss = warp_sum(ss);
    if (threadIdx.x % 32 == 0) sh[threadIdx.x / 32] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float t = threadIdx.x < blockDim.x / 32 ? sh[threadIdx.x] : 0.f;
        t = warp_sum(t);
        if (threadIdx.x == 0) sh[0] = t;
    }
    __syncthreads();
    const float rr = 1.0f / sqrtf(sh[0] / (float)d + RMS_EPS_D);
    for (int j = threadIdx.x; j < d; j += blockDim.x) y[(long)b * d + j] = from_f<T>(xt[(long)j * Bp + b] * rr);
}

// c = [q | k | v]^T [3d][Bp] of position pos -> q [Bp][d] with RoPE, and k (with RoPE), v
// appended to the cache at row (b, pos).  One thread per (b, head, rotation pair).
template <typename T>
__global__ void qkv_post_kernel(const T* c, int B, int Bp, int d, int H, int Dh, int pos_arg,
                                const int* pos_dev, const float2* rope, int rope_ld, T* q, T* kc, T* vc,
                                int cache_T) {
    const int pos = pos_dev ? *pos_dev : pos_arg;   // (a replayed step reads its position)
    const int half = Dh / 2;
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long)Bp * H * half) return;
    const int b = idx % Bp;                  // (consecutive threads read one row of c)
    const int j = (idx / Bp) % half;
    const int h = idx / ((long)Bp * half);
    const int c1 = h * Dh + j, c2 = c1 + half;
    if (b >= B) {
        q[(long)b * d + c1] = from_f<T>(0.f);
        q[(long)b * d + c2] = from_f<T>(0.f);
        return;
    }
    const float2 cs = rope[(long)j * rope_ld + pos];
    const long row = (long)b * cache_T + pos;
    {
        const float x1 = to_f<T>(c[(long)c1 * Bp + b]), x2 = to_f<T>(c[(long)c2 * Bp + b]);
        q[(long)b * d + c1] = from_f<T>(x1 * cs.x - x2 * cs.y);
        q[(long)b * d + c2] = from_f<T>(x2 * cs.x + x1 * cs.y);
    }
    {
        const float x1 = to_f<T>(c[(long)(d + c1) * Bp + b]), x2 = to_f<T>(c[(long)(d + c2) * Bp + b]);
        kc[row * d + c1] = from_f<T>(x1 * cs.x - x2 * cs.y);
        kc[row * d + c2] = from_f<T>(x2 * cs.x + x1 * cs.y);
    }
    vc[row * d + c1] = c[(long)(2 * d + c1) * Bp + b];
    vc[row * d + c2] = c[(long)(2 * d + c2) * Bp + b];
}

// --------------------------------------------------------------------- decode attention
// One query per (b, head) against its n cached keys (causal: every cached position is at
// or before the query's).  CTA (chunk, head, b) takes keys [chunk*kc, min(n, (chunk+1)*kc));
// its 8 groups of 16 lanes take every 8th key, each lane 8 of the 128 dimensions, and keep
// an online softmax (log2 domain); the groups are merged in shared memory and the chunk's
// unnormalised (max, sum, o) go to the workspace for the combine kernel.
constexpr int DA_THREADS = 128;
constexpr int DA_GROUPS = DA_THREADS / 16;
constexpr int DA_HD = 128;

template <typename T> struct Vec8;
template <> struct Vec8<bf16> {
    __device__ static void load(const bf16* p, float* f) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            f[2 * e] = x.x;
            f[2 * e + 1] = x.y;
        }
    }
};
template <> struct Vec8<float> {
    __device__ static void load(const float* p, float* f) {
        const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
};

template <typename T>
__global__ void __launch_bounds__(DA_THREADS) decode_attn_kernel(const T* q, const T* kc, const T* vc, int d,
                                                                 int cache_T, int n_arg, const int* pos_dev,
                                                                 int kchunk, float scale, float* part_o,
                                                                 float2* part_ml) {
    // a replayed step reads its position; the grid then covers the whole cache and the
    // chunks past the last key leave an empty partial (max -inf, sum 0)
    const int n = pos_dev ? *pos_dev + 1 : n_arg;
    __shared__ float s_o[DA_GROUPS][DA_HD];
    __shared__ float s_m[DA_GROUPS], s_l[DA_GROUPS];
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z, H = gridDim.y, nchunk = gridDim.x;
    const int g = threadIdx.x / 16, lane = threadIdx.x % 16;
    const int k0 = chunk * kchunk, k1 = min(n, k0 + kchunk);
    const long base = (long)b * cache_T * d + h * DA_HD + lane * 8;
    float qf[8];
    Vec8<T>::load(q + (long)b * d + h * DA_HD + lane * 8, qf);
    const float c2 = scale * LOG2E_D;
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[e] *= c2;
    float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = 0.f;
    // the loop bound is the same for the whole CTA (every lane reaches every shuffle);
    // a group whose key is past the chunk's end takes no part in the update
    for (int k = k0 + g; k - g < k1; k += 2 * DA_GROUPS) {
        const int kb = k + DA_GROUPS;
        const bool one = k < k1, two = kb < k1;
        float kf[8], kf2[8], vf[8], vf2[8];
        if (one) {
            Vec8<T>::load(kc + base + (long)k * d, kf);
            Vec8<T>::load(vc + base + (long)k * d, vf);
        }
        if (two) {
            Vec8<T>::load(kc + base + (long)kb * d, kf2);
            Vec8<T>::load(vc + base + (long)kb * d, vf2);
        }
        float s = 0.f, s2 = 0.f;
        if (one) {
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(qf[e], kf[e], s);
        }
        if (two) {
#pragma unroll
            for (int e = 0; e < 8; ++e) s2 = fmaf(qf[e], kf2[e], s2);
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {   // sum over the group's 16 lanes
            s += __shfl_xor_sync(0xffffffffu, s, off);
            s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        }
        if (!one) continue;                        // (then two is false as well)
        const float mn = two ? fmaxf(m, fmaxf(s, s2)) : fmaxf(m, s);
        const float corr = exp2f(m - mn);          // m = -inf before the first key: 0
        const float p = exp2f(s - mn), p2 = two ? exp2f(s2 - mn) : 0.f;
        l = l * corr + p + p2;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = fmaf(o[e], corr, fmaf(p, vf[e], two ? p2 * vf2[e] : 0.f));
        m = mn;
    }
    // merge the groups
#pragma unroll
    for (int e = 0; e < 8; ++e) s_o[g][lane * 8 + e] = o[e];
    if (lane == 0) { s_m[g] = m; s_l[g] = l; }
    __syncthreads();
    float mm = -INFINITY;
#pragma unroll
    for (int i = 0; i < DA_GROUPS; ++i) mm = fmaxf(mm, s_m[i]);
    const int dim = threadIdx.x;   // DA_THREADS == DA_HD
    float acc = 0.f, ll = 0.f;
#pragma unroll
    for (int i = 0; i < DA_GROUPS; ++i) {
        const float w = s_m[i] == -INFINITY ? 0.f : exp2f(s_m[i] - mm);
        acc = fmaf(s_o[i][dim], w, acc);
        ll = fmaf(s_l[i], w, ll);
    }
    const long pc = ((long)b * H + h) * nchunk + chunk;
    part_o[pc * DA_HD + dim] = acc;
    if (dim == 0) part_ml[pc] = make_float2(mm, ll);
}

// The same chunked one-query attention for bf16 caches with the cache rows brought in
// by TMA: tiles of 32 keys x 128 dims of k and of v (two 64-dim atoms each, 128-byte
// swizzle) in a ring of DT_ST stages, so the copies run ahead of the arithmetic instead
// of each group waiting on its own loads.  Group g (16 lanes, 8 dims each) takes keys
// g, g+8, g+16 and g+24 of every tile, four at a time.
constexpr int DT_KEYS = 32;
constexpr int DT_ST = 4;
constexpr int DT_TILE = DT_KEYS * DA_HD * 2;          // 8 KB
// tiles | barriers (64 B) | group merge [DA_GROUPS][DA_HD] + m, l | abort word
constexpr int DT_SMEM = DT_ST * 2 * DT_TILE + 64 + (DA_GROUPS * DA_HD + 2 * DA_GROUPS + 4) * 4;

// this lane's 8 dims of key row r of a swizzled tile (atom = dims 64a .. 64a+63)
__device__ __forceinline__ const uint8_t* dt_addr(const uint8_t* tile, int r, int lane16) {
    const int a = lane16 >> 3, c = lane16 & 7;
    return tile + a * (DT_KEYS * 128) + r * 128 + ((c ^ (r & 7)) << 4);
}

__global__ void __launch_bounds__(DA_THREADS) decode_attn_tma_kernel(
    const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv, const bf16* q, int d,
    int cache_T, int n_arg, const int* pos_dev, int kchunk, float scale, float* part_o, float2* part_ml) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(dsm + DT_ST * 2 * DT_TILE);
    float (*s_o)[DA_HD] = reinterpret_cast<float (*)[DA_HD]>(dsm + DT_ST * 2 * DT_TILE + 64);
    float* s_m = &s_o[DA_GROUPS][0];
    float* s_l = s_m + DA_GROUPS;
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_l + DA_GROUPS);
    // the swizzled tiles need a 1024-byte aligned base; without it the chunk reports NaN
    const bool bad = (tc::smem_u32(dsm) & 1023u) != 0;
    const int n = pos_dev ? *pos_dev + 1 : n_arg;
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z, H = gridDim.y, nchunk = gridDim.x;
    const int g = threadIdx.x / 16, lane = threadIdx.x % 16;
    const int k0 = chunk * kchunk, k1 = min(n, k0 + kchunk);
    const int ntile = bad ? 0 : k1 > k0 ? (k1 - k0 + DT_KEYS - 1) / DT_KEYS : 0;
    const int row0 = b * cache_T + k0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < DT_ST; ++i) tc::mbar_init(&full[i], 1);
        *s_abort = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    auto issue = [&](int i) {
        uint8_t* kt = dsm + (i % DT_ST) * 2 * DT_TILE;
        uint64_t* bar = &full[i % DT_ST];
        tc::mbar_expect_tx(bar, 2 * DT_TILE);
        const int y = row0 + i * DT_KEYS;
        tc::tma_load_3d(kt, &mk, bar, h * DA_HD, y, 0);
        tc::tma_load_3d(kt + DT_TILE / 2, &mk, bar, h * DA_HD + 64, y, 0);
        tc::tma_load_3d(kt + DT_TILE, &mv, bar, h * DA_HD, y, 0);
        tc::tma_load_3d(kt + DT_TILE + DT_TILE / 2, &mv, bar, h * DA_HD + 64, y, 0);
    };
    if (threadIdx.x == 0)
        for (int i = 0; i < DT_ST && i < ntile; ++i) issue(i);
    float qf[8];
    Vec8<bf16>::load(q + (long)b * d + h * DA_HD + lane * 8, qf);
    const float c2 = scale * LOG2E_D;
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[e] *= c2;
    float m = bad ? NAN : -INFINITY, l = 0.f, o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = 0.f;
    for (int i = 0; i < ntile; ++i) {
        if (!tc::mbar_wait(&full[i % DT_ST], (i / DT_ST) & 1, s_abort)) {
            m = NAN;   // a copy that never landed: the step's logits come out NaN (flagged)
            break;
        }
        const uint8_t* kt = dsm + (i % DT_ST) * 2 * DT_TILE;
        const uint8_t* vt = kt + DT_TILE;
        const int kbase = k0 + i * DT_KEYS;
        float sc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float kf[8];
            Vec8<bf16>::load(reinterpret_cast<const bf16*>(dt_addr(kt, g + 8 * u, lane)), kf);
            float x = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) x = fmaf(qf[e], kf[e], x);
            sc[u] = x;
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)   // sums over the group's 16 lanes
#pragma unroll
            for (int u = 0; u < 4; ++u) sc[u] += __shfl_xor_sync(0xffffffffu, sc[u], off);
        float mn = m;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (kbase + g + 8 * u >= k1) sc[u] = -INFINITY;
            mn = fmaxf(mn, sc[u]);
        }
        if (mn != -INFINITY) {
            const float corr = exp2f(m - mn);   // m = -inf before the first key: 0
            l *= corr;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] *= corr;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (sc[u] == -INFINITY) continue;   // past the chunk's end: the row is not read
                const float pr = exp2f(sc[u] - mn);
                float vf[8];
                Vec8<bf16>::load(reinterpret_cast<const bf16*>(dt_addr(vt, g + 8 * u, lane)), vf);
                l += pr;
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = fmaf(pr, vf[e], o[e]);
            }
            m = mn;
        }
        __syncthreads();   // every thread is done with this stage
        if (threadIdx.x == 0 && i + DT_ST < ntile) {
            tc::fence_async_smem();
            issue(i + DT_ST);
        }
    }
    // merge the groups
#pragma unroll
    for (int e = 0; e < 8; ++e) s_o[g][lane * 8 + e] = o[e];
    if (lane == 0) { s_m[g] = m; s_l[g] = l; }
    __syncthreads();
    float mm = -INFINITY;
#pragma unroll
    for (int i = 0; i < DA_GROUPS; ++i) mm = fmaxf(mm, s_m[i]);
    const int dim = threadIdx.x;   // DA_THREADS == DA_HD
    float acc = 0.f, ll = 0.f;
#pragma unroll
    for (int i = 0; i < DA_GROUPS; ++i) {
        const float w = s_m[i] == -INFINITY ? 0.f : exp2f(s_m[i] - mm);
        acc = fmaf(s_o[i][dim], w, acc);
        ll = fmaf(s_l[i], w, ll);
    }
    const long pc = ((long)b * H + h) * nchunk + chunk;
    part_o[pc * DA_HD + dim] = acc;
    if (dim == 0) part_ml[pc] = make_float2(mm, ll);
}

// out[b][h*128 + dim] = sum_c o_c 2^(m_c - M) / sum_c l_c 2^(m_c - M); zero rows b >= B
template <typename T>
__global__ void __launch_bounds__(DA_HD) decode_combine_kernel(const float* part_o, const float2* part_ml,
                                                                int nchunk, int B, int d, T* out) {
    const int h = blockIdx.x, b = blockIdx.y, H = gridDim.x, dim = threadIdx.x;
    T* dst = out + (long)b * d + h * DA_HD + dim;
    if (b >= B) { *dst = from_f<T>(0.f); return; }
    const long p0 = ((long)b * H + h) * nchunk;
    float mm = -INFINITY;
    for (int c = 0; c < nchunk; ++c) mm = fmaxf(mm, part_ml[p0 + c].x);
    float acc = 0.f, ll = 0.f;
    for (int c = 0; c < nchunk; ++c) {
        const float2 ml = part_ml[p0 + c];
        const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mm);
        acc = fmaf(part_o[(p0 + c) * DA_HD + dim], w, acc);
        ll = fmaf(ml.y, w, ll);
    }
    *dst = from_f<T>(acc / ll);
}

// --------------------------------------------------------------------- greedy token
// logits^T [V][Bp]: CTA (part, b) scans its rows of column b; ties go to the lowest id
constexpr int AM_THREADS = 256;

__device__ __forceinline__ void am_pick(float& v, int& i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i) || (v != v && v2 == v2)) { v = v2; i = i2; }
}

__global__ void __launch_bounds__(AM_THREADS) argmax_part_kernel(const float* lt, int V, int Bp, int rows_per_part,
                                                                 float* pv, int* pi) {
    __shared__ float sv[AM_THREADS / 32];
    __shared__ int si[AM_THREADS / 32];
    const int part = blockIdx.x, b = blockIdx.y, nparts = gridDim.x;
    const int r0 = part * rows_per_part, r1 = min(V, r0 + rows_per_part);
    float v = -INFINITY;
    int i = 0x7fffffff;
    for (int r = r0 + threadIdx.x; r < r1; r += AM_THREADS) am_pick(v, i, lt[(long)r * Bp + b], r);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, off);
        am_pick(v, i, v2, i2);
    }
    if (threadIdx.x % 32 == 0) { sv[threadIdx.x / 32] = v; si[threadIdx.x / 32] = i; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < AM_THREADS / 32; ++w) am_pick(v, i, sv[w], si[w]);
        pv[(long)b * nparts + part] = v;
        pi[(long)b * nparts + part] = i;
    }
}

__global__ void argmax_final_kernel(const float* pv, const int* pi, int nparts, int V, int32_t* next,
                                    uint32_t* flag) {
    const int b = blockIdx.x;
    float v = -INFINITY;
    int i = 0x7fffffff;
    for (int p = threadIdx.x; p < nparts; p += 32) am_pick(v, i, pv[(long)b * nparts + p], pi[(long)b * nparts + p]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, off);
        am_pick(v, i, v2, i2);
    }
    if (threadIdx.x == 0) {
        if (!(v == v) || i < 0 || i >= V) {   // no finite logit: flag it, emit token 0
            flag_or(flag, NC_FLAG_NONFINITE);
            i = 0;
        }
        next[b] = i;
    }
}

// out [B][V] fp32 = logits^T [V][Bp] transposed (32 x 32 tiles)
__global__ void transpose_logits_kernel(const float* lt, int V, int Bp, int B, float* out) {
    __shared__ float t[32][33];
    const int r0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    for (int k = threadIdx.y; k < 32; k += blockDim.y) {
        const int r = r0 + k, c = c0 + threadIdx.x;
        t[k][threadIdx.x] = (r < V && c < Bp) ? lt[(long)r * Bp + c] : 0.f;
    }
    __syncthreads();
    for (int k = threadIdx.y; k < 32; k += blockDim.y) {
        const int c = c0 + k, r = r0 + threadIdx.x;
        if (c < B && r < V) out[(long)c * V + r] = t[threadIdx.x][k];
    }
}

// --------------------------------------------------------------------- prefill helpers
// cache row (b, t) <- k, v of row b*T0 + t of the projection output [B*T0][3d]
template <typename T>
__global__ void kv_store_kernel(const T* qkv, int B, int T0, int d, T* kc, T* vc, int cache_T) {
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    const long per_row = d;
    if (idx >= (long)B * T0 * per_row) return;
    const long row = idx / per_row;
    const int j = idx % per_row;
    const int b = row / T0, t = row % T0;
    const long dst = ((long)b * cache_T + t) * d + j;
    kc[dst] = qkv[row * 3 * d + d + j];
    vc[dst] = qkv[row * 3 * d + 2 * d + j];
}

// out [Bp][d] <- row b*T0 + T0-1 of y for b < B, zero rows B .. Bp-1
template <typename T>
__global__ void gather_last_kernel(const T* y, int B, int Bp, int T0, int d, T* out) {
    const int b = blockIdx.y, j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= d) return;
    out[(long)b * d + j] = b < B ? y[((long)b * T0 + T0 - 1) * d + j] : from_f<T>(0.f);
}

}  // namespace

// ------------------------------------------------------------------------------ host
template <typename T>
int decode_embed_t(const int32_t* tok, const T* wte, float* xt, int B, int Bp, int d, int V, uint32_t* flag,
                   cudaStream_t s) {
    embed_t_kernel<T><<<dim3(ceil_div(d, 256), Bp), 256, 0, s>>>(tok, wte, xt, B, Bp, d, V, flag);
    note_launch();
    NC_LAUNCH_CHECK("decode_embed_t");
    return NC_OK;
}

template <typename T>
int decode_rmsnorm_cols(const float* xt, T* y, int Bp, int d, cudaStream_t s) {
    rmsnorm_cols_kernel<T><<<Bp, 256, 0, s>>>(xt, y, Bp, d);
    note_launch();
    NC_LAUNCH_CHECK("decode_rmsnorm_cols");
    return NC_OK;
}

template <typename T>
int decode_qkv_post(const T* c, int B, int Bp, int d, int H, int Dh, int pos, const int* pos_dev,
                    const float2* rope, int rope_ld, T* q, T* kc, T* vc, int cache_T, cudaStream_t s) {
    const long total = (long)Bp * H * (Dh / 2);
    qkv_post_kernel<T><<<ceil_div(total, 256), 256, 0, s>>>(c, B, Bp, d, H, Dh, pos, pos_dev, rope, rope_ld, q,
                                                           kc, vc, cache_T);
    note_launch();
    NC_LAUNCH_CHECK("decode_qkv_post");
    return NC_OK;
}

int decode_attention_chunks(int B, int H, int n) {
    // keys per CTA: the largest power of two (16 .. 512) that gives >= 16 CTAs per SM, so
    // that the cache rows in flight cover the memory latency (each group has two rows of k
    // and two of v in flight)
    int kc = 512;
    while (kc > 16 && (long)B * H * ceil_div(n, kc) < 16L * num_sms()) kc /= 2;
    return kc;
}

size_t decode_attention_ws_bytes(int B, int H, int n) {
    const int kc = decode_attention_chunks(B, H, n);
    const long parts = (long)B * H * ceil_div(n, kc);
    return (((size_t)parts * DA_HD * 4 + 255) & ~(size_t)255) + (size_t)parts * 8;
}

template <typename T>
int decode_attention(const T* q, const T* kc, const T* vc, int B, int Bp, int d, int H, int Dh, int cache_T,
                     int n, const int* pos_dev, T* out, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (Dh != DA_HD) return set_error(NC_ERR_UNSUPPORTED, "decode attention: head dim %d (128 only)", Dh);
    // chunk boundaries from the cache length, so a replayed step (grid over the whole cache,
    // the chunks past the last key empty) adds up exactly as a direct one
    const int kch = decode_attention_chunks(B, H, cache_T);
    const int nchunk = ceil_div(pos_dev ? cache_T : n, kch);
    const long parts = (long)B * H * nchunk;
    if (decode_attention_ws_bytes(B, H, cache_T) > ws_bytes) return set_error(NC_ERR_ARG, "decode attention workspace");
    float* po = reinterpret_cast<float*>(ws);
    float2* pml = reinterpret_cast<float2*>(reinterpret_cast<char*>(ws) + (((size_t)parts * DA_HD * 4 + 255) & ~(size_t)255));
    if constexpr (sizeof(T) == 2) {
        // bf16: the cache rows come in by TMA (d and the cache base allow the copies)
        static DeviceOnce init;
        NC_TRY(init.run([] {
            return cuda_check(cudaFuncSetAttribute(decode_attn_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   DT_SMEM), "decode attention smem attribute");
        }));
        CUtensorMap mk, mv;
        const long rows = (long)B * cache_T;   // the sequences in use (rows past them read as zeros)
        NC_TRY(make_map(&mk, kc, d, rows, 1, d, 0, 64, DT_KEYS));
        NC_TRY(make_map(&mv, vc, d, rows, 1, d, 0, 64, DT_KEYS));
        decode_attn_tma_kernel<<<dim3(nchunk, H, B), DA_THREADS, DT_SMEM, s>>>(
            mk, mv, q, d, cache_T, n, pos_dev, kch, 1.0f / sqrtf((float)Dh), po, pml);
    } else {
        decode_attn_kernel<T><<<dim3(nchunk, H, B), DA_THREADS, 0, s>>>(q, kc, vc, d, cache_T, n, pos_dev, kch,
                                                                       1.0f / sqrtf((float)Dh), po, pml);
    }
    decode_combine_kernel<T><<<dim3(H, Bp), DA_HD, 0, s>>>(po, pml, nchunk, B, d, out);
    note_launch(2);
    NC_LAUNCH_CHECK("decode_attention");
    return NC_OK;
}

int decode_argmax(const float* lt, int V, int B, int Bp, int32_t* next, void* ws, size_t ws_bytes, uint32_t* flag,
                  cudaStream_t s) {
    const int nparts = 64;
    if ((size_t)B * nparts * 8 > ws_bytes) return set_error(NC_ERR_ARG, "argmax workspace");
    float* pv = reinterpret_cast<float*>(ws);
    int* pi = reinterpret_cast<int*>(pv + (long)B * nparts);
    argmax_part_kernel<<<dim3(nparts, B), AM_THREADS, 0, s>>>(lt, V, Bp, ceil_div(V, nparts), pv, pi);
    argmax_final_kernel<<<B, 32, 0, s>>>(pv, pi, nparts, V, next, flag);
    note_launch(2);
    NC_LAUNCH_CHECK("decode_argmax");
    return NC_OK;
}

int decode_logits_out(const float* lt, int V, int B, int Bp, float* out, cudaStream_t s) {
    transpose_logits_kernel<<<dim3(ceil_div(V, 32), ceil_div(Bp, 32)), dim3(32, 8), 0, s>>>(lt, V, Bp, B, out);
    note_launch();
    NC_LAUNCH_CHECK("decode_logits_out");
    return NC_OK;
}

template <typename T>
int prefill_kv_store(const T* qkv, int B, int T0, int d, T* kc, T* vc, int cache_T, cudaStream_t s) {
    const long total = (long)B * T0 * d;
    kv_store_kernel<T><<<ceil_div(total, 256), 256, 0, s>>>(qkv, B, T0, d, kc, vc, cache_T);
    note_launch();
    NC_LAUNCH_CHECK("prefill_kv_store");
    return NC_OK;
}

template <typename T>
int prefill_gather_last(const T* y, int B, int Bp, int T0, int d, T* out, cudaStream_t s) {
    gather_last_kernel<T><<<dim3(ceil_div(d, 256), Bp), 256, 0, s>>>(y, B, Bp, T0, d, out);
    note_launch();
    NC_LAUNCH_CHECK("prefill_gather_last");
    return NC_OK;
}

__global__ void set_int_kernel(int* p, int v) { *p = v; }

int decode_set_pos(int* pos_dev, int pos, cudaStream_t s) {
    set_int_kernel<<<1, 1, 0, s>>>(pos_dev, pos);
    note_launch();
    NC_LAUNCH_CHECK("decode_set_pos");
    return NC_OK;
}

#define NC_DEC_INST(T)                                                                                       \
    template int decode_embed_t<T>(const int32_t*, const T*, float*, int, int, int, int, uint32_t*,         \
                                   cudaStream_t);                                                            \
    template int decode_rmsnorm_cols<T>(const float*, T*, int, int, cudaStream_t);                           \
    template int decode_qkv_post<T>(const T*, int, int, int, int, int, int, const int*, const float2*, int, \
                                    T*, T*, T*, int, cudaStream_t);                                          \
    template int decode_attention<T>(const T*, const T*, const T*, int, int, int, int, int, int, int,       \
                                     const int*, T*, void*, size_t, cudaStream_t);                           \
    template int prefill_kv_store<T>(const T*, int, int, int, T*, T*, int, cudaStream_t);                    \
    template int prefill_gather_last<T>(const T*, int, int, int, int, T*, cudaStream_t);
NC_DEC_INST(float)
NC_DEC_INST(bf16)

}  // namespace nc
