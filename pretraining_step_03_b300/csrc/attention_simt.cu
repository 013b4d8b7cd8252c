// Causal multi-head attention on CUDA cores, any even head dim <= 128.
// It is the fp32-mode path (exact enough for 1e-5 loss parity) and the
// path for head dims the tensor-core kernels do not take.
//
// Source: nanochat speedrun walkthrough (lyylswood.com), section 预搜检
// (pretraining): multi-head attention, 10 heads of dim 128 at d20.
//   forward:  O_t = sum_{s<=t} softmax_s(q_t.k_s / sqrt(D)) v_s, lse_t kept;
//   backward: P_ts = exp(q_t.k_s/sqrt(D) - lse_t), dP_ts = dO_t.v_s,
//             D_t = dO_t.O_t, dS = P (dP - D_t); dq_t = sum_s dS k_s / sqrt(D),
//             dk_s = sum_t dS q_t / sqrt(D), dv_s = sum_t P dO_t.
#include "kernels.cuh"

#include <math.h>

namespace nc {
namespace {

constexpr int WARPS = 8;

template <typename T>
__global__ void __launch_bounds__(WARPS * 32) attn_fwd_simt(const T* q, const T* k, const T* v,
                                                            long ld, T* o, long ldo, float* lse,
                                                            int T_, int H, int D) {
    const int lane = threadIdx.x % 32, b = blockIdx.z, h = blockIdx.y;
    const int t = blockIdx.x * WARPS + threadIdx.x / 32;
    if (t >= T_) return;
    const float scale = 1.0f / sqrtf((float)D);
    const long rowq = ((long)b * T_ + t) * ld + (long)h * D;
    float qv[4], acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int j = lane + 32 * i;
        qv[i] = j < D ? to_f<T>(q[rowq + j]) : 0.f;
        acc[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int s = 0; s <= t; ++s) {
        const long rk = ((long)b * T_ + s) * ld + (long)h * D;
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int j = lane + 32 * i;
            if (j < D) p += qv[i] * to_f<T>(k[rk + j]);
        }
        p = warp_sum(p) * scale;
        const float mn = fmaxf(m, p), c = expf(m - mn), e = expf(p - mn);
        l = l * c + e;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int j = lane + 32 * i;
            if (j < D) acc[i] = acc[i] * c + e * to_f<T>(v[rk + j]);
        }
        m = mn;
    }
    const long ro = ((long)b * T_ + t) * ldo + (long)h * D;
    const float inv = 1.0f / l;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int j = lane + 32 * i;
        if (j < D) o[ro + j] = from_f<T>(acc[i] * inv);
    }
    if (lane == 0) lse[((long)b * H + h) * T_ + t] = m + logf(l);
}

template <typename T>
__global__ void attn_delta_simt(const T* o, const T* dout, long ldo, float* delta, int T_, int H,
                                int D) {
    const int lane = threadIdx.x % 32, b = blockIdx.z, h = blockIdx.y;
    const int t = blockIdx.x * WARPS + threadIdx.x / 32;
    if (t >= T_) return;
    const long r = ((long)b * T_ + t) * ldo + (long)h * D;
    float s = 0.f;
    for (int j = lane; j < D; j += 32) s += to_f<T>(o[r + j]) * to_f<T>(dout[r + j]);
    s = warp_sum(s);
    if (lane == 0) delta[((long)b * H + h) * T_ + t] = s;
}

// one warp per query row: dq_t = scale * sum_{s<=t} P (dP - D_t) k_s
template <typename T>
__global__ void __launch_bounds__(WARPS * 32) attn_dq_simt(const T* q, const T* k, const T* v,
                                                           long ld, const T* dout, long ldo,
                                                           const float* lse, const float* delta,
                                                           T* dq, long ldd, int T_, int H, int D) {
    const int lane = threadIdx.x % 32, b = blockIdx.z, h = blockIdx.y;
    const int t = blockIdx.x * WARPS + threadIdx.x / 32;
    if (t >= T_) return;
    const float scale = 1.0f / sqrtf((float)D);
    const long rq = ((long)b * T_ + t) * ld + (long)h * D;
    const long rdo = ((long)b * T_ + t) * ldo + (long)h * D;
    const long st = ((long)b * H + h) * T_ + t;
    const float L = lse[st], Dt = delta[st];
    float qv[4], dov[4], acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int j = lane + 32 * i;
        qv[i] = j < D ? to_f<T>(q[rq + j]) : 0.f;
        dov[i] = j < D ? to_f<T>(dout[rdo + j]) : 0.f;
        acc[i] = 0.f;
    }
    for (int s = 0; s <= t; ++s) {
        const long rk = ((long)b * T_ + s) * ld + (long)h * D;
        float sc = 0.f, dp = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int j = lane + 32 * i;
            if (j < D) {
                sc += qv[i] * to_f<T>(k[rk + j]);
                dp += dov[i] * to_f<T>(v[rk + j]);
            }
        }
        sc = warp_sum(sc);
        dp = warp_sum(dp);
        const float p = expf(sc * scale - L), ds = p * (dp - Dt);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int j = lane + 32 * i;
            if (j < D) acc[i] += ds * to_f<T>(k[rk + j]);
        }
    }
    const long rd = ((long)b * T_ + t) * ldd + (long)h * D;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int j = lane + 32 * i;
        if (j < D) dq[rd + j] = from_f<T>(acc[i] * scale);
    }
}

// one warp per key row s: dv_s = sum_{t>=s} P dO_t; dk_s = scale * sum_{t>=s} dS q_t
template <typename T>
__global__ void __launch_bounds__(WARPS * 32) attn_dkdv_simt(const T* q, const T* k, const T* v,
                                                             long ld, const T* dout, long ldo,
                                                             const float* lse, const float* delta,
                                                             T* dk, T* dv, long ldd, int T_, int H,
                                                             int D) {
    const int lane = threadIdx.x % 32, b = blockIdx.z, h = blockIdx.y;
    const int s = blockIdx.x * WARPS + threadIdx.x / 32;
    if (s >= T_) return;
    const float scale = 1.0f / sqrtf((float)D);
    const long rk = ((long)b * T_ + s) * ld + (long)h * D;
    float kv[4], vv[4], adk[4], adv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int j = lane + 32 * i;
        kv[i] = j < D ? to_f<T>(k[rk + j]) : 0.f;
        vv[i] = j < D ? to_f<T>(v[rk + j]) : 0.f;
        adk[i] = adv[i] = 0.f;
    }
    for (int t = s; t < T_; ++t) {
        const long rq = ((long)b * T_ + t) * ld + (long)h * D;
        const long rdo = ((long)b * T_ + t) * ldo + (long)h * D;
        const long st = ((long)b * H + h) * T_ + t;
        float sc = 0.f, dp = 0.f, qx[4], dox[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int j = lane + 32 * i;
            qx[i] = j < D ? to_f<T>(q[rq + j]) : 0.f;
            dox[i] = j < D ? to_f<T>(dout[rdo + j]) : 0.f;
            sc += qx[i] * kv[i];
            dp += dox[i] * vv[i];
        }
        sc = warp_sum(sc);
        dp = warp_sum(dp);
        const float p = expf(sc * scale - lse[st]), ds = p * (dp - delta[st]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            adv[i] += p * dox[i];
            adk[i] += ds * qx[i];
        }
    }
    const long rd = ((long)b * T_ + s) * ldd + (long)h * D;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int j = lane + 32 * i;
        if (j < D) {
            dk[rd + j] = from_f<T>(adk[i] * scale);
            dv[rd + j] = from_f<T>(adv[i]);
        }
    }
}

}  // namespace

template <typename T>
int attention_forward_simt(const T* q, const T* k, const T* v, long ld, T* o, long ldo, float* lse,
                           int B, int T_, int H, int D, cudaStream_t s) {
    dim3 grid(ceil_div(T_, WARPS), H, B);
    attn_fwd_simt<T><<<grid, WARPS * 32, 0, s>>>(q, k, v, ld, o, ldo, lse, T_, H, D);
    note_launch();
    NC_LAUNCH_CHECK("attention_forward_simt");
    return NC_OK;
}

template <typename T>
int attention_backward_simt(const T* q, const T* k, const T* v, long ld, const T* o, const T* dout,
                            long ldo, const float* lse, T* dq, T* dk, T* dv, long ldd, float* delta,
                            int B, int T_, int H, int D, cudaStream_t s) {
    dim3 grid(ceil_div(T_, WARPS), H, B);
    attn_delta_simt<T><<<grid, WARPS * 32, 0, s>>>(o, dout, ldo, delta, T_, H, D);
    attn_dq_simt<T><<<grid, WARPS * 32, 0, s>>>(q, k, v, ld, dout, ldo, lse, delta, dq, ldd, T_, H, D);
    attn_dkdv_simt<T><<<grid, WARPS * 32, 0, s>>>(q, k, v, ld, dout, ldo, lse, delta, dk, dv, ldd, T_,
                                                  H, D);
    note_launch(3);
    NC_LAUNCH_CHECK("attention_backward_simt");
    return NC_OK;
}

int attention_delta_simt_bf16(const bf16* o, const bf16* dout, long ldo, float* delta, int B, int T_,
                              int H, int D, cudaStream_t s) {
    dim3 grid(ceil_div(T_, WARPS), H, B);
    attn_delta_simt<bf16><<<grid, WARPS * 32, 0, s>>>(o, dout, ldo, delta, T_, H, D);
    note_launch();
    NC_LAUNCH_CHECK("attention_delta");
    return NC_OK;
}

template int attention_forward_simt<float>(const float*, const float*, const float*, long, float*,
                                           long, float*, int, int, int, int, cudaStream_t);
template int attention_forward_simt<bf16>(const bf16*, const bf16*, const bf16*, long, bf16*, long,
                                          float*, int, int, int, int, cudaStream_t);
template int attention_backward_simt<float>(const float*, const float*, const float*, long,
                                            const float*, const float*, long, const float*, float*,
                                            float*, float*, long, float*, int, int, int, int,
                                            cudaStream_t);
template int attention_backward_simt<bf16>(const bf16*, const bf16*, const bf16*, long, const bf16*,
                                           const bf16*, long, const float*, bf16*, bf16*, bf16*, long,
                                           float*, int, int, int, int, cudaStream_t);

}  // namespace nc
