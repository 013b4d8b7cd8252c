// Attention dispatch: tensor-core kernels for bf16 head dim 128, CUDA-core
// kernels otherwise (fp32 mode, other head dims).
#include "kernels.cuh"

namespace nc {

template <typename T>
int attention_forward_simt(const T* q, const T* k, const T* v, long ld, T* o, long ldo, float* lse,
                           int B, int T_, int H, int D, cudaStream_t s);
template <typename T>
int attention_backward_simt(const T* q, const T* k, const T* v, long ld, const T* o, const T* dout,
                            long ldo, const float* lse, T* dq, T* dk, T* dv, long ldd, float* delta,
                            int B, int T_, int H, int D, cudaStream_t s);

int attention_delta_simt_bf16(const bf16* o, const bf16* dout, long ldo, float* delta, int B, int T_,
                              int H, int D, cudaStream_t s);
bool attention_tc_supported(long ld, long ldo, long ldd, const void* q, const void* k, const void* v,
                            int D);
int attention_forward_tc(const bf16* q, const bf16* k, const bf16* v, long ld, bf16* o, long ldo,
                         float* lse, int B, int T, int H, cudaStream_t s, uint32_t* flag);
int attention_backward_tc(const bf16* q, const bf16* k, const bf16* v, long ld, const bf16* dout,
                          long ldo, const float* lse, const float* delta, bf16* dq, bf16* dk, bf16* dv,
                          long ldd, int B, int T, int H, const float2* rope, int rope_ld, bf16* ds,
                          cudaStream_t s, uint32_t* flag);
size_t attention_tc_ds_bytes(int B, int T, int H);

template <typename T>
int attention_forward(const T* q, const T* k, const T* v, long ld, T* o, long ldo, float* lse,
                      int B, int T_, int H, int D, cudaStream_t s, uint32_t* flag) {
    if (B <= 0 || T_ <= 0) return NC_OK;
    if constexpr (sizeof(T) == 2) {
        if (attention_tc_supported(ld, ldo, ldo, q, k, v, D))
            return attention_forward_tc(q, k, v, ld, o, ldo, lse, B, T_, H, s, flag);
    }
    return attention_forward_simt<T>(q, k, v, ld, o, ldo, lse, B, T_, H, D, s);
}

template <typename T>
int attention_backward(const T* q, const T* k, const T* v, long ld, const T* o, const T* dout,
                       long ldo, const float* lse, T* dq, T* dk, T* dv, long ldd, float* delta,
                       int B, int T_, int H, int D, cudaStream_t s, uint32_t* flag, const float2* rope,
                       int rope_ld, int* rope_done, bool delta_ready, void* ds) {
    if (rope_done) *rope_done = 0;
    if (B <= 0 || T_ <= 0) return NC_OK;
    if constexpr (sizeof(T) == 2) {
        if (attention_tc_supported(ld, ldo, ldd, q, k, v, D)) {
            if (!delta_ready) NC_TRY(attention_delta_simt_bf16(o, dout, ldo, delta, B, T_, H, D, s));
            if (rope_done) *rope_done = rope != nullptr;
            return attention_backward_tc(q, k, v, ld, dout, ldo, lse, delta, dq, dk, dv, ldd, B, T_, H,
                                         rope, rope_ld, (bf16*)ds, s, flag);
        }
    }
    return attention_backward_simt<T>(q, k, v, ld, o, dout, ldo, lse, dq, dk, dv, ldd, delta, B, T_,
                                      H, D, s);
}

template int attention_forward<float>(const float*, const float*, const float*, long, float*, long,
                                      float*, int, int, int, int, cudaStream_t, uint32_t*);
template int attention_forward<bf16>(const bf16*, const bf16*, const bf16*, long, bf16*, long,
                                     float*, int, int, int, int, cudaStream_t, uint32_t*);
template int attention_backward<float>(const float*, const float*, const float*, long, const float*,
                                       const float*, long, const float*, float*, float*, float*,
                                       long, float*, int, int, int, int, cudaStream_t, uint32_t*,
                                       const float2*, int, int*, bool, void*);
template int attention_backward<bf16>(const bf16*, const bf16*, const bf16*, long, const bf16*,
                                      const bf16*, long, const float*, bf16*, bf16*, bf16*, long,
                                      float*, int, int, int, int, cudaStream_t, uint32_t*,
                                      const float2*, int, int*, bool, void*);

size_t attention_ds_bytes(int B, int T_, int H, int D) {
    if (D != 128 || B <= 0 || T_ <= 0) return 0;
    return attention_tc_ds_bytes(B, T_, H);
}

}  // namespace nc
