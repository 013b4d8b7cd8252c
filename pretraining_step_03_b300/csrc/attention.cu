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

template <typename T>
int attention_forward(const T* q, const T* k, const T* v, long ld, T* o, long ldo, float* lse,
                      int B, int T_, int H, int D, cudaStream_t s) {
    if (B <= 0 || T_ <= 0) return NC_OK;
    return attention_forward_simt<T>(q, k, v, ld, o, ldo, lse, B, T_, H, D, s);
}

template <typename T>
int attention_backward(const T* q, const T* k, const T* v, long ld, const T* o, const T* dout,
                       long ldo, const float* lse, T* dq, T* dk, T* dv, long ldd, float* delta,
                       int B, int T_, int H, int D, cudaStream_t s) {
    if (B <= 0 || T_ <= 0) return NC_OK;
    return attention_backward_simt<T>(q, k, v, ld, o, dout, ldo, lse, dq, dk, dv, ldd, delta, B, T_,
                                      H, D, s);
}

template int attention_forward<float>(const float*, const float*, const float*, long, float*, long,
                                      float*, int, int, int, int, cudaStream_t);
template int attention_forward<bf16>(const bf16*, const bf16*, const bf16*, long, bf16*, long,
                                     float*, int, int, int, int, cudaStream_t);
template int attention_backward<float>(const float*, const float*, const float*, long, const float*,
                                       const float*, long, const float*, float*, float*, float*,
                                       long, float*, int, int, int, int, cudaStream_t);
template int attention_backward<bf16>(const bf16*, const bf16*, const bf16*, long, const bf16*,
                                      const bf16*, long, const float*, bf16*, bf16*, bf16*, long,
                                      float*, int, int, int, int, cudaStream_t);

}  // namespace nc
