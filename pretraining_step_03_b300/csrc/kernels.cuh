// Internal launch interface of libnc's kernels (raw pointers + a stream).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "optim.cuh"

namespace nc {

// ------------------------------------------------------------ GEMM
// C = alpha * op(A) op(B)^T (+ epilogue), op(A) [M, K], op(B) [N, K].
enum EpiKind {
    EPI_STORE = 0,      // C = alpha*acc + beta*aux            (aux may alias C)
    EPI_RELU2 = 1,      // C = relu(alpha*acc)^2 (the activation a; h itself is not kept)
    EPI_RELU2_BWD = 2,  // C = alpha*acc * 2*sqrt(aux)          (aux = a = relu(h)^2, so 2 sqrt(a) = 2 relu(h))
    EPI_ROPE = 3,       // C = alpha*acc with columns < rope_cols rotated by RoPE (head dim 128)
    EPI_DELTA = 4,      // C = alpha*acc (bf16) and delta[b, h, t] = sum over head h of bf16(C) * aux
    EPI_LSE = 5,        // C = alpha*acc (bf16) and, per row and 128-column group k, lse_part[row][k] =
                        //   (max z, sum exp(z - max)) over the stored (rounded) values z
    EPI_NORMB = 6,      // the RMSNorm backward finished in the dX product: with dy = alpha*acc,
                        //   y = aux (bf16), r = nb_r[row], D = sum of nb_part[row][0 .. nb_nparts):
                        //   C (fp32) = nb_gin + r (dy - y D nb_inv_d), nb_gt = bf16(C)
};

struct Gemm {
    int M = 0, N = 0, K = 0, batch = 1;
    const void* A = nullptr; long lda = 0, sA = 0; bool a_t = false;  // a_t: A stored [K, M]
    const void* B = nullptr; long ldb = 0, sB = 0; bool b_t = false;  // b_t: B stored [K, N]
    int in_dtype = NC_BF16;
    void* C = nullptr; long ldc = 0, sC = 0; int c_dtype = NC_BF16;
    const void* aux = nullptr; long ldaux = 0, sAux = 0; int aux_dtype = NC_BF16;
    float alpha = 1.f, beta = 0.f;
    int epi = EPI_STORE;
    const float2* rope = nullptr;  // EPI_ROPE: (cos, sin) of pair j at position t is rope[j * rope_ld + t];
    int rope_T = 0, rope_cols = 0; //   row position = row % rope_T
    int rope_ld = 0;
    float* delta = nullptr;        // EPI_DELTA: [B, N/128, rope_T] row statistics (row = b*rope_T + t)
    // C is symmetric (M == N, e.g. X X^T): the CTA-pair path computes only the 256 x 256
    // tiles on and above the diagonal and writes each off-diagonal tile a second time,
    // transposed.  Ignored (full computation) where the pair path does not apply.
    bool sym = false;
    float2* lse_part = nullptr;    // EPI_LSE: [M][N/128]
    uint32_t* flag = nullptr;      // device flag word for aborted waits (may be null)
    // EPI_RELU2_BWD (optional): per row and 128-column group k, dot_out[row][k] = sum of
    // bf16(C) * sqrt(aux), i.e. <dh, relu(h)> (the row dot of the next RMSNorm's backward)
    float* dot_out = nullptr;
    // EPI_NORMB (see above); nb_gin may alias C (the residual gradient updated in place)
    const float* nb_r = nullptr;
    const float* nb_part = nullptr;
    int nb_nparts = 0;
    float nb_inv_d = 0.f;
    const float* nb_gin = nullptr;
    bf16* nb_gt = nullptr;
};
// Fraction of the 2*M*N*K products gemm_tc executes for g (below 1 for symmetric C).
double gemm_tc_work_fraction(const Gemm& g);

int gemm_simt(const Gemm& g, cudaStream_t s);
// 3-D bf16 TMA map over [batch][outer][inner], 128-byte swizzle, zero OOB fill.
int make_map(CUtensorMap* m, const void* ptr, long inner, long outer, long batch, long ld, long bs,
             int box_inner, int box_outer);
int num_sms();
// tcgen05/TMA path (bf16 operands).  ws: fp32 split-K scratch (may be null).
int gemm_tc(const Gemm& g, void* ws, size_t ws_bytes, cudaStream_t s);
size_t gemm_tc_splitk_bytes(const Gemm& g);
bool gemm_tc_supported(const Gemm& g);

// ------------------------------------------------------------ row ops
template <typename T>
int embed_forward(const int32_t* tok, const T* wte, float* x, int M, int d, int V,
                  uint32_t* flag, cudaStream_t s);
template <typename T>
int rmsnorm_forward(const float* x, T* y, float* r, int M, int d, cudaStream_t s);
// g_out = g_in + r*(dy - y*mean(dy*y)); g_out may alias g_in; gT optional copy
template <typename T>
int rmsnorm_backward(const T* dy, const T* y, const float* r, const float* g_in,
                     float* g_out, T* gT, int M, int d, cudaStream_t s);
// in place on the q and k thirds of qkv rows (row stride ld): sign +1 fwd, -1 bwd
template <typename T>
int rope_apply(T* qkv, long ld, int M, int T_, int H, int Dh, const float2* table, int table_ld, float sign,
               cudaStream_t s);
// logits [M, V] -> dlogits in place; nll [M].  lse_part (bf16 only, optional): the
// per-row (max, sum exp) partials of every 128-column group, left by the LM-head GEMM
// (EPI_LSE); with them the logits are read once instead of twice.  grad = false: nll
// only, the logits are left untouched.  zdot (optional, with grad): per row <dz, z> =
// scale * sum of (softmax - onehot) * logits (dz before its bf16 rounding), the row dot
// <dy, y> of the final RMSNorm's backward by the adjoint identity
// <dz W, y> = <dz, y W^T> = <dz, z>.
template <typename T>
int cross_entropy(T* logits, const int32_t* tgt, float* nll, int M, int V, float scale,
                  uint32_t* flag, cudaStream_t s, const float2* lse_part = nullptr, bool grad = true,
                  float* zdot = nullptr);
// out (optional): {mean nll, bpb of this batch}; sums (optional): device double[3]
// {sum nll, sum nll over targets with bytes > 0, sum bytes}, set (accumulate = 0) or
// added to (accumulate = 1).  One CTA, fixed summation order.
int loss_reduce(const float* nll, const int32_t* tgt, const int32_t* token_bytes, int M, int V,
                float* out, uint32_t* flag, cudaStream_t s, double* sums = nullptr, int accumulate = 0);
// ------------------------------------------------------------ inference (decode.cu)
// Decode works on B sequences in a transposed layout with Bp = B rounded up to 8 columns:
// residual x^T [d][Bp] fp32, projections [N][Bp] = W [N, K] x Y[Bp, K]^T.
template <typename T>
int decode_embed_t(const int32_t* tok, const T* wte, float* xt, int B, int Bp, int d, int V, uint32_t* flag,
                   cudaStream_t s);
template <typename T>
int decode_rmsnorm_cols(const float* xt, T* y, int Bp, int d, cudaStream_t s);
// [q|k|v]^T [3d][Bp] at position pos -> q [Bp][d] (RoPE), cache rows (b, pos) of k (RoPE) and v.
// pos_dev (optional): the position is read from device memory instead (a replayed graph).
template <typename T>
int decode_qkv_post(const T* c, int B, int Bp, int d, int H, int Dh, int pos, const int* pos_dev,
                    const float2* rope, int rope_ld, T* q, T* kc, T* vc, int cache_T, cudaStream_t s);
// out [Bp][d] = softmax(q k^T / sqrt(Dh)) v over cache rows 0 .. n-1 of each of the B sequences
// (rows B .. Bp-1 of out are zeroed); head dim 128.  Key chunks are sized from cache_T, so the
// sums do not depend on n's grid.  pos_dev (optional): n = *pos_dev + 1 at run time, the grid
// covering the whole cache.
size_t decode_attention_ws_bytes(int B, int H, int n);
template <typename T>
int decode_attention(const T* q, const T* kc, const T* vc, int B, int Bp, int d, int H, int Dh, int cache_T,
                     int n, const int* pos_dev, T* out, void* ws, size_t ws_bytes, cudaStream_t s);
int decode_set_pos(int* pos_dev, int pos, cudaStream_t s);
// next[b] = argmax_v logits^T[v][b] (lowest id on ties); ws >= B * 512 bytes
int decode_argmax(const float* lt, int V, int B, int Bp, int32_t* next, void* ws, size_t ws_bytes, uint32_t* flag,
                  cudaStream_t s);
int decode_logits_out(const float* lt, int V, int B, int Bp, float* out, cudaStream_t s);
template <typename T>
int prefill_kv_store(const T* qkv, int B, int T0, int d, T* kc, T* vc, int cache_T, cudaStream_t s);
template <typename T>
int prefill_gather_last(const T* y, int B, int Bp, int T0, int d, T* out, cudaStream_t s);

struct EmbedBwdWs {
    int* hist;       // [nchunks * V]
    int* rank;       // [M]
    int* offsets;    // [V + 1]
    int* sorted;     // [M]
    float* head;     // [npieces * d]
    float* tail;     // [npieces * d]
    int* bsum;       // [ceil(V / 256)] token counts per 256 ids
};
size_t embed_backward_ws_bytes(int M, int d, int V);
EmbedBwdWs embed_backward_ws(void* base, int M, int d, int V);
int embed_backward(const int32_t* tok, const float* g, float* dwte, int M, int d, int V,
                   int accumulate, const EmbedBwdWs& ws, cudaStream_t s);

// ------------------------------------------------------------ attention
// flag: device flag word that an aborted wait or misaligned shared memory sets (may be null).
template <typename T>
int attention_forward(const T* q, const T* k, const T* v, long ld, T* o, long ldo, float* lse,
                      int B, int T_, int H, int D, cudaStream_t s, uint32_t* flag);
// rope: optional RoPE table ((cos, sin) of pair j at position t at rope[j * rope_ld + t]);
// when the kernel can rotate dq, dk back itself it does so and sets *rope_done = 1
// (else the caller applies the inverse RoPE).
// delta_ready: delta already holds dO.O per row (computed by the producer of dO)
// ds: optional scratch of attention_ds_bytes(B, T_, H) bytes; with it the bf16
// head-dim-128 path keeps dS from the dK/dV pass and forms dq as a plain product
// instead of recomputing the scores.
template <typename T>
int attention_backward(const T* q, const T* k, const T* v, long ld, const T* o, const T* dout,
                       long ldo, const float* lse, T* dq, T* dk, T* dv, long ldd, float* delta,
                       int B, int T_, int H, int D, cudaStream_t s, uint32_t* flag,
                       const float2* rope = nullptr,
                       int rope_ld = 0, int* rope_done = nullptr, bool delta_ready = false,
                       void* ds = nullptr);
// bytes of the dS scratch above (0 where it would not be used)
size_t attention_ds_bytes(int B, int T_, int H, int D);

// ------------------------------------------------------------ optimizers
// Muon, phase 1: buf = mu*buf + g; g <- g + mu*buf (nesterov) or buf; per-CTA
// sums of squares of the new g into partial[mat * chunks + chunk].
int muon_momentum(float* g, float* buf, const MuonMat* mats, int nmat, float mu, int nesterov,
                  float* partial, int chunks, cudaStream_t s);
// Muon, phase 2: X = g / (|g|_F + 1e-7), written (transposed when tr) into x.
template <typename T>
int muon_normalize(const float* g, const MuonMat* mats, int nmat, const float* partial, int chunks,
                   T* x, int blocks_per_mat, cudaStream_t s);
// Muon, phase 4: W -= lr*scale*X (X read transposed when tr); refresh the bf16 copy.
template <typename T>
int muon_apply(float* w, bf16* w16, const MuonMat* mats, int nmat, const T* x, float lr,
               int blocks_per_mat, cudaStream_t s);
int adamw(float* w, bf16* w16, const float* g, float* m, float* v, long n, float lr, float b1,
          float b2, float eps, float wd, float bc1, float bc2, cudaStream_t s);
int cast_f32_bf16(const float* x, bf16* y, long n, cudaStream_t s);

}  // namespace nc
