// The step engine and the C ABI of libnc.so.
//
// One model = one caller-owned device arena laid out here (parameters,
// optimizer state, activation stash, scratch) and one CUDA stream.  The
// schedule follows the nanochat speedrun walkthrough (lyylswood.com):
//   section 预搜检 (pretraining): token embedding; per layer a pre-norm
//   attention block and a pre-norm 4x MLP block, both residual; a final norm
//   and an untied LM head; next-token cross-entropy reported as bits per
//   byte; backward; Muon on the block matrices, AdamW on the embedding and
//   unembedding; no biases and no norm gains;
//   section 该你了 (depth scaling): gradient accumulation over micro-batches.
// Readings where the pages are silent (RoPE, ReLU^2, eps, Muon/AdamW details)
// are the same as the fp64 oracle's and are stated next to each kernel.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "kernels.cuh"

using namespace nc;

struct nc_model {
    int depth, d, H, Dh, V, F, dtype, maxB, maxT;
    long maxM;
    cudaStream_t stream;
    char* arena;
    size_t arena_bytes;
    // parameters
    int nparams;
    std::vector<long> poff, prows, pcols;
    std::vector<int> pkind;
    long P;
    float* master;
    bf16* shadow;      // bf16 compute copy (bf16 mode)
    float* grads;
    float* momentum;   // Muon buffers (same offsets as master)
    float* adam_m;     // [2, V*d]: wte then lm_head
    float* adam_v;
    // Muon
    MuonMat* mats;
    int nmat;
    float* muon_partial;
    int muon_chunks;
    void* nsX;         // [square group | wide group], act type
    void* nsX2;
    void* nsA;         // [6L, d, d]
    void* nsB;
    // misc
    float2* rope;      // [Dh/2, maxT]: (cos, sin) of pair j at position t at j * maxT + t
    float* loss;       // [2 * 64] micro-step {loss, bpb}
    uint32_t* flag;
    int32_t* tok_stage;  // [2, maxM] tokens, targets (nc_train_step)
    // activations (act type unless noted)
    struct Layer {
        void *y1, *qkv, *o, *y2, *a;
        float *r1, *r2, *lse;
    };
    std::vector<Layer> L;
    float* x;          // residual stream fp32 [M, d]
    void* yf;
    float* rf;
    void* logits;      // [M, V]
    float2* lse_part;  // [M, V/128] (max, sum exp) partials from the LM-head GEMM (bf16 mode)
    float* nll;
    float* g;          // residual gradient fp32 [M, d]
    void* gT;          // its act-type copy (bf16 mode)
    void* dy;          // gradient at a norm output [M, d] (act type)
    float* nb_dot;     // bf16 mode: <dlogits, logits> per row [M] (the final norm's row dot)
    float* nb_part;    // bf16 mode: <dh, relu(h)> per row and 128 columns [M, 4d/128]
    void* dqkv;
    void* dO;
    void* dh;
    float* delta;      // attention row statistics [M * H]
    void* ds;          // attention dS store for (maxB, maxT) (bf16, head dim 128)
    size_t ds_bytes;
    void* ebws;
    size_t ebws_bytes;
    void* splitk;
    size_t splitk_bytes;
    // decode steps replayed as CUDA graphs, one per (cache, batch, token/output buffers)
    struct DecGraph {
        const void* cache; int cache_B, cache_T, B; const void* tok; const void* logits; const void* next;
        int uses; cudaGraphExec_t exec; int kernels;
    };
    std::vector<DecGraph> dec_graphs;
    bool dec_graph_on = true;
    int* pos_dev = nullptr;
    cudaStream_t cap_stream = nullptr;   // recording needs a stream of its own (not the legacy one)
    // measurement: CUDA event pairs around kernel classes
    struct ProfRec { cudaEvent_t a, b; int cat; double flops, bytes; };
    bool prof_on = false;
    std::vector<cudaEvent_t> ev_pool;
    size_t ev_used = 0;
    std::vector<ProfRec> recs;
};

namespace {

size_t al(size_t b) { return (b + 255) & ~(size_t)255; }

struct Carver {
    size_t off = 0;
    char* base = nullptr;
    void* take(size_t bytes) {
        void* p = base ? base + off : nullptr;
        off += al(bytes);
        return p;
    }
};

int check_dims(int depth, int d, int H, int V, int maxB, int maxT, int dtype) {
    if (depth < 1 || depth > 1024) return set_error(NC_ERR_ARG, "depth %d out of range", depth);
    if (d < 32 || d % 32) return set_error(NC_ERR_ARG, "d_model %d must be a positive multiple of 32", d);
    if (H < 1 || d % H) return set_error(NC_ERR_ARG, "d_model %d not divisible by n_head %d", d, H);
    int Dh = d / H;
    if (Dh % 2 || Dh > 128) return set_error(NC_ERR_ARG, "head_dim %d must be even and <= 128", Dh);
    if (V < 8 || V % 8) return set_error(NC_ERR_ARG, "vocab %d must be a positive multiple of 8", V);
    if (maxB < 0 || maxT < 0 || (long)maxB * maxT > (1L << 24))
        return set_error(NC_ERR_ARG, "max_B*max_T out of range");
    if (dtype != NC_BF16 && dtype != NC_FP32) return set_error(NC_ERR_ARG, "dtype %d", dtype);
    return NC_OK;
}

// Lays the arena out; with base == nullptr only measures.
void layout(nc_model* m, char* base, size_t* total) {
    Carver c;
    c.base = base;
    const int d = m->d, V = m->V, Ld = m->depth;
    const size_t act = m->dtype == NC_BF16 ? 2 : 4;
    const long P = m->P;
    m->master = (float*)c.take(P * 4);
    m->shadow = m->dtype == NC_BF16 ? (bf16*)c.take(P * 2) : nullptr;
    m->grads = (float*)c.take(P * 4);
    m->momentum = (float*)c.take(P * 4);
    m->adam_m = (float*)c.take((size_t)2 * V * d * 4);
    m->adam_v = (float*)c.take((size_t)2 * V * d * 4);
    m->nmat = 6 * Ld;
    m->muon_chunks = 32;
    m->mats = (MuonMat*)c.take(sizeof(MuonMat) * m->nmat);
    m->muon_partial = (float*)c.take((size_t)m->nmat * m->muon_chunks * 4);
    const size_t nsx = ((size_t)4 * Ld * d * d + (size_t)2 * Ld * d * 4 * d) * act;
    m->nsX = c.take(nsx);
    m->nsX2 = c.take(nsx);
    m->nsA = c.take((size_t)6 * Ld * d * d * act);
    m->nsB = c.take((size_t)6 * Ld * d * d * act);
    m->rope = (float2*)c.take((size_t)(m->maxT > 0 ? m->maxT : 1) * (m->Dh / 2) * 8);
    m->loss = (float*)c.take(128 * 4);
    m->flag = (uint32_t*)c.take(16);
    m->pos_dev = (int*)c.take(16);
    const long M = m->maxM;
    m->L.assign(Ld, nc_model::Layer{});
    m->tok_stage = nullptr;
    if (M > 0) {
        m->tok_stage = (int32_t*)c.take((size_t)2 * M * 4);
        for (int l = 0; l < Ld; ++l) {
            auto& y = m->L[l];
            y.y1 = c.take(M * d * act);
            y.r1 = (float*)c.take(M * 4);
            y.qkv = c.take(M * 3 * d * act);
            y.o = c.take(M * d * act);
            y.lse = (float*)c.take(M * m->H * 4);
            y.y2 = c.take(M * d * act);
            y.r2 = (float*)c.take(M * 4);
            y.a = c.take(M * 4 * d * act);
        }
        m->x = (float*)c.take(M * d * 4);
        m->yf = c.take(M * d * act);
        m->rf = (float*)c.take(M * 4);
        m->logits = c.take(M * V * act);
        m->lse_part = m->dtype == NC_BF16 && V % 128 == 0 ? (float2*)c.take((size_t)M * (V / 128) * 8) : nullptr;
        m->nll = (float*)c.take(M * 4);
        m->g = (float*)c.take(M * d * 4);
        m->gT = m->dtype == NC_BF16 ? c.take(M * d * act) : nullptr;
        m->dy = c.take(M * d * act);
        m->nb_dot = m->dtype == NC_BF16 ? (float*)c.take(M * 4) : nullptr;
        m->nb_part = m->dtype == NC_BF16 ? (float*)c.take(M * ceil_div(4 * d, 128) * 4) : nullptr;
        m->dqkv = c.take(M * 3 * d * act);
        m->dO = c.take(M * d * act);
        m->dh = c.take(M * 4 * d * act);
        m->delta = (float*)c.take(M * m->H * 4);
        m->ds_bytes = m->dtype == NC_BF16 ? attention_ds_bytes(m->maxB, m->maxT, m->H, m->Dh) : 0;
        m->ds = m->ds_bytes ? c.take(m->ds_bytes) : nullptr;
        m->ebws_bytes = embed_backward_ws_bytes((int)M, d, V);
        m->ebws = c.take(m->ebws_bytes);
    }
    // split-K scratch: the largest need among the step's GEMMs
    size_t sk = 0;
    if (m->dtype == NC_BF16) {
        const long mm = M > 0 ? M : 1;
        const int shapes[][3] = {{3 * d, d, (int)mm}, {d, d, (int)mm}, {4 * d, d, (int)mm},
                                 {d, 4 * d, (int)mm}, {V, d, (int)mm}};
        for (auto& s : shapes) {
            Gemm g;
            g.M = s[0]; g.N = s[1]; g.K = s[2];
            size_t b = gemm_tc_splitk_bytes(g);
            if (b > sk) sk = b;
        }
    }
    m->splitk_bytes = sk;
    m->splitk = sk ? c.take(sk) : nullptr;
    *total = c.off;
}

cudaEvent_t prof_event(nc_model* m) {
    if (m->ev_used == m->ev_pool.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        m->ev_pool.push_back(e);
    }
    return m->ev_pool[m->ev_used++];
}

// Records a CUDA event pair around the launches made during its lifetime.
struct Prof {
    nc_model* m;
    int cat;
    double flops, bytes;
    cudaEvent_t a = nullptr;
    Prof(nc_model* m_, int cat_, double flops_, double bytes_) : m(m_), cat(cat_), flops(flops_), bytes(bytes_) {
        if (m->prof_on && (a = prof_event(m))) cudaEventRecord(a, m->stream);
    }
    ~Prof() {
        if (!a) return;
        cudaEvent_t b = prof_event(m);
        if (!b) return;
        cudaEventRecord(b, m->stream);
        m->recs.push_back({a, b, cat, flops, bytes});
    }
};

template <typename T> T* W(nc_model* m, int i) {
    if (m->dtype == NC_BF16) return (T*)(m->shadow + m->poff[i]);
    return (T*)(m->master + m->poff[i]);
}

int run_gemm(nc_model* m, const Gemm& g, int cat = NC_PROF_GEMM) {
    // FLOPs actually executed (a symmetric product computes only its upper tiles)
    const double frac = m->dtype == NC_BF16 ? gemm_tc_work_fraction(g) : 1.0;
    Prof pr(m, cat, 2.0 * g.M * g.N * g.K * g.batch * frac, 0.0);
    if (g.in_dtype == NC_BF16) return gemm_tc(g, m->splitk, m->splitk_bytes, m->stream);
    return gemm_simt(g, m->stream);
}

// C[M,N] = A[M,K] (row-major, lda) * B[N,K]^T, or with a_t/b_t as stored [K, .]
Gemm mk(nc_model* m, int M, int N, int K, const void* A, long lda, bool a_t, const void* B, long ldb,
        bool b_t, void* C, long ldc, int c_dtype) {
    Gemm g;
    g.M = M; g.N = N; g.K = K;
    g.A = A; g.lda = lda; g.a_t = a_t;
    g.B = B; g.ldb = ldb; g.b_t = b_t;
    g.in_dtype = m->dtype;
    g.C = C; g.ldc = ldc; g.c_dtype = c_dtype;
    g.flag = m->flag;
    return g;
}

// weight gradient dW[N_out, K_out] (+)= dY^T X over M rows
int weight_grad(nc_model* m, float* dW, int rows, int cols, const void* dY, long ldy, const void* X,
                long ldx, int M, int accumulate) {
    Gemm g = mk(m, rows, cols, M, dY, ldy, true, X, ldx, true, dW, cols, NC_FP32);
    g.aux = dW; g.ldaux = cols; g.aux_dtype = NC_FP32; g.beta = accumulate ? 1.f : 0.f;
    return run_gemm(m, g);
}

template <typename T>
// backward = false: the forward and the loss only (the evaluation pass); the logits are
// not turned into their gradient and no gradient is touched.  sums (optional): running
// loss totals, see loss_reduce.
int forward_backward(nc_model* m, const int32_t* tok, const int32_t* tgt, const int32_t* tb, int B,
                     int T_, int accumulate, float grad_scale, float* out, bool backward = true,
                     double* sums = nullptr, int sum_acc = 0) {
    const int d = m->d, H = m->H, Dh = m->Dh, V = m->V, F = m->F;
    const int M = B * T_;
    const int act = m->dtype;
    const double ab = m->dtype == NC_BF16 ? 2.0 : 4.0;   // bytes per activation element
    const double Md = (double)M * d;
    const double attn_fl = 4.0 * B * H * Dh * (0.5 * T_ * (T_ + 1.0));  // causal q.k and p.v
    cudaStream_t s = m->stream;
    const int iw = 0, iu = 1 + 6 * m->depth;
    T* gop = m->dtype == NC_BF16 ? (T*)m->gT : (T*)m->g;  // residual gradient as GEMM operand
    T* gT = m->dtype == NC_BF16 ? (T*)m->gT : nullptr;
    const bool fuse_rope = m->dtype == NC_BF16 && Dh == 128;
    const int rope_ld = m->maxT > 0 ? m->maxT : 1;   // stride of the pair-major RoPE table
    auto norm_f = [&](const float* x, void* y, float* r) {
        Prof pr(m, NC_PROF_NORM, 0, Md * (4 + ab) + M * 4.0);
        return rmsnorm_forward<T>(x, (T*)y, r, M, d, s);
    };
    auto norm_b = [&](void* y, float* r, const float* gin) {
        Prof pr(m, NC_PROF_NORM, 0, Md * (ab + ab + (gin ? 4 : 0) + 4 + (gT ? ab : 0)) + M * 4.0);
        return rmsnorm_backward<T>((const T*)m->dy, (T*)y, r, gin, m->g, gT, M, d, s);
    };
    // dy = (the product g0) and then the norm's backward; in bf16 mode, given each row's
    // <dy, y> as partials (part, nparts per row), the product's epilogue finishes the norm
    // and dy is never stored
    auto dx_norm_b = [&](Gemm g0, void* y, float* r, const float* gin, const float* part, int nparts) {
        if (part && gT) {
            Gemm g = g0;
            g.epi = EPI_NORMB; g.C = m->g; g.ldc = d; g.c_dtype = NC_FP32;
            g.aux = y; g.ldaux = d; g.aux_dtype = act;
            g.nb_r = r; g.nb_part = part; g.nb_nparts = nparts; g.nb_inv_d = 1.f / (float)d;
            g.nb_gin = gin; g.nb_gt = (bf16*)gT;
            if (gemm_tc_supported(g)) return run_gemm(m, g);
        }
        NC_TRY(run_gemm(m, g0));
        return norm_b(y, r, gin);
    };
    auto rope = [&](void* qkv, float sign) {
        Prof pr(m, NC_PROF_ROPE, 0, 4.0 * Md * ab);
        return rope_apply<T>((T*)qkv, 3 * d, M, T_, H, Dh, m->rope, rope_ld, sign, s);
    };

    // ------------------------------------------------ forward
    {
        Prof pr(m, NC_PROF_EMBED, 0, Md * (ab + 4) + M * 4.0);
        NC_TRY(embed_forward<T>(tok, W<T>(m, iw), m->x, M, d, V, m->flag, s));
    }
    for (int l = 0; l < m->depth; ++l) {
        auto& Ly = m->L[l];
        const int b0 = 1 + 6 * l;
        NC_TRY(norm_f(m->x, Ly.y1, Ly.r1));
        {   // q|k|v = y1 Wqkv^T, RoPE on q and k (in the GEMM epilogue when it can)
            Gemm g = mk(m, M, 3 * d, d, Ly.y1, d, false, W<T>(m, b0), d, false, Ly.qkv, 3 * d, act);
            if (fuse_rope) {
                g.epi = EPI_ROPE; g.rope = m->rope; g.rope_T = T_; g.rope_cols = 2 * d;
                g.rope_ld = rope_ld;
            }
            NC_TRY(run_gemm(m, g));
            if (!fuse_rope) NC_TRY(rope(Ly.qkv, 1.f));
        }
        T* q = (T*)Ly.qkv;
        {
            Prof pr(m, NC_PROF_ATTN_FWD, attn_fl, 0);
            NC_TRY(attention_forward<T>(q, q + d, q + 2 * d, 3 * d, (T*)Ly.o, d, Ly.lse, B, T_, H, Dh, s, m->flag));
        }
        {   // x += o Wo^T
            Gemm g = mk(m, M, d, d, Ly.o, d, false, W<T>(m, b0 + 3), d, false, m->x, d, NC_FP32);
            g.aux = m->x; g.ldaux = d; g.aux_dtype = NC_FP32; g.beta = 1.f;
            NC_TRY(run_gemm(m, g));
        }
        NC_TRY(norm_f(m->x, Ly.y2, Ly.r2));
        {   // h = y2 W1^T, a = relu(h)^2
            Gemm g = mk(m, M, F, d, Ly.y2, d, false, W<T>(m, b0 + 4), d, false, Ly.a, F, act);
            g.epi = EPI_RELU2;
            NC_TRY(run_gemm(m, g));
        }
        {   // x += a W2^T
            Gemm g = mk(m, M, d, F, Ly.a, F, false, W<T>(m, b0 + 5), F, false, m->x, d, NC_FP32);
            g.aux = m->x; g.ldaux = d; g.aux_dtype = NC_FP32; g.beta = 1.f;
            NC_TRY(run_gemm(m, g));
        }
    }
    NC_TRY(norm_f(m->x, m->yf, m->rf));
    const float2* lse_part = nullptr;
    {   // logits; in bf16 mode the epilogue also leaves each row's softmax partials
        Gemm g = mk(m, M, V, d, m->yf, d, false, W<T>(m, iu), d, false, m->logits, V, act);
        if (m->lse_part) {
            g.epi = EPI_LSE;
            g.lse_part = m->lse_part;
            if (gemm_tc_supported(g)) lse_part = m->lse_part;
            else g.epi = EPI_STORE;
        }
        NC_TRY(run_gemm(m, g));
    }
    {
        const double ce_bytes = backward ? 2.0 * M * V * ab
                                         : (lse_part ? M * (V / 128) * 8.0 : (double)M * V * ab);
        Prof pr(m, NC_PROF_CE, 0, ce_bytes + M * 16.0);
        NC_TRY(cross_entropy<T>((T*)m->logits, tgt, m->nll, M, V, grad_scale / (float)M, m->flag, s,
                                lse_part, backward, m->nb_dot));
        NC_TRY(loss_reduce(m->nll, tgt, tb, M, V, out, m->flag, s, sums, sum_acc));
    }
    if (!backward) return NC_OK;

    // ------------------------------------------------ backward
    float* G = m->grads;
    NC_TRY(weight_grad(m, G + m->poff[iu], V, d, m->logits, V, m->yf, d, M, accumulate));
    NC_TRY(dx_norm_b(mk(m, M, d, V, m->logits, V, false, W<T>(m, iu), d, true, m->dy, d, act), m->yf, m->rf,
                     nullptr, m->nb_dot, 1));
    for (int l = m->depth - 1; l >= 0; --l) {
        auto& Ly = m->L[l];
        const int b0 = 1 + 6 * l;
        // MLP block
        NC_TRY(weight_grad(m, G + m->poff[b0 + 5], d, F, gop, d, Ly.a, F, M, accumulate));
        bool dots = false;
        {   // dh = (g W2) * 2 relu(h); in bf16 mode also <dh, relu(h)> per row and 128 columns
            Gemm g = mk(m, M, F, d, gop, d, false, W<T>(m, b0 + 5), F, true, m->dh, F, act);
            g.epi = EPI_RELU2_BWD; g.aux = Ly.a; g.ldaux = F; g.aux_dtype = act;
            if (m->nb_part) {
                g.dot_out = m->nb_part;
                dots = gemm_tc_supported(g);
                if (!dots) g.dot_out = nullptr;
            }
            NC_TRY(run_gemm(m, g));
        }
        NC_TRY(weight_grad(m, G + m->poff[b0 + 4], F, d, m->dh, F, Ly.y2, d, M, accumulate));
        NC_TRY(dx_norm_b(mk(m, M, d, F, m->dh, F, false, W<T>(m, b0 + 4), d, true, m->dy, d, act), Ly.y2, Ly.r2,
                         m->g, dots ? m->nb_part : nullptr, F / 128));
        // attention block
        NC_TRY(weight_grad(m, G + m->poff[b0 + 3], d, d, gop, d, Ly.o, d, M, accumulate));
        {   // dO = g Wo; with head dim 128 the epilogue also leaves D_t = dO_t . O_t per head
            Gemm g = mk(m, M, d, d, gop, d, false, W<T>(m, b0 + 3), d, true, m->dO, d, act);
            if (fuse_rope) {
                g.epi = EPI_DELTA; g.aux = Ly.o; g.ldaux = d; g.aux_dtype = act; g.delta = m->delta;
                g.rope_T = T_;
            }
            NC_TRY(run_gemm(m, g));
        }
        T* q = (T*)Ly.qkv;
        T* dq = (T*)m->dqkv;
        int unroped = 0;
        {
            Prof pr(m, NC_PROF_ATTN_BWD, 2.5 * attn_fl, 0);
            NC_TRY(attention_backward<T>(q, q + d, q + 2 * d, 3 * d, (T*)Ly.o, (T*)m->dO, d, Ly.lse, dq,
                                         dq + d, dq + 2 * d, 3 * d, m->delta, B, T_, H, Dh, s, m->flag, m->rope,
                                         rope_ld, &unroped, fuse_rope,
                                         attention_ds_bytes(B, T_, H, Dh) <= m->ds_bytes ? m->ds : nullptr));
        }
        if (!unroped) NC_TRY(rope(m->dqkv, -1.f));
        NC_TRY(weight_grad(m, G + m->poff[b0], 3 * d, d, m->dqkv, 3 * d, Ly.y1, d, M, accumulate));
        NC_TRY(run_gemm(m, mk(m, M, d, 3 * d, m->dqkv, 3 * d, false, W<T>(m, b0), d, true, m->dy, d, act)));
        NC_TRY(norm_b(Ly.y1, Ly.r1, m->g));
    }
    {
        Prof pr(m, NC_PROF_EMBED, 0, Md * 4.0 + (double)V * d * 4.0 + M * 24.0);
        NC_TRY(embed_backward(tok, m->g, G + m->poff[iw], M, d, V, accumulate,
                              embed_backward_ws(m->ebws, M, d, V), s));
    }
    return NC_OK;
}

template <typename T>
int muon(nc_model* m, float lr, float mu, int nesterov, int steps, const float* coef) {
    cudaStream_t s = m->stream;
    const int d = m->d, Ld = m->depth;
    const double nm = 12.0 * d * d * Ld;   // matrix parameters
    const double xb = m->dtype == NC_BF16 ? 2.0 : 4.0;
    {
        Prof pr(m, NC_PROF_MUON_ELEM, 0, nm * (16.0 + 4.0 + xb));
        NC_TRY(muon_momentum(m->grads, m->momentum, m->mats, m->nmat, mu, nesterov, m->muon_partial,
                             m->muon_chunks, s));
        NC_TRY(muon_normalize<T>(m->grads, m->mats, m->nmat, m->muon_partial, m->muon_chunks, (T*)m->nsX,
                                 32, s));
    }
    T* X = (T*)m->nsX;
    T* Y = (T*)m->nsX2;
    const long sq = (long)4 * Ld * d * d;  // elements of the square group
    const int act = m->dtype;
    for (int it = 0; it < steps; ++it) {
        for (int grp = 0; grp < 2; ++grp) {
            const int n = grp == 0 ? 4 * Ld : 2 * Ld, r = d, c = grp == 0 ? d : 4 * d;
            T* x = X + (grp == 0 ? 0 : sq);
            T* y = Y + (grp == 0 ? 0 : sq);
            T* A = (T*)m->nsA + (grp == 0 ? 0 : (long)4 * Ld * d * d);
            T* Bm = (T*)m->nsB + (grp == 0 ? 0 : (long)4 * Ld * d * d);
            {   // A = X X^T (symmetric: upper tiles computed, mirrored)
                Gemm g = mk(m, r, r, c, x, c, false, x, c, false, A, r, act);
                g.batch = n; g.sA = g.sB = (long)r * c; g.sC = (long)r * r; g.sym = true;
                NC_TRY(run_gemm(m, g, NC_PROF_MUON_NS));
            }
            {   // B = c2 A A + c1 A (symmetric, as A is)
                Gemm g = mk(m, r, r, r, A, r, false, A, r, true, Bm, r, act);
                g.batch = n; g.sA = g.sB = g.sC = (long)r * r; g.sym = true;
                g.alpha = coef[2]; g.aux = A; g.ldaux = r; g.sAux = (long)r * r; g.aux_dtype = act;
                g.beta = coef[1];
                NC_TRY(run_gemm(m, g, NC_PROF_MUON_NS));
            }
            {   // Y = B X + c0 X
                Gemm g = mk(m, r, c, r, Bm, r, false, x, c, true, y, c, act);
                g.batch = n; g.sA = (long)r * r; g.sB = (long)r * c; g.sC = (long)r * c;
                g.aux = x; g.ldaux = c; g.sAux = (long)r * c; g.aux_dtype = act; g.beta = coef[0];
                NC_TRY(run_gemm(m, g, NC_PROF_MUON_NS));
            }
        }
        T* t = X; X = Y; Y = t;
    }
    {
        Prof pr(m, NC_PROF_MUON_ELEM, 0, nm * (xb + 8.0 + (m->shadow ? 2.0 : 0.0)));
        NC_TRY(muon_apply<T>(m->master, m->shadow, m->mats, m->nmat, X, lr, 32, s));
    }
    return NC_OK;
}

int upload_f32(nc_model* m, float* dst, const float* host, size_t n) {
    NC_TRY(cuda_check(cudaMemcpyAsync(dst, host, n * 4, cudaMemcpyHostToDevice, m->stream), "H2D"));
    return cuda_check(cudaStreamSynchronize(m->stream), "sync");
}
int download_f32(nc_model* m, float* host, const float* src, size_t n) {
    NC_TRY(cuda_check(cudaMemcpyAsync(host, src, n * 4, cudaMemcpyDeviceToHost, m->stream), "D2H"));
    return cuda_check(cudaStreamSynchronize(m->stream), "sync");
}

// splitmix64 is counter-based: output i (0-based) of the stream seeded with s is
// mix(s + (i + 1) * golden), so any element of the weight stream can be drawn on its own.
__host__ __device__ __forceinline__ uint64_t splitmix_at(uint64_t seed, uint64_t i) {
    uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Weights N(0, std): value pair k of the model (parameters in index order, pairs
// numbered from pair0 for this tensor) is the Box-Muller transform of outputs 2k and
// 2k + 1 of the splitmix64 stream seeded with `seed`.
__global__ void init_normal_kernel(float* w, long n, uint64_t seed, long pair0, double std) {
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (2 * i >= n) return;
    const uint64_t k = (uint64_t)(pair0 + i);
    const double u1 = ((splitmix_at(seed, 2 * k) >> 11) + 1.0) * (1.0 / 9007199254740993.0);
    const double u2 = (splitmix_at(seed, 2 * k + 1) >> 11) * (1.0 / 9007199254740992.0);
    const double rr = sqrt(-2.0 * log(u1)) * std;
    double sn, cs;
    sincospi(2.0 * u2, &sn, &cs);
    w[2 * i] = (float)(rr * cs);
    if (2 * i + 1 < n) w[2 * i + 1] = (float)(rr * sn);
}

int check_param(nc_model* m, int index, size_t n) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    if (index < 0 || index >= m->nparams) return set_error(NC_ERR_ARG, "param index %d", index);
    if (n != (size_t)(m->prows[index] * m->pcols[index]))
        return set_error(NC_ERR_ARG, "param %d has %ld elements, got %zu", index,
                         m->prows[index] * m->pcols[index], n);
    return NC_OK;
}

void init_geometry(nc_model* m, int depth, int d, int H, int V, int dtype, int maxB, int maxT) {
    m->depth = depth; m->d = d; m->H = H; m->Dh = d / H; m->V = V; m->F = 4 * d;
    m->dtype = dtype; m->maxB = maxB; m->maxT = maxT; m->maxM = (long)maxB * maxT;
    m->nparams = 6 * depth + 2;
    m->poff.clear(); m->prows.clear(); m->pcols.clear(); m->pkind.clear();
    long off = 0;
    auto add = [&](long r, long c, int k) {
        m->poff.push_back(off); m->prows.push_back(r); m->pcols.push_back(c); m->pkind.push_back(k);
        off += (r * c + 63) / 64 * 64;
    };
    add(V, d, NC_KIND_EMB);
    for (int l = 0; l < depth; ++l) {
        for (int j = 0; j < 4; ++j) add(d, d, NC_KIND_MATRIX);
        add(4 * d, d, NC_KIND_MATRIX);
        add(d, 4 * d, NC_KIND_MATRIX);
    }
    add(V, d, NC_KIND_UNEMB);
    m->P = off;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

int nc_arena_bytes(int depth, int d_model, int n_head, int vocab, int max_B, int max_T, int dtype,
                   size_t* out_bytes) {
    NC_TRY(check_dims(depth, d_model, n_head, vocab, max_B, max_T, dtype));
    if (!out_bytes) return set_error(NC_ERR_ARG, "null out_bytes");
    nc_model m{};
    init_geometry(&m, depth, d_model, n_head, vocab, dtype, max_B, max_T);
    size_t total = 0;
    layout(&m, nullptr, &total);
    *out_bytes = total;
    return NC_OK;
}

int nc_init_model(int depth, int d_model, int n_head, int vocab, uint64_t seed, void* arena,
                  size_t arena_bytes, int dtype, int max_B, int max_T, void* stream, nc_model** out) {
    NC_TRY(check_dims(depth, d_model, n_head, vocab, max_B, max_T, dtype));
    if (!out) return set_error(NC_ERR_ARG, "null out");
    if (!arena || (uintptr_t)arena % 256) return set_error(NC_ERR_ARG, "arena must be 256-byte aligned device memory");
    nc_model* m = new nc_model();
    init_geometry(m, depth, d_model, n_head, vocab, dtype, max_B, max_T);
    size_t need = 0;
    layout(m, nullptr, &need);
    if (arena_bytes < need) {
        delete m;
        return set_error(NC_ERR_OOM, "arena has %zu bytes, the model needs %zu", arena_bytes, need);
    }
    m->arena = (char*)arena;
    m->arena_bytes = arena_bytes;
    m->stream = (cudaStream_t)stream;
    layout(m, m->arena, &need);
    int rc = NC_OK;
    do {
        cudaStream_t s = m->stream;
        // weights N(0, 0.02) drawn on the device, one tensor at a time (init_normal_kernel)
        long pair0 = 0;
        for (int i = 0; i < m->nparams && rc == NC_OK; ++i) {
            const long n = m->prows[i] * m->pcols[i];
            init_normal_kernel<<<ceil_div((n + 1) / 2, 256), 256, 0, s>>>(m->master + m->poff[i], n, seed, pair0, 0.02);
            note_launch();
            rc = cuda_check(cudaGetLastError(), "init_normal_kernel");
            pair0 += (n + 1) / 2;
        }
        if (rc) break;
        if (m->shadow && (rc = cast_f32_bf16(m->master, m->shadow, m->P, s))) break;
        if ((rc = cuda_check(cudaMemsetAsync(m->grads, 0, m->P * 4, s), "memset"))) break;
        if ((rc = cuda_check(cudaMemsetAsync(m->momentum, 0, m->P * 4, s), "memset"))) break;
        if ((rc = cuda_check(cudaMemsetAsync(m->adam_m, 0, (size_t)2 * m->V * m->d * 4, s), "memset"))) break;
        if ((rc = cuda_check(cudaMemsetAsync(m->adam_v, 0, (size_t)2 * m->V * m->d * 4, s), "memset"))) break;
        if ((rc = cuda_check(cudaMemsetAsync(m->flag, 0, 16, s), "memset"))) break;
        // Muon table: q, k, v, o, w2 in the wide orientation already; w1 transposed
        std::vector<MuonMat> mats;
        long sq = 0, wide = (long)4 * depth * d_model * d_model;
        for (int l = 0; l < depth; ++l)
            for (int j = 0; j < 6; ++j) {
                const int idx = 1 + 6 * l + j;
                MuonMat mm;
                mm.off = m->poff[idx];
                mm.rows = (int)m->prows[idx];
                mm.cols = (int)m->pcols[idx];
                mm.tr = mm.rows > mm.cols;
                mm.scale = (float)sqrt(mm.rows > mm.cols ? (double)mm.rows / mm.cols : 1.0);
                if (j < 4) { mm.x_off = sq; sq += (long)d_model * d_model; }
                else { mm.x_off = wide; wide += (long)4 * d_model * d_model; }
                mats.push_back(mm);
            }
        if ((rc = cuda_check(cudaMemcpyAsync(m->mats, mats.data(), mats.size() * sizeof(MuonMat),
                                             cudaMemcpyHostToDevice, s), "H2D mats"))) break;
        // RoPE table: angle t * 10000^(-2j/Dh), computed in double; pair-major
        // ([j][t]) so that kernels whose lanes hold consecutive positions read it
        // contiguously
        const int half = m->Dh / 2, Tt = m->maxT > 0 ? m->maxT : 1;
        std::vector<float2> rt((size_t)Tt * half);
        for (int t = 0; t < Tt; ++t)
            for (int j = 0; j < half; ++j) {
                double ang = t * pow(10000.0, -2.0 * j / m->Dh);
                rt[(size_t)j * Tt + t] = make_float2((float)cos(ang), (float)sin(ang));
            }
        if ((rc = cuda_check(cudaMemcpyAsync(m->rope, rt.data(), rt.size() * 8, cudaMemcpyHostToDevice, s),
                             "H2D rope"))) break;
        rc = cuda_check(cudaStreamSynchronize(s), "init sync");
    } while (0);
    if (rc) { delete m; return rc; }
    *out = m;
    return NC_OK;
}

int nc_free(nc_model* m) {
    if (m) for (auto e : m->ev_pool) cudaEventDestroy(e);
    if (m) for (auto& g : m->dec_graphs) if (g.exec) cudaGraphExecDestroy(g.exec);
    if (m && m->cap_stream) cudaStreamDestroy(m->cap_stream);
    delete m;
    return NC_OK;
}

int nc_profile(nc_model* m, int enable) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    if (enable) {
        NC_TRY(cuda_check(cudaStreamSynchronize(m->stream), "sync"));
        m->recs.clear();
        m->ev_used = 0;
    }
    m->prof_on = enable != 0;
    return NC_OK;
}

int nc_profile_read(nc_model* m, int category, double* ms, long* launches, double* flops, double* bytes) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    if (category < 0 || category >= NC_PROF_COUNT) return set_error(NC_ERR_ARG, "category %d", category);
    NC_TRY(cuda_check(cudaStreamSynchronize(m->stream), "sync"));
    double t = 0, fl = 0, by = 0;
    long n = 0;
    for (auto& r : m->recs) {
        if (r.cat != category) continue;
        float e = 0.f;
        NC_TRY(cuda_check(cudaEventElapsedTime(&e, r.a, r.b), "event time"));
        t += e; fl += r.flops; by += r.bytes; ++n;
    }
    if (ms) *ms = t;
    if (launches) *launches = n;
    if (flops) *flops = fl;
    if (bytes) *bytes = by;
    return NC_OK;
}

int nc_num_params(nc_model* m, int* out_n) {
    if (!m || !out_n) return set_error(NC_ERR_ARG, "null argument");
    *out_n = m->nparams;
    return NC_OK;
}

int nc_param_info(nc_model* m, int index, int* rows, int* cols, int* kind) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    if (index < 0 || index >= m->nparams) return set_error(NC_ERR_ARG, "param index %d", index);
    if (rows) *rows = (int)m->prows[index];
    if (cols) *cols = (int)m->pcols[index];
    if (kind) *kind = m->pkind[index];
    return NC_OK;
}

int nc_forward_backward(nc_model* m, const int32_t* tokens, const int32_t* targets,
                        const int32_t* token_bytes, int B, int T, int accumulate, float grad_scale,
                        float* loss_bpb_out) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    if (!tokens || !targets || !token_bytes || !loss_bpb_out) return set_error(NC_ERR_ARG, "null pointer");
    if (B < 1 || T < 1 || T > m->maxT || (long)B * T > m->maxM)
        return set_error(NC_ERR_ARG, "B=%d T=%d exceeds the arena's max_B*max_T=%ld / max_T=%d", B, T,
                         m->maxM, m->maxT);
    if (accumulate != 0 && accumulate != 1) return set_error(NC_ERR_ARG, "accumulate must be 0 or 1");
    if (m->dtype == NC_BF16)
        return forward_backward<bf16>(m, tokens, targets, token_bytes, B, T, accumulate, grad_scale, loss_bpb_out);
    return forward_backward<float>(m, tokens, targets, token_bytes, B, T, accumulate, grad_scale, loss_bpb_out);
}

int nc_eval_loss(nc_model* m, const int32_t* tokens, const int32_t* targets, const int32_t* token_bytes,
                 int B, int T, int accumulate, double* sums, float* loss_bpb_out) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    if (!tokens || !targets || !token_bytes || !sums) return set_error(NC_ERR_ARG, "null pointer");
    if (B < 1 || T < 1 || T > m->maxT || (long)B * T > m->maxM)
        return set_error(NC_ERR_ARG, "B=%d T=%d exceeds the arena's max_B*max_T=%ld / max_T=%d", B, T,
                         m->maxM, m->maxT);
    if (accumulate != 0 && accumulate != 1) return set_error(NC_ERR_ARG, "accumulate must be 0 or 1");
    if (m->dtype == NC_BF16)
        return forward_backward<bf16>(m, tokens, targets, token_bytes, B, T, 0, 1.f, loss_bpb_out, false,
                                      sums, accumulate);
    return forward_backward<float>(m, tokens, targets, token_bytes, B, T, 0, 1.f, loss_bpb_out, false,
                                   sums, accumulate);
}

int nc_muon_step(nc_model* m, float lr, float momentum, int nesterov, int ns_steps, const float ns_coef[3]) {
    if (!m || !ns_coef) return set_error(NC_ERR_ARG, "null argument");
    if (ns_steps < 0 || ns_steps > 100) return set_error(NC_ERR_ARG, "ns_steps %d", ns_steps);
    if (m->dtype == NC_BF16) return muon<bf16>(m, lr, momentum, nesterov, ns_steps, ns_coef);
    return muon<float>(m, lr, momentum, nesterov, ns_steps, ns_coef);
}

int nc_adamw_step(nc_model* m, float lr_emb, float lr_unemb, float beta1, float beta2, float eps,
                  float weight_decay, int step) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    if (step < 1) return set_error(NC_ERR_ARG, "step must be >= 1");
    const float bc1 = (float)(1.0 - pow((double)beta1, step));
    const float bc2 = (float)(1.0 - pow((double)beta2, step));
    const long n = (long)m->V * m->d;
    const int idx[2] = {0, m->nparams - 1};
    const float lrs[2] = {lr_emb, lr_unemb};
    Prof pr(m, NC_PROF_ADAMW, 0, 2.0 * n * (28.0 + (m->shadow ? 2.0 : 0.0)));
    for (int k = 0; k < 2; ++k) {
        const long o = m->poff[idx[k]];
        NC_TRY(adamw(m->master + o, m->shadow ? m->shadow + o : nullptr, m->grads + o,
                     m->adam_m + k * n, m->adam_v + k * n, n, lrs[k], beta1, beta2, eps,
                     weight_decay, bc1, bc2, m->stream));
    }
    return NC_OK;
}

int nc_train_step(nc_model* m, const int32_t* tokens_host, const int32_t* targets_host,
                  const int32_t* token_bytes, int B, int T, int n_micro, float muon_lr,
                  float muon_momentum, int ns_steps, const float ns_coef[3], float lr_emb,
                  float lr_unemb, float beta1, float beta2, float eps, float weight_decay,
                  int adam_step, float* loss_bpb_host) {
    if (!m || !tokens_host || !targets_host || !loss_bpb_host) return set_error(NC_ERR_ARG, "null argument");
    if (n_micro < 1 || n_micro > 64) return set_error(NC_ERR_ARG, "n_micro %d out of [1, 64]", n_micro);
    if (B < 1 || T < 1 || (long)B * T > m->maxM || T > m->maxT) return set_error(NC_ERR_ARG, "batch too large");
    const long n = (long)B * T;
    for (int i = 0; i < n_micro; ++i) {
        NC_TRY(cuda_check(cudaMemcpyAsync(m->tok_stage, tokens_host + i * n, n * 4, cudaMemcpyHostToDevice,
                                          m->stream), "H2D tokens"));
        NC_TRY(cuda_check(cudaMemcpyAsync(m->tok_stage + m->maxM, targets_host + i * n, n * 4,
                                          cudaMemcpyHostToDevice, m->stream), "H2D targets"));
        NC_TRY(nc_forward_backward(m, m->tok_stage, m->tok_stage + m->maxM, token_bytes, B, T, i > 0,
                                   1.0f / n_micro, m->loss + 2 * i));
    }
    NC_TRY(nc_muon_step(m, muon_lr, muon_momentum, 1, ns_steps, ns_coef));
    NC_TRY(nc_adamw_step(m, lr_emb, lr_unemb, beta1, beta2, eps, weight_decay, adam_step));
    float tmp[128];
    NC_TRY(cuda_check(cudaMemcpyAsync(tmp, m->loss, (size_t)n_micro * 2 * 4, cudaMemcpyDeviceToHost, m->stream),
                      "D2H loss"));
    NC_TRY(cuda_check(cudaStreamSynchronize(m->stream), "sync"));
    double a = 0, b = 0;
    for (int i = 0; i < n_micro; ++i) { a += tmp[2 * i]; b += tmp[2 * i + 1]; }
    loss_bpb_host[0] = (float)(a / n_micro);
    loss_bpb_host[1] = (float)(b / n_micro);
    return NC_OK;
}

}  // extern "C"

namespace {

// ---------------------------------------------------------------- inference with a KV cache
// Cache layout: [layer][k | v][cache_B][cache_T][d] in the model's activation type.
template <typename T>
struct Cache {
    T* base;
    int B, T_, d;
    T* k(int l) const { return base + (size_t)l * 2 * B * T_ * d; }
    T* v(int l) const { return k(l) + (size_t)B * T_ * d; }
};

int round8(int b) { return (b + 7) & ~7; }

// greedy token and (optionally) the logits of the Bp token rows in y [Bp][d]
template <typename T>
int lm_head_rows(nc_model* m, const void* y, int B, int Bp, float* logits_out, int32_t* next_out) {
    const int d = m->d, V = m->V, iu = 1 + 6 * m->depth;
    float* lt = reinterpret_cast<float*>(m->logits);   // logits^T [V][Bp]
    NC_TRY(run_gemm(m, mk(m, V, Bp, d, W<T>(m, iu), d, false, y, d, false, lt, Bp, NC_FP32)));
    Prof pr(m, NC_PROF_CE, 0, (double)V * Bp * 4);
    // (the argmax partials use the attention-gradient scratch, idle outside the backward)
    const size_t ws_bytes = (size_t)m->maxM * 3 * d * (m->dtype == NC_BF16 ? 2 : 4);
    if (next_out) NC_TRY(decode_argmax(lt, V, B, Bp, next_out, m->dqkv, ws_bytes, m->flag, m->stream));
    if (logits_out) NC_TRY(decode_logits_out(lt, V, B, Bp, logits_out, m->stream));
    return NC_OK;
}

template <typename T>
int prefill(nc_model* m, const Cache<T>& c, const int32_t* tok, int B, int T0, float* logits_out,
            int32_t* next_out) {
    const int d = m->d, H = m->H, Dh = m->Dh, F = m->F, V = m->V;
    const int M = B * T0, act = m->dtype, Bp = round8(B);
    const double ab = m->dtype == NC_BF16 ? 2.0 : 4.0;
    const double Md = (double)M * d;
    cudaStream_t s = m->stream;
    const bool fuse_rope = m->dtype == NC_BF16 && Dh == 128;
    const int rope_ld = m->maxT > 0 ? m->maxT : 1;
    {
        Prof pr(m, NC_PROF_EMBED, 0, Md * (ab + 4) + M * 4.0);
        NC_TRY(embed_forward<T>(tok, W<T>(m, 0), m->x, M, d, V, m->flag, s));
    }
    for (int l = 0; l < m->depth; ++l) {
        auto& Ly = m->L[l];
        const int b0 = 1 + 6 * l;
        {
            Prof pr(m, NC_PROF_NORM, 0, Md * (4 + ab) + M * 4.0);
            NC_TRY(rmsnorm_forward<T>(m->x, (T*)Ly.y1, Ly.r1, M, d, s));
        }
        {
            Gemm g = mk(m, M, 3 * d, d, Ly.y1, d, false, W<T>(m, b0), d, false, Ly.qkv, 3 * d, act);
            if (fuse_rope) {
                g.epi = EPI_ROPE; g.rope = m->rope; g.rope_T = T0; g.rope_cols = 2 * d; g.rope_ld = rope_ld;
            }
            NC_TRY(run_gemm(m, g));
            if (!fuse_rope) {
                Prof pr(m, NC_PROF_ROPE, 0, 4.0 * Md * ab);
                NC_TRY(rope_apply<T>((T*)Ly.qkv, 3 * d, M, T0, H, Dh, m->rope, rope_ld, 1.f, s));
            }
        }
        T* q = (T*)Ly.qkv;
        {
            Prof pr(m, NC_PROF_ROPE, 0, 4.0 * Md * ab);
            NC_TRY(prefill_kv_store<T>(q, B, T0, d, c.k(l), c.v(l), c.T_, s));
        }
        {
            Prof pr(m, NC_PROF_ATTN_FWD, 4.0 * B * H * Dh * (0.5 * T0 * (T0 + 1.0)), 0);
            NC_TRY(attention_forward<T>(q, q + d, q + 2 * d, 3 * d, (T*)Ly.o, d, Ly.lse, B, T0, H, Dh, s, m->flag));
        }
        {
            Gemm g = mk(m, M, d, d, Ly.o, d, false, W<T>(m, b0 + 3), d, false, m->x, d, NC_FP32);
            g.aux = m->x; g.ldaux = d; g.aux_dtype = NC_FP32; g.beta = 1.f;
            NC_TRY(run_gemm(m, g));
        }
        {
            Prof pr(m, NC_PROF_NORM, 0, Md * (4 + ab) + M * 4.0);
            NC_TRY(rmsnorm_forward<T>(m->x, (T*)Ly.y2, Ly.r2, M, d, s));
        }
        {
            Gemm g = mk(m, M, F, d, Ly.y2, d, false, W<T>(m, b0 + 4), d, false, Ly.a, F, act);
            g.epi = EPI_RELU2;
            NC_TRY(run_gemm(m, g));
        }
        {
            Gemm g = mk(m, M, d, F, Ly.a, F, false, W<T>(m, b0 + 5), F, false, m->x, d, NC_FP32);
            g.aux = m->x; g.ldaux = d; g.aux_dtype = NC_FP32; g.beta = 1.f;
            NC_TRY(run_gemm(m, g));
        }
    }
    {
        Prof pr(m, NC_PROF_NORM, 0, Md * (4 + ab) + M * 4.0);
        NC_TRY(rmsnorm_forward<T>(m->x, (T*)m->yf, m->rf, M, d, s));
        NC_TRY(prefill_gather_last<T>((const T*)m->yf, B, Bp, T0, d, (T*)m->dy, s));
    }
    return lm_head_rows<T>(m, m->dy, B, Bp, logits_out, next_out);
}

// pos_dev (a step recorded for replay): the position is read from device memory by the
// kernels that need it, and pos is only its upper bound (cache_T - 1)
template <typename T>
int decode_step(nc_model* m, const Cache<T>& c, const int32_t* tok, int B, int pos, float* logits_out,
                int32_t* next_out, const int* pos_dev = nullptr) {
    const int d = m->d, H = m->H, Dh = m->Dh, F = m->F, V = m->V;
    const int Bp = round8(B), n = pos + 1, act = m->dtype;
    const double ab = m->dtype == NC_BF16 ? 2.0 : 4.0;
    cudaStream_t s = m->stream;
    const int rope_ld = m->maxT > 0 ? m->maxT : 1;
    // scratch in the training activations: x^T, the normed rows, [q|k|v]^T, q, the attention
    // output, a^T (relu(h)^2), and the attention partials
    float* xt = m->x;
    T* y = (T*)m->yf;
    T* cq = (T*)m->L[0].qkv;
    T* q = (T*)m->L[0].o;
    T* att = (T*)m->L[0].y2;
    T* at = (T*)m->L[0].a;
    void* ws = m->dqkv;
    const size_t ws_bytes = (size_t)m->maxM * 3 * d * (size_t)ab;
    {
        Prof pr(m, NC_PROF_EMBED, 0, (double)B * d * (ab + 4));
        NC_TRY(decode_embed_t<T>(tok, W<T>(m, 0), xt, B, Bp, d, V, m->flag, s));
    }
    auto norm = [&]() {
        Prof pr(m, NC_PROF_NORM, 0, (double)Bp * d * (4 + ab));
        return decode_rmsnorm_cols<T>(xt, y, Bp, d, s);
    };
    for (int l = 0; l < m->depth; ++l) {
        const int b0 = 1 + 6 * l;
        NC_TRY(norm());
        NC_TRY(run_gemm(m, mk(m, 3 * d, Bp, d, W<T>(m, b0), d, false, y, d, false, cq, Bp, act)));
        {
            Prof pr(m, NC_PROF_ROPE, 0, (double)Bp * 3 * d * ab * 2);
            NC_TRY(decode_qkv_post<T>(cq, B, Bp, d, H, Dh, pos, pos_dev, m->rope, rope_ld, q, c.k(l), c.v(l), c.T_,
                                      s));
        }
        {
            Prof pr(m, NC_PROF_ATTN_FWD, 4.0 * B * H * Dh * n, 2.0 * B * n * d * ab);
            NC_TRY(decode_attention<T>(q, c.k(l), c.v(l), B, Bp, d, H, Dh, c.T_, n, pos_dev, att, ws, ws_bytes, s));
        }
        {   // x^T += Wo att^T
            Gemm g = mk(m, d, Bp, d, W<T>(m, b0 + 3), d, false, att, d, false, xt, Bp, NC_FP32);
            g.aux = xt; g.ldaux = Bp; g.aux_dtype = NC_FP32; g.beta = 1.f;
            NC_TRY(run_gemm(m, g));
        }
        NC_TRY(norm());
        {   // a^T = relu(W1 y^T)^2
            Gemm g = mk(m, F, Bp, d, W<T>(m, b0 + 4), d, false, y, d, false, at, Bp, act);
            g.epi = EPI_RELU2;
            NC_TRY(run_gemm(m, g));
        }
        {   // x^T += W2 a^T (a^T stored [F][Bp]: the K x N layout of the second operand)
            Gemm g = mk(m, d, Bp, F, W<T>(m, b0 + 5), F, false, at, Bp, true, xt, Bp, NC_FP32);
            g.aux = xt; g.ldaux = Bp; g.aux_dtype = NC_FP32; g.beta = 1.f;
            NC_TRY(run_gemm(m, g));
        }
    }
    NC_TRY(norm());
    return lm_head_rows<T>(m, y, B, Bp, logits_out, next_out);
}

int check_cache(nc_model* m, const void* cache, int cache_B, int cache_T, int B) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    if (!cache) return set_error(NC_ERR_ARG, "null cache");
    if ((uintptr_t)cache % 16) return set_error(NC_ERR_ARG, "cache must be 16-byte aligned");
    if (cache_B < 1 || cache_T < 1) return set_error(NC_ERR_ARG, "cache_B %d, cache_T %d", cache_B, cache_T);
    if (cache_T > m->maxT) return set_error(NC_ERR_ARG, "cache_T %d > the model's max_T %d", cache_T, m->maxT);
    if (B < 1 || B > cache_B) return set_error(NC_ERR_ARG, "B = %d outside [1, cache_B = %d]", B, cache_B);
    const long Bp = round8(B);
    const double ab = m->dtype == NC_BF16 ? 2.0 : 4.0;
    if (Bp > m->maxM || Bp * 4.0 > m->maxM * ab)
        return set_error(NC_ERR_ARG, "B = %d too large for the arena (max_B*max_T = %ld)", B, m->maxM);
    if (m->Dh != 128) return set_error(NC_ERR_UNSUPPORTED, "inference path: head dim %d (128 only)", m->Dh);
    return NC_OK;
}

}  // namespace

extern "C" {

int nc_kv_cache_bytes(nc_model* m, int cache_B, int cache_T, size_t* out) {
    if (!m || !out) return set_error(NC_ERR_ARG, "null argument");
    if (cache_B < 1 || cache_T < 1) return set_error(NC_ERR_ARG, "cache_B %d, cache_T %d", cache_B, cache_T);
    *out = (size_t)m->depth * 2 * cache_B * cache_T * m->d * (m->dtype == NC_BF16 ? 2 : 4);
    return NC_OK;
}

int nc_prefill(nc_model* m, void* cache, int cache_B, int cache_T, const int32_t* tokens, int B, int T0,
               float* logits_out, int32_t* next_out) {
    NC_TRY(check_cache(m, cache, cache_B, cache_T, B));
    if (!tokens) return set_error(NC_ERR_ARG, "null tokens");
    if (T0 < 1 || T0 > cache_T || (long)B * T0 > m->maxM)
        return set_error(NC_ERR_ARG, "T0 = %d: needs 1 <= T0 <= cache_T and B*T0 <= max_B*max_T", T0);
    if (m->dtype == NC_BF16)
        return prefill<bf16>(m, Cache<bf16>{(bf16*)cache, cache_B, cache_T, m->d}, tokens, B, T0, logits_out, next_out);
    return prefill<float>(m, Cache<float>{(float*)cache, cache_B, cache_T, m->d}, tokens, B, T0, logits_out,
                          next_out);
}

int nc_decode_step(nc_model* m, void* cache, int cache_B, int cache_T, const int32_t* tokens, int B, int pos,
                   float* logits_out, int32_t* next_out) {
    NC_TRY(check_cache(m, cache, cache_B, cache_T, B));
    if (!tokens) return set_error(NC_ERR_ARG, "null tokens");
    if (pos < 0 || pos >= cache_T) return set_error(NC_ERR_ARG, "pos %d outside [0, cache_T = %d)", pos, cache_T);
    if (decode_attention_ws_bytes(B, m->H, cache_T) > (size_t)m->maxM * 3 * m->d * (m->dtype == NC_BF16 ? 2 : 4))
        return set_error(NC_ERR_ARG, "decode workspace too small for B = %d", B);
    auto run = [&](int p, const int* pd) {
        if (m->dtype == NC_BF16)
            return decode_step<bf16>(m, Cache<bf16>{(bf16*)cache, cache_B, cache_T, m->d}, tokens, B, p, logits_out,
                                     next_out, pd);
        return decode_step<float>(m, Cache<float>{(float*)cache, cache_B, cache_T, m->d}, tokens, B, p,
                                  logits_out, next_out, pd);
    };
    if (!m->dec_graph_on || m->prof_on) return run(pos, nullptr);
    // The second call with the same buffers records the step (the position read from device
    // memory, the attention grid sized for the whole cache) as a CUDA graph; later calls set
    // the position and replay it: ~13 launches per layer become one.
    nc_model::DecGraph* gr = nullptr;
    for (auto& g : m->dec_graphs)
        if (g.cache == cache && g.cache_B == cache_B && g.cache_T == cache_T && g.B == B && g.tok == tokens &&
            g.logits == logits_out && g.next == next_out)
            gr = &g;
    if (!gr) {
        if (m->dec_graphs.size() >= 8) {
            if (m->dec_graphs.front().exec) cudaGraphExecDestroy(m->dec_graphs.front().exec);
            m->dec_graphs.erase(m->dec_graphs.begin());
        }
        m->dec_graphs.push_back({cache, cache_B, cache_T, B, tokens, logits_out, next_out, 0, nullptr, 0});
        gr = &m->dec_graphs.back();
    }
    if (gr->exec == nullptr && gr->uses++ == 0) return run(pos, nullptr);   // the first call runs directly
    if (gr->exec == nullptr) {
        if (!m->cap_stream)
            NC_TRY(cuda_check(cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking), "capture stream"));
        cudaStream_t s = m->cap_stream, user = m->stream;
        NC_TRY(cuda_check(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal), "decode capture"));
        const uint64_t l0 = nc_launch_count();
        m->stream = s;   // the step's launches go to the recording stream
        const int rc = run(cache_T - 1, m->pos_dev);
        m->stream = user;
        cudaGraph_t graph = nullptr;
        const cudaError_t e = cudaStreamEndCapture(s, &graph);
        const int k = (int)(nc_launch_count() - l0);
        note_launch(-k);   // recorded, not launched
        if (rc != NC_OK) {
            if (graph) cudaGraphDestroy(graph);
            return rc;
        }
        NC_TRY(cuda_check(e, "decode capture end"));
        const cudaError_t e2 = cudaGraphInstantiate(&gr->exec, graph, 0);
        cudaGraphDestroy(graph);
        NC_TRY(cuda_check(e2, "decode graph instantiate"));
        gr->kernels = k;
    }
    NC_TRY(decode_set_pos(m->pos_dev, pos, m->stream));
    NC_TRY(cuda_check(cudaGraphLaunch(gr->exec, m->stream), "decode graph launch"));
    note_launch(gr->kernels);
    return NC_OK;
}

int nc_decode_graphs(nc_model* m, int enable) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    m->dec_graph_on = enable != 0;
    return NC_OK;
}

int nc_lr_schedule(int step, int n_steps, float warmdown_frac, int d_model, int d_ref, const float base[3],
                   float out[3]) {
    if (!base || !out) return set_error(NC_ERR_ARG, "null pointer");
    if (n_steps < 1 || step < 0 || step >= n_steps)
        return set_error(NC_ERR_ARG, "step %d outside [0, n_steps = %d)", step, n_steps);
    if (!(warmdown_frac >= 0.f && warmdown_frac <= 1.f))
        return set_error(NC_ERR_ARG, "warmdown_frac %g outside [0, 1]", (double)warmdown_frac);
    if (d_model < 1 || d_ref < 1) return set_error(NC_ERR_ARG, "d_model %d, d_ref %d", d_model, d_ref);
    const long w = lround((double)warmdown_frac * n_steps);
    const double lrm = (w == 0 || step < n_steps - w) ? 1.0 : (double)(n_steps - step) / (double)w;
    const double width = sqrt((double)d_ref / (double)d_model);
    out[0] = (float)(lrm * base[0]);
    out[1] = (float)(lrm * base[1] * width);
    out[2] = (float)(lrm * base[2] * width);
    return NC_OK;
}

int nc_get_params(nc_model* m, int index, float* host, size_t n) {
    NC_TRY(check_param(m, index, n));
    if (!host) return set_error(NC_ERR_ARG, "null host buffer");
    return download_f32(m, host, m->master + m->poff[index], n);
}

int nc_set_params(nc_model* m, int index, const float* host, size_t n) {
    NC_TRY(check_param(m, index, n));
    if (!host) return set_error(NC_ERR_ARG, "null host buffer");
    NC_TRY(upload_f32(m, m->master + m->poff[index], host, n));
    if (m->shadow) {
        NC_TRY(cast_f32_bf16(m->master + m->poff[index], m->shadow + m->poff[index], (long)n, m->stream));
        return cuda_check(cudaStreamSynchronize(m->stream), "sync");
    }
    return NC_OK;
}

int nc_get_grads(nc_model* m, int index, float* host, size_t n) {
    NC_TRY(check_param(m, index, n));
    if (!host) return set_error(NC_ERR_ARG, "null host buffer");
    return download_f32(m, host, m->grads + m->poff[index], n);
}

int nc_set_grads(nc_model* m, int index, const float* host, size_t n) {
    NC_TRY(check_param(m, index, n));
    if (!host) return set_error(NC_ERR_ARG, "null host buffer");
    return upload_f32(m, m->grads + m->poff[index], host, n);
}

static float* state_ptr(nc_model* m, int index, int slot) {
    const int kind = m->pkind[index];
    if (kind == NC_KIND_MATRIX) return slot == NC_STATE_MOMENTUM ? m->momentum + m->poff[index] : nullptr;
    if (slot != NC_STATE_ADAM_M && slot != NC_STATE_ADAM_V) return nullptr;
    const long n = (long)m->V * m->d;
    float* base = slot == NC_STATE_ADAM_M ? m->adam_m : m->adam_v;
    return base + (kind == NC_KIND_EMB ? 0 : n);
}

int nc_get_state(nc_model* m, int index, int slot, float* host, size_t n) {
    NC_TRY(check_param(m, index, n));
    float* p = state_ptr(m, index, slot);
    if (!p || !host) return set_error(NC_ERR_ARG, "param %d has no state slot %d", index, slot);
    return download_f32(m, host, p, n);
}

int nc_set_state(nc_model* m, int index, int slot, const float* host, size_t n) {
    NC_TRY(check_param(m, index, n));
    float* p = state_ptr(m, index, slot);
    if (!p || !host) return set_error(NC_ERR_ARG, "param %d has no state slot %d", index, slot);
    return upload_f32(m, p, host, n);
}

int nc_check_device_flag(nc_model* m, uint32_t* flags) {
    if (!m) return set_error(NC_ERR_ARG, "null model");
    uint32_t f = 0;
    NC_TRY(cuda_check(cudaMemcpyAsync(&f, m->flag, 4, cudaMemcpyDeviceToHost, m->stream), "D2H flag"));
    NC_TRY(cuda_check(cudaMemsetAsync(m->flag, 0, 4, m->stream), "clear flag"));
    NC_TRY(cuda_check(cudaStreamSynchronize(m->stream), "sync"));
    if (flags) *flags = f;
    if (f) return set_error(NC_ERR_DEVICE_FLAG, "device flag 0x%x", f);
    return NC_OK;
}

// ------------------------------------------------------------ kernel-level
int nc_attention_forward(const void* q, const void* k, const void* v, int ld_qkv, void* o, int ld_o,
                         float* lse, int B, int T, int H, int D, int dtype, void* stream) {
    if (!q || !k || !v || !o || !lse) return set_error(NC_ERR_ARG, "null pointer");
    if (B < 0 || T < 0 || H < 1 || D < 2 || D > 128 || D % 2 || ld_qkv < H * D || ld_o < H * D)
        return set_error(NC_ERR_ARG, "bad attention shape");
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t* flag = nullptr;
    NC_TRY(kernel_flag(&flag));
    if (dtype == NC_BF16)
        return attention_forward<bf16>((const bf16*)q, (const bf16*)k, (const bf16*)v, ld_qkv, (bf16*)o,
                                       ld_o, lse, B, T, H, D, s, flag);
    if (dtype == NC_FP32)
        return attention_forward<float>((const float*)q, (const float*)k, (const float*)v, ld_qkv,
                                        (float*)o, ld_o, lse, B, T, H, D, s, flag);
    return set_error(NC_ERR_ARG, "dtype %d", dtype);
}

// [row statistics: B*H*T floats | dS store of the bf16 head-dim-128 path]
size_t nc_attention_workspace_bytes(int B, int T, int H) {
    if (B <= 0 || T <= 0 || H <= 0) return 256;
    return al((size_t)B * T * H * 4) + attention_ds_bytes(B, T, H, 128);
}

int nc_attention_backward(const void* q, const void* k, const void* v, int ld_qkv, const void* o,
                          const void* dout, int ld_o, const float* lse, void* dq, void* dk, void* dv,
                          int ld_dqkv, void* workspace, int B, int T, int H, int D, int dtype,
                          void* stream) {
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
        return set_error(NC_ERR_ARG, "null pointer");
    if (B < 0 || T < 0 || H < 1 || D < 2 || D > 128 || D % 2 || ld_qkv < H * D || ld_o < H * D ||
        ld_dqkv < H * D)
        return set_error(NC_ERR_ARG, "bad attention shape");
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t* flag = nullptr;
    NC_TRY(kernel_flag(&flag));
    if (dtype == NC_BF16)
        return attention_backward<bf16>((const bf16*)q, (const bf16*)k, (const bf16*)v, ld_qkv,
                                        (const bf16*)o, (const bf16*)dout, ld_o, lse, (bf16*)dq,
                                        (bf16*)dk, (bf16*)dv, ld_dqkv, (float*)workspace, B, T, H, D, s,
                                        flag, nullptr, 0, nullptr, false,
                                        (char*)workspace + al((size_t)B * T * H * 4));
    if (dtype == NC_FP32)
        return attention_backward<float>((const float*)q, (const float*)k, (const float*)v, ld_qkv,
                                         (const float*)o, (const float*)dout, ld_o, lse, (float*)dq,
                                         (float*)dk, (float*)dv, ld_dqkv, (float*)workspace, B, T, H, D,
                                         s, flag);
    return set_error(NC_ERR_ARG, "dtype %d", dtype);
}

int nc_gemm_bf16(int M, int N, int K, int batch, const void* A, long lda, long stride_a, int trans_a,
                 const void* B, long ldb, long stride_b, int trans_b, void* C, long ldc, long stride_c,
                 int c_dtype, float alpha, float beta, void* workspace, size_t workspace_bytes,
                 void* stream) {
    if (!A || !B || !C) return set_error(NC_ERR_ARG, "null pointer");
    if (M < 1 || N < 1 || K < 1 || batch < 1) return set_error(NC_ERR_ARG, "bad GEMM shape");
    if (c_dtype != NC_BF16 && c_dtype != NC_FP32) return set_error(NC_ERR_ARG, "c_dtype");
    if (lda < (trans_a ? M : K) || ldb < (trans_b ? N : K) || ldc < N)
        return set_error(NC_ERR_ARG, "leading dimension too small");
    Gemm g;
    g.M = M; g.N = N; g.K = K; g.batch = batch;
    g.A = A; g.lda = lda; g.sA = stride_a; g.a_t = trans_a != 0;
    g.B = B; g.ldb = ldb; g.sB = stride_b; g.b_t = trans_b != 0;
    g.in_dtype = NC_BF16;
    g.C = C; g.ldc = ldc; g.sC = stride_c; g.c_dtype = c_dtype;
    g.alpha = alpha; g.beta = beta;
    if (beta != 0.f) { g.aux = C; g.ldaux = ldc; g.sAux = stride_c; g.aux_dtype = c_dtype; }
    if (!gemm_tc_supported(g))
        return set_error(NC_ERR_UNSUPPORTED, "operands must be 16-byte aligned with leading dims % 8 == 0");
    NC_TRY(kernel_flag(&g.flag));
    return gemm_tc(g, workspace, workspace_bytes, (cudaStream_t)stream);
}

}  // extern "C"
