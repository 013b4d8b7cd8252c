/*
 * nc_api.h -- C ABI of libnc.so, one nanochat pretraining step on one B300.
 *
 * The step (nanochat speedrun walkthrough, lyylswood.com, section 预搜检
 * "pretraining"): a Llama-like, bias-free decoder-only transformer with
 * parameter-free RMSNorm; next-token cross-entropy, also reported as bits
 * per byte; full backward; Muon (Newton-Schulz orthogonalised momentum) for
 * the 2-D block matrices and AdamW for the embedding and unembedding.  The
 * section 该你了 (depth scaling) adds gradient accumulation when the device
 * batch is smaller than the optimizer batch.  Around the step: an evaluation
 * pass (loss and bits per byte, no backward), the run's learning-rate
 * schedule, and inference with a KV cache (prefill and greedy decode).
 *
 * Conventions for every entry point:
 *  - Every function returns an int status: NC_OK (0) or one of NC_ERR_*.
 *    nc_last_error() returns a thread-local message for the last failure.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns NC_ERR_ARG and launches nothing.
 *  - "device" pointers are CUDA device memory owned by the caller; "host"
 *    pointers are ordinary (or pinned) host memory owned by the caller.
 *  - Calls on a model enqueue work on the model's stream and return without
 *    waiting, unless the comment says the call synchronises.
 *  - The library allocates no device memory for data: the caller passes one
 *    arena (e.g. a torch uint8 tensor) of nc_arena_bytes() bytes and the
 *    library lays every parameter, optimizer state and activation out inside
 *    it (a KV cache is a second caller-owned buffer).  The one exception is
 *    the CUDA graphs (and their recording stream) that nc_decode_step keeps,
 *    which the CUDA runtime backs with its own memory; nc_decode_graphs(m, 0)
 *    turns them off.
 *  - Conditions found on the device (a token id >= vocab, a non-finite loss,
 *    a bounded wait that ran out) set bits of a device flag word instead of
 *    trapping; nc_check_device_flag() reads and clears a model's word, and
 *    nc_check_kernel_flag() the per-device word of the kernel-level entry
 *    points (attention, GEMM), which belong to no model.
 */
#ifndef NC_API_H
#define NC_API_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NC_API __attribute__((visibility("default")))
#else
#define NC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum {
    NC_OK = 0,
    NC_ERR_ARG = 1,          /* invalid argument (checked on the host) */
    NC_ERR_CUDA = 2,         /* a CUDA runtime/driver call failed */
    NC_ERR_OOM = 3,          /* the arena is smaller than nc_arena_bytes() */
    NC_ERR_DEVICE_FLAG = 4,  /* nc_check_device_flag found a flag set */
    NC_ERR_TIMEOUT = 5,      /* a bounded device wait ran out */
    NC_ERR_UNSUPPORTED = 6   /* shape not supported by this build */
};

enum { NC_BF16 = 0, NC_FP32 = 1 };              /* compute mode */
enum { NC_KIND_EMB = 0, NC_KIND_MATRIX = 1, NC_KIND_UNEMB = 2 };
enum { NC_STATE_MOMENTUM = 0, NC_STATE_ADAM_M = 1, NC_STATE_ADAM_V = 2 };

/* device flag bits */
#define NC_FLAG_TOKEN_RANGE 0x1u  /* a token or target id outside [0, vocab) */
#define NC_FLAG_NONFINITE   0x2u  /* the loss came out NaN or Inf */
#define NC_FLAG_TIMEOUT     0x4u  /* a pipeline wait inside a kernel gave up */
#define NC_FLAG_SMEM_ALIGN  0x8u  /* a kernel found its shared memory misaligned and skipped its work */

typedef struct nc_model nc_model;   /* opaque, owned by the library (host memory) */

NC_API const char* nc_last_error(void);

/* Number of kernels this process has launched through the library so far. */
NC_API uint64_t nc_launch_count(void);

/*
 * Bytes of device arena a model needs.  depth >= 1; d_model % n_head == 0;
 * head_dim = d_model / n_head even and <= 128; d_model % 8 == 0;
 * 1 <= vocab < 2^31 and vocab % 8 == 0.  max_B * max_T is the largest
 * micro-batch nc_forward_backward will be given (0 for an optimizer-only
 * model).  dtype is NC_BF16 or NC_FP32.
 */
NC_API int nc_arena_bytes(int depth, int d_model, int n_head, int vocab, int max_B, int max_T,
                   int dtype, size_t* out_bytes);

/*
 * Create a model (section 预搜检: depth layers of width d_model with n_head
 * heads; section 该你了: depth is the one size knob).  Weights are drawn
 * N(0, 0.02) on the device: value pair k (parameters in index order) is the
 * Box-Muller transform of outputs 2k and 2k+1 of the splitmix64 stream
 * seeded by `seed`; optimizer state is zero.
 * arena: device pointer, 256-byte aligned, arena_bytes >= nc_arena_bytes().
 * stream: a cudaStream_t (NULL = legacy default stream) all work is put on.
 * Synchronises the stream before returning.  *out receives the handle.
 */
NC_API int nc_init_model(int depth, int d_model, int n_head, int vocab, uint64_t seed,
                  void* arena, size_t arena_bytes, int dtype, int max_B, int max_T,
                  void* stream, nc_model** out);

NC_API int nc_free(nc_model* m);   /* frees the host-side handle; the arena stays the caller's */

/* Parameter tensors: 0 = wte [V, d]; 1 + 6*l + {0..5} = wq, wk, wv, wo [d, d],
 * w1 [4d, d], w2 [d, 4d] of layer l; 6*depth + 1 = lm_head [V, d]. */
NC_API int nc_num_params(nc_model* m, int* out_n);
NC_API int nc_param_info(nc_model* m, int index, int* rows, int* cols, int* kind);

/*
 * Forward, loss and backward for one micro-batch (section 预搜检: predict the
 * next token; validation loss reported as bits per byte).
 * tokens, targets: device int32 [B*T], row b*T + t.  token_bytes: device
 * int32 [vocab], the UTF-8 length of each token id (0 = excluded from bpb).
 * B*T <= max_B*max_T, T <= max_T.  accumulate = 0 overwrites the gradients,
 * 1 adds to them; the gradient is grad_scale * d(mean loss).
 * loss_bpb_out: device float[2] <- {mean cross-entropy (nats), bits per byte}
 * of this micro-batch.  Asynchronous.
 */
NC_API int nc_forward_backward(nc_model* m, const int32_t* tokens, const int32_t* targets,
                        const int32_t* token_bytes, int B, int T, int accumulate,
                        float grad_scale, float* loss_bpb_out);

/*
 * Evaluation pass (section 预搜检: the run reports validation bits per byte
 * from time to time): forward and loss of one batch, no backward.  The
 * gradients, optimizer state and weights are not touched.
 * tokens, targets, token_bytes: as for nc_forward_backward.
 * sums: device double[3], required: {sum of nll (nats), sum of nll over the
 * targets with token_bytes > 0, sum of token_bytes}, set (accumulate = 0) or
 * added to (accumulate = 1), so that bits per byte over many batches is the
 * ratio of sums sums[1] / (ln 2 * sums[2]).
 * loss_bpb_out: device float[2] or NULL <- {mean nll, bpb} of this batch,
 * bit-identical to what nc_forward_backward reports for the same batch and
 * weights.  Asynchronous.
 */
NC_API int nc_eval_loss(nc_model* m, const int32_t* tokens, const int32_t* targets,
                        const int32_t* token_bytes, int B, int T, int accumulate, double* sums,
                        float* loss_bpb_out);

/*
 * Muon on every block matrix (section 预搜检: Muon optimises the matrices):
 * buf = momentum*buf + g; g' = g + momentum*buf if nesterov else buf;
 * X = g'/(|g'|_F + 1e-7), transposed when rows > cols; ns_steps iterations of
 * A = X X^T, B = c1*A + c2*A A, X = c0*X + B X with ns_coef = {c0, c1, c2};
 * W -= lr * sqrt(max(1, rows/cols)) * X.  q, k and v are three matrices.
 * The gradient buffers are consumed (overwritten with g').  Asynchronous.
 */
NC_API int nc_muon_step(nc_model* m, float lr, float momentum, int nesterov, int ns_steps,
                 const float ns_coef[3]);

/*
 * AdamW on wte (lr_emb) and lm_head (lr_unemb), section 预搜检: AdamW
 * optimises the embedding and unembedding.  step is 1-based (bias
 * correction 1 - beta^step); decoupled decay W *= 1 - lr*weight_decay.
 * Asynchronous.
 */
NC_API int nc_adamw_step(nc_model* m, float lr_emb, float lr_unemb, float beta1, float beta2,
                  float eps, float weight_decay, int step);

/*
 * One whole optimizer step from HOST buffers: copies n_micro micro-batches of
 * tokens/targets (host int32 [n_micro*B*T]) to the device, runs
 * nc_forward_backward on each with grad_scale 1/n_micro, then nc_muon_step
 * and nc_adamw_step with the given hyper-parameters, and copies the mean
 * {loss, bpb} over the micro-batches to loss_bpb_host (host float[2]).
 * token_bytes is a device pointer (uploaded once by the caller).
 * Synchronises the stream.
 */
NC_API int nc_train_step(nc_model* m, const int32_t* tokens_host, const int32_t* targets_host,
                  const int32_t* token_bytes, int B, int T, int n_micro,
                  float muon_lr, float muon_momentum, int ns_steps, const float ns_coef[3],
                  float lr_emb, float lr_unemb, float beta1, float beta2, float eps,
                  float weight_decay, int adam_step, float* loss_bpb_host);

/*
 * Inference with a KV cache (section 预搜检, on sampling from the base model: an
 * Engine with a KV cache runs prefill and decode).  The cache is caller-owned
 * device memory of nc_kv_cache_bytes(m, cache_B, cache_T) bytes, 16-byte
 * aligned, laid out [layer][k | v][cache_B][cache_T][d_model] in the model's
 * activation type, k after RoPE.  cache_T <= the model's max_T.  Both calls
 * use the model's training activations as scratch (a training step in between
 * is fine; the cache holds all state of the sequences) and are asynchronous.
 */
NC_API int nc_kv_cache_bytes(nc_model* m, int cache_B, int cache_T, size_t* out);

/*
 * Prefill: B prompts of T0 tokens (tokens: device int32 [B*T0], row b*T0 + t),
 * 1 <= B <= cache_B, T0 <= cache_T, B*T0 <= max_B*max_T.  Writes k and v of
 * positions 0 .. T0-1 of sequence b into cache row b, and for the last
 * position of every prompt the logits (logits_out: device float [B*V] or
 * NULL) and the greedy next token (next_out: device int32 [B] or NULL; the
 * lowest id among equal maxima).
 */
NC_API int nc_prefill(nc_model* m, void* cache, int cache_B, int cache_T, const int32_t* tokens, int B,
                      int T0, float* logits_out, int32_t* next_out);

/*
 * Decode: tokens (device int32 [B]) is the token at position pos of each of the
 * sequences in cache rows 0 .. B-1, whose positions 0 .. pos-1 are cached.
 * Appends its k and v at position pos and returns the logits of the next
 * position and the greedy next token as nc_prefill does.  0 <= pos < cache_T.
 * Errors: NC_ERR_ARG for a bad cache, B, pos or pointer; NC_ERR_UNSUPPORTED
 * for head dims other than 128.  An out-of-range token sets
 * NC_FLAG_TOKEN_RANGE (its row embeds as zeros).
 */
NC_API int nc_decode_step(nc_model* m, void* cache, int cache_B, int cache_T, const int32_t* tokens, int B,
                          int pos, float* logits_out, int32_t* next_out);

/*
 * Decode steps as CUDA graphs (default on): the second nc_decode_step call with the
 * same cache, B and token/logit/next-token buffers records the step once; later
 * calls set the position and replay it, with results bit-identical to direct
 * launches.  enable = 0 launches every kernel directly (as does every call while
 * the profiler is on).  New weights need no re-recording.
 */
NC_API int nc_decode_graphs(nc_model* m, int enable);

/*
 * Learning rates of optimizer step `step` (0-based) of an n_steps run (section
 * 预搜检: the rate scales as 1/sqrt(dim), and the multiplier lrm falls
 * linearly to 0 near the end of training).  Host arithmetic, no device work.
 *   lrm = 1 for step < n_steps - W, else (n_steps - step) / W, where
 *   W = round(warmdown_frac * n_steps) warm-down steps (W = 0: lrm = 1).
 *   out[0] = lrm * base[0]                          (Muon; its update size is
 *            already fixed by the orthogonalisation and sqrt(max(1, rows/cols)))
 *   out[1] = lrm * base[1] * sqrt(d_ref / d_model)  (AdamW, embedding)
 *   out[2] = lrm * base[2] * sqrt(d_ref / d_model)  (AdamW, unembedding)
 * base: host float[3], the rates at width d_ref.  out: host float[3].
 * Errors: NC_ERR_ARG for n_steps < 1, step outside [0, n_steps),
 * warmdown_frac outside [0, 1], d_model or d_ref < 1, or null pointers.
 */
NC_API int nc_lr_schedule(int step, int n_steps, float warmdown_frac, int d_model, int d_ref,
                          const float base[3], float out[3]);

/* Host <-> device copies of one tensor as fp32 (n = rows*cols elements).
 * nc_set_params also refreshes the bf16 compute copy.  slot is one of
 * NC_STATE_* (momentum for matrices, Adam m/v for wte and lm_head).
 * All synchronise the stream. */
NC_API int nc_get_params(nc_model* m, int index, float* host, size_t n);
NC_API int nc_set_params(nc_model* m, int index, const float* host, size_t n);
NC_API int nc_get_grads(nc_model* m, int index, float* host, size_t n);
NC_API int nc_set_grads(nc_model* m, int index, const float* host, size_t n);
NC_API int nc_get_state(nc_model* m, int index, int slot, float* host, size_t n);
NC_API int nc_set_state(nc_model* m, int index, int slot, const float* host, size_t n);

/* Reads and clears the device flag word (NC_FLAG_*).  Synchronises.
 * Returns NC_ERR_DEVICE_FLAG when any bit was set, NC_OK otherwise. */
NC_API int nc_check_device_flag(nc_model* m, uint32_t* flags);

/* ------------------------------------------------------------------ */
/* Kernel-level entry points (the same kernels the step runs).         */
/* ------------------------------------------------------------------ */

/* Reads and clears the flag word (NC_FLAG_*) that the kernels of the
 * kernel-level entry points below set on the current device (one word per
 * device in the library's own memory; a kernel that gave up a bounded wait,
 * or found its shared memory misaligned, leaves its outputs unwritten and
 * sets a bit here).  Synchronises `stream`, which should be the stream the
 * calls were made on.  Returns NC_ERR_DEVICE_FLAG when any bit was set. */
NC_API int nc_check_kernel_flag(void* stream, uint32_t* flags);

/* Failure-detection self-test: launches one CTA on `stream` that waits on an
 * mbarrier nothing arrives on, through the library's bounded wait (about 4 s
 * of %globaltimer), which then gives up; the kernel sets NC_FLAG_TIMEOUT in
 * the per-device word of nc_check_kernel_flag() and returns, leaving the
 * context usable.  No fault, trap or unbounded wait is involved.
 * Asynchronous; returns NC_ERR_CUDA if the launch fails. */
NC_API int nc_selftest_wait_timeout(void* stream);

/*
 * Causal multi-head attention forward (section 预搜检: 10 heads of dim 128):
 * O = softmax(Q K^T / sqrt(D), keys s <= query t) V per (b, h).
 * q, k, v: device bf16 (dtype NC_BF16) or fp32 (NC_FP32); element (b, t, h, j)
 * at ptr[(b*T + t)*ld + h*D + j] with ld = ld_qkv (elements, >= H*D).
 * o: same layout with ld_o.  lse: device fp32 [B, H, T], natural-log
 * sum-exp of the scaled scores of each query row.  D <= 128, even.
 */
NC_API int nc_attention_forward(const void* q, const void* k, const void* v, int ld_qkv,
                         void* o, int ld_o, float* lse, int B, int T, int H, int D,
                         int dtype, void* stream);

/*
 * Gradients of the attention above given dO (layout of o, ld_o): dq, dk, dv
 * in the layout of q, k, v with ld_dqkv.  workspace: device scratch of
 * nc_attention_workspace_bytes() bytes, 16-byte aligned: the row statistics
 * D_t = dO_t.O_t, then (bf16, head dim 128) a store for the score gradients
 * dS of every causal 128x128 block (B*H*nb(nb+1)/2 tiles of 32 KB, nb =
 * ceil(T/128)), which lets dq be formed without recomputing the scores.
 * Deterministic.
 */
NC_API size_t nc_attention_workspace_bytes(int B, int T, int H);
NC_API int nc_attention_backward(const void* q, const void* k, const void* v, int ld_qkv,
                          const void* o, const void* dout, int ld_o, const float* lse,
                          void* dq, void* dk, void* dv, int ld_dqkv, void* workspace,
                          int B, int T, int H, int D, int dtype, void* stream);

/*
 * The attention backward above, for callers that cannot allocate device
 * memory (no counterpart on the pages: it only changes where the scratch
 * lives).  Same arguments and results as nc_attention_backward minus the
 * workspace: the B*H*T row statistics go to a fixed array compiled into the
 * library, which every GPU that loads it holds until the process exits.
 * B*H*T must not exceed NC_ATTN_NOALLOC_MAX_ROWS (NC_ERR_ARG otherwise).
 * Allocates nothing.  The first call on a device looks up the array's device
 * address (with that device current), so make it before any stream capture.
 * All calls share the array: calls that overlap on the GPU (different
 * streams) race; calls on one stream are safe.  Nothing needs clearing: each
 * call overwrites every element it reads.
 */
#define NC_ATTN_NOALLOC_MAX_ROWS (1L << 20)
NC_API int nc_attention_backward_noalloc(const void* q, const void* k, const void* v, int ld_qkv,
                                         const void* o, const void* dout, int ld_o, const float* lse,
                                         void* dq, void* dk, void* dv, int ld_dqkv, int B, int T, int H,
                                         int D, int dtype, void* stream);

/*
 * Dense GEMM on the tensor cores (bf16 in, fp32 accumulate):
 * C[b] = alpha * op(A[b]) op(B[b])^T + beta * C_in[b] for b < batch, where
 * op(A) is [M, K] and op(B) is [N, K].  trans_a = 0: A row-major [M, K] with
 * leading dimension lda; trans_a = 1: A row-major [K, M] (lda >= M).
 * trans_b = 0: B row-major [N, K]; trans_b = 1: B row-major [K, N].
 * c_dtype NC_BF16 or NC_FP32 (C row-major [M, N], ldc).  beta != 0 reads C
 * before writing it.  stride_* are element strides between batch entries.
 * Leading dimensions must be multiples of 8 and pointers 16-byte aligned.
 * workspace: device scratch for split-K partial sums (fp32); pass NULL and
 * 0 to disable split-K.
 */
NC_API int nc_gemm_bf16(int M, int N, int K, int batch, const void* A, long lda, long stride_a,
                 int trans_a, const void* B, long ldb, long stride_b, int trans_b,
                 void* C, long ldc, long stride_c, int c_dtype, float alpha, float beta,
                 void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------ */
/* Measurement: CUDA events around each kernel class of a model.       */
/* ------------------------------------------------------------------ */
enum {
    NC_PROF_GEMM = 0,        /* step GEMMs (projections, LM head, their backward) */
    NC_PROF_ATTN_FWD = 1,    /* causal attention forward */
    NC_PROF_ATTN_BWD = 2,    /* causal attention backward */
    NC_PROF_NORM = 3,        /* RMSNorm forward and backward */
    NC_PROF_ROPE = 4,        /* RoPE on q, k and on their gradients */
    NC_PROF_CE = 5,          /* softmax cross-entropy, loss and bpb reduction */
    NC_PROF_EMBED = 6,       /* embedding lookup and its backward */
    NC_PROF_MUON_NS = 7,     /* Newton-Schulz GEMMs */
    NC_PROF_MUON_ELEM = 8,   /* Muon momentum, normalisation, update */
    NC_PROF_ADAMW = 9,       /* AdamW */
    NC_PROF_COUNT = 10
};

/* enable = 1 clears the counters and records a CUDA event pair around every
 * kernel class launched on the model's stream from now on; 0 stops. */
NC_API int nc_profile(nc_model* m, int enable);

/* Totals since nc_profile(m, 1) for one class: device milliseconds (sum of
 * event-pair durations), launch sites timed, algorithmic FLOPs and bytes
 * (the work the class must do: 2*M*N*K per GEMM, the causal half of the
 * attention products, the bytes an elementwise kernel must read and write).
 * Synchronises the stream. */
NC_API int nc_profile_read(nc_model* m, int category, double* ms, long* launches, double* flops,
                           double* bytes);

#ifdef __cplusplus
}
#endif
#endif /* NC_API_H */
