"""Model geometry: parameter order, shapes and the FLOP convention used for MFU.

Geometry from the nanochat speedrun walkthrough (lyylswood.com):
  * section 预搜检 (pretraining): 20 layers, 1280 channels, 10 heads of
    dim 128, ~560M parameters, 32 x 2048 tokens per GPU per step;
  * section 该你了 (depth scaling): depth is the single knob, channels follow
    it (64 * depth), and deeper models use smaller device batches with
    gradient accumulation to keep the 0.5M-token optimizer batch.

The parameter count 12*d^2*L + 2*V*d (untied embedding and unembedding,
non-gated 4x MLP) gives 560,988,160 at d20, the page's "~560M".

MFU convention: FLOP/token = 6 * N_matmul + 12 * L * d * T, with N_matmul the
block matrices plus the LM head (the embedding lookup is not a matmul).  At
d20 this is 3.492e9 FLOP/token; times 21,400 steps of 524,288 tokens it gives
3.9e19, the page's "~4e19 FLOPs", and with ~0.5 s per step on 8 GPUs the
"nearly half" bf16 utilisation it reports.
"""

EMB, MATRIX, UNEMB = 0, 1, 2


def param_shapes(depth, d_model, n_head, vocab):
    d, V = d_model, vocab
    shapes = [(V, d)]
    for _ in range(depth):
        shapes += [(d, d), (d, d), (d, d), (d, d), (4 * d, d), (d, 4 * d)]
    shapes.append((V, d))
    return shapes


def param_kinds(depth):
    return [EMB] + [MATRIX] * (6 * depth) + [UNEMB]


def n_params(depth, d_model, n_head, vocab):
    return sum(r * c for r, c in param_shapes(depth, d_model, n_head, vocab))


def flops_per_token(depth, d_model, vocab, seq_len, causal=False):
    """Model FLOPs per trained token (forward + backward).

    causal=False is the pages' convention (attention counted as dense,
    12*L*d*T); causal=True counts only the unmasked half (6*L*d*T).
    """
    n_matmul = 12 * d_model * d_model * depth + vocab * d_model
    attn = (6 if causal else 12) * depth * d_model * seq_len
    return 6 * n_matmul + attn


def chinchilla_steps(depth, d_model, n_head, vocab, tokens_per_step, tokens_per_param=20):
    """Optimizer steps of a run that trains on tokens_per_param tokens per
    parameter (section 预搜检: 560M x 20 ~ 11.2B tokens, ~21,400 steps of
    524,288 tokens at d20)."""
    return round(tokens_per_param * n_params(depth, d_model, n_head, vocab) / tokens_per_step)


def eval_flops_per_token(depth, d_model, vocab, seq_len, causal=False):
    """Forward-only FLOPs per evaluated token: a third of flops_per_token."""
    return flops_per_token(depth, d_model, vocab, seq_len, causal) / 3

