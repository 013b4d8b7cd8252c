"""fp64 forward and hand-derived backward of the nanochat decoder step.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources (nanochat speedrun walkthrough, lyylswood.com):
  * intro, the author's comment under the release: the model is Llama-like
    but simpler and borrows parts of modded-nanoGPT.
  * section 预搜检 (pretraining): a 20-layer transformer, 1280 channels,
    10 heads of dim 128, ~560M parameters; each GPU runs 32 rows of 2048
    tokens; Muon for the matrices, AdamW for embedding and unembedding, no
    other trainable parameters (no biases, no RMSNorm gains); validation
    loss is reported as bits per byte, i.e. the per-token loss normalised by
    the bytes each token stands for.

Readings taken where the pages are silent (each one is also listed in the
design notes):
  * positional encoding: RoPE, base 10000, rotate-half pairing (dims j and
    j + Dh/2), positions 0..T-1 within each row, applied to q and k after
    the projection;
  * pre-norm blocks (norm before attention and before the MLP) and a final
    norm before the LM head; RMSNorm eps = 1e-6 inside the square root;
  * untied embedding / unembedding and a non-gated 4x MLP with ReLU^2: the
    ~560M count fixes untied + non-gated (12*d^2*L + 2*V*d = 560,988,160);
  * multi-head attention with as many k/v heads as q heads, scale 1/sqrt(Dh);
  * loss = mean over all B*T next-token targets;
  * bpb = sum(nll over targets with bytes > 0) / (ln 2 * sum(bytes[target]))
    (corpus ratio of sums, bytes looked up by the target id).

Parameters are a flat list in a fixed order:
  0                wte      [V, d]
  1 + 6*l + 0..5   wq, wk, wv, wo [d, d]; w1 [4d, d]; w2 [d, 4d]   (layer l)
  1 + 6*L          lm_head  [V, d]
Rows of activations are tokens in (b, t) order: row = b*T + t.
"""

from dataclasses import dataclass

import numpy as np

EPS = 1e-6
ROPE_BASE = 10000.0


@dataclass(frozen=True)
class Config:
    depth: int
    d_model: int
    n_head: int
    vocab: int

    @property
    def head_dim(self):
        return self.d_model // self.n_head

    @property
    def d_ff(self):
        return 4 * self.d_model


def param_shapes(cfg):
    d, V = cfg.d_model, cfg.vocab
    shapes = [(V, d)]
    for _ in range(cfg.depth):
        shapes += [(d, d), (d, d), (d, d), (d, d), (4 * d, d), (d, 4 * d)]
    shapes.append((V, d))
    return shapes


# ---------------------------------------------------------------- RMSNorm
def rmsnorm(x):
    """Parameter-free RMSNorm over the last axis: y = x / sqrt(mean(x^2) + eps).

    Returns (y, r) with r = 1 / sqrt(mean(x^2) + eps) per row.
    """
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS)
    return x * r, r


def rmsnorm_backward(dy, y, r):
    """dL/dx of y = x * r(x).

    With y = x r and dr/dx_j = -r^3 x_j / d:
      dx_j = r * (dy_j - y_j * mean_i(dy_i * y_i)).
    """
    return r * (dy - y * np.mean(dy * y, axis=-1, keepdims=True))


# ---------------------------------------------------------------- RoPE
def rope_tables(T, head_dim):
    """cos/sin of angle t * base^(-2j/Dh) for t < T, j < Dh/2, in fp64."""
    half = head_dim // 2
    inv_freq = ROPE_BASE ** (-np.arange(half, dtype=np.float64) * 2.0 / head_dim)
    ang = np.arange(T, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def rope(x, cos, sin):
    """Rotate pairs (j, j + Dh/2) of x [B, T, H, Dh] by the angle of position t."""
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    c = cos[None, :, None, :]
    s = sin[None, :, None, :]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_backward(dy, cos, sin):
    """Adjoint of ``rope``: the rotation is orthogonal, so rotate by -angle."""
    return rope(dy, cos, -sin)


# ---------------------------------------------------------------- attention
def causal_attention(q, k, v):
    """O = softmax(q k^T / sqrt(Dh), keys s <= query t) v.

    q, k, v: [B, T, H, Dh].  Returns (O [B, T, H, Dh], P [B, H, T, T],
    lse [B, H, T]) where lse is the natural-log sum-exp of the scaled,
    masked scores of each query row.
    """
    B, T, H, Dh = q.shape
    scale = 1.0 / np.sqrt(Dh)
    qh = q.transpose(0, 2, 1, 3)
    kh = k.transpose(0, 2, 1, 3)
    vh = v.transpose(0, 2, 1, 3)
    s = np.matmul(qh, kh.transpose(0, 1, 3, 2)) * scale
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    s = np.where(mask[None, None], -np.inf, s)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=-1, keepdims=True)
    p = e / z
    lse = (m + np.log(z))[..., 0]
    o = np.matmul(p, vh).transpose(0, 2, 1, 3)
    return o, p, lse


def causal_attention_backward(do, q, k, v, p):
    """Gradients of O = P v with P = softmax(S), S = q k^T / sqrt(Dh) (masked).

    dP = dO v^T; dv = P^T dO; dS = P * (dP - rowsum(P * dP));
    dq = dS k / sqrt(Dh); dk = dS^T q / sqrt(Dh).  All [B, T, H, Dh].
    """
    Dh = q.shape[-1]
    scale = 1.0 / np.sqrt(Dh)
    qh = q.transpose(0, 2, 1, 3)
    kh = k.transpose(0, 2, 1, 3)
    vh = v.transpose(0, 2, 1, 3)
    doh = do.transpose(0, 2, 1, 3)
    dp = np.matmul(doh, vh.transpose(0, 1, 3, 2))
    dv = np.matmul(p.transpose(0, 1, 3, 2), doh)
    ds = p * (dp - np.sum(p * dp, axis=-1, keepdims=True))
    dq = np.matmul(ds, kh) * scale
    dk = np.matmul(ds.transpose(0, 1, 3, 2), qh) * scale
    tr = (0, 2, 1, 3)
    return dq.transpose(tr), dk.transpose(tr), dv.transpose(tr)


# ---------------------------------------------------------------- model
def forward(params, cfg, tokens, targets, token_bytes):
    """Forward pass.  tokens, targets: int [B, T]; token_bytes: int [V].

    Returns (loss, bpb, cache) where cache holds what ``backward`` needs and
    the logits ``z`` [B*T, V].
    """
    p = [np.asarray(w, dtype=np.float64) for w in params]
    B, T = tokens.shape
    d, H, Dh = cfg.d_model, cfg.n_head, cfg.head_dim
    N = B * T
    tok = tokens.reshape(N)
    tgt = targets.reshape(N)
    cos, sin = rope_tables(T, Dh)

    x = p[0][tok]                                   # embedding lookup
    layers = []
    for l in range(cfg.depth):
        wq, wk, wv, wo, w1, w2 = p[1 + 6 * l: 7 + 6 * l]
        c = {}
        y1, r1 = rmsnorm(x)
        q = rope((y1 @ wq.T).reshape(B, T, H, Dh), cos, sin)
        k = rope((y1 @ wk.T).reshape(B, T, H, Dh), cos, sin)
        v = (y1 @ wv.T).reshape(B, T, H, Dh)
        o, P, lse = causal_attention(q, k, v)
        o = o.reshape(N, d)
        x = x + o @ wo.T
        y2, r2 = rmsnorm(x)
        h = y2 @ w1.T
        a = np.maximum(h, 0.0) ** 2
        x = x + a @ w2.T
        c.update(y1=y1, r1=r1, q=q, k=k, v=v, P=P, lse=lse, o=o,
                 y2=y2, r2=r2, h=h, a=a)
        layers.append(c)
    yf, rf = rmsnorm(x)
    z = yf @ p[-1].T
    zmax = np.max(z, axis=-1, keepdims=True)
    lse = (zmax + np.log(np.sum(np.exp(z - zmax), axis=-1, keepdims=True)))[:, 0]
    nll = lse - z[np.arange(N), tgt]
    loss = float(np.mean(nll))
    nbytes = np.asarray(token_bytes, dtype=np.int64)[tgt]
    bpb = float(np.sum(nll[nbytes > 0]) / (np.log(2.0) * np.sum(nbytes)))
    cache = dict(p=p, B=B, T=T, tok=tok, tgt=tgt, cos=cos, sin=sin,
                 layers=layers, yf=yf, rf=rf, z=z, lse=lse, nll=nll)
    return loss, bpb, cache


def backward(cache, cfg, grad_scale=1.0):
    """Exact gradients of grad_scale * mean(nll) w.r.t. every parameter."""
    p = cache["p"]
    B, T = cache["B"], cache["T"]
    d, H, Dh = cfg.d_model, cfg.n_head, cfg.head_dim
    N = B * T
    tgt = cache["tgt"]
    cos, sin = cache["cos"], cache["sin"]
    grads = [None] * len(p)

    # softmax cross-entropy: d nll_i / d z_i = softmax(z_i) - onehot(t_i)
    z = cache["z"]
    dz = np.exp(z - cache["lse"][:, None])
    dz[np.arange(N), tgt] -= 1.0
    dz *= grad_scale / N
    grads[-1] = dz.T @ cache["yf"]
    dyf = dz @ p[-1]
    dx = rmsnorm_backward(dyf, cache["yf"], cache["rf"])

    for l in reversed(range(cfg.depth)):
        wq, wk, wv, wo, w1, w2 = p[1 + 6 * l: 7 + 6 * l]
        c = cache["layers"][l]
        base = 1 + 6 * l
        # MLP block: x_out = x_mid + relu(h)^2 w2^T, h = y2 w1^T
        grads[base + 5] = dx.T @ c["a"]
        da = dx @ w2
        dh = da * 2.0 * np.maximum(c["h"], 0.0)
        grads[base + 4] = dh.T @ c["y2"]
        dy2 = dh @ w1
        dx = dx + rmsnorm_backward(dy2, c["y2"], c["r2"])
        # attention block: x_mid = x_in + o wo^T
        grads[base + 3] = dx.T @ c["o"]
        do = (dx @ wo).reshape(B, T, H, Dh)
        dqr, dkr, dv = causal_attention_backward(do, c["q"], c["k"], c["v"], c["P"])
        dq = rope_backward(dqr, cos, sin).reshape(N, d)
        dk = rope_backward(dkr, cos, sin).reshape(N, d)
        dv = dv.reshape(N, d)
        grads[base + 0] = dq.T @ c["y1"]
        grads[base + 1] = dk.T @ c["y1"]
        grads[base + 2] = dv.T @ c["y1"]
        dy1 = dq @ wq + dk @ wk + dv @ wv
        dx = dx + rmsnorm_backward(dy1, c["y1"], c["r1"])

    dwte = np.zeros_like(p[0])
    np.add.at(dwte, cache["tok"], dx)               # segment sum by token id
    grads[0] = dwte
    return grads


def loss_and_grads(params, cfg, tokens, targets, token_bytes, grad_scale=1.0):
    loss, bpb, cache = forward(params, cfg, tokens, targets, token_bytes)
    return loss, bpb, backward(cache, cfg, grad_scale)


def eval_sums(params, cfg, tokens, targets, token_bytes):
    """Evaluation pass of one batch (section 预搜检: validation bits per byte).

    Returns (sum nll, sum nll over targets with bytes > 0, sum bytes), so that
    bits per byte over several batches is the corpus ratio of sums,
    sums[1] / (ln 2 * sums[2]).
    """
    _, _, cache = forward(params, cfg, tokens, targets, token_bytes)
    nll = cache["nll"]
    nbytes = np.asarray(token_bytes, dtype=np.int64)[cache["tgt"]]
    return float(np.sum(nll)), float(np.sum(nll[nbytes > 0])), float(np.sum(nbytes))


def bpb_of_sums(sums):
    """Bits per byte from the running sums of ``eval_sums``."""
    return sums[1] / (np.log(2.0) * sums[2])

