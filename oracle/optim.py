"""fp64 Muon (Newton-Schulz orthogonalised momentum) and AdamW.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: nanochat speedrun walkthrough (lyylswood.com), section 预搜检
(pretraining): Muon optimises the 2-D matrices, AdamW the embedding and
unembedding; no other trainable parameters.  The Newton-Schulz quintic
coefficients (3.4445, -4.7750, 2.0315) and 5 iterations are the optimizer
microbenchmark's workload definition.

Readings where the pages are silent:
  * Muon: buf <- mu*buf + g; Nesterov g' = g + mu*buf (mu = 0.95 by default);
    X0 = g' / (||g'||_F + 1e-7); iterate in the wide orientation
    (transpose when rows > cols): A = X X^T, B = b A + c A A, X = a X + B X;
    W <- W - lr * sqrt(max(1, rows/cols)) * X; no weight decay.
  * AdamW: m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2; bias-corrected
    m_hat = m/(1-b1^t), v_hat = v/(1-b2^t); decoupled decay
    W <- W (1 - lr*wd) - lr * m_hat / (sqrt(v_hat) + eps).
"""

import numpy as np

NS_COEFS = (3.4445, -4.7750, 2.0315)
NORM_EPS = 1e-7


def newton_schulz(g, steps=5, coefs=NS_COEFS):
    """Approximate orthogonalisation of g by the quintic Newton-Schulz map."""
    a, b, c = coefs
    x = np.asarray(g, dtype=np.float64)
    x = x / (np.linalg.norm(x) + NORM_EPS)
    tall = x.shape[0] > x.shape[1]
    if tall:
        x = x.T
    for _ in range(steps):
        A = x @ x.T
        Bm = b * A + c * (A @ A)
        x = a * x + Bm @ x
    return x.T if tall else x


def muon_step(w, g, buf, lr, momentum=0.95, nesterov=True, ns_steps=5,
              coefs=NS_COEFS):
    """One Muon update of one matrix.  Returns (w_new, buf_new, X)."""
    w = np.asarray(w, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    buf = momentum * np.asarray(buf, dtype=np.float64) + g
    geff = g + momentum * buf if nesterov else buf
    x = newton_schulz(geff, ns_steps, coefs)
    rows, cols = w.shape
    scale = np.sqrt(max(1.0, rows / cols))
    return w - lr * scale * x, buf, x


def adamw_step(w, g, m, v, lr, beta1=0.9, beta2=0.95, eps=1e-8,
               weight_decay=0.0, step=1):
    """One AdamW update (1-based ``step``).  Returns (w_new, m_new, v_new)."""
    w = np.asarray(w, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** step)
    vhat = v / (1.0 - beta2 ** step)
    w = w * (1.0 - lr * weight_decay) - lr * mhat / (np.sqrt(vhat) + eps)
    return w, m, v
