"""Learning-rate schedule of the pretraining run, as plain definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: nanochat speedrun walkthrough (lyylswood.com), section 预搜检:
  * the optimizer step takes 32 x 2048 = 524,288 tokens; the Chinchilla
    advice of 20 training tokens per parameter gives 560M x 20 ~ 11.2B
    tokens, i.e. ~21,400 steps;
  * the learning rate scales automatically as 1/sqrt(dim): larger models
    prefer smaller rates;
  * lrm is the learning-rate multiplier that falls linearly to 0 near the
    end of training.

Readings where the pages stop short (also listed in the design notes):
  * "near the end" = the last W = round(warmdown_frac * n_steps) of the
    n_steps optimizer steps; before them lrm = 1; step s of the warm-down
    has lrm = (n_steps - s) / W, which is 1 where it starts and reaches 0 at
    s = n_steps, one step past the last;
  * "1/sqrt(dim)" applies to the AdamW rates (embedding and unembedding) as
    a factor sqrt(d_ref / d_model) on rates given at a reference width
    d_ref; the Muon rate is not width-scaled, since the orthogonalised
    update and its sqrt(max(1, rows/cols)) factor already fix its size.
"""

import math


def chinchilla_steps(n_params, tokens_per_step, tokens_per_param=20):
    """Optimizer steps for tokens_per_param training tokens per parameter."""
    return round(tokens_per_param * n_params / tokens_per_step)


def lrm(step, n_steps, warmdown_frac):
    """Learning-rate multiplier of 0-based optimizer step ``step``."""
    assert 0 <= step < n_steps and 0.0 <= warmdown_frac <= 1.0
    w = round(warmdown_frac * n_steps)
    if w == 0 or step < n_steps - w:
        return 1.0
    return (n_steps - step) / w


def learning_rates(step, n_steps, warmdown_frac, d_model, d_ref, base):
    """(Muon, embedding AdamW, unembedding AdamW) rates; ``base`` at width d_ref."""
    m = lrm(step, n_steps, warmdown_frac)
    width = math.sqrt(d_ref / d_model)
    return m * base[0], m * base[1] * width, m * base[2] * width
