"""Oracle: plain, slow, fp64 CPU implementation of one nanochat pretraining step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code, table or helper with the CUDA
path in ``pretraining_step_03_b300``.

What it computes follows the nanochat speedrun walkthrough (lyylswood.com),
section 预搜检 (pretraining): a Llama-like, bias-free decoder-only
transformer with parameter-free RMSNorm, next-token cross-entropy reported
as bits per byte, Muon for the 2-D block matrices and AdamW for the
embedding and unembedding.  Every reading the pages leave open is listed in
``model.py`` / ``optim.py`` next to the code that takes it.

Every function here is pinned by a ``-m "not gpu"`` test against something
other than itself (finite differences, closed forms, brute force, the SVD
spectral map); none is "parity unpinned".
"""

from .model import (  # noqa: F401
    Config,
    param_shapes,
    rmsnorm,
    rmsnorm_backward,
    rope_tables,
    rope,
    rope_backward,
    causal_attention,
    causal_attention_backward,
    forward,
    backward,
    loss_and_grads,
    eval_sums,
    bpb_of_sums,
)
from .optim import newton_schulz, muon_step, adamw_step  # noqa: F401
from . import schedule  # noqa: F401
from . import generate  # noqa: F401
