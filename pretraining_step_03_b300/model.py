"""Convenience wrapper over the C ABI: one model in a torch-allocated arena.

PyTorch only provides the device memory (the arena and small I/O tensors)
and the stream; every computation runs in libnc's CUDA kernels.
"""

import numpy as np

from . import _lib as L

NS_COEFS = (3.4445, -4.7750, 2.0315)


class Model:
    def __init__(self, depth, d_model, n_head, vocab, max_B, max_T, dtype="bf16", seed=0,
                 device="cuda"):
        import torch

        self.torch = torch
        self.dtype = L.NC_BF16 if dtype == "bf16" else L.NC_FP32
        self.depth, self.d_model, self.n_head, self.vocab = depth, d_model, n_head, vocab
        self.max_B, self.max_T = max_B, max_T
        self.device = torch.device(device)
        self.arena_bytes = L.nc_arena_bytes(depth, d_model, n_head, vocab, max_B, max_T, self.dtype)
        self.arena = torch.empty(self.arena_bytes, dtype=torch.uint8, device=self.device)
        self.stream = torch.cuda.current_stream(self.device).cuda_stream
        self.h = L.nc_init_model(depth, d_model, n_head, vocab, seed, self.arena.data_ptr(),
                                 self.arena_bytes, self.dtype, max_B, max_T, self.stream)
        self.n_params = L.nc_num_params(self.h)
        self.shapes = [L.nc_param_info(self.h, i)[:2] for i in range(self.n_params)]
        self.loss_buf = torch.zeros(2, dtype=torch.float32, device=self.device)

    # ---------------------------------------------------------------- host I/O
    def _get(self, fn, i):
        r, c = self.shapes[i]
        out = np.empty((r, c), dtype=np.float32)
        fn(self.h, i, out.ctypes.data, out.size)
        return out

    def get_param(self, i):
        return self._get(L.nc_get_params, i)

    def get_grad(self, i):
        return self._get(L.nc_get_grads, i)

    def get_state(self, i, slot):
        r, c = self.shapes[i]
        out = np.empty((r, c), dtype=np.float32)
        L.nc_get_state(self.h, i, slot, out.ctypes.data, out.size)
        return out

    def set_param(self, i, a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        assert a.shape == tuple(self.shapes[i]), (a.shape, self.shapes[i])
        L.nc_set_params(self.h, i, a.ctypes.data, a.size)

    def set_grad(self, i, a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        assert a.shape == tuple(self.shapes[i])
        L.nc_set_grads(self.h, i, a.ctypes.data, a.size)

    def set_state(self, i, slot, a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        L.nc_set_state(self.h, i, slot, a.ctypes.data, a.size)

    def set_params(self, params):
        for i, p in enumerate(params):
            self.set_param(i, p)

    # ---------------------------------------------------------------- the step
    def device_i32(self, a):
        return self.torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32).reshape(-1)).to(self.device)

    def forward_backward(self, tokens, targets, token_bytes, B, T, accumulate=0, grad_scale=1.0,
                         out=None):
        """tokens/targets/token_bytes: device int32 tensors.  Returns the device {loss, bpb} tensor."""
        out = self.loss_buf if out is None else out
        L.nc_forward_backward(self.h, tokens.data_ptr(), targets.data_ptr(), token_bytes.data_ptr(), B, T,
                              accumulate, grad_scale, out.data_ptr())
        return out

    def eval_loss(self, tokens, targets, token_bytes, B, T, accumulate=0, sums=None, out=None):
        """Forward and loss only.  Returns the device double[3] running sums
        {sum nll, sum nll over byte-counted targets, sum bytes}; ``out`` (device
        float[2], optional) receives this batch's {loss, bpb}."""
        if sums is None:
            sums = self.torch.zeros(3, dtype=self.torch.float64, device=self.device)
        L.nc_eval_loss(self.h, tokens.data_ptr(), targets.data_ptr(), token_bytes.data_ptr(), B, T,
                       accumulate, sums.data_ptr(), 0 if out is None else out.data_ptr())
        return sums

    # ---------------------------------------------------------------- inference
    def kv_cache(self, cache_B, cache_T):
        """A device KV cache for cache_B sequences of up to cache_T positions."""
        n = L.nc_kv_cache_bytes(self.h, cache_B, cache_T)
        return KVCache(self.torch.empty(n, dtype=self.torch.uint8, device=self.device), cache_B, cache_T)

    def prefill(self, cache, tokens, B, T0, logits=None, next_tok=None):
        """tokens: device int32 [B*T0].  Fills positions 0..T0-1 of cache rows 0..B-1."""
        L.nc_prefill(self.h, cache.buf.data_ptr(), cache.B, cache.T, tokens.data_ptr(), B, T0,
                     0 if logits is None else logits.data_ptr(), 0 if next_tok is None else next_tok.data_ptr())

    def decode_step(self, cache, tokens, B, pos, logits=None, next_tok=None):
        """tokens: device int32 [B], the tokens at position pos."""
        L.nc_decode_step(self.h, cache.buf.data_ptr(), cache.B, cache.T, tokens.data_ptr(), B, pos,
                         0 if logits is None else logits.data_ptr(), 0 if next_tok is None else next_tok.data_ptr())

    def generate(self, cache, prompt, n_new):
        """Greedy continuation of B equal-length prompts (device int32 [B, T0]) by n_new
        tokens; returns the device int32 [n_new, B] tokens (step-major).  The steps take
        their input from and write their output to two fixed buffers in turn, so from the
        third token on each step is a replay of a recorded graph."""
        torch = self.torch
        B, T0 = prompt.shape
        out = torch.empty(n_new, B, dtype=torch.int32, device=self.device)
        buf = [torch.empty(B, dtype=torch.int32, device=self.device) for _ in range(2)]
        self.prefill(cache, prompt.reshape(-1).contiguous(), B, T0, next_tok=buf[0])
        out[0].copy_(buf[0])
        for i in range(1, n_new):
            self.decode_step(cache, buf[(i - 1) % 2], B, T0 + i - 1, next_tok=buf[i % 2])
            out[i].copy_(buf[i % 2])
        return out

    def decode_graphs(self, enable):
        L.nc_decode_graphs(self.h, int(enable))

    def muon_step(self, lr, momentum=0.95, nesterov=True, ns_steps=5, coefs=NS_COEFS):
        L.nc_muon_step(self.h, lr, momentum, int(nesterov), ns_steps, coefs)

    def adamw_step(self, lr_emb, lr_unemb, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0, step=1):
        L.nc_adamw_step(self.h, lr_emb, lr_unemb, beta1, beta2, eps, weight_decay, step)

    def train_step(self, tokens_host, targets_host, token_bytes, B, T, n_micro, muon_lr, lr_emb,
                   lr_unemb, step, momentum=0.95, ns_steps=5, coefs=NS_COEFS, beta1=0.9, beta2=0.95,
                   eps=1e-8, weight_decay=0.0):
        """Whole optimizer step from host int32 arrays (pinned torch tensors or numpy)."""
        out = np.zeros(2, dtype=np.float32)
        tp = tokens_host.data_ptr() if hasattr(tokens_host, "data_ptr") else tokens_host.ctypes.data
        gp = targets_host.data_ptr() if hasattr(targets_host, "data_ptr") else targets_host.ctypes.data
        L.nc_train_step(self.h, tp, gp, token_bytes.data_ptr(), B, T, n_micro, muon_lr, momentum, ns_steps,
                        coefs, lr_emb, lr_unemb, beta1, beta2, eps, weight_decay, step, out.ctypes.data)
        return float(out[0]), float(out[1])

    def check_flag(self):
        return L.nc_check_device_flag(self.h)

    def close(self):
        if self.h is not None:
            L.nc_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KVCache:
    """Device buffer of a KV cache and its geometry (see nc_kv_cache_bytes)."""

    def __init__(self, buf, B, T):
        self.buf, self.B, self.T = buf, B, T

