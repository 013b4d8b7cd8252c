"""ctypes binding of libnc.so: the C ABI functions under their own names.

Argument marshalling only -- every step of the computation runs in the
library's CUDA kernels.  Device pointers are passed as integers (e.g.
``tensor.data_ptr()``), streams as ``torch.cuda.Stream.cuda_stream`` or 0.
Each wrapper raises ``NcError`` when the C call returns a non-zero status.
"""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnc.so")

NC_OK, NC_ERR_ARG, NC_ERR_CUDA, NC_ERR_OOM, NC_ERR_DEVICE_FLAG, NC_ERR_TIMEOUT, NC_ERR_UNSUPPORTED = range(7)
NC_BF16, NC_FP32 = 0, 1
NC_KIND_EMB, NC_KIND_MATRIX, NC_KIND_UNEMB = 0, 1, 2
NC_STATE_MOMENTUM, NC_STATE_ADAM_M, NC_STATE_ADAM_V = 0, 1, 2
NC_FLAG_TOKEN_RANGE, NC_FLAG_NONFINITE, NC_FLAG_TIMEOUT, NC_FLAG_SMEM_ALIGN = 1, 2, 4, 8
PROF_NAMES = ["gemm", "attn_fwd", "attn_bwd", "norm", "rope", "ce", "embed", "muon_ns", "muon_elem",
              "adamw"]


class NcError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libnc error {code}: {msg}")
        self.code = code


_V, _I, _F, _SZ, _U64, _L = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                             ctypes.c_uint64, ctypes.c_long)

# name -> (restype, argtypes)
SIGNATURES = {
    "nc_last_error": (ctypes.c_char_p, []),
    "nc_launch_count": (_U64, []),
    "nc_arena_bytes": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "nc_init_model": (_I, [_I, _I, _I, _I, _U64, _V, _SZ, _I, _I, _I, _V, ctypes.POINTER(_V)]),
    "nc_free": (_I, [_V]),
    "nc_num_params": (_I, [_V, ctypes.POINTER(_I)]),
    "nc_param_info": (_I, [_V, _I, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "nc_forward_backward": (_I, [_V, _V, _V, _V, _I, _I, _I, _F, _V]),
    "nc_eval_loss": (_I, [_V, _V, _V, _V, _I, _I, _I, _V, _V]),
    "nc_lr_schedule": (_I, [_I, _I, _F, _I, _I, ctypes.POINTER(_F), ctypes.POINTER(_F)]),
    "nc_kv_cache_bytes": (_I, [_V, _I, _I, ctypes.POINTER(_SZ)]),
    "nc_prefill": (_I, [_V, _V, _I, _I, _V, _I, _I, _V, _V]),
    "nc_decode_step": (_I, [_V, _V, _I, _I, _V, _I, _I, _V, _V]),
    "nc_decode_graphs": (_I, [_V, _I]),
    "nc_muon_step": (_I, [_V, _F, _F, _I, _I, ctypes.POINTER(_F)]),
    "nc_adamw_step": (_I, [_V, _F, _F, _F, _F, _F, _F, _I]),
    "nc_train_step": (_I, [_V, _V, _V, _V, _I, _I, _I, _F, _F, _I, ctypes.POINTER(_F), _F, _F, _F,
                           _F, _F, _F, _I, ctypes.POINTER(_F)]),
    "nc_get_params": (_I, [_V, _I, _V, _SZ]),
    "nc_set_params": (_I, [_V, _I, _V, _SZ]),
    "nc_get_grads": (_I, [_V, _I, _V, _SZ]),
    "nc_set_grads": (_I, [_V, _I, _V, _SZ]),
    "nc_get_state": (_I, [_V, _I, _I, _V, _SZ]),
    "nc_set_state": (_I, [_V, _I, _I, _V, _SZ]),
    "nc_check_device_flag": (_I, [_V, ctypes.POINTER(ctypes.c_uint32)]),
    "nc_check_kernel_flag": (_I, [_V, ctypes.POINTER(ctypes.c_uint32)]),
    "nc_selftest_wait_timeout": (_I, [_V]),
    "nc_attention_forward": (_I, [_V, _V, _V, _I, _V, _I, _V, _I, _I, _I, _I, _I, _V]),
    "nc_attention_workspace_bytes": (_SZ, [_I, _I, _I]),
    "nc_attention_backward": (_I, [_V, _V, _V, _I, _V, _V, _I, _V, _V, _V, _V, _I, _V, _I, _I, _I,
                                   _I, _I, _V]),
    "nc_attention_backward_noalloc": (_I, [_V, _V, _V, _I, _V, _V, _I, _V, _V, _V, _V, _I, _I, _I, _I,
                                           _I, _I, _V]),
    "nc_profile": (_I, [_V, _I]),
    "nc_profile_read": (_I, [_V, _I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_L),
                             ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
    "nc_gemm_bf16": (_I, [_I, _I, _I, _I, _V, _L, _L, _I, _V, _L, _L, _I, _V, _L, _L, _I, _F, _F,
                          _V, _SZ, _V]),
}

_lib = None


def lib():
    """Loads libnc.so (built in-tree by ``python -m pretraining_step_03_b300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run python -m pretraining_step_03_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc):
    if rc != NC_OK:
        raise NcError(rc, lib().nc_last_error().decode(errors="replace"))


def _f3(v):
    return (ctypes.c_float * 3)(*[float(x) for x in v])


def nc_last_error():
    return lib().nc_last_error().decode(errors="replace")


def nc_launch_count():
    return int(lib().nc_launch_count())


def nc_arena_bytes(depth, d_model, n_head, vocab, max_B, max_T, dtype):
    out = ctypes.c_size_t(0)
    _check(lib().nc_arena_bytes(depth, d_model, n_head, vocab, max_B, max_T, dtype, ctypes.byref(out)))
    return out.value


def nc_init_model(depth, d_model, n_head, vocab, seed, arena, arena_bytes, dtype, max_B, max_T, stream):
    h = ctypes.c_void_p()
    _check(lib().nc_init_model(depth, d_model, n_head, vocab, seed, arena, arena_bytes, dtype, max_B,
                               max_T, stream, ctypes.byref(h)))
    return h


def nc_free(m):
    _check(lib().nc_free(m))


def nc_num_params(m):
    n = ctypes.c_int()
    _check(lib().nc_num_params(m, ctypes.byref(n)))
    return n.value


def nc_param_info(m, index):
    r, c, k = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().nc_param_info(m, index, ctypes.byref(r), ctypes.byref(c), ctypes.byref(k)))
    return r.value, c.value, k.value


def nc_forward_backward(m, tokens, targets, token_bytes, B, T, accumulate, grad_scale, loss_bpb_out):
    _check(lib().nc_forward_backward(m, tokens, targets, token_bytes, B, T, accumulate, grad_scale,
                                     loss_bpb_out))


def nc_eval_loss(m, tokens, targets, token_bytes, B, T, accumulate, sums, loss_bpb_out):
    _check(lib().nc_eval_loss(m, tokens, targets, token_bytes, B, T, accumulate, sums, loss_bpb_out))


def nc_kv_cache_bytes(m, cache_B, cache_T):
    n = ctypes.c_size_t()
    _check(lib().nc_kv_cache_bytes(m, cache_B, cache_T, ctypes.byref(n)))
    return n.value


def nc_prefill(m, cache, cache_B, cache_T, tokens, B, T0, logits_out, next_out):
    _check(lib().nc_prefill(m, cache, cache_B, cache_T, tokens, B, T0, logits_out, next_out))


def nc_decode_step(m, cache, cache_B, cache_T, tokens, B, pos, logits_out, next_out):
    _check(lib().nc_decode_step(m, cache, cache_B, cache_T, tokens, B, pos, logits_out, next_out))


def nc_decode_graphs(m, enable):
    _check(lib().nc_decode_graphs(m, enable))


def nc_lr_schedule(step, n_steps, warmdown_frac, d_model, d_ref, base):
    """Returns (muon_lr, lr_emb, lr_unemb) of optimizer step `step` (0-based)."""
    out = (ctypes.c_float * 3)()
    _check(lib().nc_lr_schedule(step, n_steps, warmdown_frac, d_model, d_ref, _f3(base), out))
    return tuple(float(x) for x in out)


def nc_muon_step(m, lr, momentum, nesterov, ns_steps, ns_coef):
    _check(lib().nc_muon_step(m, lr, momentum, nesterov, ns_steps, _f3(ns_coef)))


def nc_adamw_step(m, lr_emb, lr_unemb, beta1, beta2, eps, weight_decay, step):
    _check(lib().nc_adamw_step(m, lr_emb, lr_unemb, beta1, beta2, eps, weight_decay, step))


def nc_train_step(m, tokens_host, targets_host, token_bytes, B, T, n_micro, muon_lr, muon_momentum,
                  ns_steps, ns_coef, lr_emb, lr_unemb, beta1, beta2, eps, weight_decay, adam_step,
                  loss_bpb_host):
    _check(lib().nc_train_step(m, tokens_host, targets_host, token_bytes, B, T, n_micro, muon_lr,
                               muon_momentum, ns_steps, _f3(ns_coef), lr_emb, lr_unemb, beta1, beta2,
                               eps, weight_decay, adam_step,
                               ctypes.cast(loss_bpb_host, ctypes.POINTER(ctypes.c_float))))


def _host_io(fn, m, index, host, n, *extra):
    _check(getattr(lib(), fn)(m, index, *extra, host, n))


def nc_get_params(m, index, host, n):
    _host_io("nc_get_params", m, index, host, n)


def nc_set_params(m, index, host, n):
    _host_io("nc_set_params", m, index, host, n)


def nc_get_grads(m, index, host, n):
    _host_io("nc_get_grads", m, index, host, n)


def nc_set_grads(m, index, host, n):
    _host_io("nc_set_grads", m, index, host, n)


def nc_get_state(m, index, slot, host, n):
    _host_io("nc_get_state", m, index, host, n, slot)


def nc_set_state(m, index, slot, host, n):
    _host_io("nc_set_state", m, index, host, n, slot)


def nc_check_device_flag(m):
    """Returns the flag bits (0 when clean); never raises for a set flag."""
    f = ctypes.c_uint32(0)
    rc = lib().nc_check_device_flag(m, ctypes.byref(f))
    if rc not in (NC_OK, NC_ERR_DEVICE_FLAG):
        _check(rc)
    return f.value


def nc_selftest_wait_timeout(stream):
    _check(lib().nc_selftest_wait_timeout(stream))


def nc_check_kernel_flag(stream):
    """Flag bits of the kernel-level entry points on the current device (0 when clean)."""
    f = ctypes.c_uint32(0)
    rc = lib().nc_check_kernel_flag(stream, ctypes.byref(f))
    if rc not in (NC_OK, NC_ERR_DEVICE_FLAG):
        _check(rc)
    return f.value


def nc_attention_forward(q, k, v, ld_qkv, o, ld_o, lse, B, T, H, D, dtype, stream):
    _check(lib().nc_attention_forward(q, k, v, ld_qkv, o, ld_o, lse, B, T, H, D, dtype, stream))


def nc_attention_workspace_bytes(B, T, H):
    return int(lib().nc_attention_workspace_bytes(B, T, H))


def nc_attention_backward(q, k, v, ld_qkv, o, dout, ld_o, lse, dq, dk, dv, ld_dqkv, workspace, B, T, H,
                          D, dtype, stream):
    _check(lib().nc_attention_backward(q, k, v, ld_qkv, o, dout, ld_o, lse, dq, dk, dv, ld_dqkv,
                                       workspace, B, T, H, D, dtype, stream))


def nc_attention_backward_noalloc(q, k, v, ld_qkv, o, dout, ld_o, lse, dq, dk, dv, ld_dqkv, B, T, H, D,
                                  dtype, stream):
    _check(lib().nc_attention_backward_noalloc(q, k, v, ld_qkv, o, dout, ld_o, lse, dq, dk, dv, ld_dqkv,
                                               B, T, H, D, dtype, stream))


def nc_gemm_bf16(M, N, K, batch, A, lda, stride_a, trans_a, B, ldb, stride_b, trans_b, C, ldc, stride_c,
                 c_dtype, alpha, beta, workspace, workspace_bytes, stream):
    _check(lib().nc_gemm_bf16(M, N, K, batch, A, lda, stride_a, trans_a, B, ldb, stride_b, trans_b, C,
                              ldc, stride_c, c_dtype, alpha, beta, workspace, workspace_bytes, stream))


def nc_profile(m, enable):
    _check(lib().nc_profile(m, int(enable)))


def nc_profile_read(m, category):
    """-> (device ms, launch sites, algorithmic FLOPs, algorithmic bytes) for one kernel class."""
    ms, n, fl, by = ctypes.c_double(), ctypes.c_long(), ctypes.c_double(), ctypes.c_double()
    _check(lib().nc_profile_read(m, category, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(fl),
                                 ctypes.byref(by)))
    return ms.value, n.value, fl.value, by.value
