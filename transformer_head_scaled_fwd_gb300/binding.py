"""Thin ctypes binding of ``libmha.so`` (the C ABI in ``include/mha.h``).

Argument marshalling only: tensors are passed as raw pointers, every step of
the forward pass runs in the library's CUDA kernels. There is no fallback:
if the library is missing or a call fails, an exception is raised.

Function names match the C entry points: ``mha_forward``,
``mha_qkv_projection``, ``mha_attention_core``, ``mha_output_projection``,
``mha_forward_host``, ``mha_workspace_size``, ``mha_host_staging_size``,
``mha_check_device_status``.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmha.so")

MHA_OK, MHA_ERR_INVALID_ARG, MHA_ERR_UNSUPPORTED, MHA_ERR_CUDA = 0, 1, 2, 3
MHA_F32, MHA_BF16 = 0, 1

# every symbol include/mha.h declares
EXPORTS = ("mha_workspace_size", "mha_forward", "mha_qkv_projection", "mha_attention_core",
           "mha_output_projection", "mha_host_staging_size", "mha_forward_host", "mha_last_error",
           "mha_check_device_status", "mha_version", "mha_forward_noalloc", "mha_ffn_workspace_size",
           "mha_ffn_forward", "mha_sublayer_workspace_size", "mha_sublayer_forward",
           "mha_decode_workspace_size", "mha_kv_cache_prefill", "mha_decode_step",
           "mha_selftest_wait_timeout")
MHA_SELFTEST_WAIT_CODE = 0x7f1


class MHAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"status {status}: {message}")
        self.status = status


class MaskT(ctypes.Structure):
    _fields_ = [("causal", ctypes.c_int), ("key_valid_lens", ctypes.c_void_p),
                ("dense", ctypes.c_void_p), ("dense_mq", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libmha.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} not found: build it with transformer_head_scaled_fwd_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.mha_workspace_size.restype = sz
        lib.mha_workspace_size.argtypes = [i] * 6
        lib.mha_forward.restype = i
        lib.mha_forward.argtypes = [i] + [vp] * 11 + [i] * 5 + [ctypes.POINTER(MaskT), vp, vp, vp, sz, vp]
        lib.mha_qkv_projection.restype = i
        lib.mha_qkv_projection.argtypes = [i] + [vp] * 9 + [i] * 5 + [vp, sz, vp]
        lib.mha_attention_core.restype = i
        lib.mha_attention_core.argtypes = [i] * 6 + [ctypes.POINTER(MaskT), vp, vp, sz, vp]
        lib.mha_output_projection.restype = i
        lib.mha_output_projection.argtypes = [i, vp, vp] + [i] * 5 + [vp, vp, sz, vp]
        lib.mha_host_staging_size.restype = sz
        lib.mha_host_staging_size.argtypes = [i] * 7
        lib.mha_forward_host.restype = i
        lib.mha_forward_host.argtypes = ([i] + [vp] * 11 + [i] * 5
                                         + [ctypes.POINTER(MaskT), vp, vp, sz, vp, sz, vp])
        lib.mha_last_error.restype = ctypes.c_char_p
        lib.mha_last_error.argtypes = []
        lib.mha_check_device_status.restype = i
        lib.mha_check_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), i]
        lib.mha_version.restype = ctypes.c_char_p
        lib.mha_version.argtypes = []
        lib.mha_ffn_workspace_size.restype = sz
        lib.mha_ffn_workspace_size.argtypes = [i] * 5
        lib.mha_ffn_forward.restype = i
        lib.mha_ffn_forward.argtypes = [i] + [vp] * 5 + [i] * 4 + [vp, vp, sz, vp]
        lib.mha_sublayer_workspace_size.restype = sz
        lib.mha_sublayer_workspace_size.argtypes = [i] * 6
        lib.mha_sublayer_forward.restype = i
        lib.mha_sublayer_forward.argtypes = ([i, vp, vp, vp, vp, ctypes.c_float, i] + [vp] * 8 + [i] * 5
                                             + [ctypes.POINTER(MaskT), vp, vp, sz, vp])
        lib.mha_decode_workspace_size.restype = sz
        lib.mha_decode_workspace_size.argtypes = [i] * 4
        lib.mha_kv_cache_prefill.restype = i
        lib.mha_kv_cache_prefill.argtypes = [i] + [vp] * 5 + [i] * 4 + [vp, vp, i, vp]
        lib.mha_decode_step.restype = i
        lib.mha_decode_step.argtypes = [i] + [vp] * 9 + [i] * 3 + [vp, vp, vp, i, vp, vp, sz, vp]
        lib.mha_selftest_wait_timeout.restype = i
        lib.mha_selftest_wait_timeout.argtypes = [vp]
        lib.mha_forward_noalloc.restype = i
        lib.mha_forward_noalloc.argtypes = [i] + [vp] * 11 + [i] * 5 + [ctypes.POINTER(MaskT), vp, vp, vp]
        _lib = lib
        return lib


def _check(status: int):
    if status != MHA_OK:
        raise MHAError(status, load().mha_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return MHA_BF16
    if t.dtype == torch.float32:
        return MHA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_mask(causal=False, key_valid_lens=None, dense=None):
    """Build the C mask struct. The struct holds references to the two tensors, so
    they stay allocated for as long as the struct is alive."""
    if not causal and key_valid_lens is None and dense is None:
        return None
    m = MaskT()
    m.causal = int(bool(causal))
    m.key_valid_lens = _ptr(key_valid_lens)
    m.dense = _ptr(dense)
    m.dense_mq = int(dense.shape[1]) if dense is not None else 0
    m._tensors = (key_valid_lens, dense)
    return m


def workspace_size(dt: int, B: int, Lq: int, Lk: int, d_model: int, h: int) -> int:
    return int(load().mha_workspace_size(dt, B, Lq, Lk, d_model, h))


def mha_forward(query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, h, *, out, workspace,
                mask=None, p_attn=None, stream=None):
    """Enqueue the whole sublayer on ``stream``. All tensors are CUDA tensors."""
    B, Lq, d = query.shape
    Lk = key.shape[1]
    _check(load().mha_forward(
        _dtype_code(query), _ptr(query), _ptr(key), _ptr(value), _ptr(w_q), _ptr(b_q), _ptr(w_k),
        _ptr(b_k), _ptr(w_v), _ptr(b_v), _ptr(w_o), _ptr(b_o), B, Lq, Lk, d, h,
        ctypes.byref(mask) if mask is not None else None, _ptr(out), _ptr(p_attn), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def mha_qkv_projection(query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, h, *, workspace, stream=None):
    B, Lq, d = query.shape
    Lk = key.shape[1]
    _check(load().mha_qkv_projection(
        _dtype_code(query), _ptr(query), _ptr(key), _ptr(value), _ptr(w_q), _ptr(b_q), _ptr(w_k),
        _ptr(b_k), _ptr(w_v), _ptr(b_v), B, Lq, Lk, d, h, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def mha_attention_core(dt: int, B, Lq, Lk, d_model, h, *, workspace, mask=None, p_attn=None, stream=None):
    _check(load().mha_attention_core(
        dt, B, Lq, Lk, d_model, h, ctypes.byref(mask) if mask is not None else None, _ptr(p_attn),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def mha_output_projection(w_o, b_o, B, Lq, Lk, h, *, out, workspace, stream=None):
    d = w_o.shape[0]
    _check(load().mha_output_projection(
        _dtype_code(w_o), _ptr(w_o), _ptr(b_o), B, Lq, Lk, d, h, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def host_staging_size(dt: int, B, Lq, Lk, d_model, kv_distinct: bool, q_distinct: bool) -> int:
    return int(load().mha_host_staging_size(dt, B, Lq, Lk, d_model, int(kv_distinct), int(q_distinct)))


def mha_forward_host(h_query, h_key, h_value, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, h, *, h_out,
                     staging, workspace, mask=None, stream=None):
    """Host activations (pinned CPU tensors) in and out; weights and workspace on the device."""
    B, Lq, d = h_query.shape
    Lk = h_key.shape[1]
    _check(load().mha_forward_host(
        _dtype_code(h_query), _ptr(h_query), _ptr(h_key), _ptr(h_value), _ptr(w_q), _ptr(b_q),
        _ptr(w_k), _ptr(b_k), _ptr(w_v), _ptr(b_v), _ptr(w_o), _ptr(b_o), B, Lq, Lk, d, h,
        ctypes.byref(mask) if mask is not None else None, _ptr(h_out), _ptr(staging),
        staging.numel() * staging.element_size(), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def mha_forward_noalloc(query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, h, *, out,
                        mask=None, p_attn=None, stream=None):
    """mha_forward without a workspace: uses the library's fixed scratch (see include/mha.h)."""
    B, Lq, d = query.shape
    Lk = key.shape[1]
    _check(load().mha_forward_noalloc(
        _dtype_code(query), _ptr(query), _ptr(key), _ptr(value), _ptr(w_q), _ptr(b_q), _ptr(w_k),
        _ptr(b_k), _ptr(w_v), _ptr(b_v), _ptr(w_o), _ptr(b_o), B, Lq, Lk, d, h,
        ctypes.byref(mask) if mask is not None else None, _ptr(out), _ptr(p_attn), _stream(stream)))


def decode_workspace_size(B: int, d_model: int, h: int, L_max: int) -> int:
    return int(load().mha_decode_workspace_size(B, d_model, h, L_max))


def mha_kv_cache_prefill(x, w_k, b_k, w_v, b_v, h, *, k_cache, v_cache, stream=None):
    """Project x [B, T, d_model] into positions 0..T-1 of the caches [B, h, L_max, 64]."""
    B, T, d = x.shape
    _check(load().mha_kv_cache_prefill(
        _dtype_code(x), _ptr(x), _ptr(w_k), _ptr(b_k), _ptr(w_v), _ptr(b_v), B, T, d, h, _ptr(k_cache),
        _ptr(v_cache), k_cache.shape[2], _stream(stream)))


def mha_decode_step(x_new, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, h, *, k_cache, v_cache, cache_len, out,
                    workspace, stream=None):
    """One decoding step: x_new [B, d_model] -> out [B, d_model]; appends to the caches, bumps cache_len."""
    B, d = x_new.shape
    _check(load().mha_decode_step(
        _dtype_code(x_new), _ptr(x_new), _ptr(w_q), _ptr(b_q), _ptr(w_k), _ptr(b_k), _ptr(w_v), _ptr(b_v),
        _ptr(w_o), _ptr(b_o), B, d, h, _ptr(k_cache), _ptr(v_cache), _ptr(cache_len), k_cache.shape[2],
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


LN_UNBIASED_STD, LN_TORCH = 0, 1


def sublayer_workspace_size(dt: int, B: int, L: int, L_mem: int, d_model: int, h: int) -> int:
    return int(load().mha_sublayer_workspace_size(dt, B, L, L_mem, d_model, h))


def mha_sublayer_forward(x, ln_gain, ln_bias, ln_eps, ln_kind, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, h, *,
                         out, workspace, memory=None, mask=None, stream=None):
    """out = x + MHA(LayerNorm(x), kv, kv, mask), kv = LayerNorm(x) or memory (CUDA tensors)."""
    B, L, d = x.shape
    L_mem = memory.shape[1] if memory is not None else 0
    _check(load().mha_sublayer_forward(
        _dtype_code(x), _ptr(x), _ptr(memory), _ptr(ln_gain), _ptr(ln_bias), float(ln_eps), int(ln_kind),
        _ptr(w_q), _ptr(b_q), _ptr(w_k), _ptr(b_k), _ptr(w_v), _ptr(b_v), _ptr(w_o), _ptr(b_o), B, L, L_mem, d, h,
        ctypes.byref(mask) if mask is not None else None, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def ffn_workspace_size(dt: int, B: int, L: int, d_model: int, d_ff: int) -> int:
    return int(load().mha_ffn_workspace_size(dt, B, L, d_model, d_ff))


def mha_ffn_forward(x, w_1, b_1, w_2, b_2, *, out, workspace, stream=None):
    """Position-wise FFN: out = max(0, x W_1^T + b_1) W_2^T + b_2 (CUDA tensors)."""
    B, L, d = x.shape
    d_ff = w_1.shape[0]
    _check(load().mha_ffn_forward(
        _dtype_code(x), _ptr(x), _ptr(w_1), _ptr(b_1), _ptr(w_2), _ptr(b_2), B, L, d, d_ff, _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def mha_selftest_wait_timeout(stream=None):
    """Enqueue the diagnostic kernel whose bounded pipeline wait runs out (it records
    MHA_SELFTEST_WAIT_CODE in the device status word)."""
    _check(load().mha_selftest_wait_timeout(_stream(stream)))


def mha_check_device_status(reset: bool = True) -> int:
    """Synchronise and return the kernels' bounded-wait status word (0 = clean)."""
    v = ctypes.c_int(0)
    _check(load().mha_check_device_status(ctypes.byref(v), int(reset)))
    return v.value


def version() -> str:
    return load().mha_version().decode()
