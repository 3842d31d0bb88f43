"""fp64 CPU oracle for the multi-head attention forward pass.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The
product path (the CUDA library and its Python binding) never imports it and
shares no code with it.

Two independent implementations live here:

* ``mha_forward`` -- ctypes wrapper around ``mha_oracle.c`` (fp64, OpenMP, no
  BLAS), usable at full workload sizes or on sampled query rows.
* ``oracle.brute`` -- pure-Python fp64 loops for tiny inputs, used to pin the C
  oracle.

Both follow "The Annotated Transformer", section "Attention" (attention():
scale by 1/sqrt(d_k), masked_fill(mask == 0, -1e9), softmax, P.V) and the
"003-Transformer" tutorial, section "Multi-head attention"
(MultiHeadedAttention.forward: Linear -> split heads -> attention -> concat ->
Linear).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mha_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmha_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mha_oracle.c`` into ``oracle/_build/libmha_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            bp = ctypes.POINTER(ctypes.c_ubyte)
            lib.oracle_mha_forward.restype = ctypes.c_int
            lib.oracle_mha_forward.argtypes = (
                [dp] * 3 + [dp] * 8
                + [ctypes.c_int] * 5
                + [ctypes.c_int, ip, bp, ctypes.c_int, ip, ctypes.c_int, dp, dp])
            lib.oracle_linear.restype = None
            lib.oracle_linear.argtypes = [dp, dp, dp, ctypes.c_long, ctypes.c_int,
                                          ctypes.c_int, dp]
            lib.oracle_ffn_forward.restype = ctypes.c_int
            lib.oracle_ffn_forward.argtypes = [dp] * 5 + [ctypes.c_long, ctypes.c_int, ctypes.c_int, dp]
            lib.oracle_layernorm.restype = ctypes.c_int
            lib.oracle_layernorm.argtypes = [dp] * 3 + [ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                                        ctypes.c_int, dp]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    """OpenMP threads the C oracle uses."""
    return int(_load().oracle_num_threads())


def linear(x, W, b=None):
    """nn.Linear in fp64: y = x W^T + b, W stored [out, in]."""
    lib = _load()
    x = _f64(x)
    W = _f64(W)
    b = _f64(b)
    rows = int(np.prod(x.shape[:-1]))
    dout, din = W.shape
    y = np.empty(x.shape[:-1] + (dout,), dtype=np.float64)
    lib.oracle_linear(_ptr(x, ctypes.c_double), _ptr(W, ctypes.c_double),
                      _ptr(b, ctypes.c_double), rows, din, dout,
                      _ptr(y, ctypes.c_double))
    return y


def mha_forward(query, key, value, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, h,
                causal=False, valid_lens=None, dense=None, rows=None,
                want_p_attn=False):
    """The multi-head attention sublayer, forward, in fp64.

    query [B, Lq, d]; key, value [B, Lk, d]; W [d, d] stored (out, in); b [d] or None.
    causal: subsequent mask j <= i.  valid_lens: [B] ints (key j allowed iff
    j < valid_lens[b]).  dense: uint8 [B, mq, Lk] with mq in {1, Lq}, 0 = masked.
    rows: optional list of query positions; the outputs are then only those rows.
    Returns ``out`` [B, nrows, d] and, if ``want_p_attn``, ``p_attn`` [B, h, nrows, Lk].
    """
    lib = _load()
    q, k, v = _f64(query), _f64(key), _f64(value)
    B, Lq, d = q.shape
    Lk = k.shape[1]
    ws = [_f64(w) for w in (w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o)]
    vl = None if valid_lens is None else np.ascontiguousarray(np.asarray(valid_lens, dtype=np.int32))
    dm = None
    mq = 0
    if dense is not None:
        dm = np.ascontiguousarray(np.asarray(dense, dtype=np.uint8))
        mq = dm.shape[1]
    rr = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    nr = Lq if rr is None else len(rr)
    out = np.empty((B, nr, d), dtype=np.float64)
    p = np.empty((B, h, nr, Lk), dtype=np.float64) if want_p_attn else None
    rc = lib.oracle_mha_forward(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        *[_ptr(w, ctypes.c_double) for w in ws],
        B, Lq, Lk, d, h, int(bool(causal)),
        _ptr(vl, ctypes.c_int), _ptr(dm, ctypes.c_ubyte), mq,
        _ptr(rr, ctypes.c_int), nr,
        _ptr(out, ctypes.c_double), _ptr(p, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_mha_forward rejected its arguments (code {rc})")
    return (out, p) if want_p_attn else out


def ffn_forward(x, w_1, b_1, w_2, b_2):
    """Position-wise FFN in fp64: max(0, x W_1^T + b_1) W_2^T + b_2 (nn.Linear layouts).
    x [..., d_model]; w_1 [d_ff, d_model]; w_2 [d_model, d_ff]; b_* or None."""
    lib = _load()
    x = _f64(x)
    w_1, b_1, w_2, b_2 = _f64(w_1), _f64(b_1), _f64(w_2), _f64(b_2)
    d_ff, d_model = w_1.shape
    rows = int(np.prod(x.shape[:-1]))
    out = np.empty(x.shape[:-1] + (d_model,), dtype=np.float64)
    rc = lib.oracle_ffn_forward(_ptr(x, ctypes.c_double), _ptr(w_1, ctypes.c_double), _ptr(b_1, ctypes.c_double),
                                _ptr(w_2, ctypes.c_double), _ptr(b_2, ctypes.c_double), rows, d_model, d_ff,
                                _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_ffn_forward rejected its arguments (code {rc})")
    return out


LN_ANNOTATED, LN_TORCH = 0, 1


def layernorm(x, a=None, b=None, eps=1e-6, kind=LN_ANNOTATED):
    """Row LayerNorm in fp64. kind 0: a (x - mean) / (std_unbiased + eps) + b ("The Annotated
    Transformer"); kind 1: nn.LayerNorm, a (x - mean) / sqrt(var_biased + eps) + b."""
    lib = _load()
    x = _f64(x)
    a, b = _f64(a), _f64(b)
    d = x.shape[-1]
    y = np.empty_like(x)
    rc = lib.oracle_layernorm(_ptr(x, ctypes.c_double), _ptr(a, ctypes.c_double), _ptr(b, ctypes.c_double),
                              int(np.prod(x.shape[:-1])), d, float(eps), int(kind), _ptr(y, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_layernorm rejected its arguments (code {rc})")
    return y


def sublayer_forward(x, ln_a, ln_b, eps, kind, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, h, memory=None,
                     causal=False, valid_lens=None, dense=None, rows=None):
    """The residual sublayer around multi-head attention ("The Annotated Transformer",
    SublayerConnection.forward): x + sublayer(norm(x)) with sublayer = self_attn(y, y, y, mask)
    when memory is None, else src_attn(y, memory, memory, mask); dropout is the identity."""
    y = layernorm(x, ln_a, ln_b, eps, kind)
    kv = y if memory is None else _f64(memory)
    att = mha_forward(y, kv, kv, w_q, b_q, w_k, b_k, w_v, b_v, w_o, b_o, h, causal=causal,
                      valid_lens=valid_lens, dense=dense, rows=rows)
    xs = _f64(x) if rows is None else _f64(x)[:, rows]
    return xs + att
