"""The C-ABI library builds, loads and exports every symbol include/mha.h declares;
host-side validation rejects bad arguments before anything touches a GPU.
No compute call is made here (no GPU in this test)."""
import ctypes
import os
import re

import pytest

from transformer_head_scaled_fwd_gb300 import binding
from transformer_head_scaled_fwd_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return binding.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "mha.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mha_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(binding.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert "sm_103a" in binding.version()


def test_workspace_size_layout(lib):
    # bf16: Qh + KVh + ctx + stats, each 256-aligned, then 256 bytes of schedule counter
    B_, Lq, Lk, d, h = 2, 10, 7, 512, 8
    es = 2
    a = lambda x: (x + 255) // 256 * 256
    q = a(es * B_ * Lq * d)
    kv = a(es * B_ * 2 * Lk * d)
    ctx = a(es * B_ * Lq * d)
    st = a(4 * 2 * B_ * h * Lq)
    assert binding.workspace_size(binding.MHA_BF16, B_, Lq, Lk, d, h) == q + kv + ctx + st + 256
    assert binding.workspace_size(binding.MHA_BF16, B_, Lq, Lk, 510, 8) == 0
    assert binding.workspace_size(binding.MHA_F32, 0, Lq, Lk, d, h) == 0


def test_workspace_size_bf16_other_head_widths(lib):
    """bf16 with d_k outside {64, 128} runs on the fp32 kernels over fp32 copies: the
    workspace is the fp32 forward's, then query, key, value, 4 weights, 4 biases and out
    in fp32, each part 256-aligned."""
    B_, Lq, Lk, d, h = 2, 10, 7, 192, 2
    a = lambda x: (x + 255) // 256 * 256
    f32 = binding.workspace_size(binding.MHA_F32, B_, Lq, Lk, d, h)
    qn, kn = 4 * B_ * Lq * d, 4 * B_ * Lk * d
    off = a(f32)
    off = a(off + qn)
    off = a(off + kn)
    off = a(off + kn)
    off = a(off + 16 * d * d)
    off = a(off + 16 * d)
    assert binding.workspace_size(binding.MHA_BF16, B_, Lq, Lk, d, h) == a(off + qn)
    assert binding.workspace_size(binding.MHA_BF16, B_, Lq, Lk, 640, 2) > 0    # sizes stay defined


def _call_forward(lib, dt=binding.MHA_BF16, B_=1, Lq=4, Lk=4, d=128, h=2, mask=None, ws=1 << 30,
                  ws_ptr=256, ptr=4096):
    P = ctypes.c_void_p(ptr)
    return lib.mha_forward(dt, P, P, P, P, None, P, None, P, None, P, None, B_, Lq, Lk, d, h,
                           ctypes.byref(mask) if mask is not None else None, P, None,
                           ctypes.c_void_p(ws_ptr), ws, None)


def test_validation_without_gpu(lib):
    assert _call_forward(lib, d=130, h=4) == binding.MHA_ERR_INVALID_ARG          # d % h != 0
    assert b"d_model % h" in lib.mha_last_error()
    assert _call_forward(lib, B_=0) == binding.MHA_ERR_INVALID_ARG
    assert _call_forward(lib, d=640, h=2) == binding.MHA_ERR_UNSUPPORTED          # d_k = 320 > 256
    assert _call_forward(lib, dt=binding.MHA_F32, d=1024, h=2) == binding.MHA_ERR_UNSUPPORTED
    assert _call_forward(lib, dt=7) == binding.MHA_ERR_INVALID_ARG
    m = binding.MaskT(); m.causal = 1
    assert _call_forward(lib, Lq=4, Lk=5, mask=m) == binding.MHA_ERR_INVALID_ARG  # causal needs Lq == Lk
    m2 = binding.MaskT(); m2.dense = 4096; m2.dense_mq = 3
    assert _call_forward(lib, mask=m2) == binding.MHA_ERR_INVALID_ARG             # dense_mq not 1 / Lq
    assert _call_forward(lib, ws=16) == binding.MHA_ERR_INVALID_ARG               # workspace too small
    assert _call_forward(lib, ws_ptr=260) == binding.MHA_ERR_INVALID_ARG          # misaligned workspace
    assert _call_forward(lib, ptr=4097) == binding.MHA_ERR_INVALID_ARG            # misaligned bf16 tensor
    P = ctypes.c_void_p(4096)
    rc = lib.mha_forward(binding.MHA_BF16, None, P, P, P, None, P, None, P, None, P, None, 1, 4, 4, 128, 2,
                         None, P, None, ctypes.c_void_p(256), 1 << 30, None)
    assert rc == binding.MHA_ERR_INVALID_ARG                                       # null query


def test_size_limits_without_gpu(lib):
    """The largest problems: activations beyond 4e9 elements, or more than 1e15 query/key pairs
    over all heads, are refused as UNSUPPORTED before anything reaches the GPU (32-bit tile
    indices); a problem just inside the limits gets past the size check (and here stops at
    the workspace check, which the caller's 1 GB does not satisfy)."""
    big = 1 << 30
    assert _call_forward(lib, B_=64, Lq=1 << 20, Lk=1 << 20, d=1024, h=16, ws=big) == binding.MHA_ERR_UNSUPPORTED
    assert b"too large" in lib.mha_last_error()
    # activations inside the limit, 1.2e15 query/key pairs outside it
    assert _call_forward(lib, B_=1, Lq=60_000_000, Lk=20_000_000, d=64, h=1, ws=big) == binding.MHA_ERR_UNSUPPORTED
    assert _call_forward(lib, B_=1, Lq=1 << 20, Lk=1 << 20, d=1024, h=16, ws=big) == binding.MHA_ERR_INVALID_ARG
    assert b"workspace too small" in lib.mha_last_error()
    assert binding.workspace_size(binding.MHA_BF16, 1, 1 << 20, 1 << 20, 1024, 16) > big


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        binding._lib = None
        try:
            binding.load(str(tmp_path / "missing.so"))
        finally:
            binding._lib = None
