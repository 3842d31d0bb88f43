"""Residual attention sublayer x + MHA(LayerNorm(x), ...) on the GPU vs the fp64 oracle
("The Annotated Transformer", SublayerConnection; both LayerNorm forms the pages use)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from transformer_head_scaled_fwd_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu

WN = ("w_q", "b_q", "w_k", "b_k", "w_v", "b_v", "w_o", "b_o")


@pytest.fixture(scope="module")
def bnd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_head_scaled_fwd_gb300 import build as B
    B.build()
    from transformer_head_scaled_fwd_gb300 import binding
    binding.load()
    return binding


def _run(bnd, inp, ln, eps, kind, *, memory=None, causal=False, valid_lens=None, inplace=False):
    dt = torch.bfloat16 if inp.wl.dtype == "bf16" else torch.float32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dt)
    x = dev(inp.query)
    B, L, d = x.shape
    mem = None if memory is None else dev(memory)
    code = bnd.MHA_BF16 if inp.wl.dtype == "bf16" else bnd.MHA_F32
    ws = torch.empty(bnd.sublayer_workspace_size(code, B, L, 0 if mem is None else mem.shape[1], d, inp.wl.h),
                     dtype=torch.uint8, device="cuda")
    out = x if inplace else torch.full_like(x, float("nan"))
    vl = None if valid_lens is None else torch.tensor(valid_lens, dtype=torch.int32, device="cuda")
    bnd.mha_sublayer_forward(x, dev(ln[0]), dev(ln[1]), eps, kind, *[dev(inp.weights[n]) for n in WN], inp.wl.h,
                             out=out, workspace=ws, memory=mem, mask=bnd.make_mask(causal, vl, None))
    torch.cuda.synchronize()
    assert bnd.mha_check_device_status(reset=True) == 0
    return out.double().cpu().numpy()


def _ref(inp, ln, eps, kind, **kw):
    return oracle.sublayer_forward(inp.query, ln[0], ln[1], eps, kind, *[inp.weights[n] for n in WN], inp.wl.h, **kw)


def _check(got, ref, atol, rtol):
    err = np.abs(got - ref)
    assert np.all(err <= atol + rtol * np.abs(ref)), f"max abs err {err.max():.3e}"


@pytest.mark.parametrize("kind,eps", [(0, 1e-6), (1, 1e-5)])
def test_self_attention_sublayer_bf16(bnd, kind, eps):
    inp = W.random_case(300 + kind, 2, 200, 200, 512, 8, self_attn=True)
    ln = W.make_ln_params(512, seed=kind)
    got = _run(bnd, inp, ln, eps, kind, causal=True, valid_lens=[200, 130])
    _check(got, _ref(inp, ln, eps, kind, causal=True, valid_lens=[200, 130]), 1.5e-2, 2e-2)


def test_source_attention_sublayer_bf16(bnd):
    inp = W.random_case(310, 2, 150, 150, 256, 4, self_attn=True)
    mem = W.random_case(311, 2, 77, 77, 256, 4, self_attn=True).query
    ln = W.make_ln_params(256, seed=5)
    got = _run(bnd, inp, ln, 1e-6, 0, memory=mem, valid_lens=[77, 30])
    _check(got, _ref(inp, ln, 1e-6, 0, memory=mem, valid_lens=[77, 30]), 1.5e-2, 2e-2)


def test_sublayer_in_place(bnd):
    inp = W.random_case(320, 2, 130, 130, 256, 4, self_attn=True)
    ln = W.make_ln_params(256, seed=6)
    got = _run(bnd, inp, ln, 1e-6, 0, causal=True, inplace=True)
    _check(got, _ref(inp, ln, 1e-6, 0, causal=True), 1.5e-2, 2e-2)


@pytest.mark.parametrize("kind", [0, 1])
def test_sublayer_fp32(bnd, kind):
    inp = W.random_case(330 + kind, 2, 23, 23, 96, 3, self_attn=True, dtype="f32")
    ln = W.make_ln_params(96, seed=7, dtype="f32")
    got = _run(bnd, inp, ln, 1e-6, kind, causal=True, valid_lens=[23, 9])
    _check(got, _ref(inp, ln, 1e-6, kind, causal=True, valid_lens=[23, 9]), 1e-4, 1e-4)


def test_sublayer_long_config_sampled_rows(bnd):
    wl = W.WORKLOADS["long"]
    inp = W.make_inputs(wl)
    ln = W.make_ln_params(wl.d_model, seed=8)
    got = _run(bnd, inp, ln, 1e-6, 0, causal=True)
    rows = W.sample_rows(wl.Lq, 32, seed=9)
    _check(got[:, rows], _ref(inp, ln, 1e-6, 0, causal=True, rows=rows), 1.5e-2, 2e-2)
