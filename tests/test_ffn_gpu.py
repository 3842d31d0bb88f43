"""Position-wise FFN on the GPU vs the fp64 oracle, through the C ABI
(max(0, x W_1 + b_1) W_2 + b_2: "003-Transformer" tutorial, feed-forward layer)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from transformer_head_scaled_fwd_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bnd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_head_scaled_fwd_gb300 import build as B
    B.build()
    from transformer_head_scaled_fwd_gb300 import binding
    binding.load()
    return binding


def _run(bnd, inp):
    dt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dt)
    x = dev(inp.x)
    B, L, d = x.shape
    d_ff = inp.w_1.shape[0]
    code = bnd.MHA_BF16 if inp.dtype == "bf16" else bnd.MHA_F32
    ws = torch.empty(bnd.ffn_workspace_size(code, B, L, d, d_ff), dtype=torch.uint8, device="cuda")
    out = torch.full_like(x, float("nan"))
    bnd.mha_ffn_forward(x, dev(inp.w_1), dev(inp.b_1), dev(inp.w_2), dev(inp.b_2), out=out, workspace=ws)
    torch.cuda.synchronize()
    assert bnd.mha_check_device_status(reset=True) == 0
    return out.double().cpu().numpy()


def _check(got, ref, atol, rtol):
    err = np.abs(got - ref)
    assert np.all(err <= atol + rtol * np.abs(ref)), f"max abs err {err.max():.3e}"


@pytest.mark.parametrize("B,L,d,d_ff", [(2, 200, 512, 2048), (3, 77, 192, 320), (1, 1, 64, 64)])
def test_ffn_bf16_matches_oracle(bnd, B, L, d, d_ff):
    inp = W.make_ffn_inputs(B, L, d, d_ff, seed=B * 1000 + L)
    got = _run(bnd, inp)
    ref = oracle.ffn_forward(inp.x, inp.w_1, inp.b_1, inp.w_2, inp.b_2)
    _check(got, ref, 1.5e-2, 2e-2)


def test_ffn_bf16_bench_size_sampled_rows(bnd):
    cfg = W.FFN_WORKLOADS["ffn_long"]
    inp = W.make_ffn_inputs(cfg["B"], cfg["L"], cfg["d_model"], cfg["d_ff"], seed=11)
    got = _run(bnd, inp)
    rows = W.sample_rows(cfg["L"], 128, seed=12)
    ref = oracle.ffn_forward(inp.x[:, rows], inp.w_1, inp.b_1, inp.w_2, inp.b_2)
    _check(got[:, rows], ref, 1.5e-2, 2e-2)


def test_ffn_bf16_odd_k_block_counts(bnd):
    """d_model 1344 (21 k-blocks) and d_ff 2752 (43): both layers run on pairs of SMs at B=4, L=1024,
    each tile ending on a ring stage that holds one k-block."""
    inp = W.make_ffn_inputs(4, 1024, 1344, 2752, seed=13)
    got = _run(bnd, inp)
    rows = W.sample_rows(1024, 64, seed=14)
    ref = oracle.ffn_forward(inp.x[:, rows], inp.w_1, inp.b_1, inp.w_2, inp.b_2)
    _check(got[:, rows], ref, 1.5e-2, 2e-2)


@pytest.mark.parametrize("B,L,d,d_ff", [(2, 37, 48, 100), (1, 5, 512, 2048)])
def test_ffn_fp32_matches_oracle(bnd, B, L, d, d_ff):
    inp = W.make_ffn_inputs(B, L, d, d_ff, seed=7 + d, dtype="f32")
    got = _run(bnd, inp)
    ref = oracle.ffn_forward(inp.x, inp.w_1, inp.b_1, inp.w_2, inp.b_2)
    _check(got, ref, 1e-4, 1e-4)


def test_ffn_relu_cuts_everything(bnd):
    inp = W.make_ffn_inputs(2, 130, 256, 512, seed=3)
    inp.b_1 = np.full_like(inp.b_1, -1e4)
    got = _run(bnd, inp)
    assert np.all(got == np.broadcast_to(inp.b_2.astype(np.float64), got.shape))
