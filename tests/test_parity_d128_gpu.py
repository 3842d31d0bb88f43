"""bf16 tensor-core path with head width d_k = 128 vs the fp64 oracle (heads wider
than 64, e.g. d_model 1024 with h = 8)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from transformer_head_scaled_fwd_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_head_scaled_fwd_gb300 import build as B
    B.build()
    from transformer_head_scaled_fwd_gb300 import binding
    binding.load()
    binding.mha_check_device_status(reset=True)


from gpu_helpers import ROWSUM_TOL, assert_close, run_gpu, run_oracle  # noqa: E402


@pytest.mark.parametrize("L", [1, 5, 128, 300])
def test_d128_causal_padding(L):
    inp = W.random_case(600 + L, 2, L, L, 512, 4, self_attn=True)
    vl = [L, max(1, L // 3)]
    got, gp = run_gpu(inp, causal=True, valid_lens=vl, want_p_attn=True)
    ref, rp = run_oracle(inp, causal=True, valid_lens=vl, want_p_attn=True)
    assert_close(got, ref, "bf16")
    assert_close(gp, rp, "bf16", "p_attn")
    np.testing.assert_allclose(gp.sum(-1), 1.0, atol=ROWSUM_TOL)


def test_d128_ragged_cross_attention_distinct_kv():
    inp = W.random_case(610, 3, 200, 77, 256, 2, kv_alias=False, bias_scale=0.1)
    vl = [77, 1, 40]
    got, _ = run_gpu(inp, valid_lens=vl)
    ref = run_oracle(inp, valid_lens=vl)
    assert_close(got, ref, "bf16")


def test_d128_dense_mask_and_fully_masked_rows():
    B, Lq, Lk = 2, 140, 260
    inp = W.random_case(620, B, Lq, Lk, 384, 3)
    rng = np.random.default_rng(621)
    dense = (rng.random((B, Lq, Lk)) < 0.7).astype(np.uint8)
    dense[1, 5, :] = 0
    got, gp = run_gpu(inp, dense=dense, want_p_attn=True)
    ref, rp = run_oracle(inp, dense=dense, want_p_attn=True)
    assert_close(got, ref, "bf16")
    np.testing.assert_allclose(gp[1, :, 5], 1.0 / Lk, rtol=1e-5, atol=0)
    vl_case = W.random_case(622, 2, 70, 150, 256, 2)
    got2, _ = run_gpu(vl_case, valid_lens=[0, 150])
    assert_close(got2, run_oracle(vl_case, valid_lens=[0, 150]), "bf16")


def test_d128_full_size_causal_sampled_rows():
    wl = W.WORKLOADS["long_d128"]
    inp = W.make_inputs(wl)
    rows = W.sample_rows(wl.Lq, 64, seed=5)
    got, _ = run_gpu(inp, causal=True)
    ref = run_oracle(inp, causal=True, rows=rows)
    assert_close(got[:, rows], ref, "bf16")
