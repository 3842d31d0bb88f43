"""bf16 heads narrower than 64 on the tensor cores vs the fp64 oracle.

Heads of width d_k = 8, 16 or 32 (with d_model a multiple of 64) run on the d_k = 64
kernels: the projection GEMM stores 64 / d_k heads per 64-column slab, and the attention
loads each head zero-padded to 64 columns (the padding columns are out of the tensor's
bounds and arrive as zeros, so the scores and P.V are the narrow head's exactly).
The d2l Transformer chapter's model uses d_k = 8 (num_hiddens 32 with 4 heads); d_model
512 with 16 heads gives d_k = 32. Tolerance |g - o| <= 1.5e-2 + 2e-2 |o|.
"""
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


def test_encoder_workload_sixteen_heads_full_size():
    """The encoder workload's shape (B 32, L 128, d_model 512, key padding U{64..128})
    with 16 heads of width 32, every output element."""
    base = W.WORKLOADS["enc"]
    wl = W.Workload("enc_h16", 11, "bf16", base.B, base.Lq, base.Lk, base.d_model, 16, False, True,
                    valid_range=base.valid_range)
    inp = W.make_inputs(wl)
    got, _ = run_gpu(inp, valid_lens=inp.valid_lens)
    assert_close(got, run_oracle(inp, valid_lens=inp.valid_lens), "bf16")


@pytest.mark.parametrize("dk", [8, 16, 32])
@pytest.mark.parametrize("L", [1, 129, 300])
def test_causal_self_attention_ragged(dk, L):
    d = 256
    inp = W.random_case(500 + dk + L, 2, L, L, d, d // dk, self_attn=True, bias_scale=0.1)
    vl = [L, max(1, L // 3)]
    got, _ = run_gpu(inp, causal=True, valid_lens=vl)
    assert_close(got, run_oracle(inp, causal=True, valid_lens=vl), "bf16")


@pytest.mark.parametrize("dk", [8, 16, 32])
def test_cross_attention_distinct_value_with_p_attn(dk):
    """Query, key and value all distinct, one fully masked sequence (uniform rows), p_attn."""
    d = 128
    inp = W.random_case(520 + dk, 3, 100, 260, d, d // dk, kv_alias=False, bias_scale=0.1)
    vl = [260, 0, 77]
    got, gp = run_gpu(inp, valid_lens=vl, want_p_attn=True)
    ref, rp = run_oracle(inp, valid_lens=vl, want_p_attn=True)
    assert_close(got, ref, "bf16")
    assert_close(gp, rp, "bf16", "p_attn")
    np.testing.assert_allclose(gp.sum(-1), 1.0, atol=ROWSUM_TOL)


def test_stage_entry_points_equal_forward():
    inp = W.random_case(530, 2, 200, 200, 512, 16, self_attn=True, bias_scale=0.1)
    a, _ = run_gpu(inp, causal=True, valid_lens=[200, 90])
    b, _ = run_gpu(inp, causal=True, valid_lens=[200, 90], stages=True)
    np.testing.assert_array_equal(a, b)


def test_long_sequence_sampled_rows():
    """One 4096-token causal sequence, d_model 1024 with 32 heads (d_k 32), on 64 sampled
    query rows (shared by every head, so W_o applies to whole rows)."""
    inp = W.random_case(540, 1, 4096, 4096, 1024, 32, self_attn=True, bias_scale=0.0)
    rows = W.sample_rows(4096, 64, 540)
    got, _ = run_gpu(inp, causal=True)
    ref = run_oracle(inp, causal=True, rows=rows)
    assert_close(got[:, rows], ref, "bf16")
