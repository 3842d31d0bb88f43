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


def test_d128_work_counter_reset_and_reuse():
    """The d_k = 128 attention is persistent: its CTAs draw query tiles from a counter in
    the workspace. With the workspace filled with 0xFF first (the projection stage zeroes
    the counter) and the attention stage run three times after one projection (each
    launch leaves the counter at zero), every run gives the same context bit for bit,
    close to the oracle, and the counter words end at zero. 256 query tiles: more than one
    per SM."""
    from gpu_helpers import to_dev
    from transformer_head_scaled_fwd_gb300 import binding
    inp = W.random_case(630, 8, 1000, 1000, 512, 4, self_attn=True)
    B, L, d, h = 8, 1000, 512, 4
    dt = torch.bfloat16
    x = to_dev(inp.query, dt)
    Wt = {n: to_dev(a, dt) for n, a in inp.weights.items()}
    size = binding.workspace_size(binding.MHA_BF16, B, L, L, d, h)
    ws = torch.full((size,), 255, dtype=torch.uint8, device="cuda")
    mask = binding.make_mask(True, None, None)
    binding.mha_qkv_projection(x, x, x, Wt["w_q"], Wt["b_q"], Wt["w_k"], Wt["b_k"], Wt["w_v"], Wt["b_v"], h,
                               workspace=ws)
    outs = []
    for _ in range(3):
        out = torch.empty(B, L, d, dtype=dt, device="cuda")
        binding.mha_attention_core(binding.MHA_BF16, B, L, L, d, h, workspace=ws, mask=mask)
        binding.mha_output_projection(Wt["w_o"], Wt["b_o"], B, L, L, h, out=out, workspace=ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert binding.mha_check_device_status(reset=True) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert ws[size - 256:size - 248].view(torch.int32).tolist() == [0, 0]
    rows = W.sample_rows(L, 48, seed=631)
    ref = run_oracle(inp, causal=True, rows=rows)
    assert_close(outs[0].double().cpu().numpy()[:, rows], ref, "bf16")


def test_d128_cuda_graph_replays_equal_eager():
    """The whole d_k = 128 forward captured once in a CUDA graph (the projection zeroes the
    attention's work counter, the persistent attention leaves it at zero) and replayed three
    times gives the eager call's output bit for bit, with more query tiles than SMs."""
    from gpu_helpers import to_dev
    from transformer_head_scaled_fwd_gb300 import binding
    B, L, d, h = 4, 1200, 512, 4
    inp = W.random_case(640, B, L, L, d, h, self_attn=True)
    dt = torch.bfloat16
    x = to_dev(inp.query, dt)
    Wt = {n: to_dev(a, dt) for n, a in inp.weights.items()}
    ws = torch.empty(binding.workspace_size(binding.MHA_BF16, B, L, L, d, h), dtype=torch.uint8, device="cuda")
    mask = binding.make_mask(True, None, None)
    args = (x, x, x, Wt["w_q"], Wt["b_q"], Wt["w_k"], Wt["b_k"], Wt["w_v"], Wt["b_v"], Wt["w_o"], Wt["b_o"], h)
    eager = torch.empty(B, L, d, dtype=dt, device="cuda")
    binding.mha_forward(*args, out=eager, workspace=ws, mask=mask)
    torch.cuda.synchronize()
    out = torch.zeros(B, L, d, dtype=dt, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            binding.mha_forward(*args, out=out, workspace=ws, mask=mask, stream=s)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert binding.mha_check_device_status(reset=True) == 0
    rows = W.sample_rows(L, 32, seed=641)
    assert_close(out.double().cpu().numpy()[:, rows], run_oracle(inp, causal=True, rows=rows), "bf16")


def test_d128_dense_mask_many_query_tiles():
    """A dense mask with more query tiles than SMs (every key tile visited, each CTA taking
    several units of different batch items) and a ragged L_q: sampled rows against the
    oracle, row sums of p_attn equal one."""
    B, Lq, Lk, d, h = 3, 1700, 900, 512, 4
    inp = W.random_case(650, B, Lq, Lk, d, h, kv_alias=False)
    rng = np.random.default_rng(651)
    dense = (rng.random((B, Lq, Lk)) < 0.5).astype(np.uint8)
    dense[2, 1699, :] = 0
    got, gp = run_gpu(inp, dense=dense, want_p_attn=True)
    rows = W.sample_rows(Lq, 40, seed=652)
    ref = run_oracle(inp, dense=dense, rows=rows)
    assert_close(got[:, rows], ref, "bf16")
    np.testing.assert_allclose(gp.sum(-1), 1.0, atol=ROWSUM_TOL)
    np.testing.assert_allclose(gp[2, :, 1699], 1.0 / Lk, rtol=1e-5, atol=0)
