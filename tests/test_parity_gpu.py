"""GPU path vs the fp64 oracle, element by element, through the C ABI.

Inputs are seeded and bf16-rounded before both paths (workloads module).
Tolerances: bf16 |g-o| <= 1.5e-2 + 2e-2|o|; fp32 |g-o| <= 1e-4 + 1e-4|o|;
p_attn rows sum to 1 within 1e-3.
"""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from transformer_head_scaled_fwd_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


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


def _worked_example_inputs(dtype):
    g = json.load(open(os.path.join(GOLDEN, "thinking_machines.json")))
    d = g["d_k"]
    wl = W.Workload("worked", 0, dtype, 1, 1, 2, d, 1, False, False)
    eye = np.eye(d, dtype=np.float32)
    q = np.zeros((1, 1, d), np.float32); q[0, 0, 0] = 1
    k = np.zeros((1, 2, d), np.float32); k[0, 0, 0] = g["raw_scores"][0]; k[0, 1, 0] = g["raw_scores"][1]
    v = np.zeros((1, 2, d), np.float32); v[0, 0, 0] = 1; v[0, 1, 1] = 1
    w = {"w_q": eye, "w_k": eye, "w_v": eye, "w_o": eye}
    for n in "qkvo":
        w["b_" + n] = np.zeros(d, np.float32)
    return W.Inputs(wl, q, k, v, w), g


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_worked_example_thinking_machines(dtype):
    inp, g = _worked_example_inputs(dtype)
    out, p = run_gpu(inp, want_p_attn=True)
    tol = 1e-6 if dtype == "f32" else 5e-3
    np.testing.assert_allclose(p[0, 0, 0], g["weights"], rtol=0, atol=tol)
    expect = np.zeros(inp.wl.d_model); expect[:2] = g["weights"]
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=tol if dtype == "f32" else 1e-2)


def test_tiny_fp32_config_with_p_attn():
    inp = W.make_inputs(W.WORKLOADS["tiny"])
    got, gp = run_gpu(inp, valid_lens=inp.valid_lens, want_p_attn=True)
    ref, rp = run_oracle(inp, valid_lens=inp.valid_lens, want_p_attn=True)
    assert_close(got, ref, "f32")
    assert_close(gp, rp, "f32", "p_attn")
    np.testing.assert_allclose(gp.sum(-1), 1.0, atol=ROWSUM_TOL)


@pytest.mark.parametrize("name", ["enc", "dec", "xattn"])
def test_bf16_configs_full(name):
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    got, _ = run_gpu(inp, causal=wl.causal, valid_lens=inp.valid_lens)
    ref = run_oracle(inp, causal=wl.causal, valid_lens=inp.valid_lens)
    assert_close(got, ref, "bf16")


def test_long_causal_sampled_rows():
    wl = W.WORKLOADS["long"]
    inp = W.make_inputs(wl)
    rows = W.sample_rows(wl.Lq, 64, seed=4)
    got, _ = run_gpu(inp, causal=True)
    ref = run_oracle(inp, causal=True, rows=rows)
    assert_close(got[:, rows], ref, "bf16")


def test_long_single_sequence_ragged_sampled_rows():
    """The longest case of the suite: one causal sequence of 32768 tokens (four times the bench
    length) whose keys stop at a valid length of 30001, so tensor-map coordinates and row offsets run
    far past those of the bench; sampled query rows include the ones around the valid length and the
    last row (its allowed keys are the first 30001)."""
    L = 32768
    inp = W.random_case(71, 1, L, L, 1024, 16, self_attn=True, bias_scale=0.05)
    vl = [30001]
    rows = np.unique(np.concatenate([W.sample_rows(L, 48, seed=9), [30000, 30001, 30002]])).astype(np.int32)
    got, _ = run_gpu(inp, causal=True, valid_lens=vl)
    ref = run_oracle(inp, causal=True, valid_lens=vl, rows=rows)
    assert_close(got[:, rows], ref, "bf16")


def test_widest_model_dimension():
    """d_model 2048 with 32 heads: projection GEMMs with 8 column tiles of 256 and K = 2048,
    attention over 64 (batch, head) planes, ragged valid lengths."""
    inp = W.random_case(72, 2, 700, 700, 2048, 32, self_attn=True, bias_scale=0.05)
    vl = [700, 333]
    got, _ = run_gpu(inp, causal=True, valid_lens=vl)
    ref = run_oracle(inp, causal=True, valid_lens=vl)
    assert_close(got, ref, "bf16")


def test_pair_gemm_odd_k_block_count():
    """d_model 1344 = 21 k-blocks of 64 with 21 heads: at B=4, L=1024 both projections run on pairs of
    SMs (288 and 96 tile pairs), whose ring stages hold two k-blocks, so the last stage of every tile
    holds one; a ragged last column tile (1344 = 5.25 x 256) and ragged valid lengths."""
    inp = W.random_case(74, 4, 1024, 1024, 1344, 21, self_attn=True, bias_scale=0.05)
    vl = [1024, 1000, 513, 77]
    rows = W.sample_rows(1024, 48, seed=74)
    got, _ = run_gpu(inp, causal=True, valid_lens=vl)
    ref = run_oracle(inp, causal=True, valid_lens=vl, rows=rows)
    assert_close(got[:, rows], ref, "bf16")


# ------------------------------------------------------------------ edge cases (bf16)
def test_ragged_cross_attention_distinct_kv_bias_p_attn():
    inp = W.random_case(1, 3, 200, 77, 512, 8, kv_alias=False, bias_scale=0.1)
    vl = [77, 1, 40]
    got, gp = run_gpu(inp, valid_lens=vl, want_p_attn=True)
    ref, rp = run_oracle(inp, valid_lens=vl, want_p_attn=True)
    assert_close(got, ref, "bf16")
    assert_close(gp, rp, "bf16", "p_attn")
    np.testing.assert_allclose(gp.sum(-1), 1.0, atol=ROWSUM_TOL)
    assert np.all(gp[1, :, :, 1:] == 0.0)


@pytest.mark.parametrize("L", [1, 2, 3, 10, 129, 300])
def test_causal_self_attention_small_and_ragged(L):
    inp = W.random_case(10 + L, 2, L, L, 256, 4, self_attn=True)
    vl = [L, max(1, L // 2)]
    got, gp = run_gpu(inp, causal=True, valid_lens=vl, want_p_attn=L <= 300)
    ref, rp = run_oracle(inp, causal=True, valid_lens=vl, want_p_attn=True)
    assert_close(got, ref, "bf16")
    assert_close(gp, rp, "bf16", "p_attn")


def test_fully_masked_rows_are_uniform():
    """valid length 0: every score is -1e9, weights 1/L_k over all keys."""
    inp = W.random_case(30, 3, 70, 150, 256, 4)
    vl = [0, 150, 3]
    got, gp = run_gpu(inp, valid_lens=vl, want_p_attn=True)
    ref, rp = run_oracle(inp, valid_lens=vl, want_p_attn=True)
    assert_close(got, ref, "bf16")
    np.testing.assert_allclose(gp[0], 1.0 / 150, rtol=1e-5, atol=0)
    assert_close(gp, rp, "bf16", "p_attn")


@pytest.mark.parametrize("mq", ["broadcast", "per_query"])
def test_dense_mask(mq):
    B, Lq, Lk = 2, 140, 260
    inp = W.random_case(40, B, Lq, Lk, 256, 4)
    rng = np.random.default_rng(41)
    dense = (rng.random((B, 1 if mq == "broadcast" else Lq, Lk)) < 0.7).astype(np.uint8)
    dense[1, 0, :] = 0                         # a fully masked row (all rows if broadcast)
    got, gp = run_gpu(inp, dense=dense, want_p_attn=True)
    ref, rp = run_oracle(inp, dense=dense, want_p_attn=True)
    assert_close(got, ref, "bf16")
    assert_close(gp, rp, "bf16", "p_attn")


@pytest.mark.parametrize("Lk", [1024, 1100])
def test_masks_on_both_sides_of_the_short_key_threshold(Lk):
    """The d_k = 64 kernel has one instance for key ranges up to 1024 and one for longer ones;
    each handles valid lengths (including 0: uniform rows), a ragged key tail and a dense mask."""
    B, Lq = 3, 200
    inp = W.random_case(44 + Lk, B, Lq, Lk, 256, 4, bias_scale=0.1)
    vl = [Lk, 0, 333]
    rng = np.random.default_rng(45)
    got, _ = run_gpu(inp, valid_lens=vl)
    ref = run_oracle(inp, valid_lens=vl)
    assert_close(got, ref, "bf16")
    dense = (rng.random((B, 1, Lk)) < 0.8).astype(np.uint8)
    got, gp = run_gpu(inp, valid_lens=vl, dense=dense, want_p_attn=True)
    ref, rp = run_oracle(inp, valid_lens=vl, dense=dense, want_p_attn=True)
    assert_close(got, ref, "bf16")
    assert_close(gp, rp, "bf16", "p_attn")
    np.testing.assert_allclose(gp[1], 1.0 / Lk, rtol=1e-5, atol=0)


@pytest.mark.parametrize("L", [1024, 1152])
def test_causal_padding_on_both_sides_of_the_short_key_threshold(L):
    inp = W.random_case(46 + L, 2, L, L, 256, 4, self_attn=True, bias_scale=0.1)
    vl = [L, 517]
    rows = [0, 1, 127, 128, 516, 517, 700, L - 1]
    got, _ = run_gpu(inp, causal=True, valid_lens=vl)
    ref = run_oracle(inp, causal=True, valid_lens=vl, rows=rows)
    assert_close(got[:, rows], ref, "bf16")


def test_dense_mask_with_causal_and_padding():
    B, L = 2, 260
    inp = W.random_case(42, B, L, L, 256, 4, self_attn=True)
    rng = np.random.default_rng(43)
    dense = (rng.random((B, L, L)) < 0.8).astype(np.uint8)
    vl = [200, 0]
    got, _ = run_gpu(inp, causal=True, valid_lens=vl, dense=dense)
    ref = run_oracle(inp, causal=True, valid_lens=vl, dense=dense)
    assert_close(got, ref, "bf16")


@pytest.mark.parametrize("h", [1, 3])
def test_odd_head_counts(h):
    d = 64 * h
    inp = W.random_case(50 + h, 2, 150, 131, d, h, bias_scale=0.2)
    got, _ = run_gpu(inp, valid_lens=[131, 60])
    ref = run_oracle(inp, valid_lens=[131, 60])
    assert_close(got, ref, "bf16")


@pytest.mark.parametrize("B,h,Lq,Lk", [(1, 3, 128, 128), (3, 1, 100, 300), (5, 2, 77, 77), (2, 8, 128, 640)])
def test_two_pairs_per_cta_for_short_queries(B, h, Lq, Lk):
    """L_q <= 128 (with L_k <= 1024): a CTA's two query tiles serve two (batch, head) pairs,
    each with its own K/V stages; an odd pair count leaves the last CTA's second tile idle.
    Per-pair valid lengths (one of them 0: uniform rows), causal when square, p_attn."""
    d = 64 * h
    inp = W.random_case(60 + 7 * B + h, B, Lq, Lk, d, h, bias_scale=0.1, self_attn=(Lq == Lk))
    vl = [max(1, (Lk * (i + 1)) // (B + 1)) for i in range(B)]
    if B >= 3:
        vl[1] = 0
    causal = Lq == Lk
    got, gp = run_gpu(inp, causal=causal, valid_lens=vl, want_p_attn=True)
    ref, rp = run_oracle(inp, causal=causal, valid_lens=vl, want_p_attn=True)
    assert_close(got, ref, "bf16")
    assert_close(gp, rp, "bf16", "p_attn")
    np.testing.assert_allclose(gp.sum(-1), 1.0, atol=ROWSUM_TOL)


def test_stage_entry_points_equal_forward():
    inp = W.random_case(60, 2, 256, 256, 512, 8, self_attn=True)
    a, _ = run_gpu(inp, causal=True)
    b, _ = run_gpu(inp, causal=True, stages=True)
    np.testing.assert_array_equal(a, b)


def test_masked_keys_do_not_change_output():
    inp = W.random_case(70, 2, 130, 300, 256, 4)
    vl = [300, 150]
    a, _ = run_gpu(inp, valid_lens=vl)
    inp.key = inp.key.copy(); inp.value = inp.key
    inp.key[1, 150:] = np.float32(7.0) * np.sign(inp.key[1, 150:])
    b, _ = run_gpu(inp, valid_lens=vl)
    np.testing.assert_array_equal(a, b)


def test_identical_query_rows_identical_outputs():
    inp = W.random_case(80, 1, 300, 200, 256, 4)
    inp.query = inp.query.copy()
    inp.query[0, 257] = inp.query[0, 3]
    out, _ = run_gpu(inp)
    np.testing.assert_array_equal(out[0, 257], out[0, 3])


# ------------------------------------------------------------------ fp32 path
@pytest.mark.parametrize("d,h", [(512, 16), (512, 4), (32, 4), (96, 1)])
def test_fp32_head_widths(d, h):
    inp = W.random_case(90 + h, 2, 37, 45, d, h, dtype="f32")
    vl = [45, 0]
    got, gp = run_gpu(inp, valid_lens=vl, want_p_attn=True)
    ref, rp = run_oracle(inp, valid_lens=vl, want_p_attn=True)
    assert_close(got, ref, "f32")
    assert_close(gp, rp, "f32", "p_attn")


def test_fp32_causal_dense():
    inp = W.random_case(99, 2, 33, 33, 128, 2, dtype="f32", self_attn=True)
    dense = (np.random.default_rng(5).random((2, 33, 33)) < 0.6).astype(np.uint8)
    got, _ = run_gpu(inp, causal=True, dense=dense)
    ref = run_oracle(inp, causal=True, dense=dense)
    assert_close(got, ref, "f32")


# ------------------------------------------------------------------ host-buffer entry point
def test_forward_host_matches_device_path():
    from transformer_head_scaled_fwd_gb300 import binding
    from gpu_helpers import to_dev
    inp = W.random_case(100, 2, 192, 192, 512, 8, self_attn=True)
    dev_out, _ = run_gpu(inp, causal=True)
    dt = torch.bfloat16
    hq = torch.from_numpy(inp.query).to(dt).pin_memory()
    hout = torch.empty_like(hq).pin_memory()
    Wd = {n: to_dev(a, dt) for n, a in inp.weights.items()}
    B, L, d = inp.query.shape
    staging = torch.empty(binding.host_staging_size(binding.MHA_BF16, B, L, L, d, False, False),
                          dtype=torch.uint8, device="cuda")
    ws = torch.empty(binding.workspace_size(binding.MHA_BF16, B, L, L, d, 8), dtype=torch.uint8, device="cuda")
    binding.mha_forward_host(hq, hq, hq, Wd["w_q"], Wd["b_q"], Wd["w_k"], Wd["b_k"], Wd["w_v"], Wd["b_v"],
                             Wd["w_o"], Wd["b_o"], 8, h_out=hout, staging=staging, workspace=ws,
                             mask=binding.make_mask(causal=True))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hout.double().numpy(), dev_out)


def test_invalid_arguments_leave_output_untouched():
    from transformer_head_scaled_fwd_gb300 import binding
    dt = torch.bfloat16
    x = torch.zeros(1, 8, 96, dtype=dt, device="cuda")
    w = torch.zeros(96, 96, dtype=dt, device="cuda")
    out = torch.full((1, 8, 96), 3.0, dtype=dt, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.MHAError) as e:
        binding.mha_forward(x, x, x, w, None, w, None, w, None, w, None, 5, out=out, workspace=ws)
    assert e.value.status == binding.MHA_ERR_INVALID_ARG
    x2 = torch.zeros(1, 8, 640, dtype=dt, device="cuda")
    w2 = torch.zeros(640, 640, dtype=dt, device="cuda")
    out2 = torch.full((1, 8, 640), 3.0, dtype=dt, device="cuda")
    with pytest.raises(binding.MHAError) as e:       # d_k = 320: above the 256 the kernels take
        binding.mha_forward(x2, x2, x2, w2, None, w2, None, w2, None, w2, None, 2, out=out2, workspace=ws)
    assert e.value.status == binding.MHA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out == 3.0) and torch.all(out2 == 3.0)


def test_forward_host_uneven_chunks_distinct_kv_and_masks():
    """Host entry point pipelined over chunks of sequences: 5 sequences, a small call -> chunks of
    3 and 2; key != value != query, per-sequence valid lengths and a per-query dense mask (offset per
    chunk)."""
    from transformer_head_scaled_fwd_gb300 import binding
    from gpu_helpers import to_dev
    B, Lq, Lk, d, h = 5, 70, 90, 256, 4
    inp = W.random_case(110, B, Lq, Lk, d, h, kv_alias=False)
    vl = [90, 3, 0, 45, 90]
    dense = (np.random.default_rng(111).random((B, Lq, Lk)) < 0.8).astype(np.uint8)
    dt = torch.bfloat16
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dt).pin_memory()
    hq, hk, hv = pin(inp.query), pin(inp.key), pin(inp.value)
    hout = torch.empty(B, Lq, d, dtype=dt).pin_memory()
    Wd = {n: to_dev(a, dt) for n, a in inp.weights.items()}
    staging = torch.empty(binding.host_staging_size(binding.MHA_BF16, B, Lq, Lk, d, True, True),
                          dtype=torch.uint8, device="cuda")
    ws = torch.empty(binding.workspace_size(binding.MHA_BF16, B, Lq, Lk, d, h), dtype=torch.uint8, device="cuda")
    vld = torch.tensor(vl, dtype=torch.int32, device="cuda")
    dmd = torch.from_numpy(dense).cuda()
    binding.mha_forward_host(hq, hk, hv, Wd["w_q"], Wd["b_q"], Wd["w_k"], Wd["b_k"], Wd["w_v"], Wd["b_v"],
                             Wd["w_o"], Wd["b_o"], h, h_out=hout, staging=staging, workspace=ws,
                             mask=binding.make_mask(False, vld, dmd))
    torch.cuda.synchronize()
    ref = run_oracle(inp, valid_lens=vl, dense=dense)
    assert_close(hout.double().numpy(), ref, "bf16")


@pytest.mark.parametrize("h,masked", [(8, "causal"), (4, "causal"), (8, "pad_dense")])   # d_k 64 and 128
def test_forward_host_row_windows(h, masked):
    """Self-attention through the host entry point: the first chunk's projections and uploads
    and the last chunk's output projection and downloads are cut into row windows (here
    [0, 256) and [256, 640)); a small call, so two chunks (2 and 1 sequences) on two compute
    streams. The result equals the device path bit for bit and matches the oracle."""
    from transformer_head_scaled_fwd_gb300 import binding
    from gpu_helpers import to_dev
    B, L, d = 3, 640, 512
    inp = W.random_case(120 + h, B, L, L, d, h, self_attn=True, bias_scale=0.1)
    if masked == "causal":
        kw = dict(causal=True)
        mk = binding.make_mask(causal=True)
    else:
        vl = [640, 300, 1]
        dense = (np.random.default_rng(121).random((B, 1, L)) < 0.7).astype(np.uint8)
        kw = dict(valid_lens=vl, dense=dense)
        vld = torch.tensor(vl, dtype=torch.int32, device="cuda")
        dmd = torch.from_numpy(dense).cuda()
        mk = binding.make_mask(False, vld, dmd)
    dev_out, _ = run_gpu(inp, **kw)
    dt = torch.bfloat16
    hq = torch.from_numpy(inp.query).to(dt).pin_memory()
    hout = torch.full((B, L, d), 7.0, dtype=dt).pin_memory()
    Wd = {n: to_dev(a, dt) for n, a in inp.weights.items()}
    staging = torch.empty(binding.host_staging_size(binding.MHA_BF16, B, L, L, d, False, False),
                          dtype=torch.uint8, device="cuda")
    ws = torch.empty(binding.workspace_size(binding.MHA_BF16, B, L, L, d, h), dtype=torch.uint8, device="cuda")
    for _ in range(2):   # a second call reuses the library's streams and events
        binding.mha_forward_host(hq, hq, hq, Wd["w_q"], Wd["b_q"], Wd["w_k"], Wd["b_k"], Wd["w_v"], Wd["b_v"],
                                 Wd["w_o"], Wd["b_o"], h, h_out=hout, staging=staging, workspace=ws, mask=mk)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(hout.double().numpy(), dev_out)
    rows = [0, 1, 255, 256, 257, 511, 512, 639]
    ref = run_oracle(inp, rows=rows, **kw)
    assert_close(hout.double().numpy()[:, rows], ref, "bf16")


def test_forward_host_large_call_four_chunks():
    """A call with at least 32 MiB of host input is pipelined over four chunks of sequences:
    5 sequences of 3328 tokens at d_model 1024 (34 MB) -> chunks of 2, 2, 1, the first and the
    last cut into row windows. Bit-equal to the device path; the last (one-sequence) chunk's
    sampled rows match the oracle."""
    from transformer_head_scaled_fwd_gb300 import binding
    from gpu_helpers import to_dev
    B, L, d, h = 5, 3328, 1024, 16
    assert 2 * B * L * d >= 32 << 20
    inp = W.random_case(140, B, L, L, d, h, self_attn=True, bias_scale=0.1)
    dev_out, _ = run_gpu(inp, causal=True)
    dt = torch.bfloat16
    hq = torch.from_numpy(inp.query).to(dt).pin_memory()
    hout = torch.full((B, L, d), 7.0, dtype=dt).pin_memory()
    Wd = {n: to_dev(a, dt) for n, a in inp.weights.items()}
    staging = torch.empty(binding.host_staging_size(binding.MHA_BF16, B, L, L, d, False, False),
                          dtype=torch.uint8, device="cuda")
    ws = torch.empty(binding.workspace_size(binding.MHA_BF16, B, L, L, d, h), dtype=torch.uint8, device="cuda")
    binding.mha_forward_host(hq, hq, hq, Wd["w_q"], Wd["b_q"], Wd["w_k"], Wd["b_k"], Wd["w_v"], Wd["b_v"],
                             Wd["w_o"], Wd["b_o"], h, h_out=hout, staging=staging, workspace=ws,
                             mask=binding.make_mask(causal=True))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hout.double().numpy(), dev_out)
    q4 = np.ascontiguousarray(inp.query[4:5])
    last = W.Inputs(inp.wl, q4, q4, q4, inp.weights)
    rows = [0, 1, 1663, 3327]
    ref = run_oracle(last, causal=True, rows=rows)
    assert_close(hout.double().numpy()[4:5, rows], ref, "bf16")


@pytest.mark.parametrize("d,h", [(256, 8), (384, 4), (512, 2)])   # d_k 32, 96, 256
def test_bf16_other_head_widths(d, h):
    """bf16 problems whose head width the tensor-core kernels do not take run on the fp32
    kernels over fp32 copies of the bf16 inputs: causal + key padding, p_attn."""
    B, L = 2, 70
    inp = W.random_case(130 + h, B, L, L, d, h, self_attn=True, bias_scale=0.1)
    vl = [70, 33]
    got, pa = run_gpu(inp, causal=True, valid_lens=vl, want_p_attn=True)
    ref, ref_pa = run_oracle(inp, causal=True, valid_lens=vl, want_p_attn=True)
    assert_close(got, ref, "bf16")
    np.testing.assert_allclose(pa.sum(-1), 1.0, atol=1e-3)
    assert np.abs(pa - ref_pa).max() < 5e-3


@pytest.mark.parametrize("d, h", [(512, 16), (512, 8)])
def test_query_is_a_prefix_of_key_buffer(d, h):
    """query and key start at the same address but the key is longer (L_k > L_q): the
    query is the first B*L_q*d_model elements of the key buffer, read as [B, L_q, d_model].
    Both the fp32-copy route (d_k = 32) and the tensor-core route (d_k = 64) must read every
    key row from the key buffer, not from a conversion sized for the query."""
    import torch as T
    from transformer_head_scaled_fwd_gb300 import binding
    B, Lq, Lk = 2, 48, 112
    inp = W.random_case(140 + h, B, Lk, Lk, d, h, self_attn=True, bias_scale=0.1)
    kv = inp.query                                          # [B, L_k, d]
    q = np.ascontiguousarray(kv.reshape(-1)[:B * Lq * d].reshape(B, Lq, d))
    dev = lambda a: T.from_numpy(np.ascontiguousarray(a)).cuda().to(T.bfloat16)
    kv_d = dev(kv)
    q_d = kv_d.reshape(-1)[:B * Lq * d].view(B, Lq, d)
    assert q_d.data_ptr() == kv_d.data_ptr()
    w = {n: dev(a) for n, a in inp.weights.items()}
    vl = [112, 57]
    mask = binding.make_mask(False, T.tensor(vl, dtype=T.int32, device="cuda"), None)
    ws = T.empty(binding.workspace_size(binding.MHA_BF16, B, Lq, Lk, d, h), dtype=T.uint8, device="cuda")
    # the workspace starts dirty, as a reused caller buffer would
    ws.fill_(0x7f)
    out = T.empty(B, Lq, d, dtype=T.bfloat16, device="cuda")
    binding.mha_forward(q_d, kv_d, kv_d, w["w_q"], w["b_q"], w["w_k"], w["b_k"], w["w_v"], w["b_v"],
                        w["w_o"], w["b_o"], h, out=out, workspace=ws, mask=mask)
    T.cuda.synchronize()
    assert binding.mha_check_device_status(reset=True) == 0
    case = W.Inputs(inp.wl, q, kv, kv, inp.weights)
    ref = run_oracle(case, valid_lens=np.asarray(vl, np.int32))
    assert_close(out.double().cpu().numpy(), ref, "bf16")
