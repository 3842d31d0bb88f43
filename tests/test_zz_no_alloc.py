"""mha_forward_noalloc: the entry point for callers that cannot allocate device
memory (their host owns the memory pool, or cudaMalloc's device-wide
synchronisation is not acceptable on their path, or their interface has no
workspace argument). It must give the same results as mha_forward with a
caller workspace, call after call, through the C ABI.

This file is named so that pytest collects it last."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from transformer_head_scaled_fwd_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_head_scaled_fwd_gb300 import build as B
    B.build()
    from transformer_head_scaled_fwd_gb300 import binding as bnd
    bnd.load()
    return bnd


def _case(seed, B, L, d, h, causal, valid_lens):
    inp = W.random_case(seed, B, L, L, d, h, self_attn=True, bias_scale=0.1)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.bfloat16)
    x = dev(inp.query)
    w = {n: dev(a) for n, a in inp.weights.items()}
    vl = torch.tensor(valid_lens, dtype=torch.int32, device="cuda")
    return x, w, vl, causal, h


def _args(x, w):
    return (x, x, x, w["w_q"], w["b_q"], w["w_k"], w["b_k"], w["w_v"], w["b_v"], w["w_o"], w["b_o"])


def test_noalloc_matches_workspace_path_two_calls_in_a_row(binding):
    cases = [_case(201, 4, 256, 512, 8, True, [256, 200, 17, 1]),
             _case(202, 3, 320, 1024, 16, False, [320, 0, 150])]
    for x, w, vl, causal, h in cases:      # two calls in a row, different shapes and masks
        B, L, d = x.shape
        mask = binding.make_mask(causal=causal, key_valid_lens=vl)
        ref = torch.empty_like(x)
        ws = torch.empty(binding.workspace_size(binding.MHA_BF16, B, L, L, d, h), dtype=torch.uint8,
                         device="cuda")
        binding.mha_forward(*_args(x, w), h, out=ref, workspace=ws, mask=mask)
        got = torch.full_like(x, float("nan"))
        binding.mha_forward_noalloc(*_args(x, w), h, out=got, mask=mask)
        torch.cuda.synchronize()
        g = got.double().cpu().numpy()
        r = ref.double().cpu().numpy()
        assert np.all(np.abs(g - r) <= 1.5e-2 + 2e-2 * np.abs(r))
    assert binding.mha_check_device_status(reset=True) == 0


def test_noalloc_rejects_problems_beyond_its_scratch(binding):
    x = torch.zeros(4, 8192, 1024, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(1024, 1024, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.MHAError) as e:
        binding.mha_forward_noalloc(x, x, x, w, None, w, None, w, None, w, None, 16, out=x)
    assert e.value.status == binding.MHA_ERR_INVALID_ARG
    assert "MHA_NOALLOC_SCRATCH_BYTES" in str(e.value)
