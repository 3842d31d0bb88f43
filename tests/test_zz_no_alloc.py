"""mha_forward_noalloc: the entry point for callers that cannot allocate device
memory (their host owns the memory pool, or cudaMalloc's device-wide
synchronisation is not acceptable on their path, or their interface has no
workspace argument). It runs the same kernels as mha_forward on the same inputs,
so its output must be bit-identical to mha_forward's with a caller workspace,
call after call, through the C ABI; one case is also held against the oracle.

The cases cover the routes whose scratch use differs: bf16 on the tensor-core
kernels (d_k = 64; d_k = 128, whose persistent attention draws its query tiles
from a counter in the scratch), bf16 with d_k = 32 (fp32 copies of the inputs in
the scratch) and fp32. Each runs twice in a row, after a different route
has left its data in the shared scratch.

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
    bnd.mha_check_device_status(reset=True)
    return bnd


def _case(seed, B, L, d, h, causal, valid_lens, dtype="bf16"):
    inp = W.random_case(seed, B, L, L, d, h, self_attn=True, bias_scale=0.1, dtype=dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(tdt)
    x = dev(inp.query)
    w = {n: dev(a) for n, a in inp.weights.items()}
    vl = torch.tensor(valid_lens, dtype=torch.int32, device="cuda")
    return inp, x, w, vl, causal, h


def _args(x, w):
    return (x, x, x, w["w_q"], w["b_q"], w["w_k"], w["b_k"], w["w_v"], w["b_v"], w["w_o"], w["b_o"])


def _both(binding, x, w, vl, causal, h):
    """(mha_forward with a caller workspace, mha_forward_noalloc) on the same inputs."""
    B, L, d = x.shape
    dt = binding.MHA_BF16 if x.dtype == torch.bfloat16 else binding.MHA_F32
    mask = binding.make_mask(causal=causal, key_valid_lens=vl)
    ref = torch.full_like(x, float("nan"))
    ws = torch.empty(binding.workspace_size(dt, B, L, L, d, h), dtype=torch.uint8, device="cuda")
    binding.mha_forward(*_args(x, w), h, out=ref, workspace=ws, mask=mask)
    got = torch.full_like(x, float("nan"))
    binding.mha_forward_noalloc(*_args(x, w), h, out=got, mask=mask)
    torch.cuda.synchronize()
    return ref, got


CASES = [
    # seed, B, L, d_model, h, causal, valid lens, dtype   (d_k = 64, 64, 32, 64, 128)
    (201, 4, 256, 512, 8, True, [256, 200, 17, 1], "bf16"),
    (202, 3, 320, 1024, 16, False, [320, 0, 150], "bf16"),
    (203, 2, 200, 512, 16, True, [200, 93], "bf16"),
    (204, 2, 96, 256, 4, False, [96, 40], "f32"),
    (205, 3, 700, 512, 4, True, [700, 333, 1], "bf16"),
]


def test_noalloc_bit_equal_to_workspace_path_two_calls_in_a_row(binding):
    cases = [_case(*c) for c in CASES]
    for rnd in range(2):                   # every route twice, each after the others
        for inp, x, w, vl, causal, h in cases:
            ref, got = _both(binding, x, w, vl, causal, h)
            assert not torch.isnan(ref).any()
            assert torch.equal(got, ref), (
                f"round {rnd}, d_k {x.shape[2] // h}, {x.dtype}: max abs diff "
                f"{(got.double() - ref.double()).abs().max().item():.3e}")
    assert binding.mha_check_device_status(reset=True) == 0


def test_noalloc_matches_the_oracle(binding):
    import oracle
    inp, x, w, vl, causal, h = _case(*CASES[0])
    _, got = _both(binding, x, w, vl, causal, h)
    ref = oracle.mha_forward(inp.query, inp.key, inp.value, *[inp.weights[n] for n in (
        "w_q", "b_q", "w_k", "b_k", "w_v", "b_v", "w_o", "b_o")], h, causal=causal,
        valid_lens=vl.cpu().numpy())
    g = got.double().cpu().numpy()
    assert np.all(np.abs(g - ref) <= 1.5e-2 + 2e-2 * np.abs(ref))
    assert binding.mha_check_device_status(reset=True) == 0


def test_noalloc_rejects_problems_beyond_its_scratch(binding):
    x = torch.zeros(4, 8192, 1024, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(1024, 1024, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.MHAError) as e:
        binding.mha_forward_noalloc(x, x, x, w, None, w, None, w, None, w, None, 16, out=x)
    assert e.value.status == binding.MHA_ERR_INVALID_ARG
    assert "MHA_NOALLOC_SCRATCH_BYTES" in str(e.value)
