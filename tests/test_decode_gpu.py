"""Incremental decoding with a key/value cache vs the fp64 oracle.

Decoding a sequence one token at a time (each new token attends to every token
so far, itself included: the d2l decoder at prediction time) must reproduce
causal self-attention over the whole sequence, row by row. Head widths 64 and 128."""
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
    binding.mha_check_device_status(reset=True)
    return binding


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.bfloat16)


class Cache:
    def __init__(self, bnd, inp, L_max):
        self.bnd = bnd
        B, _, d = inp.query.shape
        h = inp.wl.h
        self.h = h
        self.w = [_dev(inp.weights[n]) for n in WN]
        self.k = torch.zeros(B, h, L_max, d // h, dtype=torch.bfloat16, device="cuda")
        self.v = torch.zeros_like(self.k)
        self.len = torch.zeros(B, dtype=torch.int32, device="cuda")
        self.ws = torch.empty(bnd.decode_workspace_size(B, d, h, L_max), dtype=torch.uint8, device="cuda")

    def prefill(self, x):
        w = self.w
        self.bnd.mha_kv_cache_prefill(_dev(x), w[2], w[3], w[4], w[5], self.h, k_cache=self.k, v_cache=self.v)
        self.len.fill_(x.shape[1])

    def step(self, x_new):
        out = torch.full((x_new.shape[0], x_new.shape[1]), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.bnd.mha_decode_step(_dev(x_new), *self.w, self.h, k_cache=self.k, v_cache=self.v,
                                 cache_len=self.len, out=out, workspace=self.ws)
        return out


def _check(got, ref):
    err = np.abs(got - ref)
    assert np.all(err <= 1.5e-2 + 2e-2 * np.abs(ref)), f"max abs err {err.max():.3e}"


@pytest.mark.parametrize("h", [4, 2])   # d_k 64, 128
def test_decode_from_empty_cache_equals_causal_attention(bnd, h):
    B, T, d = 3, 40, 256
    inp = W.random_case(400, B, T, T, d, h, self_attn=True)
    c = Cache(bnd, inp, L_max=64)
    outs = [c.step(inp.query[:, t]) for t in range(T)]
    torch.cuda.synchronize()
    got = torch.stack(outs, 1).double().cpu().numpy()
    w = [inp.weights[n] for n in WN]
    ref = oracle.mha_forward(inp.query, inp.query, inp.query, *w, h, causal=True)
    _check(got, ref)
    assert c.len.cpu().tolist() == [T] * B
    assert bnd.mha_check_device_status(reset=True) == 0


@pytest.mark.parametrize("h", [8, 4])   # d_k 64, 128
def test_decode_after_prefill_with_ragged_histories(bnd, h):
    B, T0, d = 3, 300, 512
    inp = W.random_case(401, B, T0 + 1, T0 + 1, d, h, self_attn=True)
    c = Cache(bnd, inp, L_max=512)
    c.prefill(inp.query[:, :T0])
    lens = [300, 257, 1]
    c.len.copy_(torch.tensor(lens, dtype=torch.int32))
    x_new = np.stack([inp.query[b, lens[b]] for b in range(B)])
    got = c.step(x_new)
    torch.cuda.synchronize()
    got = got.double().cpu().numpy()
    w = [inp.weights[n] for n in WN]
    for b in range(B):
        xb = inp.query[b:b + 1, :lens[b] + 1]
        ref = oracle.mha_forward(xb, xb, xb, *w, h, causal=True, rows=[lens[b]])
        _check(got[b], ref[0, 0])
    assert c.len.cpu().tolist() == [l + 1 for l in lens]
    assert bnd.mha_check_device_status(reset=True) == 0


@pytest.mark.parametrize("h", [16, 8])   # d_k 64, 128
def test_decode_long_cache(bnd, h):
    """The bench's cache length (8192) with d_model 1024, on two sequences."""
    B, T0, d = 2, 8192, 1024
    inp = W.random_case(402, B, T0 + 1, T0 + 1, d, h, self_attn=True, bias_scale=0.0)
    c = Cache(bnd, inp, L_max=T0 + 64)
    c.prefill(inp.query[:, :T0])
    got = c.step(inp.query[:, T0])
    torch.cuda.synchronize()
    w = [inp.weights[n] for n in WN]
    ref = oracle.mha_forward(inp.query, inp.query, inp.query, *w, h, causal=True, rows=[T0])
    _check(got.double().cpu().numpy(), ref[:, 0])
    assert bnd.mha_check_device_status(reset=True) == 0


@pytest.mark.parametrize("d", [128, 256])   # d_k 64, 128
def test_full_cache_is_reported_not_written(bnd, d):
    B, h = 2, 2
    inp = W.random_case(403, B, 8, 8, d, h, self_attn=True)
    c = Cache(bnd, inp, L_max=8)
    c.prefill(inp.query)
    k_before = c.k.clone()
    c.step(inp.query[:, 0])
    torch.cuda.synchronize()
    assert c.len.cpu().tolist() == [8, 8]
    assert torch.equal(c.k, k_before)
    assert bnd.mha_check_device_status(reset=True) == 0x301


@pytest.mark.parametrize("B,h", [(17, 8), (40, 8), (64, 8), (70, 8), (40, 4), (70, 4)])
def test_decode_batch_sizes(bnd, B, h):
    """Projections of the step: up to 64 new tokens stream W over many CTAs in passes of
    16 rows (17, 40: a partial last pass); 70 tokens use the tiled projection GEMM.
    h 8 / 4 at d_model 512: d_k 64 / 128."""
    T0, d = 100, 512
    inp = W.random_case(410 + B + h, B, T0 + 1, T0 + 1, d, h, self_attn=True, bias_scale=0.1)
    c = Cache(bnd, inp, L_max=128)
    c.prefill(inp.query[:, :T0])
    got = c.step(inp.query[:, T0])
    torch.cuda.synchronize()
    w = [inp.weights[n] for n in WN]
    ref = oracle.mha_forward(inp.query, inp.query, inp.query, *w, h, causal=True, rows=[T0])
    _check(got.double().cpu().numpy(), ref[:, 0])
    assert c.len.cpu().tolist() == [T0 + 1] * B
    assert bnd.mha_check_device_status(reset=True) == 0
